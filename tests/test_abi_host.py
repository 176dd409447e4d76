"""Host-side checks of the C ABI: the library builds and loads, exports every entry point
include/fa.h declares, and rejects bad arguments before anything is launched.  No call here
reaches a kernel (every one fails validation first), so these run without a GPU."""

import ctypes
import os
import re

import pytest

from exact_attention_96_gb300 import abi, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fa.h")
FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails before any use


@pytest.fixture(scope="module")
def lib():
    build.build()
    return abi.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    names = declared_functions()
    assert names == sorted(abi.SIGNATURES), names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in [(0, "FA_OK"), (1, "FA_ERR_INVALID_ARG"), (2, "FA_ERR_UNSUPPORTED"),
                       (3, "FA_ERR_MISALIGNED"), (4, "FA_ERR_CUDA"), (5, "FA_ERR_TIMEOUT")]:
        assert abi.status_string(code) == name
    assert abi.status_string(99) == "FA_ERR_UNKNOWN"


def fwd(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N=128, d=64, scale=0.125,
             causal=0, stream=None)
    a.update(kw)
    return abi.fa_fwd(*a.values())


def bwd(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, do=FAKE, lse=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
             B=1, H=1, N=128, d=64, scale=0.125, causal=0, ws=FAKE, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return abi.fa_bwd(*a.values())


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), abi.FA_ERR_INVALID_ARG),
    (dict(lse=None), abi.FA_ERR_INVALID_ARG),
    (dict(B=0), abi.FA_ERR_INVALID_ARG),
    (dict(H=-1), abi.FA_ERR_INVALID_ARG),
    (dict(N=0), abi.FA_ERR_INVALID_ARG),
    (dict(d=96), abi.FA_ERR_UNSUPPORTED),
    (dict(d=32), abi.FA_ERR_UNSUPPORTED),
    (dict(B=300, H=300), abi.FA_ERR_UNSUPPORTED),
    (dict(N=(1 << 20) + 1), abi.FA_ERR_UNSUPPORTED),
    (dict(scale=0.0), abi.FA_ERR_INVALID_ARG),
    (dict(scale=-1.0), abi.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), abi.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), abi.FA_ERR_INVALID_ARG),
    (dict(k=FAKE + 8), abi.FA_ERR_MISALIGNED),
    (dict(o=FAKE + 2), abi.FA_ERR_MISALIGNED),
])
def test_forward_validation(lib, kw, status):
    assert fwd(**kw) == status


@pytest.mark.parametrize("kw,status", [
    (dict(do=None), abi.FA_ERR_INVALID_ARG),
    (dict(ws=None), abi.FA_ERR_INVALID_ARG),
    (dict(ws_bytes=16), abi.FA_ERR_INVALID_ARG),
    (dict(d=80), abi.FA_ERR_UNSUPPORTED),
    (dict(scale=0.0), abi.FA_ERR_INVALID_ARG),
    (dict(dv=FAKE + 4), abi.FA_ERR_MISALIGNED),
    (dict(ws=FAKE + 16), abi.FA_ERR_MISALIGNED),
])
def test_backward_validation(lib, kw, status):
    assert bwd(**kw) == status


def test_workspace_bytes(lib):
    def expected(B, H, N, d):
        r256 = lambda x: (x + 255) // 256 * 256
        Np = (N + 3) // 4 * 4
        tiles = (N + 127) // 128
        # D and LSE*log2(e) rows (fp32, padded to 4), then the fp32 dQ accumulator tiles
        return 2 * r256(B * H * Np * 4) + B * H * tiles * 128 * d * 4
    for shape in [(1, 1, 1, 64), (4, 16, 8192, 128), (2, 3, 17, 64), (1, 8, 65536, 64)]:
        assert abi.fa_bwd_workspace_bytes(*shape) == expected(*shape)
    assert abi.fa_bwd_workspace_bytes(0, 1, 1, 64) == 0
    assert abi.fa_bwd_workspace_bytes(1, 1, 1, 48) == 0


def test_wait_limit_round_trip(lib):
    prev = abi.fa_set_wait_limit_ns(5_000_000_000)
    assert abi.fa_set_wait_limit_ns(10) == 5_000_000_000  # raised to the 1 ms floor on store
    assert abi.fa_set_wait_limit_ns(prev) == 1_000_000


def test_withhold_hook_is_one_shot_request(lib):
    assert abi.fa_test_withhold_kv_tile(3) == -1
    assert abi.fa_test_withhold_kv_tile(-5) == 3   # cancel
    assert abi.fa_test_withhold_kv_tile(-1) == -1


def test_accumulate_and_convert_validate_before_launching(lib):
    def acc(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, do=FAKE, lse=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
                 B=1, H=1, N=128, d=64, scale=0.125, causal=0, ws=FAKE, ws_bytes=1 << 30, stream=None)
        a.update(kw)
        return abi.fa_bwd_accumulate(*a.values())
    assert acc(dq=None) == abi.FA_ERR_INVALID_ARG
    assert acc(dv=None) == abi.FA_ERR_INVALID_ARG
    assert acc(dk=FAKE + 4) == abi.FA_ERR_MISALIGNED
    assert acc(N=0) == abi.FA_ERR_INVALID_ARG
    assert acc(d=96) == abi.FA_ERR_UNSUPPORTED
    assert acc(ws_bytes=16) == abi.FA_ERR_INVALID_ARG
    assert abi.fa_convert_f32_to_bf16(FAKE, FAKE, 0, None) == abi.FA_ERR_INVALID_ARG
    assert abi.fa_convert_f32_to_bf16(None, FAKE, 8, None) == abi.FA_ERR_INVALID_ARG
    assert abi.fa_convert_f32_to_bf16(FAKE + 8, FAKE, 8, None) == abi.FA_ERR_MISALIGNED


def test_fp8_quantiser_validates_before_launching(lib):
    q = abi.fa_quantize_e4m3
    assert q(None, FAKE, 1, 1, 16, 128, 0, 0, FAKE, None) == abi.FA_ERR_INVALID_ARG
    assert q(FAKE, FAKE, 1, 1, 16, 128, 0, 0, None, None) == abi.FA_ERR_INVALID_ARG
    assert q(FAKE, FAKE, 1, 1, 0, 128, 0, 0, FAKE, None) == abi.FA_ERR_INVALID_ARG
    assert q(FAKE, FAKE, 1, 1, 16, 96, 0, 0, FAKE, None) == abi.FA_ERR_UNSUPPORTED
    assert q(FAKE, FAKE, 1, 1, 20, 128, 1, 16, FAKE, None) == abi.FA_ERR_INVALID_ARG   # ld < N
    assert q(FAKE, FAKE, 1, 1, 20, 128, 1, 40, FAKE, None) == abi.FA_ERR_INVALID_ARG   # ld % 16
    assert q(FAKE + 2, FAKE, 1, 1, 16, 128, 0, 0, FAKE, None) == abi.FA_ERR_MISALIGNED
    assert abi.fa_e4m3_descale(FAKE, 0, FAKE, None) == abi.FA_ERR_INVALID_ARG
    assert abi.fa_e4m3_descale(FAKE, 8, None, None) == abi.FA_ERR_INVALID_ARG
    assert abi.fa_e4m3_descale(FAKE + 8, 8, FAKE, None) == abi.FA_ERR_MISALIGNED


def test_profile_hook_wants_both_events_or_neither(lib):
    assert abi.fa_profile_next_bwd_main(FAKE, None) == abi.FA_ERR_INVALID_ARG
    assert abi.fa_profile_next_bwd_main(None, FAKE) == abi.FA_ERR_INVALID_ARG
    assert abi.fa_profile_next_bwd_main(None, None) == abi.FA_OK  # cancels


def test_split_plan(lib):
    # every range non-empty; auto picks about two CTAs per SM for decode shapes
    n = abi.fa_fwd_splitkv_num_splits
    assert n(1, 1, 1, 1000, 64, 0) == 16            # 16 tiles of 64 keys, all used
    assert n(4, 16, 1, 65536, 128, 0) == 5          # 64 CTAs per split -> ceil(304/64)
    assert n(1, 1, 1, 500, 128, 7) == 4             # 4 tiles: 7 requested, 4 effective
    assert n(1, 1, 1, 500, 128, 3) == 2             # 2 tiles per range -> 2 ranges
    assert n(1, 1, 1, 10, 64, 0) == 1
    assert abi.fa_fwd_splitkv_workspace_bytes(1, 1, 0, 10, 64, 0) == 0
    assert abi.fa_fwd_splitkv_workspace_bytes(1, 1, 1, 10, 48, 0) == 0
    ws = abi.fa_fwd_splitkv_workspace_bytes(2, 3, 5, 1000, 64, 4)
    rows = 2 * 3 * 5
    assert ws == (4 * rows * 64 * 4 + 255) // 256 * 256 + 4 * rows * 4


@pytest.mark.parametrize("p", [1.0, 1.5, -0.1, float("nan"), float("inf")])
def test_dropout_probability_is_validated(lib, p):
    assert abi.fa_fwd_dropout(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 64, 0.125, 0, p, 1, None) == \
        abi.FA_ERR_INVALID_ARG
    assert abi.fa_bwd_dropout(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 64, 0.125, 0,
                              p, 1, FAKE, 1 << 30, None) == abi.FA_ERR_INVALID_ARG


def test_dropout_argument_checks_before_launch(lib):
    # the backward dropout path takes the plain path's head dims
    assert abi.fa_bwd_dropout(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 96, 0.125, 0,
                              0.1, 1, FAKE, 1 << 30, None) == abi.FA_ERR_UNSUPPORTED
    # the usual size, pointer and alignment checks still come first
    assert abi.fa_fwd_dropout(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 0, 64, 0.125, 0, 0.1, 1, None) == \
        abi.FA_ERR_INVALID_ARG
    assert abi.fa_fwd_dropout(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 96, 0.125, 0, 0.1, 1, None) == \
        abi.FA_ERR_UNSUPPORTED
    assert abi.fa_fwd_dropout(FAKE + 8, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 64, 0.125, 0, 0.1, 1, None) == \
        abi.FA_ERR_MISALIGNED
    assert abi.fa_bwd_dropout(0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 64, 0.125, 0,
                              0.1, 1, FAKE, 1 << 30, None) == abi.FA_ERR_INVALID_ARG


def test_fp8_forward_argument_checks_before_launch(lib):
    def call(**kw):
        a = dict(q8=FAKE, k8=FAKE, vt8=FAKE, ldv=128, o=FAKE, lse=FAKE, B=1, H=1, N=128, d=128,
                 scale=0.125, qd=1.0, kd=1.0, vd=1.0, causal=0, stream=None)
        a.update(kw)
        return abi.fa_fwd_fp8(*a.values())
    assert call(d=64) == abi.FA_ERR_UNSUPPORTED
    assert call(d=256) == abi.FA_ERR_UNSUPPORTED
    assert call(ldv=112) == abi.FA_ERR_INVALID_ARG        # ldv < N
    assert call(N=100, ldv=104) == abi.FA_ERR_INVALID_ARG  # not a multiple of 16
    assert call(qd=0.0) == abi.FA_ERR_INVALID_ARG
    assert call(vd=float("nan")) == abi.FA_ERR_INVALID_ARG
    assert call(q8=0) == abi.FA_ERR_INVALID_ARG
    assert call(vt8=FAKE + 8) == abi.FA_ERR_MISALIGNED
    assert call(N=0) == abi.FA_ERR_INVALID_ARG


def test_step_host_argument_checks_before_launch(lib):
    def call(**kw):
        a = dict(ptrs=[FAKE] * 18, B=1, H=2, N=128, d=64, scale=0.125, causal=0, chunks=0, ws=FAKE,
                 ws_bytes=1 << 30, stream=None)
        a.update(kw)
        return abi.fa_step_host(a["ptrs"][:9], a["ptrs"][9:], a["B"], a["H"], a["N"], a["d"], a["scale"],
                                a["causal"], a["chunks"], a["ws"], a["ws_bytes"], a["stream"])
    assert call(ptrs=[FAKE] * 17 + [0]) == abi.FA_ERR_INVALID_ARG
    assert call(ws=0) == abi.FA_ERR_INVALID_ARG
    assert call(N=0) == abi.FA_ERR_INVALID_ARG
    assert call(chunks=65) == abi.FA_ERR_UNSUPPORTED
    assert call(d=96) == abi.FA_ERR_UNSUPPORTED
    assert call(ws_bytes=16) == abi.FA_ERR_INVALID_ARG
    # the workspace covers the largest chunk's backward
    def two(n):  # one 256-byte aligned workspace per compute stream
        return 2 * ((n + 255) // 256 * 256)
    assert abi.fa_step_host_workspace_bytes(1, 8, 128, 64, 4) == two(abi.fa_bwd_workspace_bytes(1, 2, 128, 64))
    assert abi.fa_step_host_workspace_bytes(1, 8, 130, 64, 4) == two(abi.fa_bwd_workspace_bytes(1, 4, 130, 64))
    assert abi.fa_step_host_workspace_bytes(1, 8, 128, 64, 65) == 0
    # default: BH / 16 heads per chunk, but at least 1.5 waves of 128-row tiles (228 tiles)
    assert abi.fa_step_host_workspace_bytes(4, 16, 8192, 128, 0) == two(abi.fa_bwd_workspace_bytes(1, 4, 8192, 128))
    assert abi.fa_step_host_workspace_bytes(2, 16, 2048, 64, 0) == two(abi.fa_bwd_workspace_bytes(1, 15, 2048, 64))
    assert abi.fa_step_host_workspace_bytes(1, 8, 128, 64, 0) == two(abi.fa_bwd_workspace_bytes(1, 8, 128, 64))
