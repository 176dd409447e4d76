"""GPU parity of the FP8 forward (fa_fwd_fp8) against the fp64 oracle.

The oracle computes exact attention of the dequantised E4M3 inputs.  The kernel rounds P to
E4M3 (after scaling by 2^8) before the P V product, so its O differs by that rounding:
each P_ij carries a relative error of at most 2^-4 (3 mantissa bits, round to nearest) and
the row's P sum to 1, so |dO_i| <= 2^-4 max|V| at worst, plus the bf16 rounding of O
(2^-9 |O|, taken as 2^-8 max|O|).  For the Frobenius norm the errors average: with
rounding errors spread over each binade the RMS relative error of an E4M3 value is about
2^-4 / sqrt(3) * 0.72 = 0.026, which carries over to rel-Frobenius(O); a CPU model of the same
rounding gives 0.019 - 0.025 on these inputs.  Bars: O rel-Frobenius <= 0.04, O max-abs <=
2^-4 max|V| + 2^-8 max|O|, LSE max-abs <= 1e-3 (S = Q K^T is exact on 8-bit inputs up to fp32
accumulation, as in the bf16 path)."""

import math

import numpy as np
import pytest
import torch

from exact_attention_96_gb300 import abi, build, inputs as I
from exact_attention_96_gb300 import attention as fa
from oracle import attention as A
from oracle import fp8
from parity_util import LSE_MAX_ABS, max_abs, rel_fro, to_f64

pytestmark = pytest.mark.gpu

O_REL_FRO_FP8 = 0.04


@pytest.fixture(scope="module", autouse=True)
def library():
    build.build()
    abi.load()


def device_fp8(B, H, N, seed):
    q8, k8, v8, scales = I.fp8_attention_inputs(B, H, N, 128, seed=seed)
    ldv = (N + 15) // 16 * 16
    vt = np.zeros((B, H, 128, ldv), np.uint8)
    vt[..., :N] = np.swapaxes(v8, -1, -2)
    dev = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (q8, k8, vt)]
    return (q8, k8, v8, scales), dev


def check(o, lse, o_ref, lse_ref, vmax, what):
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), what
    bar = 2.0 ** -4 * vmax + 2.0 ** -8 * np.max(np.abs(o_ref))
    assert max_abs(o, o_ref) <= bar, (what, max_abs(o, o_ref), bar)
    assert rel_fro(o, o_ref) <= O_REL_FRO_FP8, (what, rel_fro(o, o_ref))
    assert max_abs(lse, lse_ref) <= LSE_MAX_ABS, (what, max_abs(lse, lse_ref))


FP8_SMALL = [
    # (B, H, N, causal)
    (1, 1, 128, False),   # one tile, second tile of the pair absent
    (1, 1, 1, True),      # single key
    (1, 2, 300, True),    # odd tile count, ragged tail
    (2, 1, 257, False),   # ragged second tile of the pair
    (1, 2, 640, True),    # five tiles: two full pairs and a half pair
    (1, 1, 1000, False),  # V^T row stride padded to 1008
    (2, 2, 768, False),
    (11, 1, 520, True),   # causal heads in a full group of eight and a partial one
]


@pytest.mark.parametrize("B,H,N,causal", FP8_SMALL)
def test_fp8_forward_small(B, H, N, causal):
    (q8, k8, v8, (qs, ks, vs)), (tq, tk, tvt) = device_fp8(B, H, N, seed=N + 3)
    o, lse = fa.forward_fp8(tq, tk, tvt, qs, ks, vs, causal=causal)
    assert fa.status_check() == abi.FA_OK
    o_ref, lse_ref = fp8.attention_fwd_fp8(q8, k8, v8, qs, ks, vs, 1 / math.sqrt(128), causal)
    vmax = np.max(np.abs(fp8.e4m3_bits_to_f64(v8))) * vs
    check(to_f64(o), to_f64(lse), o_ref, lse_ref, vmax, (B, H, N, causal))


def test_fp8_forward_scale_and_descales():
    # the softmax scale and the three descale factors enter only as the real inputs do
    (q8, k8, v8, _), (tq, tk, tvt) = device_fp8(1, 2, 384, seed=11)
    qs, ks, vs, scale = 0.013, 0.021, 0.5, 0.2
    o, lse = fa.forward_fp8(tq, tk, tvt, qs, ks, vs, causal=True, scale=scale)
    o_ref, lse_ref = fp8.attention_fwd_fp8(q8, k8, v8, qs, ks, vs, scale, True)
    vmax = np.max(np.abs(fp8.e4m3_bits_to_f64(v8))) * vs
    check(to_f64(o), to_f64(lse), o_ref, lse_ref, vmax, "descales")


@pytest.mark.parametrize("B,causal", [(4, True), (2, False)])
def test_fp8_forward_full_size_sampled_rows(B, causal):
    # the long causal language-model shape, 4 x 16 x 8192 x 128, and its non-causal half-batch
    # sibling: heads checked on sampled rows (each row of attention depends only on its query
    # and all keys)
    H, N = 16, 8192
    (q8, k8, v8, (qs, ks, vs)), (tq, tk, tvt) = device_fp8(B, H, N, seed=42 + B)
    o, lse = fa.forward_fp8(tq, tk, tvt, qs, ks, vs, causal=causal)
    assert fa.status_check() == abi.FA_OK
    o, lse = to_f64(o), to_f64(lse)
    rng = np.random.default_rng(7)
    vmax = np.max(np.abs(fp8.e4m3_bits_to_f64(v8))) * vs
    num = den = 0.0
    for b in range(B):
        for h in range(0, H, 3):
            rows = np.sort(rng.choice(N, 48, replace=False))
            rows[0], rows[-1] = 0, N - 1
            qh, kh, vh = (fp8.e4m3_bits_to_f64(x[b, h]) * s for x, s in ((q8, qs), (k8, ks), (v8, vs)))
            o_ref, lse_ref = A.attention_fwd_rows(qh, kh, vh, 1 / math.sqrt(128), causal, rows)
            bar = 2.0 ** -4 * vmax + 2.0 ** -8 * np.max(np.abs(o_ref))
            assert max_abs(o[b, h, rows], o_ref) <= bar, (b, h)
            assert max_abs(lse[b, h, rows], lse_ref) <= LSE_MAX_ABS, (b, h)
            num += np.sum((o[b, h, rows] - o_ref) ** 2)
            den += np.sum(o_ref ** 2)
    assert math.sqrt(num / den) <= O_REL_FRO_FP8


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_is_repeatable_bitwise(causal):
    # the two query tiles of a CTA have their own issuers and take turns; the result must not
    # depend on how their work interleaves
    (_, (tq, tk, tvt)) = device_fp8(2, 4, 1100, seed=6)
    a1 = fa.forward_fp8(tq, tk, tvt, 0.01, 0.01, 0.01, causal=causal)
    a2 = fa.forward_fp8(tq, tk, tvt, 0.01, 0.01, 0.01, causal=causal)
    assert torch.equal(a1[0], a2[0]) and torch.equal(a1[1], a2[1])
