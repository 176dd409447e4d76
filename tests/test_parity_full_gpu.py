"""GPU parity at the full sizes of the five workloads, in the call configuration bench.py
times (fa.forward / fa.backward on the whole batch).  The GPU runs the whole problem; the
oracle checks sampled heads exactly (whole heads where N <= 16384; sampled query rows and
key columns at N = 65536) plus the size-free identities
  sum over keys of dV = sum over queries of dO,   sum over keys of dK = 0
on every head.  Bars as in test_parity_gpu.py."""

import math

import numpy as np
import pytest
import torch

from exact_attention_96_gb300 import abi, build, inputs as I
from exact_attention_96_gb300 import attention as fa
from oracle import attention as A
from parity_util import (GRAD_REL_FRO, LSE_MAX_ABS, O_MAX_ABS, O_REL_FRO, max_abs, rel_fro,
                         to_device, to_f64, widen)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def library():
    build.build()
    abi.load()


def run(B, H, N, d, causal, mult=1.0, seed=0, bwd=True):
    host = I.attention_inputs(B, H, N, d, seed=seed, multiplier=mult, with_grad=bwd)
    tq, tk, tv = (to_device(x) for x in host[:3])
    o, lse = fa.forward(tq, tk, tv, causal=causal)
    grads = None
    if bwd:
        tdo = to_device(host[3])
        grads = fa.backward(tq, tk, tv, o, tdo, lse, causal=causal)
    assert fa.status_check() == abi.FA_OK
    return host, o, lse, grads


def head(x, b, h):
    return widen(x[b, h])


def check_identities(grads, do_bits):
    dk, dv = (to_f64(g) for g in grads[1:])
    do = widen(do_bits)
    assert np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))
    for b in range(dk.shape[0]):
        for h in range(dk.shape[1]):
            dv_sum_err = np.linalg.norm(dv[b, h].sum(0) - do[b, h].sum(0))
            assert dv_sum_err <= GRAD_REL_FRO * np.linalg.norm(dv[b, h]), (b, h, dv_sum_err)
            dk_sum = np.linalg.norm(dk[b, h].sum(0))
            assert dk_sum <= GRAD_REL_FRO * np.linalg.norm(dk[b, h]), (b, h, dk_sum)


def check_whole_heads(host, o, lse, grads, heads, d, causal):
    q, k, v = host[:3]
    scale = 1 / math.sqrt(d)
    o, lse = to_f64(o), to_f64(lse)
    for b, h in heads:
        o_ref, lse_ref = A.attention_fwd(head(q, b, h)[None, None], head(k, b, h)[None, None],
                                         head(v, b, h)[None, None], scale, causal)
        assert max_abs(o[b, h], o_ref[0, 0]) <= O_MAX_ABS, (b, h)
        assert rel_fro(o[b, h], o_ref[0, 0]) <= O_REL_FRO, (b, h)
        assert max_abs(lse[b, h], lse_ref[0, 0]) <= LSE_MAX_ABS, (b, h)
        if grads is None:
            continue
        refs = A.attention_bwd_head(head(q, b, h), head(k, b, h), head(v, b, h),
                                    head(host[3], b, h), scale, causal)
        for name, g, r in zip(("dq", "dk", "dv"), grads, refs[:3]):
            err = rel_fro(to_f64(g[b, h]), r)
            assert err <= GRAD_REL_FRO, (b, h, name, err)


def test_gpt2_medium_shape_fwd_bwd():
    # B=64, H=16, N=1024, d=64, non-causal
    host, o, lse, grads = run(64, 16, 1024, 64, False, seed=20)
    check_whole_heads(host, o, lse, grads, [(0, 0), (31, 7), (63, 15)], 64, False)
    check_identities(grads, host[3])


@pytest.mark.parametrize("N", [1024, 2048, 4096])
def test_memory_scaling_shape_fwd_bwd(N):
    # B=16, H=8, d=64, non-causal
    host, o, lse, grads = run(16, 8, N, 64, False, seed=30 + N)
    check_whole_heads(host, o, lse, grads, [(0, 0), (15, 7)], 64, False)
    check_identities(grads, host[3])


def test_long_causal_shape_fwd_bwd():
    # B=4, H=16, N=8192, d=128, causal, inputs x0.5 (the bench workload)
    host, o, lse, grads = run(4, 16, 8192, 128, True, mult=0.5, seed=40)
    check_whole_heads(host, o, lse, grads, [(0, 0), (3, 15)], 128, True)
    check_identities(grads, host[3])


def test_long_sequence_d64_noncausal_fwd():
    # B=1, H=8, N=65536, d=64, non-causal forward: sampled rows of two heads
    host, o, lse, _ = run(1, 8, 65536, 64, False, seed=50, bwd=False)
    q, k, v = host[:3]
    o, lse = to_f64(o), to_f64(lse)
    rows = np.r_[0:64, 32768:32832, 65472:65536]
    for h in (0, 7):
        o_ref, lse_ref = A.attention_fwd_rows(head(q, 0, h), head(k, 0, h), head(v, 0, h), 0.125, False, rows)
        assert max_abs(o[0, h, rows], o_ref) <= O_MAX_ABS
        assert rel_fro(o[0, h, rows], o_ref) <= O_REL_FRO
        assert max_abs(lse[0, h, rows], lse_ref) <= LSE_MAX_ABS


def test_long_sequence_d64_causal_fwd_bwd():
    # B=1, H=8, N=65536, d=64, causal forward + backward: sampled query rows (O, LSE, dQ)
    # and key columns (dK, dV) of one head, identities on all heads
    host, o, lse, grads = run(1, 8, 65536, 64, True, seed=60)
    q, k, v, do = host
    o, lse = to_f64(o), to_f64(lse)
    dq, dk, dv = (to_f64(g) for g in grads)
    h = 3
    rows = np.r_[0:32, 30000:30032, 65504:65536]
    o_ref, lse_ref = A.attention_fwd_rows(head(q, 0, h), head(k, 0, h), head(v, 0, h), 0.125, True, rows)
    assert max_abs(o[0, h, rows], o_ref) <= O_MAX_ABS
    assert rel_fro(o[0, h, rows], o_ref) <= O_REL_FRO
    assert max_abs(lse[0, h, rows], lse_ref) <= LSE_MAX_ABS
    dq_ref, _ = A.attention_bwd_rows(head(q, 0, h), head(k, 0, h), head(v, 0, h), head(do, 0, h),
                                     0.125, True, rows[1:])  # row 0 has dQ = 0 exactly
    assert rel_fro(dq[0, h, rows[1:]], dq_ref) <= GRAD_REL_FRO
    keys = np.r_[0:16, 40000:40016, 65520:65536]
    dk_ref, dv_ref = A.attention_bwd_key_columns(head(q, 0, h), head(k, 0, h), head(v, 0, h),
                                                 head(do, 0, h), 0.125, True, keys, row_chunk=1024)
    assert rel_fro(dk[0, h, keys], dk_ref) <= GRAD_REL_FRO
    assert rel_fro(dv[0, h, keys], dv_ref) <= GRAD_REL_FRO
    check_identities(grads, do)


@pytest.mark.parametrize("causal", [False, True])
def test_wide_head_d256_fwd(causal):
    # B=2, H=8, N=16384, d=256 forward: sampled rows of two heads
    host, o, lse, _ = run(2, 8, 16384, 256, causal, seed=70 + causal, bwd=False)
    q, k, v = host[:3]
    o, lse = to_f64(o), to_f64(lse)
    rows = np.r_[0:64, 8000:8064, 16320:16384]
    for b, h in ((0, 0), (1, 7)):
        o_ref, lse_ref = A.attention_fwd_rows(head(q, b, h), head(k, b, h), head(v, b, h),
                                              1 / 16, causal, rows)
        assert max_abs(o[b, h, rows], o_ref) <= O_MAX_ABS
        assert rel_fro(o[b, h, rows], o_ref) <= O_REL_FRO
        assert max_abs(lse[b, h, rows], lse_ref) <= LSE_MAX_ABS


def test_wide_head_d256_causal_fwd_bwd():
    # B=2, H=8, N=16384, d=256, causal forward + backward: one whole head against the oracle,
    # key-sum identities on every head
    host, o, lse, grads = run(2, 8, 16384, 256, True, seed=80)
    check_whole_heads(host, o, lse, grads, [(1, 5)], 256, True)
    check_identities(grads, host[3])


def test_wide_head_d256_causal_dispatch_groups():
    # The d = 256 backward dispatches causal heads in groups whose streamed tensors fit L2:
    # two heads at N = 16384, so three heads leave a last group of one; one head from
    # N ~ 42k on.  Both launch orders must give the same gradients as the oracle.
    host, o, lse, grads = run(1, 3, 16384, 256, True, seed=90)
    check_whole_heads(host, o, lse, grads, [(0, 2)], 256, True)
    check_identities(grads, host[3])

    N = 42000  # a ragged length (not a multiple of the 64-row query tile)
    host, o, lse, grads = run(1, 2, N, 256, True, seed=91)
    q, k, v, do = host
    dq, dk, dv = (to_f64(g) for g in grads)
    h = 1
    rows = np.r_[1:33, 20000:20032, N - 32:N]
    dq_ref, _ = A.attention_bwd_rows(head(q, 0, h), head(k, 0, h), head(v, 0, h), head(do, 0, h),
                                     1 / 16, True, rows)
    assert rel_fro(dq[0, h, rows], dq_ref) <= GRAD_REL_FRO
    keys = np.r_[0:16, 21000:21016, N - 16:N]
    dk_ref, dv_ref = A.attention_bwd_key_columns(head(q, 0, h), head(k, 0, h), head(v, 0, h),
                                                 head(do, 0, h), 1 / 16, True, keys, row_chunk=1024)
    assert rel_fro(dk[0, h, keys], dk_ref) <= GRAD_REL_FRO
    assert rel_fro(dv[0, h, keys], dv_ref) <= GRAD_REL_FRO
    check_identities(grads, do)
