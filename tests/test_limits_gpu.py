"""The ABI's size limits on the GPU: B*H = 65535 heads (the largest grid dimension the kernels
use) and N = 2^20 positions (the longest sequence accepted), each against the fp64 oracle on
sampled heads or rows, plus the size-free key-sum identity of dK.  Bars as in
test_parity_gpu.py."""

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


@pytest.mark.parametrize("causal", [False, True])
def test_most_heads(causal):
    B, H, N, d = 65535, 1, 3, 64
    host = I.attention_inputs(B, H, N, d, seed=31)
    tq, tk, tv, tdo = (to_device(x) for x in host)
    o, lse = fa.forward(tq, tk, tv, causal=causal)
    dq, dk, dv = fa.backward(tq, tk, tv, o, tdo, lse, causal=causal)
    assert fa.status_check() == abi.FA_OK
    o, lse, dq, dk, dv = (to_f64(t) for t in (o, lse, dq, dk, dv))
    scale = 1 / math.sqrt(d)
    for b in (0, 1, 32767, 65533, 65534):
        q, k, v, do = (widen(x[b, 0]) for x in host)
        o_ref, lse_ref = A.attention_fwd(q[None, None], k[None, None], v[None, None], scale, causal)
        assert max_abs(o[b, 0], o_ref[0, 0]) <= O_MAX_ABS, b
        assert max_abs(lse[b, 0], lse_ref[0, 0]) <= LSE_MAX_ABS, b
        refs = A.attention_bwd_head(q, k, v, do, scale, causal)
        for g, r in zip((dq[b, 0], dk[b, 0], dv[b, 0]), refs[:3]):
            assert rel_fro(g, r) <= GRAD_REL_FRO or max_abs(g, r) <= 1e-3, b


def test_longest_sequence():
    B, H, N, d = 1, 1, 1 << 20, 64
    host = I.attention_inputs(B, H, N, d, seed=32)
    tq, tk, tv, tdo = (to_device(x) for x in host)
    o, lse = fa.forward(tq, tk, tv, causal=True)
    dq, dk, dv = fa.backward(tq, tk, tv, o, tdo, lse, causal=True)
    assert fa.status_check() == abi.FA_OK
    q, k, v, do = (widen(x[0, 0]) for x in host)
    rows = np.r_[1:9, 524284:524292, N - 8:N]  # row 0 has dQ = 0 exactly
    o_ref, lse_ref = A.attention_fwd_rows(q, k, v, 0.125, True, rows)
    o_r = to_f64(o)[0, 0, rows]
    assert max_abs(o_r, o_ref) <= O_MAX_ABS and rel_fro(o_r, o_ref) <= O_REL_FRO
    assert max_abs(to_f64(lse)[0, 0, rows], lse_ref) <= LSE_MAX_ABS
    dq_ref, _ = A.attention_bwd_rows(q, k, v, do, 0.125, True, rows)
    assert rel_fro(to_f64(dq)[0, 0, rows], dq_ref) <= GRAD_REL_FRO
    dk64 = to_f64(dk)[0, 0]
    assert np.all(np.isfinite(dk64)) and np.all(np.isfinite(to_f64(dv)))
    assert np.linalg.norm(dk64.sum(0)) <= GRAD_REL_FRO * np.linalg.norm(dk64)
