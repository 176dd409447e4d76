"""Dropout at the full size of the long causal language-model shape, 4 x 16 x 8192 x 128
causal (inputs x0.5), p = 0.1, in the call configuration bench.py times (fa.forward /
fa.backward with dropout on the whole batch).  The oracle checks sampled query rows (O, LSE,
dQ) and key columns (dK, dV) of heads spread over the batch, each with its own generator
mask, and the identity sum over keys of dK = 0 on every head (with dropout it still holds:
D = rowsum(dO * O) = rowsum(P * Z * dP)).  Bars as in test_dropout_gpu.py."""

import math

import numpy as np
import pytest

from exact_attention_96_gb300 import abi, build, inputs as I
from exact_attention_96_gb300 import attention as fa
from oracle import attention as A
from oracle import philox
from parity_util import (GRAD_REL_FRO, LSE_MAX_ABS, O_MAX_ABS, O_REL_FRO, max_abs, rel_fro,
                         to_device, to_f64, widen)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def library():
    build.build()
    abi.load()


def test_long_causal_shape_with_dropout():
    B, H, N, d, p, seed = 4, 16, 8192, 128, 0.1, 20261202
    scale = 1 / math.sqrt(d)
    host = I.attention_inputs(B, H, N, d, seed=90, multiplier=0.5)
    tq, tk, tv, tdo = (to_device(x) for x in host)
    o, lse = fa.forward(tq, tk, tv, causal=True, dropout_p=p, seed=seed)
    grads = fa.backward(tq, tk, tv, o, tdo, lse, causal=True, dropout_p=p, seed=seed)
    assert fa.status_check() == abi.FA_OK
    q, k, v, do = (widen(x) for x in host)
    o, lse = to_f64(o), to_f64(lse)
    dq, dk, dv = (to_f64(g) for g in grads)
    assert all(np.all(np.isfinite(x)) for x in (o, lse, dq, dk, dv))
    rows = np.r_[1:17, 4000:4016, 8176:8192]  # row 0 has dQ = 0 exactly
    for b, h in ((0, 0), (1, 7), (3, 15)):
        bh = b * H + h
        o_ref, lse_ref = A.attention_fwd_rows(q[b, h], k[b, h], v[b, h], scale, True, rows,
                                              dropout_p=p, seed=seed, bh=bh)
        assert max_abs(o[b, h, rows], o_ref) <= O_MAX_ABS * philox.keep_scale(p), (b, h)
        assert rel_fro(o[b, h, rows], o_ref) <= O_REL_FRO, (b, h)
        assert max_abs(lse[b, h, rows], lse_ref) <= LSE_MAX_ABS, (b, h)
        dq_ref, _ = A.attention_bwd_rows(q[b, h], k[b, h], v[b, h], do[b, h], scale, True, rows,
                                         dropout_p=p, seed=seed, bh=bh)
        assert rel_fro(dq[b, h, rows], dq_ref) <= GRAD_REL_FRO, (b, h)
    keys = np.r_[0:16, 5000:5016, 8176:8192]
    for b, h in ((0, 3), (2, 11)):
        bh = b * H + h
        dk_ref, dv_ref = A.attention_bwd_key_columns(q[b, h], k[b, h], v[b, h], do[b, h], scale, True,
                                                     keys, row_chunk=1024, dropout_p=p, seed=seed, bh=bh)
        assert rel_fro(dk[b, h, keys], dk_ref) <= GRAD_REL_FRO, (b, h)
        assert rel_fro(dv[b, h, keys], dv_ref) <= GRAD_REL_FRO, (b, h)
    for b in range(B):
        for h in range(H):
            assert np.linalg.norm(dk[b, h].sum(0)) <= GRAD_REL_FRO * np.linalg.norm(dk[b, h]), (b, h)
