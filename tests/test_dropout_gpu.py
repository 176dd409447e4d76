"""GPU parity of dropout (fa_fwd_dropout, fa_bwd_dropout) against the oracle.

The mask is compared bit for bit: with Q = 0 every score is equal, so P is uniform, and a
one-hot V (forward) or dO (backward) turns O, or dV, into the mask itself scaled by a positive
constant; its zero pattern must equal the oracle's generator mask exactly, key tile by key
tile, for several heads.  Values are then compared with the fp64 oracle on seeded random
inputs under the plain path's bars (O rel-Frobenius <= 5e-3, LSE max-abs <= 1e-3, dQ/dK/dV
rel-Frobenius <= 2e-2), with one change: O's max-abs bar, 1e-2 for the plain path, is applied
to O / s with s = 1 / q_keep the dropout scale.  Dropout multiplies the kept terms by s, so
|O| is bounded by s * max|V| instead of max|V|, and the bf16 rounding of O (up to 2^-9 |O|)
grows with it: at p = 0.5 outputs in [4, 8) round by up to 0.0156."""

import math

import numpy as np
import pytest
import torch

from exact_attention_96_gb300 import abi, build, inputs as I
from exact_attention_96_gb300 import attention as fa
from oracle import attention as A
from oracle import philox
from parity_util import (GRAD_REL_FRO, LSE_MAX_ABS, O_MAX_ABS, O_REL_FRO, max_abs, rel_fro,
                         to_device, to_f64, widen)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    build.build()
    abi.load()


def oracle_mask(B, H, N, p, seed):
    """keep[b, h, i, j] of the oracle's generator."""
    return np.stack([np.stack([philox.dropout_keep(b * H + h, np.arange(N), np.arange(N), p, seed)
                               for h in range(H)]) for b in range(B)])


# ------------------------------------------------------------------ mask ---

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("p,seed", [(0.3, 1234), (0.5, (7 << 32) | 99)])
def test_forward_mask_bit_exact(causal, p, seed):
    B, H, N, d = 2, 2, 1000, 256
    keep = oracle_mask(B, H, N, p, seed)
    if causal:
        keep = keep & (np.arange(N)[None, :] <= np.arange(N)[:, None])
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    k = to_device(I.normal_bf16((B, H, N, d), seed=5))
    for t in range(0, N, d):  # V one-hot over keys [t, t + d)
        n = min(d, N - t)
        v = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
        v[:, :, t:t + n, :n] = torch.eye(n, dtype=torch.bfloat16, device="cuda")
        o, _ = fa.forward(q, k, v, causal=causal, dropout_p=p, seed=seed)
        assert fa.status_check() == abi.FA_OK
        got = to_f64(o)[..., :n] > 0
        assert np.array_equal(got, keep[..., t:t + n]), (t, np.argwhere(got != keep[..., t:t + n])[:5])


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_mask_bit_exact(d, causal):
    B, H, N, p, seed = 1, 3, 700, 0.4, 424242
    keep = oracle_mask(B, H, N, p, seed)
    if causal:
        keep = keep & (np.arange(N)[None, :] <= np.arange(N)[:, None])
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    k = to_device(I.normal_bf16((B, H, N, d), seed=6))
    v = to_device(I.normal_bf16((B, H, N, d), seed=7))
    o, lse = fa.forward(q, k, v, causal=causal, dropout_p=p, seed=seed)
    for t in range(0, N, d):  # dO one-hot over queries [t, t + d): dV[j, c] ~ keep[t + c, j]
        n = min(d, N - t)
        do = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
        do[:, :, t:t + n, :n] = torch.eye(n, dtype=torch.bfloat16, device="cuda")
        _, _, dv = fa.backward(q, k, v, o, do, lse, causal=causal, dropout_p=p, seed=seed)
        assert fa.status_check() == abi.FA_OK
        got = to_f64(dv)[..., :n] != 0            # [b, h, key j, c]
        want = np.swapaxes(keep[:, :, t:t + n, :], -1, -2)
        assert np.array_equal(got, want), (t, np.argwhere(got != want)[:5])


def test_keep_rate_and_scale_on_device():
    # uniform P and all-ones V: O_i = scale * (kept keys of row i) / N
    B, H, N, d, p, seed = 1, 4, 4096, 64, 0.25, 77
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    k = to_device(I.normal_bf16((B, H, N, d), seed=8))
    v = torch.ones((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    o, _ = fa.forward(q, k, v, dropout_p=p, seed=seed)
    kept = oracle_mask(B, H, N, p, seed).sum(-1)
    want = philox.keep_scale(p) * kept / N
    got = to_f64(o)[..., 0]
    assert np.max(np.abs(got - want) / want) < 2 ** -8
    assert abs(kept.mean() / N - (1 - p)) < 1e-2


# ---------------------------------------------------------------- values ---

FWD = [
    # (B, H, N, d, causal, p)
    (1, 2, 300, 128, False, 0.1),
    (2, 1, 257, 64, True, 0.5),
    (1, 1, 333, 256, True, 0.2),
    (1, 2, 640, 64, False, 0.3),
    (1, 1, 1, 128, True, 0.5),
]


def check_fwd(o, lse, o_ref, lse_ref, what, p):
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), what
    assert max_abs(o, o_ref) <= O_MAX_ABS * philox.keep_scale(p), (what, max_abs(o, o_ref))
    assert rel_fro(o, o_ref) <= O_REL_FRO, (what, rel_fro(o, o_ref))
    assert max_abs(lse, lse_ref) <= LSE_MAX_ABS, (what, max_abs(lse, lse_ref))


@pytest.mark.parametrize("B,H,N,d,causal,p", FWD)
def test_forward_values(B, H, N, d, causal, p):
    seed = 1000 + N
    q, k, v, _ = I.attention_inputs(B, H, N, d, seed=N + d, with_grad=False)
    o, lse = fa.forward(to_device(q), to_device(k), to_device(v), causal=causal, dropout_p=p, seed=seed)
    assert fa.status_check() == abi.FA_OK
    o_ref, lse_ref = A.attention_fwd(widen(q), widen(k), widen(v), 1 / math.sqrt(d), causal,
                                     dropout_p=p, seed=seed)
    check_fwd(to_f64(o), to_f64(lse), o_ref, lse_ref, (B, H, N, d, causal, p), p)


BWD = [
    (1, 2, 300, 128, False, 0.1),
    (2, 1, 257, 64, True, 0.5),
    (1, 1, 640, 128, True, 0.2),
    (1, 2, 383, 64, False, 0.3),
    (2, 4, 1024, 128, True, 0.1),
    (3, 3, 260, 64, True, 0.2),  # causal heads in a full group of eight and a partial one
    (1, 2, 300, 256, True, 0.2),
    (2, 1, 200, 256, False, 0.3),
]


@pytest.mark.parametrize("B,H,N,d,causal,p", BWD)
def test_backward_values(B, H, N, d, causal, p):
    seed = 31 * N + d
    q, k, v, do = I.attention_inputs(B, H, N, d, seed=N + 7)
    tq, tk, tv, tdo = (to_device(x) for x in (q, k, v, do))
    scale = 1 / math.sqrt(d)
    o, lse = fa.forward(tq, tk, tv, causal=causal, dropout_p=p, seed=seed)
    dq, dk, dv = fa.backward(tq, tk, tv, o, tdo, lse, causal=causal, dropout_p=p, seed=seed)
    assert fa.status_check() == abi.FA_OK
    o_ref, lse_ref = A.attention_fwd(widen(q), widen(k), widen(v), scale, causal, dropout_p=p, seed=seed)
    check_fwd(to_f64(o), to_f64(lse), o_ref, lse_ref, (B, H, N, d, causal, p), p)
    ref = A.attention_bwd(widen(q), widen(k), widen(v), widen(do), scale, causal, dropout_p=p, seed=seed)
    for name, g, r in (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
        assert np.all(np.isfinite(to_f64(g))), name
        assert rel_fro(to_f64(g), r) <= GRAD_REL_FRO, (name, rel_fro(to_f64(g), r))


# ------------------------------------------------------------ properties ---

def test_zero_probability_equals_plain_path_bitwise():
    B, H, N, d = 1, 2, 517, 128
    q, k, v, do = (to_device(x) for x in I.attention_inputs(B, H, N, d, seed=3))
    o0, l0 = fa.forward(q, k, v, causal=True)
    # p below 2^-17 rounds to threshold 0: every element kept, scale 1
    o1, l1 = fa.forward(q, k, v, causal=True, dropout_p=1e-7, seed=5)
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    g0 = fa.backward(q, k, v, o0, do, l0, causal=True)
    g1 = fa.backward(q, k, v, o0, do, l0, causal=True, dropout_p=1e-7, seed=5)
    assert all(torch.equal(a, b) for a, b in zip(g0, g1))


def test_same_seed_repeats_and_new_seed_changes():
    B, H, N, d = 1, 2, 384, 64
    q, k, v, do = (to_device(x) for x in I.attention_inputs(B, H, N, d, seed=4))
    a = fa.forward(q, k, v, dropout_p=0.2, seed=11)[0]
    b = fa.forward(q, k, v, dropout_p=0.2, seed=11)[0]
    c = fa.forward(q, k, v, dropout_p=0.2, seed=12)[0]
    assert torch.equal(a, b) and not torch.equal(a, c)
