"""The method's degenerate cases on the GPU, checked against closed forms rather than only
against the oracle:

- every key equal: the probabilities are uniform over the visible keys, so O is the mean of
  the visible value rows (the whole column mean, or the prefix mean when causal), LSE is
  ln(visible keys) + scale * q.k, dV_j is the sum of dO_i / (visible keys of i) over the
  queries that see key j, and dQ vanishes (each row of dS sums to zero and every key is the
  same vector);
- one dominant key per query (a large dot product with it): O is that key's value row;
- scores of several hundred (large inputs, scale 1): the running maximum keeps the
  exponentials finite, and the result matches the fp64 oracle.

Bars as in test_parity_gpu.py."""

import math

import numpy as np
import pytest

from exact_attention_96_gb300 import abi, build, inputs as I
from exact_attention_96_gb300 import attention as fa
from oracle import attention as A
from parity_util import (GRAD_REL_FRO, LSE_MAX_ABS, O_MAX_ABS, O_REL_FRO, max_abs, rel_fro,
                         to_device, to_f64, widen)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    build.build()
    abi.load()


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_equal_keys_give_uniform_average(d, causal):
    B, H, N = 1, 2, 300
    q, k, v, do = I.attention_inputs(B, H, N, d, seed=500 + d)
    k = np.ascontiguousarray(np.broadcast_to(k[:, :, :1, :], k.shape))  # every key = key 0
    tq, tk, tv, tdo = (to_device(x) for x in (q, k, v, do))
    scale = 1 / math.sqrt(d)
    o, lse = fa.forward(tq, tk, tv, causal=causal)
    dq, dk, dv = fa.backward(tq, tk, tv, o, tdo, lse, causal=causal)
    assert fa.status_check() == abi.FA_OK
    qf, kf, vf, dof = (widen(x) for x in (q, k, v, do))
    n_vis = np.arange(1, N + 1, dtype=np.float64) if causal else np.full(N, float(N))
    if causal:
        o_ref = np.cumsum(vf, axis=2) / n_vis[None, None, :, None]
    else:
        o_ref = np.broadcast_to(vf.mean(axis=2, keepdims=True), vf.shape)
    lse_ref = np.log(n_vis)[None, None, :] + scale * np.einsum("bhnd,bhd->bhn", qf, kf[:, :, 0])
    o64, lse64 = to_f64(o), to_f64(lse)
    assert max_abs(o64, o_ref) <= O_MAX_ABS and rel_fro(o64, o_ref) <= O_REL_FRO
    assert max_abs(lse64, lse_ref) <= LSE_MAX_ABS
    # dV_j = sum over the queries i that see key j of dO_i / (keys i sees)
    w = dof / n_vis[None, None, :, None]
    dv_ref = (np.cumsum(w[:, :, ::-1], axis=2)[:, :, ::-1] if causal
              else np.broadcast_to(w.sum(axis=2, keepdims=True), w.shape))
    assert rel_fro(to_f64(dv), dv_ref) <= GRAD_REL_FRO
    # dQ = scale * dS K with every key equal and each row of dS summing to zero: dQ = 0, up
    # to the rounding of P and dS (measured against the size dK takes)
    dq64, dk64 = to_f64(dq), to_f64(dk)
    assert np.linalg.norm(dq64) <= GRAD_REL_FRO * np.linalg.norm(dk64)
    _, dk_ref, _, _ = A.attention_bwd(qf, kf, vf, dof, scale, causal)
    assert rel_fro(dk64, dk_ref) <= GRAD_REL_FRO


@pytest.mark.parametrize("d", [64, 128])
def test_dominant_key_selects_its_value(d):
    # key j = the query row i's own direction scaled up, for a permutation of the keys:
    # query i sees key perm[i] with score ~ 16 * |q_i|^2 / sqrt(d), far above the rest
    B, H, N = 1, 1, 256
    rng = np.random.default_rng(7)
    q, _, v, _ = I.attention_inputs(B, H, N, d, seed=600 + d, with_grad=False)
    perm = rng.permutation(N)
    qf = widen(q)
    kf = np.zeros_like(qf)
    kf[:, :, perm] = 16.0 * qf  # exact in bf16: a power-of-two multiple of bf16 values
    k = I.f32_to_bf16_bits(kf.astype(np.float32))
    assert np.array_equal(widen(k), kf)
    o, lse = fa.forward(to_device(q), to_device(k), to_device(v), causal=False)
    assert fa.status_check() == abi.FA_OK
    o_ref, lse_ref = A.attention_fwd(qf, kf, widen(v), 1 / math.sqrt(d), False)
    o64 = to_f64(o)
    assert max_abs(o64, o_ref) <= O_MAX_ABS and max_abs(to_f64(lse), lse_ref) <= LSE_MAX_ABS
    # the winner takes (nearly) all: O_i is within the parity bar of V[perm[i]]
    assert max_abs(o64[0, 0], widen(v)[0, 0, perm]) <= 2 * O_MAX_ABS


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_large_scores_stay_finite_and_exact(d, causal):
    # inputs x4 and scale 1: scores of several hundred, far past exp's fp32 range without
    # the running maximum
    B, H, N = 1, 2, 333
    q, k, v, do = I.attention_inputs(B, H, N, d, seed=700 + d, multiplier=4.0)
    tq, tk, tv, tdo = (to_device(x) for x in (q, k, v, do))
    o, lse = fa.forward(tq, tk, tv, causal=causal, scale=1.0)
    dq, dk, dv = fa.backward(tq, tk, tv, o, tdo, lse, causal=causal, scale=1.0)
    assert fa.status_check() == abi.FA_OK
    qf, kf, vf, dof = (widen(x) for x in (q, k, v, do))
    o_ref, lse_ref = A.attention_fwd(qf, kf, vf, 1.0, causal)
    assert np.max(np.abs(lse_ref)) > 200  # the case is what it claims
    o64, lse64 = to_f64(o), to_f64(lse)
    assert np.all(np.isfinite(o64)) and np.all(np.isfinite(lse64))
    # |V| reaches ~18 here, where bf16 rounding alone is up to 2^-8 of the value: the
    # absolute bar grows with it
    assert np.all(np.abs(o64 - o_ref) <= 2.0 ** -8 * np.abs(o_ref) + O_MAX_ABS)
    assert rel_fro(o64, o_ref) <= O_REL_FRO
    # LSE error model.  LSE is a smooth maximum of the row's scores (its derivative in S_ij is
    # P_ij), so it inherits the largest score error, plus the fp32 roundings of quantities of
    # its own size (the scaled maximum, the final change of base): about 2^-24 |LSE|.  A score
    # is an fp32 sum of d exact products; its rounding error is of the order of
    # 2^-24 sqrt(d) ||q_i * k_j||_2.  Measured on these inputs (d = 64 .. 256, |LSE| up to
    # ~1100): at most 1.15 times 2^-24 (|LSE_i| + sqrt(d) max_j ||q_i * k_j||_2), 4.0e-4 in
    # absolute terms.  The bar is 8 times that model per row, and the target's absolute bar.
    err = np.abs(lse64 - lse_ref)
    qk = np.sqrt(np.einsum("bhic,bhjc->bhij", qf ** 2, kf ** 2))
    if causal:
        qk = np.where(np.tril(np.ones((N, N), bool)), qk, 0.0)
    model = 2.0 ** -24 * (np.abs(lse_ref) + math.sqrt(d) * qk.max(-1))
    assert np.all(err <= 8 * model), float(np.max(err / model))
    assert np.max(err) <= LSE_MAX_ABS
    refs = A.attention_bwd(qf, kf, vf, dof, 1.0, causal)
    for name, g, r in (("dq", dq, refs[0]), ("dk", dk, refs[1]), ("dv", dv, refs[2])):
        g = to_f64(g)
        assert np.all(np.isfinite(g)), name
        assert rel_fro(g, r) <= GRAD_REL_FRO, (name, rel_fro(g, r))
