"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each check is chosen so that a plausible slip in the oracle (a dropped scale, a
transposed operand, a sign error in the softmax Jacobian, the wrong side of the causal
mask, a missing rescale in the streaming softmax) fails at least one of them:

* invariants the pages state (rows of P sum to 1; blockwise softmax equals whole-row
  softmax; causal zeros),
* closed forms and special cases (N = 1, equal keys, a dominant key, d = 1 by hand),
* an independent library implementation (torch's CPU math attention in float64 and
  torch.autograd),
* central finite differences of L = sum(O * dO) for the gradients,
* the worked numbers printed on the pages (tests/golden/pages_numbers.json).
"""

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attention as A
from oracle import io_model as IO
from oracle import online_softmax as OS
from exact_attention_96_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.json")


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# ---------------------------------------------------------------- invariants ---

@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one_and_causal_zeros(causal):
    # With V = identity (d = N) the output O is P itself.
    N = 24
    q = rnd((1, 1, N, N), 1)
    k = rnd((1, 1, N, N), 2)
    v = np.eye(N)[None, None]
    o, _ = A.attention_fwd(q, k, v, scale=0.3, causal=causal, row_chunk=7)
    p = o[0, 0]
    assert np.max(np.abs(p.sum(axis=1) - 1.0)) < 1e-14
    assert np.all(p >= 0)
    if causal:
        assert np.all(p[np.triu_indices(N, 1)] == 0.0)
        assert np.all(p[np.tril_indices(N)] > 0.0)


@pytest.mark.parametrize("seed", range(4))
def test_streaming_softmax_equals_whole_row_every_block_size(seed):
    n = 37
    x = rnd(n, seed, scale=[1.0, 5.0, 30.0, 0.01][seed])
    ref = OS.full_softmax_row(x)
    for block in range(1, n + 1):
        got = OS.online_softmax_row(x, block)
        assert np.max(np.abs(got - ref)) < 1e-12, block
        m, l = OS.online_row_stats(x, block)
        assert m == x.max()
        assert abs(l - np.exp(x - x.max()).sum()) < 1e-12 * max(1.0, l)


def test_streaming_softmax_increasing_and_decreasing_rows():
    # Increasing scores force a rescale on every block; decreasing scores never do.
    for x in (np.linspace(-3, 4, 16), np.linspace(4, -3, 16)):
        for block in (1, 2, 3, 16):
            assert np.max(np.abs(OS.online_softmax_row(x, block) - OS.full_softmax_row(x))) < 1e-15


def test_streaming_softmax_page_example_shape():
    # "FlashAttention 与显存" §08: one row of 8 scores taken 2 at a time; after the four
    # steps the blockwise result differs from the whole row by less than 1e-15.  The
    # page does not print the 8 scores, so its m = 3.4 and l = 2.170462 stay unpinned;
    # the invariant is checked on rows whose maximum is 3.4.
    bound = json.load(open(GOLDEN))["online_softmax_equal_within"]["value"]
    rng = np.random.default_rng(8)
    for _ in range(50):
        x = rng.uniform(-2, 3.4, size=8)
        x[rng.integers(8)] = 3.4
        m, l = OS.online_row_stats(x, 2)
        assert m == 3.4
        assert np.max(np.abs(OS.online_softmax_row(x, 2) - OS.full_softmax_row(x))) < bound


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("br,bc", [(1, 1), (4, 3), (5, 8), (16, 16), (7, 50)])
def test_tiled_forward_both_loop_orders_equal_definition(causal, br, bc):
    N, d = 29, 6
    q, k, v = rnd((N, d), 3), rnd((N, d), 4), rnd((N, d), 5)
    o_ref, lse_ref = A.attention_fwd(q[None, None], k[None, None], v[None, None], 0.4, causal)
    for fn in (OS.tiled_forward_q_outer, OS.tiled_forward_kv_outer):
        o, lse = fn(q, k, v, 0.4, causal, br, bc)
        assert np.max(np.abs(o - o_ref[0, 0])) < 1e-12, fn.__name__
        assert np.max(np.abs(lse - lse_ref[0, 0])) < 1e-12, fn.__name__


# ------------------------------------------------------- independent library ---

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(2, 3, 17, 8), (1, 2, 64, 16), (1, 1, 5, 3)])
def test_forward_and_backward_match_torch_math_attention(causal, shape):
    B, H, N, d = shape
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (rnd(shape, s) for s in (11, 12, 13, 14))
    o, lse = A.attention_fwd(q, k, v, scale, causal, row_chunk=6)
    dq, dk, dv, dvec = A.attention_bwd(q, k, v, do, scale, causal, row_chunk=5)

    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    to = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    to.backward(torch.tensor(do))
    s = scale * torch.tensor(q) @ torch.tensor(k).transpose(-1, -2)
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    tlse = torch.logsumexp(s, dim=-1)

    assert np.max(np.abs(o - to.detach().numpy())) < 1e-12
    assert np.max(np.abs(lse - tlse.numpy())) < 1e-12
    assert np.max(np.abs(dq - tq.grad.numpy())) < 1e-11
    assert np.max(np.abs(dk - tk.grad.numpy())) < 1e-11
    assert np.max(np.abs(dv - tv.grad.numpy())) < 1e-11
    assert np.max(np.abs(dvec - np.sum(do * to.detach().numpy(), axis=-1))) < 1e-11


def test_sampled_rows_match_whole_tensor():
    N, d = 70, 8
    q, k, v, do = (rnd((N, d), s) for s in (21, 22, 23, 24))
    rows = np.array([0, 1, 33, 69])
    for causal in (False, True):
        o, lse = A.attention_fwd(q[None, None], k[None, None], v[None, None], 0.35, causal)
        o_r, lse_r = A.attention_fwd_rows(q, k, v, 0.35, causal, rows)
        assert np.max(np.abs(o_r - o[0, 0, rows])) < 1e-14
        assert np.max(np.abs(lse_r - lse[0, 0, rows])) < 1e-14
        dq, _, _, dvec = A.attention_bwd_head(q, k, v, do, 0.35, causal, row_chunk=16)
        dq_r, d_r = A.attention_bwd_rows(q, k, v, do, 0.35, causal, rows)
        assert np.max(np.abs(dq_r - dq[rows])) < 1e-13
        assert np.max(np.abs(d_r - dvec[rows])) < 1e-13


def test_sampled_key_columns_match_whole_head():
    N, d = 90, 8
    q, k, v, do = (rnd((N, d), s) for s in (25, 26, 27, 28))
    keys = np.array([0, 5, 44, 89])
    for causal in (False, True):
        _, dk, dv, _ = A.attention_bwd_head(q, k, v, do, 0.3, causal, row_chunk=32)
        dk_c, dv_c = A.attention_bwd_key_columns(q, k, v, do, 0.3, causal, keys, row_chunk=17)
        assert np.max(np.abs(dk_c - dk[keys])) < 1e-13
        assert np.max(np.abs(dv_c - dv[keys])) < 1e-13


def test_gradient_sums_over_keys():
    # Rows of P sum to one and rows of dS sum to zero, so summed over keys dV equals the
    # sum of dO over queries and dK sums to zero -- identities usable at any size.
    N, d = 40, 6
    q, k, v, do = (rnd((N, d), s) for s in (29, 30, 31, 32))
    for causal in (False, True):
        _, dk, dv, _ = A.attention_bwd_head(q, k, v, do, 0.5, causal)
        assert np.max(np.abs(dv.sum(axis=0) - do.sum(axis=0))) < 1e-12
        assert np.max(np.abs(dk.sum(axis=0))) < 1e-12


def test_queries_and_keys_of_different_lengths_match_torch():
    # the decoding shape: few queries against a long key sequence (no mask)
    q, k, v = rnd((2, 3, 5, 8), 91), rnd((2, 3, 37, 8), 92), rnd((2, 3, 37, 8), 93)
    o, lse = A.attention_fwd(q, k, v, 0.4, False)
    tq, tk, tv = (torch.tensor(x) for x in (q, k, v))
    ref = F.scaled_dot_product_attention(tq, tk, tv, scale=0.4).numpy()
    tlse = torch.logsumexp(0.4 * tq @ tk.transpose(-1, -2), dim=-1).numpy()
    assert np.max(np.abs(o - ref)) < 1e-12
    assert np.max(np.abs(lse - tlse)) < 1e-12


@pytest.mark.parametrize("cuts", [[0, 37], [0, 1, 37], [0, 10, 11, 30, 37], list(range(38))])
def test_split_key_ranges_merge_to_whole(cuts):
    q, k, v = rnd((1, 2, 6, 4), 94), rnd((1, 2, 37, 4), 95), rnd((1, 2, 37, 4), 96)
    o, lse = A.attention_fwd(q, k, v, 0.7, False)
    parts = [A.attention_fwd(q, k[:, :, a:b], v[:, :, a:b], 0.7, False) for a, b in zip(cuts, cuts[1:])]
    o_m, lse_m = A.lse_merge([p[0] for p in parts], [p[1] for p in parts])
    assert np.max(np.abs(o_m - o)) < 1e-12
    assert np.max(np.abs(lse_m - lse)) < 1e-12


def test_merge_is_not_a_plain_average():
    # planted slip: averaging the parts (dropping the exp(LSE_s - LSE) weights) must differ
    q, k, v = rnd((1, 1, 4, 4), 97), rnd((1, 1, 20, 4), 98), rnd((1, 1, 20, 4), 99)
    o, _ = A.attention_fwd(q, k, v, 1.0, False)
    parts = [A.attention_fwd(q, k[:, :, a:b], v[:, :, a:b], 1.0, False) for a, b in ((0, 3), (3, 20))]
    assert np.max(np.abs(np.mean([p[0] for p in parts], axis=0) - o)) > 1e-2


# ------------------------------------------------------- finite differences ---

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(1, 1), (3, 2), (6, 4), (5, 3)])
def test_gradients_match_central_finite_differences(causal, N, d):
    q, k, v, do = (rnd((N, d), s) for s in (31, 32, 33, 34))
    scale = 0.7
    h = 1e-6

    def loss(q_, k_, v_):
        o, _ = A.attention_fwd(q_[None, None], k_[None, None], v_[None, None], scale, causal)
        return float(np.sum(o[0, 0] * do))

    dq, dk, dv, _ = A.attention_bwd_head(q, k, v, do, scale, causal)
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        num = np.zeros_like(grad)
        for idx in np.ndindex(*grad.shape):
            args_p = [q.copy(), k.copy(), v.copy()]
            args_m = [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.linalg.norm(num - grad) / max(np.linalg.norm(grad), 1e-12)
        assert err < 1e-7 or np.max(np.abs(num - grad)) < 1e-8, (which, err)


# ---------------------------------------------------------- causal structure ---

def test_causal_first_row_and_key_independence():
    N, d = 12, 5
    q, k, v, do = (rnd((N, d), s) for s in (41, 42, 43, 44))
    scale = 0.5
    o, lse = A.attention_fwd(q[None, None], k[None, None], v[None, None], scale, True)
    assert np.array_equal(o[0, 0, 0], v[0])
    assert abs(lse[0, 0, 0] - scale * float(q[0] @ k[0])) < 1e-15
    _, dk, dv, _ = A.attention_bwd_head(q, k, v, do, scale, True)
    # Queries before position t never see keys at or after t: changing them (and their
    # upstream gradients) leaves dK and dV of keys t.. unchanged.
    t = 5
    q2, do2 = q.copy(), do.copy()
    q2[:t] = rnd((t, d), 45)
    do2[:t] = rnd((t, d), 46)
    _, dk2, dv2, _ = A.attention_bwd_head(q2, k, v, do2, scale, True)
    assert np.max(np.abs(dk2[t:] - dk[t:])) < 1e-15
    assert np.max(np.abs(dv2[t:] - dv[t:])) < 1e-15
    assert np.max(np.abs(dk2[:t] - dk[:t])) > 1e-3


# ---------------------------------------------------------- closed forms ---

def test_single_key_output_is_value():
    q, k, v = rnd((1, 1, 1, 7), 51), rnd((1, 1, 1, 7), 52), rnd((1, 1, 1, 7), 53)
    for causal in (False, True):
        o, lse = A.attention_fwd(q, k, v, 0.9, causal)
        assert np.array_equal(o, v)
        assert abs(lse[0, 0, 0] - 0.9 * float(q[0, 0, 0] @ k[0, 0, 0])) < 1e-15


def test_equal_keys_give_uniform_weights():
    N, d = 9, 4
    q = rnd((1, 1, N, d), 61)
    k = np.tile(rnd((1, 1, 1, d), 62), (1, 1, N, 1))
    v = rnd((1, 1, N, d), 63)
    scale = 0.6
    s = scale * (q[0, 0] @ k[0, 0, 0])
    o, lse = A.attention_fwd(q, k, v, scale, False)
    assert np.max(np.abs(o[0, 0] - v[0, 0].mean(axis=0))) < 1e-14
    assert np.max(np.abs(lse[0, 0] - (np.log(N) + s))) < 1e-13
    o, lse = A.attention_fwd(q, k, v, scale, True)
    prefix_mean = np.cumsum(v[0, 0], axis=0) / np.arange(1, N + 1)[:, None]
    assert np.max(np.abs(o[0, 0] - prefix_mean)) < 1e-14
    assert np.max(np.abs(lse[0, 0] - (np.log(np.arange(1, N + 1)) + s))) < 1e-13


def test_zero_scale_is_mean_of_values():
    q, k, v = rnd((1, 1, 6, 3), 64), rnd((1, 1, 6, 3), 65), rnd((1, 1, 6, 3), 66)
    o, lse = A.attention_fwd(q, k, v, 0.0, False)
    assert np.max(np.abs(o[0, 0] - v[0, 0].mean(axis=0))) < 1e-15
    assert np.max(np.abs(lse - np.log(6))) < 1e-15


def test_dominant_key_selects_its_value():
    N, d = 8, 4
    k = np.zeros((1, 1, N, d))
    k[0, 0, 5] = 1.0
    q = np.ones((1, 1, N, d))
    v = rnd((1, 1, N, d), 67)
    o, _ = A.attention_fwd(q, k, v, 100.0, False)  # score gap 400
    assert np.max(np.abs(o[0, 0] - v[0, 0, 5])) < 1e-150 + 1e-15


def test_scalar_two_keys_by_hand():
    # d = 1, N = 2, non-causal: o_i = (e^{s_i0} v_0 + e^{s_i1} v_1) / (e^{s_i0} + e^{s_i1})
    q = [0.3, -1.2]
    k = [0.8, 0.5]
    v = [2.0, -1.0]
    scale = 1.5
    exp_o, exp_lse = [], []
    for qi in q:
        s0, s1 = scale * qi * k[0], scale * qi * k[1]
        e0, e1 = math.exp(s0), math.exp(s1)
        exp_o.append((e0 * v[0] + e1 * v[1]) / (e0 + e1))
        exp_lse.append(math.log(e0 + e1))
    arr = lambda x: np.array(x, dtype=np.float64).reshape(1, 1, 2, 1)
    o, lse = A.attention_fwd(arr(q), arr(k), arr(v), scale, False)
    assert np.max(np.abs(o.ravel() - exp_o)) < 1e-15
    assert np.max(np.abs(lse.ravel() - exp_lse)) < 1e-15
    # causal: row 0 sees only key 0
    o, lse = A.attention_fwd(arr(q), arr(k), arr(v), scale, True)
    assert o.ravel()[0] == v[0]
    assert abs(o.ravel()[1] - exp_o[1]) < 1e-15


def test_rowsum_identity_for_D():
    N, d = 20, 6
    q, k, v, do = (rnd((N, d), s) for s in (71, 72, 73, 74))
    for causal in (False, True):
        _, _, _, dvec = A.attention_bwd_head(q, k, v, do, 0.4, causal, row_chunk=6)
        s = A.scores(q, k, 0.4, causal, np.arange(N))
        p = np.exp(s - s.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        dp = do @ v.T
        assert np.max(np.abs(dvec - np.sum(p * dp, axis=1))) < 1e-13


# ------------------------------------------------------------- IO model ---

def test_io_model_reproduces_printed_numbers():
    g = json.load(open(GOLDEN))
    ridge = IO.ridge_flop_per_byte(g["h100_dense_fp16_tflops"]["value"] * 1e12,
                                   g["h100_hbm_tb_per_s"]["value"] * 1e12)
    assert round(ridge) == g["h100_ridge_flop_per_byte"]["value"]
    assert round(IO.standard_intensity(4096, 128)) == g["standard_intensity_flop_per_byte_d128"]["value"]
    s_bytes = IO.score_matrix_bytes(4096, 2)
    assert round(s_bytes / 1e6, 1) == g["score_matrix_mb_N4096_fp16"]["value"]
    assert round(s_bytes / (4096 * 128 * 2)) == g["score_over_q_ratio"]["value"]
    round_trip = 4 * s_bytes  # S written + read, P written + read
    assert round(round_trip / 1e6) == g["s_and_p_round_trip_mb"]["value"]
    assert round(IO.transfer_seconds(round_trip, 3.35e12) * 1e6) == g["s_and_p_round_trip_us"]["value"]
    assert round(IO.matmul_seconds(4096, 128, 989e12) * 1e6, 1) == g["two_matmuls_us"]["value"]
    assert IO.score_matrix_bytes(8192, 4) / 2**20 == g["score_matrix_mb_N8192_fp32"]["value"]


def test_flop_convention_and_flash_io():
    assert IO.attention_flops(1, 1, 1024, 64) == 4 * 1024 * 1024 * 64
    assert IO.attention_flops(2, 3, 128, 64, causal=True) == 2 * 3 * 2 * 128 * 128 * 64
    assert IO.attention_flops(1, 1, 8, 8, which="bwd") == 2.5 * IO.attention_flops(1, 1, 8, 8)
    # doubling N: standard traffic ~4x for N >> d, tiled traffic ~4x too (K, V once per
    # query block) but far smaller in absolute terms.
    assert IO.flash_fwd_hbm_bytes(4096, 128, 128) < IO.standard_hbm_bytes(4096, 128)
    assert IO.flash_fwd_hbm_bytes(128, 64, 128) == 2 * (128 * 64 * 4)


# ------------------------------------------------------------- inputs ---

def test_bf16_rounding_matches_torch_and_widening_is_exact():
    x = np.random.default_rng(5).standard_normal(4096, dtype=np.float32) * 3
    x[:4] = [1.0 + 2**-8, 1.0 + 3 * 2**-8, -(1.0 + 2**-8), 0.0]  # ties
    bits = I.f32_to_bf16_bits(x)
    t = torch.tensor(x).to(torch.bfloat16)
    assert np.array_equal(bits, t.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(A.bf16_bits_to_f64(bits), t.to(torch.float64).numpy())


def test_inputs_are_seeded_and_scaled_exactly():
    q, k, v, do = I.attention_inputs(1, 2, 5, 8, seed=3)
    q2, _, _, _ = I.attention_inputs(1, 2, 5, 8, seed=3)
    assert np.array_equal(q, q2)
    assert not np.array_equal(q, k)
    qh, _, _, doh = I.attention_inputs(1, 2, 5, 8, seed=3, multiplier=0.5)
    assert np.array_equal(A.bf16_bits_to_f64(qh), 0.5 * A.bf16_bits_to_f64(q))
    assert np.array_equal(doh, do)


# ---------------------------------------------------- planted mistakes ---

def test_pins_catch_a_planted_transpose(monkeypatch):
    # Plant a plausible slip in the oracle (K used untransposed through a wrong axis
    # order of the product) and check the torch comparison above would reject it.
    N, d = 6, 6
    q, k, v = rnd((1, 1, N, d), 81), rnd((1, 1, N, d), 82), rnd((1, 1, N, d), 83)
    good, _ = A.attention_fwd(q, k, v, 0.5, False)

    def bad_scores(q_rows, kk, scale, causal, row_index):
        return scale * (q_rows @ kk)
    monkeypatch.setattr(A, "scores", bad_scores)
    bad, _ = A.attention_fwd(q, k, v, 0.5, False)
    ref = F.scaled_dot_product_attention(*(torch.tensor(x) for x in (q, k, v)), scale=0.5).numpy()
    assert np.max(np.abs(good - ref)) < 1e-12
    assert np.max(np.abs(bad - ref)) > 1e-3


def test_pins_catch_a_planted_missing_rescale(monkeypatch):
    # Plant a streaming softmax that never re-bases earlier blocks when the maximum
    # grows; the whole-row comparison must reject it.
    x = np.linspace(-3, 4, 16)
    original = OS.fold_block

    def no_rescale_fold(m, l, block):
        m_new, l_new, _, b = original(m, l, block)
        return m_new, l_new, 1.0, b
    monkeypatch.setattr(OS, "fold_block", no_rescale_fold)
    bad = OS.online_softmax_row(x, 2)
    monkeypatch.undo()
    assert np.max(np.abs(bad - OS.full_softmax_row(x))) > 1e-3
