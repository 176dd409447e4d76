"""Pins of the oracle's dropout (mask generator and dropout arithmetic).

The generator is checked against an independent implementation of the same published
generator, cuRAND's host-side PHILOX4_32_10 generator (run on the CPU, no GPU needed), and by
its statistics and its dependence on every counter field; the arithmetic by reduction to the
plain path at p = 0, by unbiasedness over seeds, by central finite differences at a fixed mask,
and by torch (softmax and autograd) applied to P * Z."""

import ctypes
import ctypes.util
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attention as A
from oracle import philox


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ----------------------------------------------------------------------------------------
# Philox4x32-10 against cuRAND's host generator.
#
# cuRAND's host generator of type CURAND_RNG_PSEUDO_PHILOX4_32_10 (created with
# curandCreateGeneratorHost, so it runs on the host) is another implementation of the
# generator of Salmon et al. (SC 2011).  With seed s its key is (s mod 2^32, s >> 32).  Its
# output stream, observed over 2^24 values and at offsets up to 2^64, is made of blocks of four
# 32-bit words: with generator offset 4m, block b = m + n (the n-th group of four outputs) is
# Philox4x32-10 of the counter (floor(b / 2^16) mod 2^32, floor(b / 2^48), b mod 2^16, 0).  So
# the comparison covers the key, both multipliers, the Weyl bumps, the round count, the output
# word order and the counter words c0, c1 and c2 -- the three the dropout mask fills (key
# tile, query row, head); c3 is always 0 there.

_CURAND_PHILOX = 161  # curandRngType_t CURAND_RNG_PSEUDO_PHILOX4_32_10


def _curand():
    names = [os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64", "libcurand.so"),
             ctypes.util.find_library("curand"), "libcurand.so.10"]
    for name in names:
        if not name:
            continue
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    pytest.skip("cuRAND (libcurand.so) not found")


def _curand_philox_blocks(lib, seed: int, offset_blocks: int, n_blocks: int) -> np.ndarray:
    gen = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), _CURAND_PHILOX) == 0
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(4 * offset_blocks)) == 0
        out = np.zeros(4 * n_blocks, np.uint32)
        assert lib.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(out.size)) == 0
    finally:
        lib.curandDestroyGenerator(gen)
    return out.reshape(-1, 4)


def _oracle_blocks(philox4x32_10, seed: int, offset_blocks: int, n_blocks: int) -> np.ndarray:
    b = [offset_blocks + n for n in range(n_blocks)]  # python ints: offsets reach 2^62
    c0 = np.array([(x >> 16) & 0xFFFFFFFF for x in b], np.uint64)
    c1 = np.array([x >> 48 for x in b], np.uint64)
    c2 = np.array([x & 0xFFFF for x in b], np.uint64)
    words = philox4x32_10(c0, c1, c2, np.zeros_like(c0), seed & 0xFFFFFFFF, seed >> 32)
    return np.stack(words, 1)


PHILOX_CASES = [  # (seed, first block, blocks): the first spans the c2 -> c0 carry at 2^16
    (0x0123456789ABCDEF, 0, 1 << 17),
    (0, 12345, 4096),
    (0xFFFFFFFFFFFFFFFF, (1 << 32) + 77, 4096),
    (0xDEADBEEF12345678, (1 << 48) + (1 << 20) + 5, 4096),
    (7, (1 << 62) - 12345, 4096),
]


@pytest.mark.parametrize("seed,first,n", PHILOX_CASES)
def test_philox_matches_curand_host_generator(seed, first, n):
    lib = _curand()
    want = _curand_philox_blocks(lib, seed, first, n)
    got = _oracle_blocks(philox.philox4x32_10, seed, first, n)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("mistake", [dict(M0=philox.M1, M1=philox.M0), dict(M0=philox.M0 + np.uint64(2)),
                                     dict(W0=philox.W1, W1=philox.W0), dict(W1=np.uint32(0))])
def test_philox_comparison_catches_planted_mistakes(mistake, monkeypatch):
    """A mistake planted in the oracle's constants (swapped or altered multipliers, swapped or
    missing key bumps) makes the comparison with cuRAND fail."""
    lib = _curand()
    seed, first, n = PHILOX_CASES[3]
    want = _curand_philox_blocks(lib, seed, first, n)
    for name, value in mistake.items():
        monkeypatch.setattr(philox, name, value)
    assert not np.array_equal(_oracle_blocks(philox.philox4x32_10, seed, first, n), want)


@pytest.mark.parametrize("p", [0.1, 0.5, 0.9])
def test_keep_rate(p):
    keep = philox.dropout_keep(3, np.arange(256), np.arange(4096), p, seed=12345)
    n = keep.size
    sigma = math.sqrt(n * p * (1 - p))
    assert abs(keep.sum() - n * (1 - p)) < 5 * sigma


def test_mask_depends_on_every_coordinate():
    base = philox.dropout_keep(0, np.arange(64), np.arange(64), 0.5, seed=7)
    assert not np.array_equal(base, philox.dropout_keep(1, np.arange(64), np.arange(64), 0.5, seed=7))
    assert not np.array_equal(base, philox.dropout_keep(0, np.arange(64), np.arange(64), 0.5, seed=8))
    assert not np.array_equal(base, philox.dropout_keep(0, np.arange(64), np.arange(64), 0.5, seed=7 << 32))
    # neighbouring rows and the eight keys that share one generator call are not copies
    assert np.mean(base[1:] == base[:-1]) < 0.6
    assert np.mean(base[:, 1:] == base[:, :-1]) < 0.6
    assert np.all(philox.dropout_keep(0, np.arange(4), np.arange(4), 0.0, seed=1))


def test_zero_dropout_is_the_plain_path():
    q, k, v, do = (rnd((1, 2, 9, 4), s) for s in (1, 2, 3, 4))
    for causal in (False, True):
        a = A.attention_fwd(q, k, v, 0.5, causal)
        b = A.attention_fwd(q, k, v, 0.5, causal, dropout_p=0.0, seed=99)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
        ga = A.attention_bwd(q, k, v, do, 0.5, causal)
        gb = A.attention_bwd(q, k, v, do, 0.5, causal, dropout_p=0.0, seed=99)
        assert all(np.array_equal(x, y) for x, y in zip(ga, gb))


def test_dropout_is_unbiased_over_seeds():
    q, k, v = (rnd((1, 1, 6, 3), s) for s in (5, 6, 7))
    o, _ = A.attention_fwd(q, k, v, 0.8, False)
    acc = np.zeros_like(o)
    n = 3000
    for seed in range(n):
        acc += A.attention_fwd(q, k, v, 0.8, False, dropout_p=0.3, seed=seed)[0]
    assert np.max(np.abs(acc / n - o)) < 0.05


@pytest.mark.parametrize("causal", [False, True])
def test_dropout_gradients_match_finite_differences(causal):
    N, d, p, seed = 6, 3, 0.4, 2024
    q, k, v, do = (rnd((N, d), s) for s in (8, 9, 10, 11))
    h = 1e-6

    def loss(q_, k_, v_):
        o, _ = A.attention_fwd(q_[None, None], k_[None, None], v_[None, None], 0.7, causal,
                               dropout_p=p, seed=seed)
        return float(np.sum(o[0, 0] * do))

    grads = A.attention_bwd_head(q, k, v, do, 0.7, causal, dropout_p=p, seed=seed, bh=0)
    for which, g in enumerate(grads[:3]):
        num = np.zeros_like(g)
        for idx in np.ndindex(*g.shape):
            a = [q.copy(), k.copy(), v.copy()]
            b = [q.copy(), k.copy(), v.copy()]
            a[which][idx] += h
            b[which][idx] -= h
            num[idx] = (loss(*a) - loss(*b)) / (2 * h)
        assert np.linalg.norm(num - g) / np.linalg.norm(g) < 1e-7, which


@pytest.mark.parametrize("causal", [False, True])
def test_dropout_matches_torch_on_the_same_mask(causal):
    B, H, N, d, p, seed = 2, 2, 11, 4, 0.25, 5
    q, k, v, do = (rnd((B, H, N, d), s) for s in (12, 13, 14, 15))
    o, lse = A.attention_fwd(q, k, v, 0.6, causal, dropout_p=p, seed=seed)
    dq, dk, dv, _ = A.attention_bwd(q, k, v, do, 0.6, causal, dropout_p=p, seed=seed)
    z = np.stack([np.stack([philox.dropout_keep(b * H + h, np.arange(N), np.arange(N), p, seed)
                            for h in range(H)]) for b in range(B)]) * philox.keep_scale(p)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    s = 0.6 * tq @ tk.transpose(-1, -2)
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    to = (torch.softmax(s, dim=-1) * torch.tensor(z)) @ tv
    to.backward(torch.tensor(do))
    assert np.max(np.abs(o - to.detach().numpy())) < 1e-12
    assert np.max(np.abs(lse - torch.logsumexp(s, -1).detach().numpy())) < 1e-12
    for g, t in ((dq, tq), (dk, tk), (dv, tv)):
        assert np.max(np.abs(g - t.grad.numpy())) < 1e-11


def test_keep_probability_times_scale_is_one():
    # E[Z] = 1 exactly: t of the 2^16 draws are dropped, the rest scaled by 2^16 / (2^16 - t)
    for p in (0.0, 1e-6, 0.1, 0.25, 0.5, 0.9, 0.99999):
        t = philox.keep_threshold(p)
        assert abs(t - p * 65536) <= 0.5
        assert (65536 - t) / 65536 * philox.keep_scale(p) == 1.0
    with pytest.raises(ValueError):
        philox.keep_threshold(1.0)


def test_every_sixteen_bit_draw_pattern_is_used():
    # over many calls the 16-bit draws of all eight slots are uniform: the slot-wise keep rates
    # at p = 0.5 agree, so no slot reads a constant or a shared half
    keep = philox.dropout_keep(5, np.arange(512), np.arange(512), 0.5, seed=99)
    rates = keep.reshape(512, 64, 8).mean(axis=(0, 1))
    sigma = math.sqrt(0.25 / (512 * 64))
    assert np.all(np.abs(rates - 0.5) < 5 * sigma)
    # the two halves of one word are not the same draw
    assert np.mean(keep[:, 0::2] == keep[:, 1::2]) < 0.55


@pytest.mark.parametrize("causal", [False, True])
def test_row_and_column_variants_with_dropout_match_the_whole_head(causal):
    # the sampled-row / sampled-key variants used at full size are the same definition
    N, d, p, seed, bh = 37, 8, 0.3, 77, 5
    q, k, v, do = (rnd((N, d), s) for s in (21, 22, 23, 24))
    dq, dk, dv, dvec = A.attention_bwd_head(q, k, v, do, 0.4, causal, dropout_p=p, seed=seed, bh=bh)
    rows = np.array([0, 3, 17, 36])
    # forward rows against the batched definition (this head placed at index bh)
    qb, kb, vb = (np.zeros((1, bh + 1, N, d)) for _ in range(3))
    qb[0, bh], kb[0, bh], vb[0, bh] = q, k, v
    o_all, lse_all = A.attention_fwd(qb, kb, vb, 0.4, causal, dropout_p=p, seed=seed)
    o_r, lse_r = A.attention_fwd_rows(q, k, v, 0.4, causal, rows, dropout_p=p, seed=seed, bh=bh)
    assert np.max(np.abs(o_r - o_all[0, bh, rows])) < 1e-12
    assert np.max(np.abs(lse_r - lse_all[0, bh, rows])) < 1e-12
    dq_r, d_r = A.attention_bwd_rows(q, k, v, do, 0.4, causal, rows, dropout_p=p, seed=seed, bh=bh)
    assert np.max(np.abs(dq_r - dq[rows])) < 1e-12 and np.max(np.abs(d_r - dvec[rows])) < 1e-12
    keys = np.array([0, 9, 30, 36])
    dk_c, dv_c = A.attention_bwd_key_columns(q, k, v, do, 0.4, causal, keys, row_chunk=10,
                                             dropout_p=p, seed=seed, bh=bh)
    assert np.max(np.abs(dk_c - dk[keys])) < 1e-12 and np.max(np.abs(dv_c - dv[keys])) < 1e-12
