"""Philox4x32-10 counter-based generator and the dropout mask built from it (test
infrastructure; the CUDA side implements the same published generator independently).

Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
SC 2011): a 128-bit counter (c0, c1, c2, c3) and a 64-bit key (k0, k1); each of ten rounds
multiplies c0 by 0xD2511F53 and c2 by 0xCD9E8D57 (64-bit products split into high and low
halves), then
    (c0, c1, c2, c3) <- (hi(c2*M1) ^ c1 ^ k0,  lo(c2*M1),  hi(c0*M0) ^ c3 ^ k1,  lo(c0*M0))
and the key is bumped by the Weyl constants (0x9E3779B9, 0xBB67AE85) between rounds.

Dropout mask ("FlashAttention 与显存" §07/§09: dropout is fused into the kernel and its mask is
not stored; the backward pass regenerates it from the generator's state).  The pages fix no
generator or bit layout; this one is chosen so that one generator call serves eight elements:
element (bh, i, j) of the attention matrix (bh = batch*H + head, i = query, j = key) reads
the 16-bit half (j % 2: 0 = low half) of word (j % 8) // 2 of
Philox(counter = (j // 8, i, bh, 0), key = (seed & 0xffffffff, seed >> 32)).  The element is
kept when that half is >= t = min(round(p * 2^16), 2^16 - 1), i.e. with probability
(2^16 - t) / 2^16, and kept elements are scaled by the inverse of that probability, so the
mask's expectation is exactly 1 (p is quantised to multiples of 2^-16).

Pinned against an independent implementation of the same generator: cuRAND's host-side
PHILOX4_32_10 generator, whose output stream is Philox4x32-10 of a known counter sequence
(tests/test_oracle_dropout.py compares them bit for bit, over the key, the three counter words
the mask fills and counters up to 2^62).  What the method needs from the mask -- keep rate,
uniform draws, dependence on every coordinate, unbiasedness -- is pinned by the same tests.
"""

from __future__ import annotations

import numpy as np

M0 = np.uint64(0xD2511F53)
M1 = np.uint64(0xCD9E8D57)
W0 = np.uint32(0x9E3779B9)
W1 = np.uint32(0xBB67AE85)
MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Vectorised over numpy arrays (uint32-valued); returns four uint32 arrays."""
    c0, c1, c2, c3 = (np.asarray(x, np.uint64) & MASK32 for x in (c0, c1, c2, c3))
    k0 = np.asarray(k0, np.uint64) & MASK32
    k1 = np.asarray(k1, np.uint64) & MASK32
    for r in range(10):
        p0 = c0 * M0
        p1 = c2 * M1
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        if r < 9:
            k0 = (k0 + np.uint64(W0)) & MASK32
            k1 = (k1 + np.uint64(W1)) & MASK32
    return tuple(x.astype(np.uint32) for x in (c0, c1, c2, c3))


def keep_threshold(p: float) -> int:
    """16-bit threshold t: an element is kept when its 16-bit draw is >= t."""
    if not 0.0 <= p < 1.0:
        raise ValueError("dropout probability must be in [0, 1)")
    return min(int(round(p * 65536.0)), 65535)


def keep_scale(p: float) -> float:
    """Inverse of the keep probability (2^16 - t) / 2^16."""
    return 65536.0 / (65536 - keep_threshold(p))


def dropout_keep(bh: int, rows, cols, p: float, seed: int) -> np.ndarray:
    """Boolean keep mask [len(rows), len(cols)] for head index bh."""
    rows = np.asarray(rows, np.uint64)[:, None]
    cols = np.asarray(cols, np.uint64)[None, :]
    t = keep_threshold(p)
    c0 = np.broadcast_to(cols >> np.uint64(3), (rows.shape[0], cols.shape[1]))
    c1 = np.broadcast_to(rows, c0.shape)
    words = philox4x32_10(c0, c1, np.full(c0.shape, bh, np.uint64), np.zeros(c0.shape, np.uint64),
                          seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    sel = np.broadcast_to((cols & np.uint64(7)) >> np.uint64(1), c0.shape)
    w = np.choose(sel.astype(np.int64), words)
    half = np.broadcast_to(cols & np.uint64(1), c0.shape).astype(np.uint32)
    draw = (w >> (np.uint32(16) * half)) & np.uint32(0xFFFF)
    return draw >= np.uint32(t) if p > 0 else np.ones(c0.shape, bool)
