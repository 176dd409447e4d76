"""Philox4x32-10 counter-based generator and the dropout mask built from it (test
infrastructure; the CUDA side implements the same published generator independently).

Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
SC 2011): a 128-bit counter (c0, c1, c2, c3) and a 64-bit key (k0, k1); each of ten rounds
multiplies c0 by 0xD2511F53 and c2 by 0xCD9E8D57 (64-bit products split into high and low
halves), then
    (c0, c1, c2, c3) <- (hi(c2*M1) ^ c1 ^ k0,  lo(c2*M1),  hi(c0*M0) ^ c3 ^ k1,  lo(c0*M0))
and the key is bumped by the Weyl constants (0x9E3779B9, 0xBB67AE85) between rounds.

Dropout mask ("FlashAttention 与显存" §07/§09: dropout is fused into the kernel and its mask is
not stored; the backward pass regenerates it from the generator's state): element (bh, i, j)
of the attention matrix (bh = batch*H + head, i = query, j = key) reads word j % 4 of
Philox(counter = (j // 4, i, bh, 0), key = (seed & 0xffffffff, seed >> 32)); the element is
kept when that word is >= threshold(p) = min(round(p * 2^32), 2^32 - 1), and kept elements are
scaled by 1 / (1 - p).
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
    return min(int(round(p * 2.0 ** 32)), 2 ** 32 - 1)


def dropout_keep(bh: int, rows, cols, p: float, seed: int) -> np.ndarray:
    """Boolean keep mask [len(rows), len(cols)] for head index bh."""
    rows = np.asarray(rows, np.uint64)[:, None]
    cols = np.asarray(cols, np.uint64)[None, :]
    c0 = np.broadcast_to(cols >> np.uint64(2), (rows.shape[0], cols.shape[1]))
    c1 = np.broadcast_to(rows, c0.shape)
    words = philox4x32_10(c0, c1, np.full(c0.shape, bh, np.uint64), np.zeros(c0.shape, np.uint64),
                          seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    sel = np.broadcast_to(cols & np.uint64(3), c0.shape)
    w = np.choose(sel.astype(np.int64), words)
    return w >= np.uint32(keep_threshold(p)) if p > 0 else np.ones(c0.shape, bool)
