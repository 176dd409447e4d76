"""Streaming softmax and the tiled forward pass, in fp64 (test infrastructure).

The recurrence ("FlashAttention 与显存" §08; "Flash Attention 原理与实践" §2.2):
keep, for each row, the largest score seen so far m and the sum l of exp(score - m)
over the scores seen so far.  A new block of scores with its own maximum m~ and its own
sum l~ (taken relative to m~) is folded in by

    m_new = max(m, m~)
    l_new = exp(m - m_new) * l + exp(m~ - m_new) * l~

and everything already accumulated relative to the old maximum (the output
accumulator of attention) is multiplied by exp(m - m_new).  When the last block is in,
the result is the full-row softmax up to rounding.

Two loop orders of the tiled forward are written out:

* ``tiled_forward_q_outer``: the order of "FlashAttention算子优化" §2 and of the second
  version in "FlashAttention 与显存" §07/§11 -- one block of query rows at a time, all
  key/value blocks streamed past it, divide by l once at the end.
* ``tiled_forward_kv_outer``: the order of "Flash Attention 原理与实践" §2.1/§2.3 --
  key/value blocks outside, query blocks inside, with O, l and m read back and written
  out for every pair of blocks, and O kept normalised after every step.

"FlashAttention算子优化" §1 prints a streaming-softmax listing that scales the earlier
partial sum twice and never rescales earlier probabilities; the functions here follow
the recurrence above instead (the reading that the other two pages support).
"""

from __future__ import annotations

import math

import numpy as np

__all__ = ["fold_block", "online_row_stats", "online_softmax_row", "full_softmax_row",
           "tiled_forward_q_outer", "tiled_forward_kv_outer"]


def fold_block(m: float, l: float, block: np.ndarray):
    """Fold one block of scores into the running (m, l) pair; returns (m_new, l_new, a, b)
    with a = exp(m - m_new) applied to the old state and b = exp(m~ - m_new) to the block.
    """
    block = np.asarray(block, np.float64)
    m_blk = float(block.max())
    l_blk = float(np.exp(block - m_blk).sum()) if m_blk != -math.inf else 0.0
    m_new = max(m, m_blk)
    if m_new == -math.inf:  # nothing visible yet
        return m_new, 0.0, 1.0, 0.0
    a = math.exp(m - m_new) if m != -math.inf else 0.0
    b = math.exp(m_blk - m_new) if m_blk != -math.inf else 0.0
    return m_new, a * l + b * l_blk, a, b


def online_row_stats(x: np.ndarray, block: int):
    """(m, l) of one row of scores, consumed ``block`` entries at a time."""
    x = np.asarray(x, np.float64)
    m, l = -math.inf, 0.0
    for c0 in range(0, x.size, block):
        m, l, _, _ = fold_block(m, l, x[c0:c0 + block])
    return m, l


def online_softmax_row(x: np.ndarray, block: int) -> np.ndarray:
    """Softmax of one row where the normaliser comes from the streaming recurrence.

    The exponentials of each block are taken against the running maximum at the time
    the block arrives and re-based every time the maximum grows, then divided once by
    the final sum.
    """
    x = np.asarray(x, np.float64)
    m, l = -math.inf, 0.0
    parts = []
    for c0 in range(0, x.size, block):
        blk = x[c0:c0 + block]
        m, l, a, _ = fold_block(m, l, blk)
        parts = [pp * a for pp in parts]
        parts.append(np.exp(blk - m))
    return np.concatenate(parts) / l


def full_softmax_row(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, np.float64)
    e = np.exp(x - x.max())
    return e / e.sum()


def _mask_block(s, r0, c0, causal, n_keys):
    rows = np.arange(r0, r0 + s.shape[0])[:, None]
    cols = np.arange(c0, c0 + s.shape[1])[None, :]
    hidden = cols >= n_keys
    if causal:
        hidden = hidden | (cols > rows)
    return np.where(hidden, -np.inf, s)


def tiled_forward_q_outer(q, k, v, scale: float, causal: bool, br: int, bc: int):
    """One head, [N, d] fp64 in; O [N, d] and LSE [N] out.

    Per block of ``br`` query rows: running max m, running sum l and an unnormalised
    accumulator acc start at (-inf, 0, 0); every block of ``bc`` keys contributes
    exp(S - m_new) and rescales what came before by exp(m - m_new); O = acc / l at the
    end.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    n, d = q.shape
    o = np.empty((n, v.shape[1]))
    lse = np.empty(n)
    for r0 in range(0, n, br):
        qi = q[r0:r0 + br]
        rb = qi.shape[0]
        m = np.full(rb, -np.inf)
        l = np.zeros(rb)
        acc = np.zeros((rb, v.shape[1]))
        for c0 in range(0, n, bc):
            s = _mask_block(scale * (qi @ k[c0:c0 + bc].T), r0, c0, causal, n)
            m_blk = s.max(axis=1)
            m_new = np.maximum(m, m_blk)
            live = m_new > -np.inf
            a = np.where(live & (m > -np.inf), np.exp(np.where(live, m - m_new, 0.0)), 0.0)
            p = np.where(live[:, None], np.exp(s - np.where(live, m_new, 0.0)[:, None]), 0.0)
            l = a * l + p.sum(axis=1)
            acc = a[:, None] * acc + p @ v[c0:c0 + bc]
            m = m_new
        o[r0:r0 + br] = acc / l[:, None]
        lse[r0:r0 + br] = m + np.log(l)
    return o, lse


def tiled_forward_kv_outer(q, k, v, scale: float, causal: bool, br: int, bc: int):
    """One head, the loop order with key/value blocks outside.

    O, m and l live in "HBM" arrays that each (key block, query block) step reads and
    writes back; O stays normalised after every step:
        O_new = (l * exp(m - m_new) * O + exp(m~ - m_new) * (P~ V)) / l_new
    where P~ = exp(S - m~) uses the block's own maximum m~.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    n, d = q.shape
    o_hbm = np.zeros((n, v.shape[1]))
    l_hbm = np.zeros(n)
    m_hbm = np.full(n, -np.inf)
    for c0 in range(0, n, bc):
        kj, vj = k[c0:c0 + bc], v[c0:c0 + bc]
        for r0 in range(0, n, br):
            oi, li, mi = o_hbm[r0:r0 + br], l_hbm[r0:r0 + br], m_hbm[r0:r0 + br]
            s = _mask_block(scale * (q[r0:r0 + br] @ kj.T), r0, c0, causal, n)
            m_blk = s.max(axis=1)
            vis = m_blk > -np.inf
            p = np.where(vis[:, None], np.exp(s - np.where(vis, m_blk, 0.0)[:, None]), 0.0)
            l_blk = p.sum(axis=1)
            m_new = np.maximum(mi, m_blk)
            live = m_new > -np.inf
            a = np.where(live & (mi > -np.inf), np.exp(np.where(live, mi - m_new, 0.0)), 0.0)
            b = np.where(vis, np.exp(np.where(vis, m_blk - m_new, 0.0)), 0.0)
            l_new = a * li + b * l_blk
            safe = np.where(l_new > 0, l_new, 1.0)
            o_hbm[r0:r0 + br] = ((li * a)[:, None] * oi + b[:, None] * (p @ vj)) / safe[:, None]
            l_hbm[r0:r0 + br] = l_new
            m_hbm[r0:r0 + br] = m_new
    return o_hbm, m_hbm + np.log(l_hbm)
