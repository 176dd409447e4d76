"""Plain fp64 definition of exact attention, forward and backward (test infrastructure).

Forward, per (batch, head), from "Flash Attention 原理与实践" §1.3 and
"FlashAttention 与显存" §04:

    S = scale * Q K^T                       [N, N]
    causal: S_ij = -inf for j > i           (top-left aligned square mask, the
                                             ``is_causal=True`` of the SDPA call shown in
                                             "Flash Attention 原理与实践" §4.2)
    m_i = max_j S_ij,  l_i = sum_j exp(S_ij - m_i)
    P = exp(S - m) / l
    O = P V
    LSE_i = m_i + ln l_i                    (natural log, in units of scaled scores; the
                                             one-number form of the (m, l) pair that
                                             "FlashAttention 与显存" §09 keeps per row)

Backward (analytic; "FlashAttention 与显存" §09 says only that S and P are recomputed
from Q, K, V block by block).  With dO the upstream gradient of O:

    dV = P^T dO
    dP = dO V^T
    D_i = sum_c dO_ic O_ic                  (equals sum_j P_ij dP_ij)
    dS = P * (dP - D 1^T)
    dQ = scale * dS K
    dK = scale * dS^T Q

S and P are materialised for a chunk of query rows at a time, over the full key
length, which is still the plain definition (no online rescaling), and keeps the
memory bounded for N = 65536.

Dropout (optional, p > 0; "FlashAttention 与显存" §07, §09): after the softmax each
probability is kept with probability 1 - p and scaled by the inverse of that probability,
Z = keep * philox.keep_scale(p) (p quantised to multiples of 2^-16), the mask drawn from the
counter-based generator in ``philox`` (so it can be regenerated instead of stored).  O = (P * Z) V; LSE is that of the undropped P.  Backward: dV = (P * Z)^T dO,
dP = dO V^T, dS = P * (dP * Z - D) with D = rowsum(dO * O) (still = rowsum(P * Z * dP)).
"""

from __future__ import annotations

import numpy as np

from . import philox

__all__ = [
    "bf16_bits_to_f64",
    "scores",
    "attention_fwd",
    "attention_fwd_rows",
    "attention_bwd",
    "attention_bwd_head",
    "attention_bwd_rows",
    "attention_bwd_key_columns",
    "lse_merge",
]


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns (uint16) to float64 exactly.

    A bfloat16 value is the upper half of the float32 with the same bits, so the
    widening is a 16-bit shift into a float32 followed by an exact float64 cast.
    """
    bits = np.asarray(bits)
    if bits.dtype != np.uint16:
        raise TypeError("expected uint16 bfloat16 bit patterns")
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def scores(q_rows: np.ndarray, k: np.ndarray, scale: float, causal: bool,
           row_index: np.ndarray) -> np.ndarray:
    """S rows for the queries whose positions are ``row_index``: scale * q k^T, masked.

    q_rows: [R, d] fp64, k: [N, d] fp64, row_index: [R] int positions of the rows.
    Masked entries are -inf.
    """
    s = scale * (q_rows @ k.T)
    if causal:
        n = k.shape[0]
        key = np.arange(n)[None, :]
        s = np.where(key > np.asarray(row_index)[:, None], -np.inf, s)
    return s


def _softmax_rows(s: np.ndarray):
    m = s.max(axis=1)
    e = np.exp(s - m[:, None])
    l = e.sum(axis=1)
    return e / l[:, None], m, l


def _dropout_z(bh, rows, n_keys, p, seed):
    keep = philox.dropout_keep(bh, rows, np.arange(n_keys), p, seed)
    return keep * philox.keep_scale(p)


def attention_fwd(q, k, v, scale: float, causal: bool, row_chunk: int = 512,
                  dropout_p: float = 0.0, seed: int = 0):
    """O [B,H,N,d] and LSE [B,H,N] in fp64 for fp64 inputs [B,H,N,d]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, N, d = q.shape
    o = np.empty((B, H, N, v.shape[-1]))
    lse = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            for r0 in range(0, N, row_chunk):
                r1 = min(N, r0 + row_chunk)
                rows = np.arange(r0, r1)
                s = scores(q[b, h, r0:r1], k[b, h], scale, causal, rows)
                p, m, l = _softmax_rows(s)
                if dropout_p > 0:
                    p = p * _dropout_z(b * H + h, rows, k.shape[2], dropout_p, seed)
                o[b, h, r0:r1] = p @ v[b, h]
                lse[b, h, r0:r1] = m + np.log(l)
    return o, lse


def attention_fwd_rows(q_head, k_head, v_head, scale: float, causal: bool, rows,
                       dropout_p: float = 0.0, seed: int = 0, bh: int = 0):
    """O and LSE for selected query rows of one head.

    q_head, k_head, v_head: [N, d] fp64 for one (batch, head); rows: positions.
    Each row of attention depends only on its own query and all keys, so a sample of
    rows is checked against the same definition as the whole tensor.  With dropout the
    mask is that of head index ``bh``.
    """
    rows = np.asarray(rows, dtype=np.int64)
    k = np.asarray(k_head, np.float64)
    s = scores(np.asarray(q_head, np.float64)[rows], k, scale, causal, rows)
    p, m, l = _softmax_rows(s)
    if dropout_p > 0:
        p = p * _dropout_z(bh, rows, k.shape[0], dropout_p, seed)
    return p @ np.asarray(v_head, np.float64), m + np.log(l)


def attention_bwd_head(q, k, v, do, scale: float, causal: bool, row_chunk: int = 512,
                       dropout_p: float = 0.0, seed: int = 0, bh: int = 0):
    """dQ, dK, dV [N, d] and D [N] for one head, all fp64 [N, d] inputs.

    D is rowsum(dO * O) with O from this same definition.  With dropout the mask is that of
    head index ``bh`` (= batch * H + head).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    N = q.shape[0]
    dq = np.empty_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dvec = np.empty(N)
    for r0 in range(0, N, row_chunk):
        r1 = min(N, r0 + row_chunk)
        rows = np.arange(r0, r1)
        s = scores(q[r0:r1], k, scale, causal, rows)
        p, _, _ = _softmax_rows(s)
        z = _dropout_z(bh, rows, k.shape[0], dropout_p, seed) if dropout_p > 0 else 1.0
        o = (p * z) @ v
        dv += (p * z).T @ do[r0:r1]
        dp = do[r0:r1] @ v.T
        drow = np.sum(do[r0:r1] * o, axis=1)
        ds = p * (dp * z - drow[:, None])
        dq[r0:r1] = scale * (ds @ k)
        dk += scale * (ds.T @ q[r0:r1])
        dvec[r0:r1] = drow
    return dq, dk, dv, dvec


def attention_bwd(q, k, v, do, scale: float, causal: bool, row_chunk: int = 512,
                  dropout_p: float = 0.0, seed: int = 0):
    """dQ, dK, dV [B,H,N,d] and D [B,H,N] for fp64 inputs [B,H,N,d]."""
    q = np.asarray(q, np.float64)
    B, H, N, d = q.shape
    dq = np.empty_like(q)
    dk = np.empty_like(q)
    dv = np.empty((B, H, N, np.asarray(v).shape[-1]))
    dvec = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h], dvec[b, h] = attention_bwd_head(
                q[b, h], k[b, h], v[b, h], do[b, h], scale, causal, row_chunk,
                dropout_p, seed, b * H + h)
    return dq, dk, dv, dvec


def attention_bwd_rows(q_head, k_head, v_head, do_head, scale: float, causal: bool, rows,
                       dropout_p: float = 0.0, seed: int = 0, bh: int = 0):
    """dQ rows and D for selected query rows of one head.

    dQ_i = scale * sum_j P_ij (dP_ij - D_i) K_j needs only row i of P, so a sample of
    rows is computed exactly from the definition without the full N x N matrices.
    """
    rows = np.asarray(rows, dtype=np.int64)
    q = np.asarray(q_head, np.float64)
    k = np.asarray(k_head, np.float64)
    v = np.asarray(v_head, np.float64)
    do = np.asarray(do_head, np.float64)[rows]
    s = scores(q[rows], k, scale, causal, rows)
    p, _, _ = _softmax_rows(s)
    z = _dropout_z(bh, rows, k.shape[0], dropout_p, seed) if dropout_p > 0 else 1.0
    o = (p * z) @ v
    dp = do @ v.T
    drow = np.sum(do * o, axis=1)
    ds = p * (dp * z - drow[:, None])
    return scale * (ds @ k), drow


def attention_bwd_key_columns(q_head, k_head, v_head, do_head, scale: float, causal: bool,
                              keys, row_chunk: int = 512, dropout_p: float = 0.0, seed: int = 0,
                              bh: int = 0):
    """dK and dV rows of selected keys of one head, exactly from the definition.

    dV_j = sum_i P_ij dO_i and dK_j = scale * sum_i dS_ij Q_i need column j of P and dS over
    every query row i, so every row's softmax (and O_i for D_i) is formed in chunks of
    rows; only the selected key columns are kept.
    """
    keys = np.asarray(keys, dtype=np.int64)
    q = np.asarray(q_head, np.float64)
    k = np.asarray(k_head, np.float64)
    v = np.asarray(v_head, np.float64)
    do = np.asarray(do_head, np.float64)
    N = q.shape[0]
    dk = np.zeros((keys.size, k.shape[1]))
    dv = np.zeros((keys.size, v.shape[1]))
    v_sel = v[keys]
    for r0 in range(0, N, row_chunk):
        r1 = min(N, r0 + row_chunk)
        rows = np.arange(r0, r1)
        s = scores(q[r0:r1], k, scale, causal, rows)
        p, _, _ = _softmax_rows(s)
        z = _dropout_z(bh, rows, N, dropout_p, seed) if dropout_p > 0 else np.ones_like(p)
        o = (p * z) @ v
        drow = np.sum(do[r0:r1] * o, axis=1)
        p_sel, z_sel = p[:, keys], z[:, keys]
        ds_sel = p_sel * ((do[r0:r1] @ v_sel.T) * z_sel - drow[:, None])
        dv += (p_sel * z_sel).T @ do[r0:r1]
        dk += scale * (ds_sel.T @ q[r0:r1])
    return dk, dv


def lse_merge(o_parts, lse_parts):
    """Merge attention computed over disjoint key ranges ("Flash Attention 原理与实践" §5.1:
    split the keys across workers, then combine with log-sum-exp).

    o_parts: [S, ..., d] outputs, each normalised within its own key range; lse_parts:
    [S, ...] the ranges' log-sum-exps.  Returns (O, LSE) of the whole key set:
    LSE = log sum_s exp(LSE_s),  O = sum_s exp(LSE_s - LSE) O_s.
    """
    o_parts = np.asarray(o_parts, np.float64)
    lse_parts = np.asarray(lse_parts, np.float64)
    m = lse_parts.max(axis=0)
    lse = m + np.log(np.exp(lse_parts - m).sum(axis=0))
    w = np.exp(lse_parts - lse)
    return (w[..., None] * o_parts).sum(axis=0), lse
