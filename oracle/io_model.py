"""FLOP and HBM-byte counters for attention (test infrastructure).

These restate the arithmetic behind the pages' worked numbers so that tests can check
them against the printed values:

* "FlashAttention 与显存" §03: the ridge point of a GPU is peak FLOP/s over HBM bytes/s,
  and standard attention (16-bit, one head, d = 128) does about 62 FLOP per byte.
* "FlashAttention 与显存" §04: at N = 4096, d = 128 one head's S is 33.6 MB (32x Q),
  writing and reading S and P is 134 MB (about 40 us at 3.35 TB/s) and the two matmuls
  take about 8.7 us at 989 TFLOP/s.
* "FlashAttention 与显存" §14: standard attention reads/writes Q, K, V, O once and
  writes and reads S and P once each; the tiled forward (second-version order) reads
  each Q block once, streams all of K and V once per Q block, writes O once, with no
  credit for L2.
* "Flash Attention 原理与实践" §1.3: an 8K x 8K fp32 score matrix is 256 MB.

FLOP convention: forward = 2 matmuls of 2*N*N*d each = 4*B*H*N^2*d, halved under a
causal mask; backward = 2.5x forward (five matmuls instead of two).
"""

from __future__ import annotations

import math

__all__ = ["attention_flops", "score_matrix_bytes", "standard_hbm_elements",
           "standard_hbm_bytes", "standard_intensity", "ridge_flop_per_byte",
           "flash_fwd_hbm_bytes", "transfer_seconds", "matmul_seconds"]


def attention_flops(B: int, H: int, N: int, d: int, causal: bool = False,
                    which: str = "fwd") -> float:
    """Convention FLOPs of one call: 'fwd', 'bwd' or 'fwd+bwd'."""
    fwd = 4.0 * B * H * N * N * d
    if causal:
        fwd *= 0.5
    if which == "fwd":
        return fwd
    if which == "bwd":
        return 2.5 * fwd
    if which == "fwd+bwd":
        return 3.5 * fwd
    raise ValueError(which)


def score_matrix_bytes(N: int, elem_bytes: int) -> int:
    """Bytes of one head's N x N score (or probability) matrix."""
    return N * N * elem_bytes


def standard_hbm_elements(N: int, d: int) -> int:
    """Elements moved by standard attention for one head: Q, K, V read and O written
    (4*N*d), S written then read and P written then read (4*N*N)."""
    return 4 * N * d + 4 * N * N


def standard_hbm_bytes(N: int, d: int, elem_bytes: int = 2) -> int:
    return standard_hbm_elements(N, d) * elem_bytes


def standard_intensity(N: int, d: int, elem_bytes: int = 2) -> float:
    """FLOP per HBM byte of standard attention, one head, forward."""
    return attention_flops(1, 1, N, d) / standard_hbm_bytes(N, d, elem_bytes)


def ridge_flop_per_byte(peak_flops: float, hbm_bytes_per_s: float) -> float:
    return peak_flops / hbm_bytes_per_s


def flash_fwd_hbm_bytes(N: int, d: int, br: int, elem_bytes: int = 2) -> int:
    """Tiled forward, one head, no L2 reuse: Q once, K and V once per query block,
    O written once."""
    n_q_blocks = math.ceil(N / br)
    return elem_bytes * (N * d + n_q_blocks * 2 * N * d + N * d)


def transfer_seconds(nbytes: float, bytes_per_s: float) -> float:
    return nbytes / bytes_per_s


def matmul_seconds(N: int, d: int, peak_flops: float) -> float:
    """Time of one head's two attention matmuls (QK^T and PV) at peak."""
    return attention_flops(1, 1, N, d) / peak_flops
