"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module draws random numbers and rounds them to bfloat16; it holds none of the
attention arithmetic.  Recipe (the same on every machine):

* numpy ``default_rng(seed)`` (PCG64), ``standard_normal(dtype=float32)`` -> iid N(0, 1)
* optional exact power-of-two multiplier (the long causal shape multiplies Q, K, V by
  0.5 before rounding)
* float32 -> bfloat16 by round-to-nearest-even on the bit pattern
* Q, K, V, dO use seeds ``seed + 0 .. seed + 3``

Returned arrays are uint16 bfloat16 bit patterns of shape [B, H, N, d].

FP8 inputs (``fp8_attention_inputs``): the same float32 draws for Q, K, V, each divided by its
per-tensor scale s = max|x| / 448 (a float32) and rounded to the nearest E4M3 value (ties to
the even code), giving uint8 codes and the descale factor s of each tensor.
"""

from __future__ import annotations

import numpy as np

__all__ = ["f32_to_bf16_bits", "normal_bf16", "attention_inputs", "f32_to_e4m3_bits",
           "fp8_attention_inputs"]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def normal_bf16(shape, seed: int, multiplier: float = 1.0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if multiplier != 1.0:
        x = x * np.float32(multiplier)
    return f32_to_bf16_bits(x)


def attention_inputs(B: int, H: int, N: int, d: int, seed: int = 0,
                     multiplier: float = 1.0, with_grad: bool = True):
    """(q, k, v, do) as uint16 bf16 bit arrays [B, H, N, d]; do is None if not asked."""
    shape = (B, H, N, d)
    q = normal_bf16(shape, seed + 0, multiplier)
    k = normal_bf16(shape, seed + 1, multiplier)
    v = normal_bf16(shape, seed + 2, multiplier)
    do = normal_bf16(shape, seed + 3) if with_grad else None
    return q, k, v, do


def _e4m3_positive_values() -> np.ndarray:
    """The 127 finite non-negative E4M3 values, indexed by code 0x00 .. 0x7E."""
    codes = np.arange(127)
    e, m = codes >> 3, (codes & 7).astype(np.float64)
    return np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))


def f32_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to E4M3 codes: nearest value, ties to the even code, magnitudes
    above 448 saturate to 448."""
    x = np.asarray(x, dtype=np.float64)
    table = _e4m3_positive_values()
    a = np.minimum(np.abs(x), table[-1])
    hi = np.clip(np.searchsorted(table, a, side="left"), 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    d_lo, d_hi = a - table[lo], table[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)


def fp8_attention_inputs(B: int, H: int, N: int, d: int, seed: int = 0):
    """(q8, k8, v8) E4M3 codes [B, H, N, d] and their descale factors (q_s, k_s, v_s)."""
    out, scales = [], []
    for i in range(3):
        x = np.random.default_rng(seed + i).standard_normal(size=(B, H, N, d), dtype=np.float32)
        s = np.float32(np.max(np.abs(x)) / np.float32(448.0)) if x.size else np.float32(1.0)
        out.append(f32_to_e4m3_bits(x / s))
        scales.append(float(s))
    return (*out, tuple(scales))
