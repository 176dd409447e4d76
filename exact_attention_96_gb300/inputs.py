"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module draws random numbers and rounds them to bfloat16; it holds none of the
attention arithmetic.  Recipe (the same on every machine):

* numpy ``default_rng(seed)`` (PCG64), ``standard_normal(dtype=float32)`` -> iid N(0, 1)
* optional exact power-of-two multiplier (the long causal shape multiplies Q, K, V by
  0.5 before rounding)
* float32 -> bfloat16 by round-to-nearest-even on the bit pattern
* Q, K, V, dO use seeds ``seed + 0 .. seed + 3``

Returned arrays are uint16 bfloat16 bit patterns of shape [B, H, N, d].
"""

from __future__ import annotations

import numpy as np

__all__ = ["f32_to_bf16_bits", "normal_bf16", "attention_inputs"]


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
