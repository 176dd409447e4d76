"""FP8 (E4M3) inputs and the FP8 forward's definition (test infrastructure: imported only by
the tests, smoke() and the bench's CPU-baseline leg; the CUDA path shares nothing with it).

E4M3 decoding follows the OCP 8-bit floating point specification (E4M3 variant): sign bit,
4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 encodes subnormals
m/8 * 2^-6; S.1111.111 is NaN (no infinities); the largest finite magnitude is 448.

The FP8 forward pass ("Flash Attention 原理与实践" §3.2, the third version's FP8 mode) takes
Q, K, V as E4M3 codes with one fp32 descale factor per tensor: the real inputs are
descale * decode(code).  What it computes is attention of those real inputs -- the same
definition as the bf16 path (``attention.attention_fwd``), applied to the dequantised
tensors.  How the kernel rounds intermediate values (P in 8 bits) is an approximation of
this definition, covered by the tolerance the tests derive.
"""

from __future__ import annotations

import numpy as np

from . import attention as A

__all__ = ["e4m3_bits_to_f64", "attention_fwd_fp8"]


def e4m3_bits_to_f64(bits) -> np.ndarray:
    """Decode E4M3 codes (uint8) to float64 exactly (NaN for S.1111.111)."""
    b = np.asarray(bits)
    if b.dtype != np.uint8:
        raise TypeError("expected uint8 E4M3 codes")
    sign = np.where(b >> 7, -1.0, 1.0)
    e = ((b >> 3) & 0xF).astype(np.int64)
    m = (b & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def attention_fwd_fp8(q8, k8, v8, q_descale: float, k_descale: float, v_descale: float,
                      scale: float, causal: bool):
    """O [B,H,N,d] and LSE [B,H,N] (fp64) of attention over the dequantised E4M3 inputs
    q8, k8, v8 (uint8 codes [B,H,N,d])."""
    q = e4m3_bits_to_f64(q8) * float(q_descale)
    k = e4m3_bits_to_f64(k8) * float(k_descale)
    v = e4m3_bits_to_f64(v8) * float(v_descale)
    return A.attention_fwd(q, k, v, scale, causal)
