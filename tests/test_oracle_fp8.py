"""Pins of the FP8 (E4M3) decode and of the FP8 forward's definition, and a check of the
seeded E4M3 input encoder.

The decode is pinned by torch's float8_e4m3fn conversion (an independent library routine)
on all 256 codes and by values the OCP FP8 specification fixes (largest finite 448, smallest
normal 2^-6, smallest subnormal 2^-9, NaN codes, signed zero)."""

import numpy as np
import pytest
import torch

from exact_attention_96_gb300 import inputs as I
from oracle import attention as A
from oracle import fp8


def test_decode_matches_torch_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours = fp8.e4m3_bits_to_f64(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_decode_special_values_of_the_specification():
    v = fp8.e4m3_bits_to_f64(np.array([0x7E, 0x08, 0x07, 0x01, 0x38, 0xB8, 0x00, 0x80, 0x7F, 0xFF],
                                      dtype=np.uint8))
    assert v[0] == 448.0 and v[1] == 2.0 ** -6 and v[2] == 7 * 2.0 ** -9 and v[3] == 2.0 ** -9
    assert v[4] == 1.0 and v[5] == -1.0
    assert v[6] == 0.0 and not np.signbit(v[6]) and v[7] == 0.0 and np.signbit(v[7])
    assert np.isnan(v[8]) and np.isnan(v[9])
    pos = fp8.e4m3_bits_to_f64(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)  # finite codes increase strictly
    # three mantissa bits: the spacing doubles every 8 codes above the subnormals
    first, nxt = np.diff(pos[8:])[::8], np.diff(pos[16:])[::8]
    assert np.array_equal(nxt, 2 * first[:len(nxt)]) and first[0] == 2.0 ** -9


def test_encoder_rounds_to_nearest_even_and_saturates():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(20000) * 60).astype(np.float32)
    x = np.concatenate([x, np.float32([0, -0.0, 448, 449, 464, 1000, -1000, 2.0 ** -10, 2.0 ** -9 * 1.5])])
    codes = I.f32_to_e4m3_bits(x)
    back = fp8.e4m3_bits_to_f64(codes)
    table = fp8.e4m3_bits_to_f64(np.arange(0x7F, dtype=np.uint8))
    a = np.minimum(np.abs(x.astype(np.float64)), 448.0)
    best = np.min(np.abs(table[None, :] - a[:, None]), axis=1)
    assert np.all(np.abs(np.abs(back) - a) == best)        # nearest representable
    assert I.f32_to_e4m3_bits(np.float32([2.0 ** -10]))[0] == 0x00    # halfway to 2^-9: even code 0
    assert I.f32_to_e4m3_bits(np.float32([2.0 ** -9 * 1.5]))[0] == 0x02  # halfway 1 and 2 -> 2
    assert I.f32_to_e4m3_bits(np.float32([1000.0]))[0] == 0x7E
    assert I.f32_to_e4m3_bits(np.float32([-1000.0]))[0] == 0xFE
    assert I.f32_to_e4m3_bits(np.float32([-0.0]))[0] == 0x80
    in_range = np.abs(x) <= 448
    ref = torch.from_numpy(x[in_range]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes[in_range], ref)


def test_fp8_inputs_use_the_range_and_are_seeded():
    q8, k8, v8, (qs, ks, vs) = I.fp8_attention_inputs(1, 2, 64, 128, seed=5)
    for c, s in ((q8, qs), (k8, ks), (v8, vs)):
        assert c.dtype == np.uint8 and c.shape == (1, 2, 64, 128)
        assert np.max(np.abs(fp8.e4m3_bits_to_f64(c))) == 448.0 and s > 0
    again = I.fp8_attention_inputs(1, 2, 64, 128, seed=5)
    assert all(np.array_equal(a, b) for a, b in zip((q8, k8, v8), again[:3]))


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_is_attention_of_the_dequantised_inputs(causal):
    q8, k8, v8, (qs, ks, vs) = I.fp8_attention_inputs(2, 1, 40, 16, seed=9)
    o, lse = fp8.attention_fwd_fp8(q8, k8, v8, qs, ks, vs, 0.25, causal)
    # torch's own conversion and softmax give the same numbers on the same real inputs
    deq = [torch.from_numpy(c.copy()).view(torch.float8_e4m3fn).to(torch.float64) * s
           for c, s in ((q8, qs), (k8, ks), (v8, vs))]
    s_ = 0.25 * deq[0] @ deq[1].transpose(-1, -2)
    if causal:
        s_ = s_.masked_fill(torch.ones(40, 40, dtype=torch.bool).triu(1), float("-inf"))
    assert np.max(np.abs(o - (torch.softmax(s_, -1) @ deq[2]).numpy())) < 1e-12
    assert np.max(np.abs(lse - torch.logsumexp(s_, -1).numpy())) < 1e-12
    # descale factors are linear in the real inputs: doubling V's doubles O
    o2, _ = fp8.attention_fwd_fp8(q8, k8, v8, qs, ks, 2 * vs, 0.25, causal)
    assert np.max(np.abs(o2 - 2 * o)) < 1e-12
