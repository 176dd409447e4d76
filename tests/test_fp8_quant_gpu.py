"""The device-side FP8 quantisation (fa_e4m3_descale, fa_quantize_e4m3) against the host
encoder of the same definition (inputs.f32_to_e4m3_bits: nearest E4M3 value, ties to the even
code, saturation at 448, pinned against torch's float8_e4m3fn conversion in
tests/test_oracle_fp8.py), bit for bit; and the FP8 forward fed by it against the oracle."""

import math

import numpy as np
import pytest
import torch

from exact_attention_96_gb300 import abi, build, inputs as I
from exact_attention_96_gb300 import attention as fa
from oracle import fp8
from parity_util import LSE_MAX_ABS, max_abs, rel_fro, to_device, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    build.build()
    abi.load()


def host_codes(bits_bf16: np.ndarray, descale: float) -> np.ndarray:
    x = (bits_bf16.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return I.f32_to_e4m3_bits(x / np.float32(descale))  # fp32 quotient, like the kernel


@pytest.mark.parametrize("B,H,N,d,mult", [(1, 2, 300, 128, 1.0), (2, 1, 77, 64, 3.0), (1, 1, 1000, 256, 0.01),
                                          (1, 3, 16, 128, 100.0)])
def test_descale_and_codes_match_the_host_encoder(B, H, N, d, mult):
    x = I.normal_bf16((B, H, N, d), seed=N + d, multiplier=mult)
    t = to_device(x)
    q8, ds = fa.quantize_fp8(t)
    vt8, ds2 = fa.quantize_fp8(t, transpose=True)
    torch.cuda.synchronize()
    assert fa.status_check() == abi.FA_OK
    xf = (x.astype(np.uint32) << np.uint32(16)).view(np.float32)
    want_ds = np.float32(np.max(np.abs(xf))) / np.float32(448.0)
    assert ds.item() == float(want_ds) and ds2.item() == float(want_ds)
    codes = host_codes(x, want_ds)
    assert np.array_equal(q8.cpu().numpy(), codes)
    ldv = (N + 15) // 16 * 16
    want_t = np.zeros((B, H, d, ldv), np.uint8)
    want_t[..., :N] = np.swapaxes(codes, -1, -2)
    assert np.array_equal(vt8.cpu().numpy(), want_t)
    # the element of largest magnitude lands on +-448 (code 0x7E / 0xFE)
    i = np.unravel_index(np.argmax(np.abs(xf)), xf.shape)
    assert codes[i] & 0x7F == 0x7E


def test_given_descale_saturates_and_wider_ld_is_zero_filled():
    B, H, N, d = 1, 2, 40, 64
    x = I.normal_bf16((B, H, N, d), seed=9, multiplier=50.0)
    t = to_device(x)
    ds = torch.tensor([0.01], dtype=torch.float32, device="cuda")  # x / 0.01 overflows E4M3 often
    q8, _ = fa.quantize_fp8(t, descale=ds)
    vt8, _ = fa.quantize_fp8(t, transpose=True, ld=80, descale=ds)
    codes = host_codes(x, np.float32(0.01))
    assert np.any(codes & 0x7F == 0x7E)
    assert np.array_equal(q8.cpu().numpy(), codes)
    want_t = np.zeros((B, H, d, 80), np.uint8)
    want_t[..., :N] = np.swapaxes(codes, -1, -2)
    assert np.array_equal(vt8.cpu().numpy(), want_t)


def test_all_zero_tensor_gets_descale_one():
    t = torch.zeros((1, 1, 33, 128), dtype=torch.bfloat16, device="cuda")
    q8, ds = fa.quantize_fp8(t)
    assert ds.item() == 1.0 and int(q8.abs().sum().item()) == 0


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_from_bf16_inputs_against_the_oracle(causal):
    B, H, N, d = 1, 2, 333, 128
    q, k, v, _ = I.attention_inputs(B, H, N, d, seed=21, with_grad=False)
    o, lse, (q8, k8, vt8), (qs, ks, vs) = fa.forward_fp8_from_bf16(to_device(q), to_device(k), to_device(v),
                                                                  causal=causal)
    assert fa.status_check() == abi.FA_OK
    v8 = np.ascontiguousarray(np.swapaxes(vt8.cpu().numpy()[..., :N], -1, -2))
    o_ref, lse_ref = fp8.attention_fwd_fp8(q8.cpu().numpy(), k8.cpu().numpy(), v8, qs, ks, vs, 1 / math.sqrt(d),
                                           causal)
    o64, l64 = to_f64(o), to_f64(lse)
    vmax = np.max(np.abs(fp8.e4m3_bits_to_f64(v8) * vs))
    assert max_abs(o64, o_ref) <= 2.0 ** -4 * vmax + 2.0 ** -8 * np.max(np.abs(o_ref))
    assert rel_fro(o64, o_ref) <= 0.04
    assert max_abs(l64, lse_ref) <= LSE_MAX_ABS
