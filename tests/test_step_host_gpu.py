"""fa_step_host: the host-buffer step (copies in, forward, backward, copies out, pipelined over
chunks of heads) against the device calls on the same inputs.  Per head the kernels are the
same launches as the whole-batch call, so O, LSE, dK and dV must match bit for bit; dQ is
summed with fp32 atomics whose order depends on scheduling, so it is compared within one bf16
rounding step.  One case is also checked against the fp64 oracle."""

import math

import numpy as np
import pytest
import torch

from exact_attention_96_gb300 import abi, build, inputs as I
from exact_attention_96_gb300 import attention as fa
from oracle import attention as A
from parity_util import (GRAD_REL_FRO, LSE_MAX_ABS, O_MAX_ABS, O_REL_FRO, max_abs, rel_fro, to_f64,
                         widen)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    build.build()
    abi.load()


def host_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).pin_memory()


@pytest.mark.parametrize("B,H,N,d,causal,chunks", [
    (2, 3, 300, 64, True, 4),     # 6 heads in 4 chunks of 2 (the last chunk smaller)
    (1, 4, 513, 128, False, 3),   # N % 4 != 0: chunks rounded to 4 heads (one chunk)
    (4, 16, 1024, 128, True, 7),  # 64 heads in 7 chunks
    (1, 2, 256, 256, True, 1),
    (4, 16, 2048, 64, True, 0),   # default plan: 15 heads per chunk (1.5 waves of tiles), 15*4+4
    (4, 16, 2047, 64, False, 0),  # default plan, N % 4 != 0: 16 heads per chunk, 4-head aligned
])
def test_step_host_matches_device_calls(B, H, N, d, causal, chunks):
    host = I.attention_inputs(B, H, N, d, seed=N + d)
    hq, hk, hv, hdo = (host_bf16(x) for x in host)
    o_h, lse_h, dq_h, dk_h, dv_h = fa.step_host(hq, hk, hv, hdo, causal=causal, num_chunks=chunks)
    torch.cuda.synchronize()
    assert fa.status_check() == abi.FA_OK
    q, k, v, do = (t.cuda() for t in (hq, hk, hv, hdo))
    o, lse = fa.forward(q, k, v, causal=causal)
    dq, dk, dv = fa.backward(q, k, v, o, do, lse, causal=causal)
    assert torch.equal(o_h, o.cpu()) and torch.equal(lse_h, lse.cpu())
    assert torch.equal(dk_h, dk.cpu()) and torch.equal(dv_h, dv.cpu())
    a, b = dq_h.float(), dq.cpu().float()
    assert torch.all((a - b).abs() <= 2 ** -7 * b.abs() + 1e-6)


def test_step_host_against_the_oracle():
    B, H, N, d, causal = 2, 2, 384, 128, True
    host = I.attention_inputs(B, H, N, d, seed=5)
    o_h, lse_h, dq_h, dk_h, dv_h = fa.step_host(*(host_bf16(x) for x in host), causal=causal, num_chunks=2)
    torch.cuda.synchronize()
    assert fa.status_check() == abi.FA_OK
    q, k, v, do = (widen(x) for x in host)
    scale = 1 / math.sqrt(d)
    o_ref, lse_ref = A.attention_fwd(q, k, v, scale, causal)
    assert max_abs(to_f64(o_h), o_ref) <= O_MAX_ABS and rel_fro(to_f64(o_h), o_ref) <= O_REL_FRO
    assert max_abs(to_f64(lse_h), lse_ref) <= LSE_MAX_ABS
    refs = A.attention_bwd(q, k, v, do, scale, causal)
    for g, r in zip((dq_h, dk_h, dv_h), refs[:3]):
        assert rel_fro(to_f64(g), r) <= GRAD_REL_FRO


def test_step_host_reuses_buffers_across_steps():
    B, H, N, d = 1, 8, 512, 64
    host = I.attention_inputs(B, H, N, d, seed=9)
    pins = [host_bf16(x) for x in host]
    bufs = [torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda") for _ in range(5)]
    bufs += [torch.empty((B, H, N), dtype=torch.float32, device="cuda")]
    bufs += [torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    ws = torch.empty(abi.fa_step_host_workspace_bytes(B, H, N, d, 0), dtype=torch.uint8, device="cuda")
    first = [t.clone() for t in fa.step_host(*pins, device_buffers=bufs, workspace=ws)]
    second = fa.step_host(*pins, device_buffers=bufs, workspace=ws)
    torch.cuda.synchronize()
    for a, b in zip(first[:2] + first[3:], second[:2] + second[3:]):  # all but dQ: bitwise
        assert torch.equal(a, b)
