"""Ring attention emulated on one GPU (fa_fwd_partial per hop, fa_merge_partials per worker)
against the fp64 oracle and against the single-call forward."""

import math

import numpy as np
import pytest
import torch

from exact_attention_96_gb300 import abi, build, inputs as I
from exact_attention_96_gb300 import attention as fa
from exact_attention_96_gb300.ring import ring_attention_forward
from oracle import attention as A
from parity_util import (GRAD_REL_FRO, LSE_MAX_ABS, O_MAX_ABS, O_REL_FRO, max_abs, rel_fro, to_device, to_f64,
                         widen)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,N,d,world,causal", [
    (1, 2, 512, 64, 2, False),
    (1, 2, 512, 128, 4, True),
    (2, 1, 1024, 128, 4, False),
    (1, 1, 768, 256, 3, True),
    (1, 2, 1000, 64, 4, True),      # shards of 250 positions: ragged tiles inside each shard
])
def test_ring_forward_matches_oracle(B, H, N, d, world, causal):
    build.build()
    abi.load()
    q, k, v, _ = I.attention_inputs(B, H, N, d, seed=N + world, with_grad=False)
    tq, tk, tv = map(to_device, (q, k, v))
    o, lse = ring_attention_forward(tq, tk, tv, world, causal=causal)
    assert fa.status_check() == abi.FA_OK
    o_ref, lse_ref = A.attention_fwd(widen(q), widen(k), widen(v), 1 / math.sqrt(d), causal)
    o, lse = to_f64(o), to_f64(lse)
    assert max_abs(o, o_ref) <= O_MAX_ABS
    assert rel_fro(o, o_ref) <= O_REL_FRO
    assert max_abs(lse, lse_ref) <= LSE_MAX_ABS
    o1, l1 = fa.forward(tq, tk, tv, causal=causal)
    assert max_abs(o, to_f64(o1)) <= 8e-3 and max_abs(lse, to_f64(l1)) <= 1e-4


@pytest.mark.parametrize("B,H,N,d,world,causal", [
    (1, 2, 512, 64, 2, False),
    (1, 2, 512, 128, 4, True),
    (2, 1, 1000, 64, 4, True),
    (1, 2, 768, 256, 3, True),
    (1, 1, 2048, 128, 8, False),
])
def test_ring_backward_matches_oracle(B, H, N, d, world, causal):
    """Each gradient of the ring backward is as close to the oracle as the single-call
    backward's: the block pairs' contributions are summed in fp32 and rounded once."""
    from exact_attention_96_gb300.ring import ring_attention_backward
    build.build()
    abi.load()
    q, k, v, do = I.attention_inputs(B, H, N, d, seed=3 * N + world)
    tq, tk, tv, tdo = map(to_device, (q, k, v, do))
    o, lse = ring_attention_forward(tq, tk, tv, world, causal=causal)
    dq, dk, dv = ring_attention_backward(tq, tk, tv, o, tdo, lse, world, causal=causal)
    single = fa.backward(tq, tk, tv, o, tdo, lse, causal=causal)
    assert fa.status_check() == abi.FA_OK
    refs = A.attention_bwd(widen(q), widen(k), widen(v), widen(do), 1 / math.sqrt(d), causal)
    for name, g, g1, r in zip(("dq", "dk", "dv"), (dq, dk, dv), single, refs[:3]):
        err, err1 = rel_fro(to_f64(g), r), rel_fro(to_f64(g1), r)
        assert err <= GRAD_REL_FRO, name
        # one bf16 rounding of an fp32 sum, like the single call: the same error level
        assert err <= 1.1 * err1 + 2e-4, (name, err, err1)


# (6, 30, 300, 64): 540 (key tile, head) items, several for every SM
@pytest.mark.parametrize("d,B,H", [(64, 2, 2), (128, 2, 2), (256, 2, 2), (64, 6, 30)])
def test_bwd_accumulate_adds_in_fp32(d, B, H):
    """fa_bwd_accumulate adds dQ, dK, dV (dQ and dK scaled) in fp32 into the caller's buffers:
    one call into zeros equals the oracle's gradients, and a second call adds them again."""
    build.build()
    abi.load()
    N, causal = 300, d != 64
    scale = 1 / math.sqrt(d)
    q, k, v, do = I.attention_inputs(B, H, N, d, seed=50 + d)
    tq, tk, tv, tdo = map(to_device, (q, k, v, do))
    o, lse = fa.forward(tq, tk, tv, causal=causal, scale=scale)
    acc = torch.zeros((3, B, H, N, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(fa.workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    refs = A.attention_bwd(widen(q), widen(k), widen(v), widen(do), scale, causal)[:3]
    firsts = None
    for call in range(2):
        st = abi.fa_bwd_accumulate(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.data_ptr(), tdo.data_ptr(),
                                   lse.data_ptr(), acc[0].data_ptr(), acc[1].data_ptr(), acc[2].data_ptr(),
                                   B, H, N, d, scale, causal, ws.data_ptr(), ws.numel(), stream)
        assert st == abi.FA_OK, abi.status_string(st)
        assert fa.status_check() == abi.FA_OK
        got = [to_f64(acc[g]) for g in range(3)]
        if call == 0:
            firsts = got
            for name, g, r in zip(("dq", "dk", "dv"), got, refs):
                assert rel_fro(g, r) <= GRAD_REL_FRO, name
        else:
            for name, g, g0 in zip(("dq", "dk", "dv"), got, firsts):
                # the same contribution added twice (up to the order of fp32 additions)
                assert rel_fro(g, 2 * g0) <= 1e-5, name
    out = torch.empty((3, B, H, N, d), dtype=torch.bfloat16, device="cuda")
    assert abi.fa_convert_f32_to_bf16(acc.data_ptr(), out.data_ptr(), acc.numel(), stream) == abi.FA_OK
    assert torch.equal(out, acc.to(torch.bfloat16))


def test_convert_f32_to_bf16_rounds_to_nearest_even_with_a_ragged_tail():
    build.build()
    abi.load()
    g = torch.Generator().manual_seed(5)
    x = (torch.randn(1037, generator=g, dtype=torch.float64) * 3).float()
    x[:4] = torch.tensor([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 65504.5])  # ties
    src = x.cuda()
    dst = torch.empty(1037, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert abi.fa_convert_f32_to_bf16(src.data_ptr(), dst.data_ptr(), x.numel(), stream) == abi.FA_OK
    torch.cuda.synchronize()
    assert torch.equal(dst.cpu(), x.to(torch.bfloat16))
