"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.

Some callers have no way to hand fa_bwd a workspace: embedders whose device memory is owned
by an allocator they cannot call, and latency-critical code that must avoid the device
synchronisation cudaMalloc/cudaFree can cause.  fa_bwd_noalloc runs the same backward pass
on a fixed scratch array in the library's static device memory instead.  This test calls it
through the C ABI twice in a row for each head dim (each dim lays the dQ accumulator out in
its own way) and checks both results against fa_bwd (the entry point that takes a caller
workspace) and against the fp64 oracle, within the gradient tolerance of the parity tests,
and that a problem too large for the scratch array is refused before anything is launched.

The file name makes pytest collect it last."""

import math

import pytest
import torch

from exact_attention_96_gb300 import abi, build, inputs as I
from exact_attention_96_gb300 import attention as fa
from oracle import attention as A
from parity_util import GRAD_REL_FRO, rel_fro, to_device, to_f64, widen

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,N,d,causal", [
    (2, 3, 300, 128, True),
    (1, 4, 333, 64, False),
    (1, 2, 260, 256, True),
])
def test_noalloc_backward_matches_workspace_backward_and_oracle_on_two_calls(B, H, N, d, causal):
    build.build()
    abi.load()
    scale = 1 / math.sqrt(d)
    q, k, v, do = I.attention_inputs(B, H, N, d, seed=11 + d)
    assert abi.fa_bwd_workspace_bytes(B, H, N, d) <= 64 * 1024 * 1024
    tq, tk, tv, tdo = map(to_device, (q, k, v, do))
    o, lse = fa.forward(tq, tk, tv, causal=causal, scale=scale)
    ref = [to_f64(g) for g in fa.backward(tq, tk, tv, o, tdo, lse, causal=causal, scale=scale)]
    oracle = A.attention_bwd(widen(q), widen(k), widen(v), widen(do), scale, causal)[:3]
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        dq, dk, dv = (torch.full_like(tq, float("nan")) for _ in range(3))
        st = abi.fa_bwd_noalloc(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.data_ptr(),
                                tdo.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                dv.data_ptr(), B, H, N, d, scale, causal, stream)
        assert st == abi.FA_OK, abi.status_string(st)
        assert fa.status_check() == abi.FA_OK
        for name, got, want, exact in zip(("dq", "dk", "dv"), (dq, dk, dv), ref, oracle):
            got = to_f64(got)
            err = rel_fro(got, want)
            assert err <= GRAD_REL_FRO, (call, name, "vs fa_bwd", err)
            err = rel_fro(got, exact)
            assert err <= GRAD_REL_FRO, (call, name, "vs oracle", err)


def test_noalloc_refuses_problems_larger_than_its_scratch():
    build.build()
    B, H, N, d = 4, 16, 8192, 128  # needs ~272 MB of workspace
    assert abi.fa_bwd_workspace_bytes(B, H, N, d) > 64 * 1024 * 1024
    t = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    p = t.data_ptr()
    st = abi.fa_bwd_noalloc(p, p, p, p, p, p, p, p, p, B, H, N, d, 0.1, 1,
                            torch.cuda.current_stream().cuda_stream)
    assert st == abi.FA_ERR_UNSUPPORTED
    # invalid sizes get the same status as every other entry point gives them
    st = abi.fa_bwd_noalloc(p, p, p, p, p, p, p, p, p, 1, 1, 0, 128, 0.1, 1,
                            torch.cuda.current_stream().cuda_stream)
    assert st == abi.FA_ERR_INVALID_ARG
    st = abi.fa_bwd_noalloc(p, p, p, p, p, p, p, p, p, 1, 1, 64, 96, 0.1, 1,
                            torch.cuda.current_stream().cuda_stream)
    assert st == abi.FA_ERR_UNSUPPORTED
