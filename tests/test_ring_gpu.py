"""Ring attention emulated on one GPU (fa_fwd_partial per hop, fa_merge_partials per worker)
against the fp64 oracle and against the single-call forward."""

import math

import numpy as np
import pytest

from exact_attention_96_gb300 import abi, build, inputs as I
from exact_attention_96_gb300 import attention as fa
from exact_attention_96_gb300.ring import ring_attention_forward
from oracle import attention as A
from parity_util import LSE_MAX_ABS, O_MAX_ABS, O_REL_FRO, max_abs, rel_fro, to_device, to_f64, widen

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
])
def test_ring_backward_matches_oracle(B, H, N, d, world, causal):
    from exact_attention_96_gb300.ring import ring_attention_backward
    build.build()
    abi.load()
    q, k, v, do = I.attention_inputs(B, H, N, d, seed=3 * N + world)
    tq, tk, tv, tdo = map(to_device, (q, k, v, do))
    o, lse = ring_attention_forward(tq, tk, tv, world, causal=causal)
    dq, dk, dv = ring_attention_backward(tq, tk, tv, o, tdo, lse, world, causal=causal)
    assert fa.status_check() == abi.FA_OK
    refs = A.attention_bwd(widen(q), widen(k), widen(v), widen(do), 1 / math.sqrt(d), causal)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), refs[:3]):
        assert rel_fro(to_f64(g), r) <= 2e-2, name
