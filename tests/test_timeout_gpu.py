"""Failure path on the GPU without a fault: the test asks the library (host-side hook) to
withhold one key/value tile from the next forward launch.  The waits that depend on it are
bounded, so the kernel must give up after the wait limit, record FA_ERR_TIMEOUT, release its
resources and exit; the context must stay usable and the next call must be correct."""

import math

import numpy as np
import pytest

from exact_attention_96_gb300 import abi, build, inputs as I
from exact_attention_96_gb300 import attention as fa
from oracle import attention as A
from parity_util import LSE_MAX_ABS, O_MAX_ABS, max_abs, to_device, to_f64, widen

pytestmark = pytest.mark.gpu


def test_withheld_tile_times_out_and_context_survives():
    build.build()
    abi.load()
    B, H, N, d = 1, 2, 512, 128
    q, k, v, _ = I.attention_inputs(B, H, N, d, seed=21, with_grad=False)
    tq, tk, tv = map(to_device, (q, k, v))
    assert fa.status_check() == abi.FA_OK
    prev = abi.fa_set_wait_limit_ns(20_000_000)  # 20 ms
    try:
        abi.fa_test_withhold_kv_tile(1)
        fa.forward(tq, tk, tv, causal=False)        # the launch itself succeeds
        assert fa.status_check() == abi.FA_ERR_TIMEOUT
        assert fa.status_check() == abi.FA_OK        # the error word was cleared
    finally:
        abi.fa_set_wait_limit_ns(prev)
        abi.fa_test_withhold_kv_tile(-1)
    o, lse = fa.forward(tq, tk, tv, causal=False)
    assert fa.status_check() == abi.FA_OK
    o_ref, lse_ref = A.attention_fwd(widen(q), widen(k), widen(v), 1 / math.sqrt(d), False)
    assert max_abs(to_f64(o), o_ref) <= O_MAX_ABS
    assert max_abs(to_f64(lse), lse_ref) <= LSE_MAX_ABS
