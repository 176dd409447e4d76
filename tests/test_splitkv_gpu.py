"""Split-KV forward (the decoding variant) against the fp64 oracle: few queries against long
key sequences, key ranges merged by log-sum-exp.  Bars as for the forward: O max-abs <= 1e-2
and rel-Frobenius <= 5e-3, LSE max-abs <= 1e-3."""

import math

import numpy as np
import pytest
import torch

from exact_attention_96_gb300 import abi, build, inputs as I
from exact_attention_96_gb300 import attention as fa
from oracle import attention as A
from parity_util import LSE_MAX_ABS, O_MAX_ABS, O_REL_FRO, max_abs, rel_fro, to_device, to_f64, widen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    build.build()
    abi.load()


def qkv(B, H, Nq, Nk, d, seed):
    q = I.normal_bf16((B, H, Nq, d), seed)
    k = I.normal_bf16((B, H, Nk, d), seed + 1)
    v = I.normal_bf16((B, H, Nk, d), seed + 2)
    return q, k, v


@pytest.mark.parametrize("B,H,Nq,Nk,d,splits", [
    (1, 1, 1, 1000, 64, 0),
    (2, 4, 1, 10007, 128, 0),
    (2, 4, 64, 10007, 64, 3),
    (1, 2, 300, 1000, 256, 0),
    (1, 1, 5, 64, 128, 0),          # one key tile: a single range
    (3, 2, 17, 4097, 128, 1000),    # more requested than tiles
])
def test_splitkv_matches_oracle(B, H, Nq, Nk, d, splits):
    q, k, v = qkv(B, H, Nq, Nk, d, seed=Nq + Nk + d)
    o, lse = fa.forward_splitkv(*(to_device(x) for x in (q, k, v)), num_splits=splits)
    assert fa.status_check() == abi.FA_OK
    o_ref, lse_ref = A.attention_fwd(widen(q), widen(k), widen(v), 1 / math.sqrt(d), False)
    o, lse = to_f64(o), to_f64(lse)
    assert max_abs(o, o_ref) <= O_MAX_ABS
    assert rel_fro(o, o_ref) <= O_REL_FRO
    assert max_abs(lse, lse_ref) <= LSE_MAX_ABS


def test_splitkv_on_square_problem_agrees_with_fa_fwd():
    q, k, v, _ = I.attention_inputs(1, 3, 700, 128, seed=5, with_grad=False)
    tq, tk, tv = map(to_device, (q, k, v))
    o1, l1 = fa.forward(tq, tk, tv)
    o2, l2 = fa.forward_splitkv(tq, tk, tv, num_splits=3)
    assert fa.status_check() == abi.FA_OK
    assert max_abs(to_f64(o1), to_f64(o2)) <= 8e-3
    assert max_abs(to_f64(l1), to_f64(l2)) <= 1e-4


def test_decode_shape_full_size():
    # decoding a batch of 4 x 16 heads against a 65536-token cache, d = 128
    B, H, Nk, d = 4, 16, 65536, 128
    q, k, v = qkv(B, H, 1, Nk, d, seed=77)
    o, lse = fa.forward_splitkv(*(to_device(x) for x in (q, k, v)))
    assert fa.status_check() == abi.FA_OK
    o, lse = to_f64(o), to_f64(lse)
    for b, h in ((0, 0), (3, 15), (2, 7)):
        o_ref, lse_ref = A.attention_fwd_rows(widen(q[b, h]), widen(k[b, h]), widen(v[b, h]),
                                              1 / math.sqrt(d), False, [0])
        assert max_abs(o[b, h], o_ref) <= O_MAX_ABS
        assert max_abs(lse[b, h], lse_ref) <= LSE_MAX_ABS
