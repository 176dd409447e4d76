"""Runs forward and/or backward passes of one attention shape on seeded inputs -- a small
driver for profilers and quick timing.

    python -m exact_attention_96_gb300.run_case --B 2 --H 16 --N 8192 --d 128 --causal \
        --passes fwd,bwd --repeat 3
"""

from __future__ import annotations

import argparse
import math

import numpy as np
import torch

from . import abi, build, inputs
from . import attention as fa


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--B", type=int, default=2)
    ap.add_argument("--H", type=int, default=16)
    ap.add_argument("--N", type=int, default=8192)
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--causal", action="store_true")
    ap.add_argument("--multiplier", type=float, default=1.0)
    ap.add_argument("--passes", default="fwd,bwd")
    ap.add_argument("--repeat", type=int, default=3)
    ap.add_argument("--fp8", action="store_true", help="time the FP8 (E4M3) forward, head dim 128")
    ap.add_argument("--dropout", type=float, default=0.0, help="dropout probability (seed 1)")
    a = ap.parse_args()

    build.build()
    abi.load()
    if a.fp8:
        run_fp8(a)
        return
    host = inputs.attention_inputs(a.B, a.H, a.N, a.d, seed=0, multiplier=a.multiplier)
    q, k, v, do = (torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda() for x in host)
    scale = 1 / math.sqrt(a.d)
    dk = dict(dropout_p=a.dropout, seed=1) if a.dropout > 0 else {}
    o, lse = fa.forward(q, k, v, causal=a.causal, scale=scale, **dk)
    ws = torch.empty(fa.workspace_bytes(a.B, a.H, a.N, a.d), dtype=torch.uint8, device="cuda")
    grads = tuple(torch.empty_like(q) for _ in range(3))
    passes = a.passes.split(",")
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(a.repeat):
        if "fwd" in passes:
            fa.forward(q, k, v, causal=a.causal, scale=scale, out=o, lse=lse, **dk)
        if "bwd" in passes:
            fa.backward(q, k, v, o, do, lse, causal=a.causal, scale=scale, workspace=ws, grads=grads, **dk)
    end.record()
    st = fa.status_check()
    if st != abi.FA_OK:
        raise SystemExit(f"device status {abi.status_string(st)}")
    print(f"{a.B}x{a.H}x{a.N}x{a.d} causal={a.causal} passes={a.passes}: "
          f"{start.elapsed_time(end) / a.repeat:.3f} ms per repeat")


def run_fp8(a):
    q8, k8, v8, (qs, ks, vs) = inputs.fp8_attention_inputs(a.B, a.H, a.N, 128, seed=0)
    ldv = (a.N + 15) // 16 * 16
    vt = np.zeros((a.B, a.H, 128, ldv), np.uint8)
    vt[..., :a.N] = np.swapaxes(v8, -1, -2)  # the caller's layout: V transposed
    tq, tk, tvt = (torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (q8, k8, vt))
    o, lse = fa.forward_fp8(tq, tk, tvt, qs, ks, vs, causal=a.causal)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(a.repeat):
        fa.forward_fp8(tq, tk, tvt, qs, ks, vs, causal=a.causal, out=o, lse=lse)
    end.record()
    st = fa.status_check()
    if st != abi.FA_OK:
        raise SystemExit(f"device status {abi.status_string(st)}")
    print(f"{a.B}x{a.H}x{a.N}x128 fp8 causal={a.causal}: {start.elapsed_time(end) / a.repeat:.3f} ms per call")


if __name__ == "__main__":
    main()
