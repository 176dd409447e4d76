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
    a = ap.parse_args()

    build.build()
    abi.load()
    host = inputs.attention_inputs(a.B, a.H, a.N, a.d, seed=0, multiplier=a.multiplier)
    q, k, v, do = (torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda() for x in host)
    scale = 1 / math.sqrt(a.d)
    o, lse = fa.forward(q, k, v, causal=a.causal, scale=scale)
    ws = torch.empty(fa.workspace_bytes(a.B, a.H, a.N, a.d), dtype=torch.uint8, device="cuda")
    grads = tuple(torch.empty_like(q) for _ in range(3))
    passes = a.passes.split(",")
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(a.repeat):
        if "fwd" in passes:
            fa.forward(q, k, v, causal=a.causal, scale=scale, out=o, lse=lse)
        if "bwd" in passes:
            fa.backward(q, k, v, o, do, lse, causal=a.causal, scale=scale, workspace=ws, grads=grads)
    end.record()
    st = fa.status_check()
    if st != abi.FA_OK:
        raise SystemExit(f"device status {abi.status_string(st)}")
    print(f"{a.B}x{a.H}x{a.N}x{a.d} causal={a.causal} passes={a.passes}: "
          f"{start.elapsed_time(end) / a.repeat:.3f} ms per repeat")


if __name__ == "__main__":
    main()
