"""Ring attention's host-side logic on CPU: the hop schedule, and a real two-rank ring over
gloo in which each rank holds one sequence shard, passes key/value shards with send/recv in
the schedule's order, computes every hop's partial with the fp64 oracle and merges them --
the exchange pattern a multi-GPU ring would run, checked against the whole definition."""

import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from exact_attention_96_gb300.ring import ring_hops  # noqa: E402


@pytest.mark.parametrize("world", [1, 2, 3, 5])
def test_ring_schedule(world):
    for r in range(world):
        full = ring_hops(r, world, causal=False)
        assert [t for t, _, _ in full] == list(range(world))
        assert sorted(s for _, s, _ in full) == list(range(world))
        assert full[0] == (0, r, True)
        causal = ring_hops(r, world, causal=True)
        assert sorted(s for _, s, _ in causal) == list(range(r + 1))
        assert [s for _, s, d in causal if d] == [r]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _ring_rank(rank, world, port, causal, out):
    sys.path.insert(0, ROOT)
    from oracle import attention as A
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    rng = np.random.default_rng(0)
    N, d, scale = 12 * world, 4, 0.5
    q, k, v = (rng.standard_normal((N, d)) for _ in range(3))
    ns = N // world
    q_r = q[rank * ns:(rank + 1) * ns]
    held = np.stack([k[rank * ns:(rank + 1) * ns], v[rank * ns:(rank + 1) * ns]])
    parts = {}
    for t in range(world):
        s = (rank - t) % world  # the shard held at hop t
        if not (causal and s > rank):
            kk, vv = held
            if causal and s == rank:
                o, l = A.attention_fwd(q_r[None, None], kk[None, None], vv[None, None], scale, True)
            else:
                o, l = A.attention_fwd(q_r[None, None], kk[None, None], vv[None, None], scale, False)
            parts[t] = (o[0, 0], l[0, 0])
        if t + 1 < world:  # pass the held shard to the next worker, receive from the previous
            send = torch.from_numpy(held.copy())
            recv = torch.empty_like(send)
            reqs = [dist.isend(send, (rank + 1) % world), dist.irecv(recv, (rank - 1) % world)]
            for rq in reqs:
                rq.wait()
            held = recv.numpy()
    assert sorted(parts) == [t for t, _, _ in ring_hops(rank, world, causal)]
    o_m, l_m = A.lse_merge([parts[t][0] for t in sorted(parts)], [parts[t][1] for t in sorted(parts)])
    o_ref, l_ref = A.attention_fwd(q[None, None], k[None, None], v[None, None], scale, causal)
    out[rank] = (float(np.max(np.abs(o_m - o_ref[0, 0, rank * ns:(rank + 1) * ns]))),
                 float(np.max(np.abs(l_m - l_ref[0, 0, rank * ns:(rank + 1) * ns]))))
    dist.destroy_process_group()


@pytest.mark.parametrize("causal", [False, True])
def test_two_rank_gloo_ring_matches_definition(causal):
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_ring_rank, args=(world, port, causal, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        assert res[r][0] < 1e-12 and res[r][1] < 1e-12
