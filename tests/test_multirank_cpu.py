"""The multi-rank path of bench.py on CPU: two gloo ranks report different timings; the job
time is the slowest rank's and the throughput counts both replicas."""

import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = [10.0 + rank, 5.0 - rank, 1.0, 2.0 * (rank + 1)]
    got = bench.ranks_max(mine, world, "cpu")
    dist.barrier()
    out[rank] = got
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    expect = [11.0, 5.0, 1.0, 4.0]
    assert res[0] == expect and res[1] == expect


def test_job_throughput_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.ranks_max([1.0, 2.0], 1) == [1.0, 2.0]
    assert bench.job_throughput(3.85e12, 1, 5.0) == pytest.approx(770.0)
    assert bench.job_throughput(3.85e12, 4, 5.0) == pytest.approx(3080.0)
