"""Host logic of the multi-rank bench (world size 2, gloo on CPU): the job's
time is the slowest rank's, and the job's throughput counts every rank's
units (weak scaling)."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        slowest = bench.max_over_ranks(times[rank], dist, torch.device("cpu"))
        rate = bench.job_rate(1000, world, slowest)
        results[rank] = (slowest, rate)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_rate_gloo():
    world = 2
    times = [2.5, 4.0]                     # ms per step on each rank
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), times, results), nprocs=world, join=True)
        got = dict(results)
    assert sorted(got) == [0, 1]
    for rank in range(world):
        slowest, rate = got[rank]
        assert slowest == 4.0
        assert rate == pytest.approx(2 * 1000 / 4.0e-3)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.25, None, None) == 3.25
    assert bench.job_rate(10, 1, 2.0) == pytest.approx(5000.0)
