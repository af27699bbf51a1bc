"""The N>1 benchmark path on CPU: two gloo ranks (replicas) time different
amounts, the job time is the slowest rank's and the job throughput counts
every rank's tokens.  No GPU; the path has no collective on its data."""
import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = 10.0 + 5.0 * rank           # rank 1 is slower
        ms = bench.max_over_ranks(my_ms, torch.device("cpu"))
        value = bench.job_throughput(world, 4448, 20, ms)
        results[rank] = (ms, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_slowest_time_and_whole_job_throughput():
    world = 2
    port = 29500 + (os.getpid() % 2000)
    with mp.get_context("spawn").Manager() as m:
        results = m.dict()
        mp.spawn(_rank, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    assert set(res) == {0, 1}
    for ms, value in res.values():
        assert ms == pytest.approx(15.0)
        assert value == pytest.approx(2 * 4448 * 20 / 0.015)


def test_single_process_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5
    assert bench.job_throughput(1, 100, 10, 1000.0) == pytest.approx(1000.0)
