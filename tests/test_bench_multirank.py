"""bench.py's multi-rank arithmetic on CPU with two gloo ranks: the job's time is the slowest
rank's (max over ranks, taken after a barrier), and the whole-job rate counts every rank's
units (weak scaling: each rank runs the full per-GPU workload, with no collective on the
data path).  Launched with spawn, addresses on 127.0.0.1."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    try:
        elapsed = [0.50, 0.80, 0.65, 0.70][rank]  # this rank's own timed region, seconds
        dist.barrier()
        t = bench.max_over_ranks(elapsed, world, "cpu")
        e2e = bench.max_over_ranks(elapsed * 2.0, world, "cpu")
        results[rank] = (t, e2e, bench.job_rate(1.5e9, 100, world, t))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_max_over_ranks_and_job_rate_gloo(world):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True,
                           start_method="spawn")
        got = dict(results)
    slowest = max([0.50, 0.80, 0.65, 0.70][:world])
    assert sorted(got) == list(range(world))
    for rank, (t, e2e, rate) in got.items():
        assert t == slowest, (rank, t)
        assert e2e == 2.0 * slowest
        assert rate == pytest.approx(1.5e9 * 100 * world / slowest)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks(0.25, 1, "cpu") == 0.25
    assert bench.job_rate(10.0, 4, 1, 2.0) == 20.0
