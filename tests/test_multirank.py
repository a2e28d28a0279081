"""The benchmark's multi-GPU path on CPU ranks (gloo, world size 2): each rank runs its own
batch against replicated weights, so the only collective is the max of the per-rank step
times, and the whole-job value is world x (work per rank) / (slowest rank's time)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        slowest = bench.max_over_ranks(times[rank], world, "cpu")
        value = bench.aggregate_tops(world, 2.0 * 4096 * 8192 * 28672, slowest)
        dist.barrier()
        out[rank] = (slowest, value)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_with_two_gloo_ranks():
    world, port = 2, _free_port()
    times = [1.25, 1.5]                                  # rank 1 is the slower one
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_rank_main, args=(world, port, times, out), nprocs=world, start_method="spawn", join=True)
    ops = 2.0 * 4096 * 8192 * 28672
    for rank in range(world):
        slowest, value = out[rank]
        assert slowest == 1.5                            # every rank sees the max
        assert value == pytest.approx(world * ops / 1.5e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, 1, "cpu") == 2.5
    assert bench.aggregate_tops(1, 1e12, 1000.0) == pytest.approx(1.0)
