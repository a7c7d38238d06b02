"""The benchmark's multi-rank host logic on CPU: two gloo ranks.

The path shards by sequence with no exchange; the only collective is the
max-over-ranks of the timings after the timed region, and the whole-job value
of weak scaling is world_size x the per-rank bytes over that time.  The
reference arm does its work on rank 0 only.
"""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench._dist_env()
        # per-rank timings (ms): rank 1 is slower in the first, rank 0 in the second
        got = bench._max_over_ranks([1.0 + rank, 5.0 - rank], dist, torch.device("cpu"))
        value = bench._weak_value(ws, 1_000_000_000, got[0])
        results[rank] = (ws, r, local, got, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_weak_scale_the_bytes():
    world, port = 2, _free_port()
    results = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
    for rank in range(world):
        ws, r, local, got, value = results[rank]
        assert (ws, r, local) == (2, rank, rank)
        assert got == [2.0, 5.0]             # the slowest rank of each timing
        assert value == pytest.approx(2 * 1.0 / 2.0e-3)  # 2 ranks x 1 GB in 2 ms = 1000 GB/s


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench._max_over_ranks([3.0, 4.0], None, None) == [3.0, 4.0]
    assert bench._weak_value(1, 2_000_000_000, 1.0) == pytest.approx(2000.0)


def test_reference_arm_works_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class Args:  # the reference arm returns before touching them on rank 1
        pass

    assert bench.run_reference(Args()) is None
    assert capsys.readouterr().out == ""
