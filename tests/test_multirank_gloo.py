"""The benchmark's multi-rank logic on CPU ranks (gloo, world size 2).

With N GPUs the path runs N independent replicas ("replicas only": no data
path collective); the ranks only agree on the job's time, the slowest rank's,
and report the whole job's rate.  Here two CPU processes run that reduction
over gloo on 127.0.0.1, and the reference arm's non-zero rank exits without
work.
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_setup(None) == (world, rank, rank)
        local_ms = [12.5, 40.0][rank]          # rank 1 is the slow one
        total = bench.max_over_ranks(local_ms, world, torch.device("cpu"))
        rate = bench.whole_job_rate(world, 128, 10, total)
        dist.barrier()
        results[rank] = (total, rate)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_whole_job_rate():
    world = 2
    with mp.get_context("spawn").Manager() as m:
        results = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), results), nprocs=world, start_method="spawn",
                           join=True)
        got = dict(results)
    assert got[0] == got[1]
    total, rate = got[0]
    assert total == 40.0
    assert rate == pytest.approx(2 * 128 * 10 / 0.040)


def test_single_rank_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, None) == 3.5
    assert bench.whole_job_rate(1, 128, 10, 1000.0) == pytest.approx(1280.0)


def test_reference_arm_on_a_nonzero_rank_exits_without_work(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    assert bench.bench_reference(bench.parse_args()) == 0
