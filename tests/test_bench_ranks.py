"""Multi-rank logic of bench.py on CPU: two gloo ranks, no GPU.

Each rank of a multi-GPU bench run is an independent replica of the whole round (weak scaling).
What the ranks share is only the timing: the job's time is the slowest rank's, and the job's
throughput counts the units of every rank over that time. These tests run that arithmetic and
the reference arm's rank gate in two real processes joined by a gloo process group.
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
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        # rank-dependent durations: rank 1 is the slow one for the first, rank 0 for the second
        times = bench.job_times([1.0 + r, 3.0 - r], "cpu")
        rate = bench.job_rate(2048 * 10, w, times[0])
        seed = bench.replica_seed(7, r)

        class Args:
            warmup, steps, workload = 3, 1, 1
        # the reference arm does its work on rank 0 only; other ranks return at once
        ref = bench.bench_reference(Args()) if r != 0 else "skipped"
        out[r] = (r, w, local, times, rate, seed, ref)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_share_max_time_and_count_all_units():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    assert sorted(res) == [0, 1]
    for r in (0, 1):
        rank, w, local, times, rate, seed, ref = res[r]
        assert (rank, w, local) == (r, 2, r)
        assert times == [2.0, 3.0]                 # max over ranks of each duration
        assert rate == pytest.approx(2 * 2048 * 10 / 2.0)
        assert seed == 7 + 1000 * r                # each replica draws its own noise
    assert res[1][6] is None                       # reference arm: rank 1 did no work
    assert res[0][5] != res[1][5]


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_times([1.5, 2.5], "cpu") == [1.5, 2.5]
    assert bench.job_rate(100.0, 1, 2.0) == 50.0
