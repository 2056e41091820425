"""The N > 1 host path of bench.py on CPU: two gloo ranks.

The path shards into independent replicas (no exchange step), so the only
cross-rank operations are the barrier and the MAX of the per-rank timings;
the reference arm runs on rank 0 alone.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        assert (r, w, lr) == (rank, world, rank)
        # Rank 0 is fast on the first value and slow on the second.
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank], dist, world, "cpu")
        dist.barrier()
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_timings_take_the_slowest_rank():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        assert out[0] == [2.0, 10.0] and out[1] == [2.0, 10.0]


def test_single_rank_keeps_its_values():
    assert bench.max_over_ranks([3.5, 4.5], None, 1, "cpu") == [3.5, 4.5]


def test_replica_throughput_counts_every_rank():
    # Weak scaling: each replica does the same work; the job's throughput is
    # all the units over the slowest rank's time.
    assert bench.job_throughput(1, 1.0e12, 0.5) == 2.0e12
    assert bench.job_throughput(4, 1.0e12, 0.5) == 8.0e12


def test_reference_arm_runs_on_rank_zero_only(capsys):
    class A:
        workload, steps, warmup = "gemm_512", 1, 0
    assert bench.run_reference(A(), rank=1, world=2) is None
    assert capsys.readouterr().out == ""
