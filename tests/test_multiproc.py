"""Host logic of bench.py for N > 1 ranks, on CPU with the gloo backend (world size 2).

The forward pass has no cross-GPU exchange: every rank runs its own replica and the job's
throughput is the tokens of all ranks divided by the slowest rank's time. These tests check the
pieces of that logic that do not need a GPU: the max-over-ranks reduction, the barrier, the
whole-job value, and that only rank 0 runs the CPU reference arm.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.dist_barrier(world)
        local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        results[rank] = bench.dist_max(local_ms, world, torch.device("cpu"))
        bench.dist_barrier(world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        mp.start_processes(_worker, args=(world, _free_port(), results), nprocs=world,
                           join=True, start_method="spawn")
        assert dict(results) == {0: 15.0, 1: 15.0}


def test_whole_job_value_counts_every_rank():
    # tokens of all ranks over the slowest rank's time
    assert bench.job_value(tokens_per_step=1000, steps=10, elapsed_ms=20.0, world=4) == \
        pytest.approx(4 * 1000 * 10 / 0.020)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    class A:
        steps, warmup, gpus = 1, 0, 2
    assert bench.run_reference(A, bench.WORKLOADS["tiny"], world=2, rank=1) == 0
    assert capsys.readouterr().out == ""
