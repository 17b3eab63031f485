"""The multi-GPU path of the benchmark is N independent replicas (the decoder does not shard):
its only cross-rank steps are the barrier and the maximum of the timed region over ranks.  Both
run here as two gloo ranks on the CPU."""
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


def _rank(rank: int, world: int, port: int, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 5.0 * rank          # rank 1 is the slower replica
        job = bench.job_time_ms(mine, world)
        dist.barrier()
        out[rank] = job
    finally:
        dist.destroy_process_group()


def test_job_time_is_max_over_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
        assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_rank_and_whole_job_value():
    assert bench.job_time_ms(12.5, 1) == 12.5
    # 2 replicas, 100 steps of one token each in 120 ms: 0.6 ms of job time per token
    assert bench.job_value_us_per_token(120.0, 100, 1, 2) == pytest.approx(600.0)
    assert bench.job_value_us_per_token(120.0, 100, 8, 1) == pytest.approx(150.0)
