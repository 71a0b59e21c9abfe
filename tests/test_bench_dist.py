"""The benchmark's multi-rank logic on CPU with two gloo ranks: the step time is the
slowest rank's and the job throughput counts every rank's batch (weak scaling)."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.max_over_ranks(1.0 + rank, dist, device="cpu")
    dist.barrier()
    out[rank] = t
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1] == 2.0


def test_job_throughput_is_weak_scaling():
    # 2 ranks x batch 1, 10 steps in 0.5 s -> 40 tokens/s
    assert bench.job_throughput(2, 1, 0.5, 10) == pytest.approx(40.0)
    assert bench.job_throughput(1, 32, 1.0, 4) == pytest.approx(128.0)
