"""The multi-rank host logic of the benchmark, with two gloo ranks on CPU:
the timed region's barriers and the max over ranks of the elapsed time, and
the weak-scaling throughput computed from it."""
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


def _rank(rank, world, port, elapsed, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dist.barrier()
    mx = bench.max_over_ranks(elapsed[rank], world)
    out[rank] = mx
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world, port = 2, _free_port()
    elapsed = [12.5, 40.25]
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank, args=(world, port, elapsed, out), nprocs=world, join=True)
    assert out[0] == out[1] == 40.25


def test_weak_scaling_throughput():
    # 1.95 GB per rank per step, 10 steps, slowest rank 4 ms -> 2 ranks * 19.5 GB / 4 ms
    assert bench.weak_scaling_tbps(1_949_696_000, 10, 2, 4.0) == pytest.approx(9.74848)
    assert bench.weak_scaling_tbps(1_949_696_000, 10, 1, 4.0) == pytest.approx(4.87424)
    assert bench.max_over_ranks(3.5, 1) == 3.5
