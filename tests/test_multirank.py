"""The benchmark's multi-rank aggregation on CPU: two gloo ranks report
different step times; every rank must see the slowest one, and the job's
throughput counts both ranks' tokens over that time."""
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


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 1.5 + rank                      # rank 1 is the slow one
        got = bench.max_over_ranks(ms, torch.device("cpu"))
        out[rank] = (got, bench.job_value(world, 90, got))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_max_over_ranks_and_job_value_gloo_two_ranks():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    assert out[0] == out[1]
    ms, v = out[0]
    assert ms == 2.5
    assert v == pytest.approx(2 * 90 / 2.5e-3)


def test_single_process_is_identity():
    assert bench.max_over_ranks(3.25, torch.device("cpu")) == 3.25
    assert bench.job_value(1, 90, 2.0) == pytest.approx(45000.0)
