"""Host logic of a multi-rank bench run on CPU: two gloo ranks (independent
replicas, weak scaling) agree on the slowest rank's time and the whole-job
throughput counts the work of both.  No GPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], world, torch.device("cpu"))
        out[rank] = (ms, bench.job_tflops(world, 2.0e12, ms))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_max_and_aggregate():
    world, times = 2, [7.5, 9.0]
    out = mp.get_context("spawn").Manager().dict()   # no fork of this (threaded) test process
    mp.spawn(_rank, args=(world, _free_port(), times, out), nprocs=world, join=True)
    for r in range(world):
        ms, value = out[r]
        assert ms == 9.0                                # the slowest rank's time on every rank
        assert value == pytest.approx(2 * 2.0e12 / 9.0e-3 / 1e12)


def test_single_rank_passthrough():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1, torch.device("cpu")) == 3.25
    assert bench.job_tflops(1, 1.0e12, 1.0) == pytest.approx(1000.0)
