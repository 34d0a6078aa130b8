"""bench.py's multi-rank logic on CPU: two gloo ranks, the job time is the slowest rank's, the value is the
aggregate over ranks, and only rank 0 runs and prints the reference arm."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = bench.max_over_ranks(times[rank], dist, "cpu")
        value = bench.job_tflops(world, 1e12, ms)
        out[rank] = (ms, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    times = [3.0, 5.0]
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, times, out), nprocs=world, join=True)
    for r in range(world):
        ms, value = out[r]
        assert ms == 5.0                                   # max over ranks, on every rank
        assert value == pytest.approx(2 * 1e12 / 5e-3 / 1e12)  # both ranks' work over the slowest time


def test_single_rank_is_unchanged():
    assert bench.max_over_ranks(2.5) == 2.5
    assert bench.job_tflops(1, 2e12, 1000.0) == pytest.approx(2.0)


def test_reference_arm_other_ranks_do_nothing():
    class A:
        workload, warmup, steps, gpus = "cfg2", 1, 1, 2
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.reference_arm(A, rank=1)
    assert buf.getvalue() == ""
