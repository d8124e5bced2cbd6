"""Replica timing aggregation of bench.py over a world-size-2 process group
(gloo on CPU): the job's time is the slowest rank's, its rate counts every
rank's rows, and a single process is its own maximum.  The step itself has no
exchange, so this is the whole multi-process path."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], "cpu")
        out[rank] = (ms, bench.whole_job_rate(world, 10, 16384, ms))
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world = 2
    times = [12.5, 17.25]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), times, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms, rate = res[rank]
        assert ms == max(times)
        assert rate == pytest.approx(world * 10 * 16384 / (max(times) / 1e3), rel=1e-12)


def test_single_process_is_its_own_max():
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.whole_job_rate(1, 100, 16384, 40.0) == pytest.approx(100 * 16384 / 0.04)
