"""The N > 1 path of bench.py on CPU: two gloo ranks on 127.0.0.1 exchange
their timings; both see the maximum, and the whole-job value counts the work
of every rank over the slowest rank's time (weak scaling, no data-path
collective)."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [10.0 + rank, 20.0 - rank]
        got = bench.max_over_ranks(mine, dist)
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_two_ranks_share_the_maximum():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    assert out[0] == out[1] == [11.0, 20.0]


def test_whole_job_value_is_weak_scaling():
    import bench
    one = bench.whole_job_tflops(1e12, 1, 2.0)
    two = bench.whole_job_tflops(1e12, 2, 2.0)
    assert abs(one - 500.0) < 1e-9 and abs(two - 2 * one) < 1e-9


def test_single_process_needs_no_process_group():
    import bench
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
