"""Replicas in several processes (torch.distributed with gloo on the CPU, two
ranks): the benchmark takes every timing's maximum over the ranks, and the
whole-job rate counts every rank's tokens over the slowest rank's time."""
import os
import socket
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank's own step time and end-to-end time; rank r is slowest on
        # the first, fastest on the second
        got = bench.max_over_ranks([10.0 + rank, 30.0 - rank], dist, "cpu")
        assert got == [10.0 + (world - 1), 30.0], got
        rate = bench.whole_job_rate(1000, 5, world, got[0])
        assert abs(rate - 1000 * 5 * world / (got[0] / 1e3)) < 1e-6 * rate
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    mp.spawn(_worker, args=(2, _free_port()), nprocs=2, join=True)


def test_one_process_keeps_its_times():
    assert bench.max_over_ranks([1.5, 2.5], None, "cpu") == [1.5, 2.5]
    assert bench.whole_job_rate(8192, 20, 1, 100.0) == 8192 * 20 / 0.1
