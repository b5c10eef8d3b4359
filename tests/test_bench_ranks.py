"""Host logic of the multi-replica benchmark (no GPU): two gloo ranks on
the CPU combine their step times with a max all-reduce, and the whole-job
throughput counts every replica's elements over the slowest replica's time.
"""

import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 5.0 * rank  # rank 1 is the slow one
        slowest = bench.max_over_ranks(dist, mine)
        out[rank] = (slowest, bench.job_gelem_s(world, 1_000_000, 4, slowest))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time_and_count_both():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    slowest, value = res[0]
    assert slowest == 15.0
    # 2 replicas x 1e6 elements x 4 steps in 15 ms
    assert value == pytest.approx(2 * 1_000_000 * 4 / 15e-3 / 1e9)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(None, 3.5) == 3.5
    assert bench.job_gelem_s(1, 524288, 200, 10.0) == pytest.approx(524288 * 200 / 10e-3 / 1e9)
