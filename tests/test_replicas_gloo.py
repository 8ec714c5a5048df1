"""The N-replica path of bench.py on CPU: two gloo ranks, each with its own
step time; the reported time is the maximum over ranks and the value counts
the units of all ranks (-m "not gpu")."""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_max, value = bench.aggregate(10.0 + rank, 4096, torch.device("cpu"))
        q.put((rank, ms_max, value))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_and_whole_job_value(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    slowest = 10.0 + (world - 1)
    for rank, ms_max, value in got:
        assert ms_max == slowest
        assert value == pytest.approx(world * 4096 / (slowest / 1e3))


def test_single_process_value():
    sys.path.insert(0, ROOT)
    import bench
    ms_max, value = bench.aggregate(8.0, 1000, torch.device("cpu"))
    assert ms_max == 8.0 and value == pytest.approx(125000.0)
