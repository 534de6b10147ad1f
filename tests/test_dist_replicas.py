"""The multi-GPU path is replicas only: each rank runs the whole step on its own GPU and
the benchmark combines the ranks on the host (a barrier around the timed region, the
slowest rank's time, the units of all ranks).  These world-size-2 tests run that host
logic over gloo on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(dist)
        ms = 10.0 + 5.0 * rank                       # rank 1 is the slowest
        ms_max = bench.max_over_ranks(ms, dist)
        value = bench.whole_job_value(1024, 100, world, ms_max)
        bench.barrier(dist)
        q.put((rank, ms_max, value))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_replicas_take_the_slowest_rank(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, ms_max, value in got:
        assert ms_max == 15.0
        assert value == pytest.approx(world * 1024 * 100 / 0.015)


def test_single_process_needs_no_group():
    assert bench.dist_init(1) == (0, 1, None)
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.whole_job_value(10, 2, 1, 1000.0) == pytest.approx(20.0)
