"""The benchmark's multi-replica aggregation (bench.py --gpus N under
torchrun) on two gloo processes on the CPU: the step time is the maximum
over ranks and the rate counts every replica's work."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 2.0 + 3.0 * rank                       # rank 1 is the slow replica
        worst = bench.max_over_ranks(ms, dist, "cpu")
        rate = bench.whole_job_rate(1e9, world, worst)
        q.put((rank, worst, rate))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, worst, rate in got:
        assert worst == 5.0                          # max over ranks
        assert rate == pytest.approx(1e9 * 2 / 5e-3)  # both replicas' work / slowest time


def test_single_process_defaults():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.whole_job_rate(2e9, 1, 4.0) == pytest.approx(5e11)
