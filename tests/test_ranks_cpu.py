"""The N > 1 bench path (replicas; barrier + max-over-ranks time) on CPU
with two gloo ranks."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    dist.barrier()
    slowest = bench.max_over_ranks(10.0 + 5 * rank, world, "cpu")
    rate = bench.whole_job_rate(60, world, slowest)
    q.put((rank, slowest, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_report_the_slowest_rank():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, slowest, rate in res:
        assert slowest == 15.0                     # max over ranks
        assert rate == pytest.approx(120 / 15.0)   # all ranks' frames / slowest time


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.whole_job_rate(60, 1, 2.0) == 30.0
