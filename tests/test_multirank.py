"""The benchmark's N > 1 path on CPU: two gloo ranks, one replica each.

The head shards by requests with no exchange, so the only cross-rank steps are
the barrier and the max over ranks of the step time; the whole-job rate counts
every rank's positions against that max."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, times, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dist.barrier()
    slowest = bench.slowest_rank_ms(times[rank], dist, "cpu")
    rate = bench.job_throughput(8, world, slowest)
    dist.barrier()
    out[rank] = (slowest, rate)
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_replica():
    world = 2
    times = [2.0, 3.5]
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        slowest, rate = out[r]
        assert slowest == 3.5
        assert rate == pytest.approx(8 * world / 3.5e-3)


def test_single_process_is_unchanged():
    import bench
    assert bench.slowest_rank_ms(1.25, None, "cpu") == 1.25
    assert bench.job_throughput(8, 1, 1.0) == pytest.approx(8000.0)
