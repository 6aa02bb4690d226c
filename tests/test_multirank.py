"""The N > 1 host path of bench.py on CPU: two gloo ranks, barrier and the
max-over-ranks timing, and the whole-job rate (replicas, no collective on the
data path)."""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env() == (world, rank, rank)
    dist.barrier()
    slowest = bench.ranks_max(10.0 + rank)          # each rank's own elapsed ms
    rate = bench.whole_job_rate(448, 100, world, slowest)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, slowest, rate))


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=90) for _ in range(world))
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for rank, slowest, rate in out:
        assert slowest == 11.0
        assert rate == pytest.approx(448 * 100 * 2 / 0.011)


def test_single_process_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.ranks_max(3.5) == 3.5
    assert bench.whole_job_rate(448, 10, 1, 1.0) == pytest.approx(4_480_000.0)
