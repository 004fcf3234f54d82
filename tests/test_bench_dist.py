"""bench.py's multi-rank aggregation on CPU: two gloo ranks, each with its own
timed total; both get the slowest rank's time and the whole-job rate."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, totals, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, value = bench.aggregate(totals[rank], 100, world)
        out.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


def test_aggregate_takes_slowest_rank_two_gloo_ranks():
    import torch.multiprocessing as mp
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    totals = [30.0, 45.0]  # ms over 100 steps on each rank
    procs = [ctx.Process(target=_rank, args=(r, 2, port, totals, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in res:
        assert ms == pytest.approx(0.45)
        assert value == pytest.approx(2 * 100 / 0.045)


def test_aggregate_single_rank_is_local():
    sys.path.insert(0, ROOT)
    import bench
    ms, value = bench.aggregate(20.0, 50, 1)
    assert ms == pytest.approx(0.4)
    assert value == pytest.approx(50 / 0.02)
