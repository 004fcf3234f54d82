"""bench.py host logic on CPU: the multi-rank aggregation (two gloo ranks, each with its own
timed total; both get the slowest rank's time and the whole-job rate) and the
per-layer byte counts of the multi-layer mode."""

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


def test_layer_bytes_counts_every_sequence_and_head():
    import bench
    import workloads as W
    w = W.get_workload("qwen3_4b_b16_8k")
    l1 = [213] * w.B
    ne = [1000] * w.B
    hbm, link = bench.layer_bytes(w, 48, l1, ne)
    # 68 B per 4-bit entry and 52 B per 3-bit summary, keys and values, per KV head
    assert hbm == w.Hkv * w.B * (213 * 2 * 68 + 1000 * 2 * 52)
    # whole group records of N tokens, 136 B each, beta per (sequence, KV head)
    assert link == w.B * w.Hkv * 48 * w.N * 136
    # uneven sequences are summed, not multiplied from the first
    hbm2, _ = bench.layer_bytes(w, 48, [0] * (w.B - 1) + [213], [0] * (w.B - 1) + [1000])
    assert hbm2 == w.Hkv * (213 * 2 * 68 + 1000 * 2 * 52)


def test_layer_meta_matches_layer_inputs():
    import numpy as np
    import workloads as W
    w = W.get_workload("tiny_1k")
    li = W.layer_inputs(w, layer=2)
    mask, signs = W.layer_meta(w, layer=2)
    np.testing.assert_array_equal(mask, li.l1_mask)
    np.testing.assert_array_equal(signs, li.signs)
    m3, s3 = W.layer_meta(w, layer=3)
    assert not np.array_equal(s3, signs) or not np.array_equal(m3, mask)
