"""The routing entry point that allocates no device memory.

Callers that cannot call cudaMalloc (a runtime that owns all device memory
through its own pool, or one that must not let a library call synchronise
the device) use hsq_route_noalloc, whose scratch is a fixed array inside the
library.  This file is collected last so that a run stopping at the first
failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest

import oracle as O
import workloads as W
from hsq_harness import abi_buffers, ensure_built, gpu_encode, make_ctx, oracle_view, sel_mismatch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny_1k", "qwen3_0p6b_4k"])
def test_route_noalloc_matches_route_on_consecutive_calls(name):
    import torch
    ensure_built()
    import hierarchical_kv_cache_hsq_gb300 as H
    w = W.get_workload(name)
    li = W.layer_inputs(w, rope=lambda x, p: O.rope(x, p, w.theta))
    ctx = make_ctx(w)
    cache = gpu_encode(ctx, w, li)
    gview = oracle_view(abi_buffers(cache), li, w)
    q, pos = W.queries(w, steps=2)
    for s in range(2):  # two calls in a row: the shared scratch keeps the previous call's contents
        qd, pd = torch.from_numpy(q[s]).cuda(), torch.from_numpy(pos[s]).cuda()
        ref = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
        scores = torch.empty((w.B, w.Hkv, cache.G), dtype=torch.float32, device="cuda")
        H.hsq_route(ctx, cache, qd, pd, ref, scores)
        got = torch.full((w.B, w.Hkv, w.beta), -7, dtype=torch.int32, device="cuda")
        H.hsq_route_noalloc(ctx.cfg, cache, qd, pd, got)
        torch.cuda.synchronize()
        r, g = ref.cpu().numpy(), got.cpu().numpy()
        # the float64 oracle on the same cache decides which differences are near-ties
        osel, oscores = O.route(gview, q[s], pos[s], w.beta)
        for b in range(w.B):
            for h in range(w.Hkv):
                valid = g[b, h][g[b, h] >= 0]
                assert np.all(np.diff(valid) > 0) and np.all(g[b, h][len(valid):] == -1)
                bad, _ = sel_mismatch(g[b, h], osel[b, h], oscores[b, h], w.beta)
                assert bad == 0, f"call {s}: selection differs from the oracle beyond near-ties at (b={b}, h={h})"
                bad, _ = sel_mismatch(g[b, h], r[b, h], oscores[b, h], w.beta)
                assert bad == 0, f"call {s}: selection differs from hsq_route beyond near-ties at (b={b}, h={h})"
    ctx.close()


def test_route_noalloc_clamps_positions_like_hsq_route():
    """A position outside [0, max_pos) routes as the nearest valid position
    (hsq_route clamps it the same way and also flags it)."""
    import torch
    ensure_built()
    import hierarchical_kv_cache_hsq_gb300 as H
    w = W.get_workload("tiny_1k")
    li = W.layer_inputs(w)
    ctx = make_ctx(w)
    cache = gpu_encode(ctx, w, li)
    q, _ = W.queries(w, steps=1)
    qd = torch.from_numpy(q[0]).cuda()
    max_pos = ctx.cfg.max_pos
    outs = {}
    for p in (-5, 0, max_pos - 1, max_pos + 50):
        got = torch.full((w.B, w.Hkv, w.beta), -7, dtype=torch.int32, device="cuda")
        H.hsq_route_noalloc(ctx.cfg, cache, qd, torch.full((w.B,), p, dtype=torch.int32, device="cuda"), got)
        outs[p] = got.cpu().numpy()
    assert np.array_equal(outs[-5], outs[0])
    assert np.array_equal(outs[max_pos + 50], outs[max_pos - 1])
    assert not np.array_equal(outs[0], outs[max_pos - 1])
    ctx.close()


def test_route_noalloc_rejects_caches_above_its_scratch():
    ensure_built()
    import hierarchical_kv_cache_hsq_gb300 as H
    lib = H.load_library()
    # 16 x 8 heads x 8192 groups of float32 scores = 4 MiB, plus the tickets: over the limit
    cfg = H.make_config(32, 8, 8, 48, 16, 65536, 100, 70000)
    c = H._binding.hsq_cache(B=16, T=65536)
    for name in H.BUFFERS + ["signs"]:
        setattr(c, name, 256)   # never dereferenced: the size check comes first
    buf = ctypes.c_void_p(256)
    st = lib.hsq_route_noalloc(ctypes.byref(cfg), ctypes.byref(c), buf, buf, buf, None)
    assert st == H._binding.HSQ_ERR_INVALID
    assert b"4 MiB" in lib.hsq_last_error(None)
