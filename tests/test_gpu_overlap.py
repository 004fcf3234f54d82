"""Overlapped decode launches (hsq_config.overlap_launch): the decode kernels
are launched with programmatic stream serialization, so a launch may be
scheduled while the stream's preceding kernel still runs and waits for it
before its first global access.  The results must be the bits of ordinary
stream order:
  * three layers' decode steps back to back, direct calls and one captured
    CUDA graph replayed with new queries, for the fused step and for the
    route + attention path (route_max);
  * a growing cache, where every step's decode launch follows the append
    kernel that wrote the token it reads, and a torch kernel that wrote its
    query.
"""

import numpy as np
import pytest

import oracle as O
import workloads as W
from hsq_harness import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _layers(H, torch, w, li, ctx, n):
    K = torch.from_numpy(li.K).cuda().to(torch.bfloat16).contiguous()
    V = torch.from_numpy(li.V).cuda().to(torch.bfloat16).contiguous()
    out = []
    for l in range(n):
        mask, signs = (li.l1_mask, li.signs) if l == 0 else W.layer_meta(w, l)
        c = H.allocate_cache(ctx, w.B, w.T, with_staging=False)
        H.set_layer_inputs(c, mask, signs)
        H.hsq_encode(ctx, c, K, V)
        out.append(c)
    return out


@pytest.mark.parametrize("route_max", [False, True])
def test_overlapped_layers_equal_stream_order(route_max):
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    w = W.get_workload("qwen3_0p6b_4k").with_(steps=3)
    li = W.layer_inputs(w, rope=lambda x, p: O.rope(x, p, w.theta))
    q, pos = W.queries(w, steps=w.steps)
    qd, pd = torch.from_numpy(q).cuda(), torch.from_numpy(pos).cuda()
    runs = {}
    for overlap in (False, True):
        ctx = H.Context(H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, w.T, w.l1_size, w.T + w.steps + 1, w.theta,
                                      route_max=route_max, overlap_launch=overlap))
        layers = _layers(H, torch, w, li, ctx, 3)
        sels = [torch.full((w.B, w.Hkv, w.beta), -7, dtype=torch.int32, device="cuda") for _ in layers]
        outs = [torch.full((w.B, w.Hq, 128), float("nan"), device="cuda") for _ in layers]
        q_in, p_in = torch.empty_like(qd[0]), torch.empty_like(pd[0])

        def step():
            for c, sel, o in zip(layers, sels, outs):
                H.hsq_decode_step(ctx, c, q_in, p_in, sel, o)

        got = []
        for s in range(w.steps):  # direct calls
            q_in.copy_(qd[s])
            p_in.copy_(pd[s])
            step()
            got.append([(x.clone(), y.clone()) for x, y in zip(sels, outs)])
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        for s in range(w.steps):  # the captured step, replayed
            q_in.copy_(qd[s])
            p_in.copy_(pd[s])
            g.replay()
            got.append([(x.clone(), y.clone()) for x, y in zip(sels, outs)])
        torch.cuda.synchronize()
        assert H.hsq_sync_status(ctx) == 0
        runs[overlap] = got
        del g
        ctx.close()
    for a, b in zip(runs[False], runs[True]):
        for (sa, oa), (sb, ob) in zip(a, b):
            assert torch.equal(sa, sb) and torch.equal(oa, ob)
    assert all(np.isfinite(o.cpu().numpy()).all() for _, o in runs[True][0])
    # graph replay equals the direct calls of the same step
    for s in range(w.steps):
        for (sa, oa), (sb, ob) in zip(runs[True][s], runs[True][w.steps + s]):
            assert torch.equal(sa, sb) and torch.equal(oa, ob)


def test_overlapped_decode_after_append_equals_stream_order():
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    T0, grow = 1000, 24
    tiny = W.get_workload("tiny_1k")
    w = tiny.with_(name="overlap_grow", B=2, Hq=4, Hkv=2, T=T0 + grow, N=16, beta=8, sinks=4, recent=64,
                   marked=32, storage="bf16", seed_tag=77)
    li = W.layer_inputs(w)
    pos = np.arange(T0)
    mask0 = (li.l1_mask[:, :T0] & (pos >= 4) & (pos < T0 - 64)) | (pos < 4) | (pos >= T0 - 64)
    rng = np.random.default_rng(5)
    qs = rng.standard_normal((grow, w.B, w.Hq, 128)).astype(np.float32)
    K = torch.from_numpy(np.ascontiguousarray(li.K, np.float32)).cuda().to(torch.bfloat16)
    V = torch.from_numpy(np.ascontiguousarray(li.V, np.float32)).cuda().to(torch.bfloat16)
    runs = {}
    for overlap in (False, True):
        ctx = H.Context(H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, w.T, 4 + 32 + 64, w.T + 8, w.theta,
                                      sinks=4, recent=64, overlap_launch=overlap))
        c = H.allocate_cache(ctx, w.B, T0, with_staging=False, t_cap=w.T)
        H.set_layer_inputs(c, mask0, li.signs)
        H.hsq_encode(ctx, c, K[:, :, :T0].contiguous(), V[:, :, :T0].contiguous())
        qh = torch.from_numpy(qs).cuda()
        q_in = torch.empty_like(qh[0])
        p_in = torch.empty((w.B,), dtype=torch.int32, device="cuda")
        sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
        o = torch.empty((w.B, w.Hq, 128), device="cuda")
        got = []
        for i in range(grow):
            p_in.fill_(T0 + i)
            H.hsq_append(ctx, c, K[:, :, T0 + i].contiguous(), V[:, :, T0 + i].contiguous())
            torch.mul(qh[i], 1.0, out=q_in)  # a kernel writes the query right before the decode launch
            H.hsq_decode_step(ctx, c, q_in, p_in, sel, o)
            got.append((sel.clone(), o.clone()))
        torch.cuda.synchronize()
        assert H.hsq_sync_status(ctx) == 0
        runs[overlap] = got
        ctx.close()
    for (sa, oa), (sb, ob) in zip(runs[False], runs[True]):
        assert torch.equal(sa, sb) and torch.equal(oa, ob)
    assert np.isfinite(runs[True][-1][1].cpu().numpy()).all()
