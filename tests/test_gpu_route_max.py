"""Routing by each KV head's best query head (cfg.route_max) on the GPU.

Against the oracle's route(agg="max") on the GPU's own cache: scores within
1e-5 of their rms, selection bit-exact except near-ties of the beta-th score
(as for the default routing); hsq_decode_step under route_max equals
hsq_route + hsq_decode_attn bit for bit and the oracle's attention on the
GPU's selection within 1e-3 relative L2.
"""

import numpy as np
import pytest

import oracle as O
import workloads as W
from hsq_harness import abi_buffers, ensure_built, oracle_view, rel_l2, sel_mismatch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _workloads():
    tiny = W.get_workload("tiny_1k")
    return {
        "tiny_1k": tiny,
        "qwen3_0p6b_4k": W.get_workload("qwen3_0p6b_4k"),
        "ragged_r5": tiny.with_(name="ragged_r5", B=2, Hq=10, Hkv=2, T=1001, N=8, beta=12, recent=40,
                                marked=17, storage="bf16", key_law="student_t", seed_tag=11),
        "r8_lowrank": tiny.with_(name="r8_lowrank", B=1, Hq=16, Hkv=2, T=600, N=16, beta=30, recent=32,
                                 marked=6, storage="bf16", key_law="lowrank", seed_tag=12),
    }


WL = _workloads()


@pytest.mark.parametrize("name", list(WL))
def test_route_max_parity_and_fallback_step(name):
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    w = WL[name]
    li = W.layer_inputs(w, rope=lambda x, p: O.rope(x, p, w.theta))
    cfg = H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, w.T, max(w.l1_size, 1), w.T + w.steps + 1, w.theta,
                        route_max=True)
    ctx = H.Context(cfg)
    cache = H.allocate_cache(ctx, w.B, w.T)
    H.set_layer_inputs(cache, li.l1_mask, li.signs)
    dt = torch.bfloat16 if w.storage == "bf16" else torch.float32
    K = torch.from_numpy(np.ascontiguousarray(li.K, np.float32)).cuda().to(dt).contiguous()
    V = torch.from_numpy(np.ascontiguousarray(li.V, np.float32)).cuda().to(dt).contiguous()
    H.hsq_encode(ctx, cache, K, V)
    gview = oracle_view(abi_buffers(cache), li, w)
    q, pos = W.queries(w, steps=3)
    near = 0
    for s in range(3):
        qd, pd = torch.from_numpy(q[s]).cuda(), torch.from_numpy(pos[s]).cuda()
        sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
        scores = torch.empty((w.B, w.Hkv, cache.G), dtype=torch.float32, device="cuda")
        H.hsq_route(ctx, cache, qd, pd, sel, scores)
        assert H.hsq_sync_status(ctx) == 0
        osel, oscores = O.route(gview, q[s], pos[s], w.beta, agg="max")
        gs = scores.cpu().numpy()
        fin = np.isfinite(oscores)
        np.testing.assert_array_equal(np.isfinite(gs), fin)
        scale = np.sqrt(np.mean(oscores[fin] ** 2))
        assert np.max(np.abs(gs[fin] - oscores[fin])) <= 1e-5 * scale
        gsel = sel.cpu().numpy()
        for b in range(w.B):
            for h in range(w.Hkv):
                bad, ties = sel_mismatch(gsel[b, h], osel[b, h], oscores[b, h], w.beta)
                assert bad == 0, f"step {s} (b={b}, h={h}): selection differs beyond near-ties"
                near += ties
        # the fused step falls back to route + attention under route_max: same bits
        out_a = torch.empty((w.B, w.Hq, 128), device="cuda")
        H.hsq_decode_attn(ctx, cache, qd, pd, sel, out_a)
        sel2 = torch.empty_like(sel)
        out_s = torch.empty_like(out_a)
        H.hsq_decode_step(ctx, cache, qd, pd, sel2, out_s)
        assert H.hsq_sync_status(ctx) == 0
        assert torch.equal(sel2, sel) and torch.equal(out_s, out_a)
        ref = O.decode_attn(gview, q[s], pos[s], gsel.astype(np.int64))
        err = rel_l2(out_s.cpu().numpy(), ref)
        assert np.all(err <= 1e-3), f"step {s}: rel L2 {err.max():.3e}"
    print(f"[{name}] route_max near-tie groups: {near}")


def test_route_max_is_refused_by_the_noalloc_call():
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    w = WL["tiny_1k"]
    cfg = H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, w.T, w.l1_size, w.T + 8, w.theta, route_max=True)
    ctx = H.Context(cfg)
    cache = H.allocate_cache(ctx, w.B, w.T)
    q = torch.zeros((w.B, w.Hq, 128), device="cuda")
    p = torch.full((w.B,), w.T, dtype=torch.int32, device="cuda")
    sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
    with pytest.raises(H.HSQError) as ei:
        H.hsq_route_noalloc(cfg, cache, q, p, sel)
    assert ei.value.status == 6
