"""Per-query-head routing (cfg.route_per_head) on the GPU.

Every query head selects its own beta groups and attends with them.  Against
the oracle's route(agg="head") and per-head decode_attn on the GPU's own
cache: scores within 1e-5 of their rms, selections bit-exact except
near-ties of the beta-th score, attention within 1e-3 relative L2; the
fused step equals route + attention; fetch_dequant and the staged attention
path work on the per-head rows; the no-alloc routing call refuses the mode.
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


class Layer:
    def __init__(self, name):
        import torch
        import hierarchical_kv_cache_hsq_gb300 as H
        w = self.w = WL[name]
        self.li = li = W.layer_inputs(w, rope=lambda x, p: O.rope(x, p, w.theta))
        cfg = H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, w.T, max(w.l1_size, 1), w.T + w.steps + 1, w.theta,
                            route_per_head=True)
        self.ctx = H.Context(cfg)
        self.cache = H.allocate_cache(self.ctx, w.B, w.T)
        H.set_layer_inputs(self.cache, li.l1_mask, li.signs)
        dt = torch.bfloat16 if w.storage == "bf16" else torch.float32
        K = torch.from_numpy(np.ascontiguousarray(li.K, np.float32)).cuda().to(dt).contiguous()
        V = torch.from_numpy(np.ascontiguousarray(li.V, np.float32)).cuda().to(dt).contiguous()
        H.hsq_encode(self.ctx, self.cache, K, V)
        self.bufs = abi_buffers(self.cache)
        self.gview = oracle_view(self.bufs, li, w)


_L = {}


def layer(name):
    if name not in _L:
        _L[name] = Layer(name)
    return _L[name]


@pytest.mark.parametrize("name", list(WL))
def test_per_head_route_and_step_parity(name):
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    L = layer(name)
    w = L.w
    q, pos = W.queries(w, steps=3)
    near, worst = 0, 0.0
    for s in range(3):
        qd, pd = torch.from_numpy(q[s]).cuda(), torch.from_numpy(pos[s]).cuda()
        sel = torch.empty((w.B, w.Hq, w.beta), dtype=torch.int32, device="cuda")
        scores = torch.empty((w.B, w.Hq, L.cache.G), dtype=torch.float32, device="cuda")
        H.hsq_route(L.ctx, L.cache, qd, pd, sel, scores)
        assert H.hsq_sync_status(L.ctx) == 0
        osel, oscores = O.route(L.gview, q[s], pos[s], w.beta, agg="head")
        gs = scores.cpu().numpy()
        fin = np.isfinite(oscores)
        np.testing.assert_array_equal(np.isfinite(gs), fin)
        assert np.max(np.abs(gs[fin] - oscores[fin])) <= 1e-5 * np.sqrt(np.mean(oscores[fin] ** 2))
        gsel = sel.cpu().numpy()
        for b in range(w.B):
            for j in range(w.Hq):
                row = gsel[b, j]
                valid = row[row >= 0]
                assert np.all(np.diff(valid) > 0) and np.all(row[len(valid):] == -1)
                bad, diff = sel_mismatch(row, osel[b, j], oscores[b, j], w.beta)
                assert bad == 0, f"step {s} (b={b}, head {j}): selection differs beyond near-ties"
                near += diff
        # heads of one KV head select differently (the mode is not the shared selection)
        if w.Hq > w.Hkv:
            r = w.Hq // w.Hkv
            assert any(not np.array_equal(gsel[0, 0], gsel[0, j]) for j in range(1, r))
        out = torch.empty((w.B, w.Hq, 128), device="cuda")
        sel_s = torch.empty_like(sel)
        H.hsq_decode_step(L.ctx, L.cache, qd, pd, sel_s, out)
        out_a = torch.empty_like(out)
        H.hsq_decode_attn(L.ctx, L.cache, qd, pd, sel, out_a)
        assert H.hsq_sync_status(L.ctx) == 0
        assert torch.equal(sel_s, sel)
        assert np.all(rel_l2(out.cpu().numpy(), out_a.cpu().numpy()) <= 1e-5)
        ref = O.decode_attn(L.gview, q[s], pos[s], gsel.astype(np.int64))
        err = rel_l2(out.cpu().numpy(), ref)
        worst = max(worst, float(err.max()))
        assert np.all(err <= 1e-3), f"step {s}: rel L2 {err.max():.3e}"
    print(f"[{name}] per-head near-tie differences {near}, attention rel L2 {worst:.2e}")


@pytest.mark.parametrize("name", ["tiny_1k", "ragged_r5"])
def test_per_head_fetch_and_staged_attention(name):
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    L = layer(name)
    w = L.w
    q, pos = W.queries(w, steps=1)
    qd, pd = torch.from_numpy(q[0]).cuda(), torch.from_numpy(pos[0]).cuda()
    sel = torch.empty((w.B, w.Hq, w.beta), dtype=torch.int32, device="cuda")
    H.hsq_route(L.ctx, L.cache, qd, pd, sel)
    shape = (w.B, w.Hq, w.beta, w.N, 128)
    k, v = torch.empty(shape, device="cuda"), torch.empty(shape, device="cuda")
    valid = torch.empty(shape[:-1], dtype=torch.uint8, device="cuda")
    H.hsq_fetch_dequant(L.ctx, L.cache, sel, k, v, valid)
    assert H.hsq_sync_status(L.ctx) == 0
    gsel = sel.cpu().numpy().astype(np.int64)
    r = w.Hq // w.Hkv
    kk, vv, va = k.cpu().numpy(), v.cpu().numpy(), valid.cpu().numpy().astype(bool)
    st = L.cache.view("staging").cpu().numpy()
    assert st.shape[1] == w.Hq
    for h in range(w.Hkv):
        # the oracle's fetch maps selection row i to KV head i: give every KV head
        # query head j's row and compare KV head h, the one j belongs to
        for j in range(h * r, (h + 1) * r):
            ok1, ov1, va1 = O.fetch_dequant(L.gview, np.repeat(gsel[:, j:j + 1], w.Hkv, axis=1))
            nz = np.linalg.norm(ok1[:, h], axis=-1) > 0
            assert np.all(rel_l2(kk[:, j], ok1[:, h])[nz] <= 1e-5)
            assert np.all(rel_l2(vv[:, j], ov1[:, h])[nz] <= 1e-5)
            np.testing.assert_array_equal(va[:, j], va1[:, h])
            for b in range(w.B):
                for i, g in enumerate(gsel[b, j]):
                    if g >= 0:
                        np.testing.assert_array_equal(st[b, j, i], L.bufs["l3"][b, h, g])
    # attention from the staged records equals attention gathering them itself
    out_g = torch.empty((w.B, w.Hq, 128), device="cuda")
    out_s = torch.empty_like(out_g)
    H.hsq_decode_attn(L.ctx, L.cache, qd, pd, sel, out_g)
    H.hsq_decode_attn(L.ctx, L.cache, qd, pd, sel, out_s, flags=H.HSQ_ATTN_FROM_STAGING)
    assert H.hsq_sync_status(L.ctx) == 0
    assert np.all(rel_l2(out_s.cpu().numpy(), out_g.cpu().numpy()) <= 1e-6)


def test_per_head_is_refused_by_the_noalloc_call():
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    L = layer("tiny_1k")
    w = L.w
    q = torch.zeros((w.B, w.Hq, 128), device="cuda")
    p = torch.full((w.B,), w.T, dtype=torch.int32, device="cuda")
    sel = torch.empty((w.B, w.Hq, w.beta), dtype=torch.int32, device="cuda")
    with pytest.raises(H.HSQError) as ei:
        H.hsq_route_noalloc(L.ctx.cfg, L.cache, q, p, sel)
    assert ei.value.status == 6
