"""TQ-QKV (cfg.qjl: a 1-bit sketch of every 4-bit key's residual and the
logit correction it carries) on the GPU.

Against the oracle on the same seeded inputs and sketch matrix:
  * sketch bits of the L3 and L1 keys bit-exact except rows whose projection
    S_i . rho lies within 1e-4 |S_i| |rho| of zero (counted), residual norms
    within 1e-4 relative -- taken against the residuals of the GPU's own
    codes (oracle.key_residuals), so a quantiser near-tie cannot cascade;
  * the fused decode step equal to route + attention, and its attention
    within 1e-3 relative L2 of the oracle's on the GPU's cache, sketches and
    selection, and measurably different from the TQ-KV output of the same cache;
  * hsq_append refuses the mode.
"""

import numpy as np
import pytest

import oracle as O
import workloads as W
from hsq_harness import abi_buffers, ensure_built, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _workloads():
    tiny = W.get_workload("tiny_1k")
    return {
        "tiny_1k": tiny,
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
        self.S = W.qjl_matrix(w)
        cfg = H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, w.T, max(w.l1_size, 1), w.T + w.steps + 1, w.theta,
                            qjl=True)
        self.ctx = H.Context(cfg)
        self.cache = H.allocate_cache(self.ctx, w.B, w.T)
        H.set_layer_inputs(self.cache, li.l1_mask, li.signs)
        H.set_qjl_matrix(self.cache, self.S)
        dt = torch.bfloat16 if w.storage == "bf16" else torch.float32
        K = torch.from_numpy(np.ascontiguousarray(li.K, np.float32)).cuda().to(dt).contiguous()
        V = torch.from_numpy(np.ascontiguousarray(li.V, np.float32)).cuda().to(dt).contiguous()
        H.hsq_encode(self.ctx, self.cache, K, V)
        assert H.hsq_sync_status(self.ctx) == 0
        self.bufs = abi_buffers(self.cache)
        for n in ("l1_qs", "l1_qn", "l3_qs", "l3_qn"):
            self.bufs[n] = self.cache.view(n).cpu().numpy()
        self.bufs["l1_qs"] = self.bufs["l1_qs"].view(np.uint32)
        self.bufs["l3_qs"] = self.bufs["l3_qs"].view(np.uint32)
        self.gview = O.cache_from_abi(self.bufs, li.l1_mask, li.signs, w.N, w.T, w.theta, qjl_S=self.S)
        # the same codes without the sketches: the TQ-KV reading of this cache
        self.plain_view = O.cache_from_abi(self.bufs, li.l1_mask, li.signs, w.N, w.T, w.theta)


_L = {}


def layer(name):
    if name not in _L:
        _L[name] = Layer(name)
    return _L[name]


def _sketch_mismatch(got: O.Sketch, rho: np.ndarray, S: np.ndarray):
    proj = rho @ S.astype(np.float64).T
    want = proj >= 0
    tie = np.abs(proj) <= 1e-4 * np.linalg.norm(S.astype(np.float64), axis=1) * \
        np.linalg.norm(rho, axis=-1, keepdims=True)
    diff = got.bits != want
    return int(np.sum(diff & ~tie)), int(np.sum(diff & tie))


@pytest.mark.parametrize("name", list(WL))
def test_qjl_sketch_parity(name):
    L = layer(name)
    w, g = L.w, L.gview
    r3, r1 = O.key_residuals(g, L.li.K)
    bad3, tie3 = _sketch_mismatch(g.l3_qjl, r3, L.S)
    assert bad3 == 0, f"L3 sketches: {bad3} bits differ outside the near-zero band"
    np.testing.assert_allclose(g.l3_qjl.norm, np.linalg.norm(r3, axis=-1), rtol=1e-4, atol=1e-6)
    bad1 = tie1 = 0
    for b in range(w.B):
        c = int(g.l1_count[b])
        sk = O.Sketch(bits=g.l1_qjl.bits[b, :, :c], norm=g.l1_qjl.norm[b, :, :c])
        r = _sketch_mismatch(sk, r1[b, :, :c], L.S)
        bad1, tie1 = bad1 + r[0], tie1 + r[1]
        np.testing.assert_allclose(sk.norm, np.linalg.norm(r1[b, :, :c], axis=-1), rtol=1e-4, atol=1e-6)
    assert bad1 == 0, f"L1 sketches: {bad1} bits differ outside the near-zero band"
    # against the oracle's own encode: the same sketches wherever the codes agree
    ora = O.encode(L.li.K, L.li.V, L.li.l1_mask, L.li.signs, w.N, w.theta, qjl_S=L.S)
    same = np.all(ora.l3_k.codes == g.l3_k.codes, axis=-1)
    assert np.mean(ora.l3_qjl.bits[same] == g.l3_qjl.bits[same]) > 0.9999
    print(f"[{name}] near-zero sketch bits that differ: L3 {tie3}, L1 {tie1}")


@pytest.mark.parametrize("name", list(WL))
def test_qjl_decode_parity(name):
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    L = layer(name)
    w = L.w
    q, pos = W.queries(w, steps=3)
    worst, moved = 0.0, 0.0
    for s in range(3):
        qd, pd = torch.from_numpy(q[s]).cuda(), torch.from_numpy(pos[s]).cuda()
        sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
        out = torch.empty((w.B, w.Hq, 128), device="cuda")
        H.hsq_decode_step(L.ctx, L.cache, qd, pd, sel, out)
        sel_r = torch.empty_like(sel)
        H.hsq_route(L.ctx, L.cache, qd, pd, sel_r)
        assert H.hsq_sync_status(L.ctx) == 0
        assert torch.equal(sel, sel_r)  # the sketch does not touch routing
        out_a = torch.empty_like(out)  # the fused step attends like the attention call
        H.hsq_decode_attn(L.ctx, L.cache, qd, pd, sel_r, out_a)
        assert H.hsq_sync_status(L.ctx) == 0
        assert np.all(rel_l2(out.cpu().numpy(), out_a.cpu().numpy()) <= 1e-5)
        gsel = sel.cpu().numpy().astype(np.int64)
        o = out.cpu().numpy()
        ref = O.decode_attn(L.gview, q[s], pos[s], gsel)
        err = rel_l2(o, ref)
        worst = max(worst, float(err.max()))
        assert np.all(err <= 1e-3), f"step {s}: rel L2 {err.max():.3e}"
        # the correction is there: the TQ-KV reading of the same cache is far off
        moved = max(moved, float(np.median(rel_l2(o, O.decode_attn(L.plain_view, q[s], pos[s], gsel)))))
    assert moved > 1e-2
    print(f"[{name}] TQ-QKV attention rel L2 {worst:.2e}; median distance to TQ-KV {moved:.2e}")


def test_qjl_refused_by_append_and_needs_turboquant():
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    w = WL["tiny_1k"]
    cfg = H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, w.T + 8, 100, w.T + 16, w.theta, sinks=4, recent=64,
                        qjl=True)
    ctx = H.Context(cfg)
    cache = H.allocate_cache(ctx, w.B, w.T, t_cap=w.T + 8)
    k = torch.zeros((w.B, w.Hkv, 128), device="cuda")
    with pytest.raises(H.HSQError) as ei:
        H.hsq_append(ctx, cache, k, k)
    assert ei.value.status == 6
    with pytest.raises(H.HSQError):
        H.Context(H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, w.T, 100, w.T + 8, w.theta, codec="plain", qjl=True))


def test_qjl_in_place_variant_equals_staged():
    """An L1 capacity of 40000 slots does not fit a split's shared memory, so the launch
    plan takes the variant that reads the tiers and the L1 sketches in place (and forms
    every row of S q~ itself); its selection and output equal the staged variant's."""
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    w = WL["tiny_1k"]
    li = W.layer_inputs(w, rope=lambda x, p: O.rope(x, p, w.theta))
    S = W.qjl_matrix(w)
    dt = torch.bfloat16 if w.storage == "bf16" else torch.float32
    K = torch.from_numpy(np.ascontiguousarray(li.K, np.float32)).cuda().to(dt).contiguous()
    V = torch.from_numpy(np.ascontiguousarray(li.V, np.float32)).cuda().to(dt).contiguous()
    q, pos = W.queries(w, steps=3)
    outs, sels = [], []
    for max_l1 in (40000, max(w.l1_size, 1)):
        cfg = H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, w.T, max_l1, w.T + w.steps + 1, w.theta, qjl=True)
        ctx = H.Context(cfg)
        cache = H.allocate_cache(ctx, w.B, w.T)
        H.set_layer_inputs(cache, li.l1_mask, li.signs)
        H.set_qjl_matrix(cache, S)
        H.hsq_encode(ctx, cache, K, V)
        o_steps, s_steps = [], []
        for s in range(3):
            sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
            out = torch.empty((w.B, w.Hq, 128), device="cuda")
            H.hsq_decode_step(ctx, cache, torch.from_numpy(q[s]).cuda(), torch.from_numpy(pos[s]).cuda(), sel, out)
            o_steps.append(out.cpu().numpy())
            s_steps.append(sel.cpu().numpy())
        assert H.hsq_sync_status(ctx) == 0
        outs.append(o_steps)
        sels.append(s_steps)
        ctx.close()
    for s in range(3):
        np.testing.assert_array_equal(sels[0][s], sels[1][s])
        assert np.all(rel_l2(outs[0][s], outs[1][s]) <= 1e-5)
