"""The Plain-KV codec (cfg.codec = plain: the codebook on unrotated unit
vectors) on the GPU, and the relMSE / cosine codec diagnostics.

Against the oracle's encode(codec="plain") with the same acceptance as the
TurboQuant path: codes bit-exact except near-ties, routing scores within
1e-5 of their rms and selection bit-exact except near-ties, fetched
originals within 1e-5 relative, attention within 1e-3 relative L2 on the
GPU's own cache and selection; the fused step equals route + attention bit
for bit; a grown cache equals the encode of the longer context bit for bit.
hsq_recover returns the oracle's L3 originals; the diagnostics of the GPU's
recovered originals equal the oracle's on the same codes, and the
heavy-tailed keys show the rotation's gain.
"""

import numpy as np
import pytest

import oracle as O
import workloads as W
from hsq_harness import abi_buffers, code_mismatch, ensure_built, rel_l2, sel_mismatch

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
    def __init__(self, name, codec):
        import torch
        import hierarchical_kv_cache_hsq_gb300 as H
        w = WL[name]
        self.w = w
        self.li = li = W.layer_inputs(w, rope=lambda x, p: O.rope(x, p, w.theta))
        self.ora = O.encode(li.K, li.V, li.l1_mask, li.signs, w.N, w.theta, codec=codec)
        cfg = H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, w.T, max(w.l1_size, 1), w.T + w.steps + 1, w.theta,
                            codec=codec)
        self.ctx = H.Context(cfg)
        self.cache = H.allocate_cache(self.ctx, w.B, w.T)
        H.set_layer_inputs(self.cache, li.l1_mask, li.signs)
        dt = torch.bfloat16 if w.storage == "bf16" else torch.float32
        K = torch.from_numpy(np.ascontiguousarray(li.K, np.float32)).cuda().to(dt).contiguous()
        V = torch.from_numpy(np.ascontiguousarray(li.V, np.float32)).cuda().to(dt).contiguous()
        H.hsq_encode(self.ctx, self.cache, K, V)
        torch.cuda.synchronize()
        self.bufs = abi_buffers(self.cache)
        self.gview = O.cache_from_abi(self.bufs, li.l1_mask, li.signs, w.N, w.T, w.theta, codec=codec)


_L = {}


def layer(name, codec="plain"):
    if (name, codec) not in _L:
        _L[(name, codec)] = Layer(name, codec)
    return _L[(name, codec)]


@pytest.mark.parametrize("name", list(WL))
def test_plain_encode_parity(name):
    L = layer(name)
    w, ora, g = L.w, L.ora, L.gview
    np.testing.assert_array_equal(g.l2_cnt, ora.l2_cnt)
    for tier, bits in (("l3_k", 4), ("l3_v", 4), ("l1_k", 4), ("l1_v", 4), ("l2_k", 3), ("l2_v", 3)):
        go, oo = getattr(g, tier), getattr(ora, tier)
        if tier.startswith("l1"):
            for b in range(w.B):
                n = int(ora.l1_count[b])
                bad, _, _ = code_mismatch(go.codes[b, :, :n], oo.codes[b, :, :n], oo.y[b, :, :n], bits,
                                          oo.norms[b, :, :n])
                assert bad == 0, f"{tier}: {bad} code mismatches outside the near-tie band"
        else:
            bad, _, _ = code_mismatch(go.codes, oo.codes, oo.y, bits, oo.norms)
            assert bad == 0, f"{tier}: {bad} code mismatches outside the near-tie band"
            np.testing.assert_allclose(go.norms, oo.norms, rtol=2e-6 if tier.startswith("l3") else 1e-5,
                                       atol=1e-30)
    # the two codecs store different codes for the same input
    T = layer(name, "tq")
    assert np.mean(T.gview.l3_k.codes != g.l3_k.codes) > 0.5


@pytest.mark.parametrize("name", list(WL))
def test_plain_route_fetch_and_decode_parity(name):
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    L = layer(name)
    w = L.w
    q, pos = W.queries(w, steps=3)
    for s in range(3):
        qd, pd = torch.from_numpy(q[s]).cuda(), torch.from_numpy(pos[s]).cuda()
        sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
        scores = torch.empty((w.B, w.Hkv, L.cache.G), dtype=torch.float32, device="cuda")
        H.hsq_route(L.ctx, L.cache, qd, pd, sel, scores)
        assert H.hsq_sync_status(L.ctx) == 0
        osel, oscores = O.route(L.gview, q[s], pos[s], w.beta)
        gs = scores.cpu().numpy()
        fin = np.isfinite(oscores)
        np.testing.assert_array_equal(np.isfinite(gs), fin)
        assert np.max(np.abs(gs[fin] - oscores[fin])) <= 1e-5 * np.sqrt(np.mean(oscores[fin] ** 2))
        gsel = sel.cpu().numpy()
        for b in range(w.B):
            for h in range(w.Hkv):
                bad, _ = sel_mismatch(gsel[b, h], osel[b, h], oscores[b, h], w.beta)
                assert bad == 0, f"step {s} (b={b}, h={h}): selection differs beyond near-ties"
        # fetch + dequant of the selected groups
        shape = (w.B, w.Hkv, w.beta, w.N, 128)
        k, v = torch.empty(shape, device="cuda"), torch.empty(shape, device="cuda")
        H.hsq_fetch_dequant(L.ctx, L.cache, sel, k, v)
        ok, ov, _ = O.fetch_dequant(L.gview, gsel.astype(np.int64))
        nz = np.linalg.norm(ok, axis=-1) > 0
        assert np.all(rel_l2(k.cpu().numpy(), ok)[nz] <= 1e-5)
        assert np.all(rel_l2(v.cpu().numpy(), ov)[nz] <= 1e-5)
        # the fused step: same selection as the routing call, same bits as the attention call
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
        assert np.all(err <= 1e-3), f"step {s}: rel L2 {err.max():.3e}"


def test_plain_noalloc_route_parity():
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    L = layer("tiny_1k")
    w = L.w
    q, pos = W.queries(w, steps=1)
    sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
    H.hsq_route_noalloc(L.ctx.cfg, L.cache, torch.from_numpy(q[0]).cuda(), torch.from_numpy(pos[0]).cuda(), sel)
    torch.cuda.synchronize()
    osel, oscores = O.route(L.gview, q[0], pos[0], w.beta)
    gsel = sel.cpu().numpy()
    for b in range(w.B):
        for h in range(w.Hkv):
            bad, _ = sel_mismatch(gsel[b, h], osel[b, h], oscores[b, h], w.beta)
            assert bad == 0


def _recover_all(L):
    """Every token's original from L3 via hsq_recover, [B, Hkv, T, 128] each."""
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    w, G = L.w, -(-L.w.T // L.w.N)
    shape = (w.B, w.Hkv, G, w.N, 128)
    k = torch.full(shape, 7.0, device="cuda")
    v = torch.full(shape, 7.0, device="cuda")
    H.hsq_recover(L.ctx, L.cache, 0, G, k, v)
    assert H.hsq_sync_status(L.ctx) == 0
    k = k.reshape(w.B, w.Hkv, G * w.N, 128).cpu().numpy()
    v = v.reshape(w.B, w.Hkv, G * w.N, 128).cpu().numpy()
    assert np.all(k[:, :, w.T:] == 0) and np.all(v[:, :, w.T:] == 0)
    return k[:, :, : w.T], v[:, :, : w.T]


@pytest.mark.parametrize("codec", list(O.CODECS))
@pytest.mark.parametrize("name", ["ragged_r5", "r8_lowrank"])
def test_recover_parity(name, codec):
    """hsq_recover returns the oracle's L3 originals (pre-RoPE, every token)."""
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    L = layer(name, codec)
    k, v = _recover_all(L)
    ok, ov = L.gview.l3_k.vectors(L.gview.Pi), L.gview.l3_v.vectors(L.gview.Pi)
    nz = np.linalg.norm(ok, axis=-1) > 0
    assert np.all(rel_l2(k, ok)[nz] <= 1e-5) and np.all(rel_l2(v, ov)[nz] <= 1e-5)
    # a sub-range lands in slots 0..ng-1
    w = L.w
    g0, ng = 3, 5
    part = torch.empty((w.B, w.Hkv, ng, w.N, 128), device="cuda")
    H.hsq_recover(L.ctx, L.cache, g0, ng, None, part)
    got = part.reshape(w.B, w.Hkv, ng * w.N, 128).cpu().numpy()
    np.testing.assert_array_equal(got, v[:, :, g0 * w.N: (g0 + ng) * w.N])
    for bad in ((-1, 2), (0, 0), (0, -(-w.T // w.N) + 1)):
        with pytest.raises(H.HSQError):
            H.hsq_recover(L.ctx, L.cache, bad[0], bad[1], part, None)


@pytest.mark.parametrize("name", ["ragged_r5", "r8_lowrank"])
def test_codec_diagnostics_of_recovered_originals(name):
    """relMSE_K / relMSE_V / cosine of every token recovered by the GPU
    against the inputs: equal to the oracle's diagnostics on the GPU's codes;
    on the heavy-tailed keys the rotation wins, on the isotropic values the
    two codecs are alike."""
    out = {}
    for codec in O.CODECS:
        L = layer(name, codec)
        k, v = _recover_all(L)
        gk, gv = O.codec_errors(L.li.K, k), O.codec_errors(L.li.V, v)
        ok = O.codec_errors(L.li.K, L.gview.l3_k.vectors(L.gview.Pi))
        ov = O.codec_errors(L.li.V, L.gview.l3_v.vectors(L.gview.Pi))
        for a, b in ((gk, ok), (gv, ov)):
            assert abs(a["relmse"] - b["relmse"]) <= 1e-5 * b["relmse"]
            assert abs(a["cosine"] - b["cosine"]) <= 1e-6
        out[codec] = (gk, gv)
    if WL[name].key_law == "student_t":
        assert out["plain"][0]["relmse"] > 3.0 * out["tq"][0]["relmse"]
    vt, vp = out["tq"][1]["relmse"], out["plain"][1]["relmse"]
    assert abs(vt - vp) <= 0.1 * vt
    print(f"[{name}] relMSE_K tq {out['tq'][0]['relmse']:.4f} plain {out['plain'][0]['relmse']:.4f}; "
          f"relMSE_V tq {vt:.4f} plain {vp:.4f}")


def test_plain_growth_equals_encode_of_longer_context():
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    T0, s, sinks, recent = 500, 37, 4, 48
    T1 = T0 + s
    w = W.get_workload("tiny_1k").with_(name="grow_plain", B=2, Hq=4, Hkv=2, T=T1, N=16, beta=8, sinks=sinks,
                                         recent=recent, marked=20, storage="bf16", key_law="student_t",
                                         seed_tag=31)
    li = W.layer_inputs(w)
    pos = np.arange(T0)
    marked = li.l1_mask[:, :T0] & (pos >= sinks) & (pos < T0 - recent)
    mask0 = marked | (pos < sinks) | (pos >= T0 - recent)
    mask1 = O.grown_l1_mask(mask0, T1, sinks, recent)
    cfg = H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, T1, sinks + 20 + recent, T1 + 8, w.theta, 0,
                        sinks=sinks, recent=recent, codec="plain")
    ctx = H.Context(cfg)
    K = torch.from_numpy(np.ascontiguousarray(li.K, np.float32)).cuda().to(torch.bfloat16)
    V = torch.from_numpy(np.ascontiguousarray(li.V, np.float32)).cuda().to(torch.bfloat16)
    a = H.allocate_cache(ctx, w.B, T0, with_staging=False, t_cap=T1)
    H.set_layer_inputs(a, mask0, li.signs)
    H.hsq_encode(ctx, a, K[:, :, :T0].contiguous(), V[:, :, :T0].contiguous())
    for i in range(s):
        H.hsq_append(ctx, a, K[:, :, T0 + i].contiguous(), V[:, :, T0 + i].contiguous())
    b = H.allocate_cache(ctx, w.B, T1, with_staging=False, t_cap=T1)
    H.set_layer_inputs(b, mask1, li.signs)
    H.hsq_encode(ctx, b, K.contiguous(), V.contiguous())
    assert H.hsq_sync_status(ctx) == 0
    for name in ("l3", "l2_kc", "l2_vc", "l2_kn", "l2_vn", "l2_cnt", "l1_count"):
        assert torch.equal(a.view(name), b.view(name)), name
    ora = O.encode(li.K, li.V, mask1, li.signs, w.N, w.theta, codec="plain")
    g = O.cache_from_abi(abi_buffers(a), mask1, li.signs, w.N, T1, w.theta, codec="plain")
    bad, _, _ = code_mismatch(g.l3_k.codes, ora.l3_k.codes, ora.l3_k.y, 4, ora.l3_k.norms)
    assert bad == 0
