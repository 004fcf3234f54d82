"""Decode-time growth (hsq_append) on the GPU.

A cache encoded at length T0 and grown by s appended tokens must be the
encode of the T0 + s context under the grown L1 set (oracle.grown_l1_mask):
  * bit-exact against the GPU's own encode of the longer context: L3
    records, L2 codes, norms and counts, the L1 bitmap and count, the
    window ring, the running sums and counts, and the L1 entries as a set keyed by
    position (an appended token takes the slot of the token that leaves);
  * within the encode parity bar against the oracle's encode of the longer
    context (codes bit-exact except near-ties);
  * the decode step on the grown cache within 1e-3 relative L2 of the
    oracle on that cache and selection.
"""

import numpy as np
import pytest

import oracle as O
import workloads as W
from hsq_harness import code_mismatch, ensure_built, rel_l2, sel_mismatch

pytestmark = pytest.mark.gpu

CASES = {
    # f32, N = 16, r = 2; T0 - recent and T0 + s - recent both inside a group
    "n16_f32": dict(B=2, Hq=4, Hkv=2, N=16, beta=8, sinks=4, recent=64, marked=32, storage="f32",
                    key_law="lognormal", T0=1000, s=45),
    # bf16, N = 8, r = 5; the growth crosses several group boundaries
    "n8_bf16_r5": dict(B=2, Hq=10, Hkv=2, N=8, beta=12, sinks=4, recent=40, marked=17, storage="bf16",
                       key_law="student_t", T0=777, s=30),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


class Grown:
    """K/V for T0 + s tokens; cache A = encode of T0 then s appends; cache B =
    encode of T0 + s under the grown L1 set; both laid out for T0 + s."""

    def __init__(self, name):
        import torch
        import hierarchical_kv_cache_hsq_gb300 as H
        c = CASES[name]
        T0, s = c["T0"], c["s"]
        T1 = T0 + s
        tiny = W.get_workload("tiny_1k")
        w = tiny.with_(name="grow_" + name, B=c["B"], Hq=c["Hq"], Hkv=c["Hkv"], T=T1, N=c["N"], beta=c["beta"],
                       sinks=c["sinks"], recent=c["recent"], marked=c["marked"], storage=c["storage"],
                       key_law=c["key_law"], seed_tag=21 + len(name))
        li = W.layer_inputs(w)
        sinks, recent = c["sinks"], c["recent"]
        # the encode-time L1 set of the T0 context: sinks, the marked tokens below
        # its window, its window
        pos = np.arange(T0)
        marked = li.l1_mask[:, :T0] & (pos >= sinks) & (pos < T0 - recent)
        mask0 = marked | (pos < sinks) | (pos >= T0 - recent)
        mask1 = O.grown_l1_mask(mask0, T1, sinks, recent)
        cfg = H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, T1, sinks + c["marked"] + recent, T1 + 8, w.theta, 0,
                            sinks=sinks, recent=recent)
        self.ctx = H.Context(cfg)
        dt = torch.bfloat16 if w.storage == "bf16" else torch.float32
        K = torch.from_numpy(np.ascontiguousarray(li.K, np.float32)).cuda().to(dt)
        V = torch.from_numpy(np.ascontiguousarray(li.V, np.float32)).cuda().to(dt)
        self.a = H.allocate_cache(self.ctx, w.B, T0, with_staging=False, t_cap=T1)
        H.set_layer_inputs(self.a, mask0, li.signs)
        H.hsq_encode(self.ctx, self.a, K[:, :, :T0].contiguous(), V[:, :, :T0].contiguous())
        for i in range(s):
            H.hsq_append(self.ctx, self.a, K[:, :, T0 + i].contiguous(), V[:, :, T0 + i].contiguous())
        assert self.a.T == T1
        self.b = H.allocate_cache(self.ctx, w.B, T1, with_staging=False, t_cap=T1)
        H.set_layer_inputs(self.b, mask1, li.signs)
        H.hsq_encode(self.ctx, self.b, K.contiguous(), V.contiguous())
        assert H.hsq_sync_status(self.ctx) == 0
        self.w, self.li, self.mask1, self.T1 = w, li, mask1, T1


_G = {}


def grown(name):
    if name not in _G:
        _G[name] = Grown(name)
    return _G[name]


def _np(cache, name):
    return cache.view(name).cpu().numpy()


def _l1_by_position(cache, b):
    """{position: slot} of sequence b's L1 entries."""
    cnt = int(_np(cache, "l1_count")[b])
    pos = _np(cache, "l1_pos")[b, :cnt]
    return {int(p): i for i, p in enumerate(pos)}


@pytest.mark.parametrize("name", list(CASES))
def test_append_equals_encode_of_longer_context(name):
    g = grown(name)
    for buf in ("l3", "l2_kc", "l2_vc", "l2_kn", "l2_vn", "l2_cnt", "l1_bitmap", "l1_count", "win_kv"):
        np.testing.assert_array_equal(_np(g.a, buf), _np(g.b, buf), err_msg=buf)
    # the running sums and member count (the last word is each cache's own slot bookkeeping)
    np.testing.assert_array_equal(_np(g.a, "gsum")[..., :257], _np(g.b, "gsum")[..., :257])
    for b in range(g.w.B):
        pa, pb = _l1_by_position(g.a, b), _l1_by_position(g.b, b)
        assert sorted(pa) == sorted(pb) == list(np.nonzero(g.mask1[b])[0])
        ia = np.array([pa[p] for p in sorted(pa)])
        ib = np.array([pb[p] for p in sorted(pb)])
        for buf in ("l1_kc", "l1_vc", "l1_kn", "l1_vn"):
            np.testing.assert_array_equal(_np(g.a, buf)[b][:, ia], _np(g.b, buf)[b][:, ib], err_msg=buf)
    # the appended tokens reused the slots of the tokens that left the window
    assert int(_np(g.a, "l1_count")[0]) == int(g.mask1[0].sum())


def _sorted_view(g):
    """The grown GPU cache read back with its L1 slots in position order."""
    bufs = {k: _np(g.a, k) for k in ("l1_kc", "l1_vc", "l1_kn", "l1_vn", "l1_pos", "l1_count", "l2_kc", "l2_vc",
                                      "l2_kn", "l2_vn", "l2_cnt", "l3")}
    for b in range(g.w.B):
        cnt = int(bufs["l1_count"][b])
        order = np.argsort(bufs["l1_pos"][b, :cnt], kind="stable")
        for k in ("l1_kc", "l1_vc", "l1_kn", "l1_vn"):
            bufs[k][b, :, :cnt] = bufs[k][b][:, order]
        bufs["l1_pos"][b, :cnt] = bufs["l1_pos"][b, :cnt][order]
    return bufs, O.cache_from_abi(bufs, g.mask1, g.li.signs, g.w.N, g.T1, g.w.theta)


@pytest.mark.parametrize("name", list(CASES))
def test_append_parity_with_oracle_encode(name):
    g = grown(name)
    w = g.w
    ora = O.encode(g.li.K, g.li.V, g.mask1, g.li.signs, w.N, w.theta)
    bufs, gv = _sorted_view(g)
    np.testing.assert_array_equal(bufs["l1_count"], ora.l1_count)
    np.testing.assert_array_equal(gv.l2_cnt, ora.l2_cnt)
    for tier, bits in (("l3_k", 4), ("l3_v", 4), ("l1_k", 4), ("l1_v", 4), ("l2_k", 3), ("l2_v", 3)):
        go, oo = getattr(gv, tier), getattr(ora, tier)
        if tier.startswith("l1"):
            for b in range(w.B):
                n = int(ora.l1_count[b])
                bad = code_mismatch(go.codes[b, :, :n], oo.codes[b, :, :n], oo.y[b, :, :n], bits, oo.norms[b, :, :n])[0]
                assert bad == 0, f"{tier}: {bad} code mismatches outside the near-tie band"
        else:
            bad = code_mismatch(go.codes, oo.codes, oo.y, bits, oo.norms)[0]
            assert bad == 0, f"{tier}: {bad} code mismatches outside the near-tie band"


@pytest.mark.parametrize("name", list(CASES))
def test_decode_step_on_grown_cache(name):
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    g = grown(name)
    w = g.w
    _, gv = _sorted_view(g)
    q, _ = W.queries(w, steps=3)
    for s in range(3):
        pos = np.full((w.B,), g.T1 + s, np.int32)
        qd, pd = torch.from_numpy(q[s]).cuda(), torch.from_numpy(pos).cuda()
        sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
        out = torch.empty((w.B, w.Hq, 128), device="cuda")
        H.hsq_decode_step(g.ctx, g.a, qd, pd, sel, out)
        assert H.hsq_sync_status(g.ctx) == 0
        gsel = sel.cpu().numpy().astype(np.int64)
        ref = O.decode_attn(gv, q[s], pos, gsel)
        err = rel_l2(out.cpu().numpy(), ref)
        assert np.all(err <= 1e-3), f"step {s}: rel L2 {err.max():.3e}"


def test_append_refuses_full_cache_and_static_context():
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    g = grown("n16_f32")
    k = torch.zeros((g.w.B, g.w.Hkv, 128), device="cuda")
    with pytest.raises(H.HSQError):
        H.hsq_append(g.ctx, g.a, k, k)  # T == t_cap
    w = g.w
    static = H.Context(H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, g.T1, 100, g.T1 + 8, w.theta, 0))
    c = H.allocate_cache(static, w.B, 100, with_staging=False, t_cap=200)
    with pytest.raises(H.HSQError):
        H.hsq_append(static, c, k, k)  # no recent window in this context


@pytest.mark.parametrize("spare", [16, 200])
def test_spare_capacity_is_invisible(spare):
    """A cache laid out for T + spare tokens (empty trailing groups and bitmap
    words) routes and attends like the oracle's cache of T tokens."""
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    w = W.get_workload("tiny_1k").with_(B=2, T=1000, steps=3)
    li = W.layer_inputs(w)
    cfg = H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, w.T + spare, w.l1_size, w.T + spare + 8, w.theta)
    ctx = H.Context(cfg)
    cache = H.allocate_cache(ctx, w.B, w.T, with_staging=False, t_cap=w.T + spare)
    H.set_layer_inputs(cache, li.l1_mask, li.signs)
    H.hsq_encode(ctx, cache, torch.from_numpy(li.K).cuda().contiguous(), torch.from_numpy(li.V).cuda().contiguous())
    G = -(-w.T // w.N)
    assert (cache.view("l2_cnt").cpu().numpy()[:, G:] == 0).all()
    bufs = {k: _np(cache, k) for k in ("l1_kc", "l1_vc", "l1_kn", "l1_vn", "l1_pos", "l1_count", "l2_kc", "l2_vc",
                                        "l2_kn", "l2_vn", "l2_cnt", "l3")}
    for k in ("l2_kc", "l2_vc", "l2_kn", "l2_vn", "l3"):
        bufs[k] = bufs[k][:, :, :G]
    bufs["l2_cnt"] = bufs["l2_cnt"][:, :G]
    gv = O.cache_from_abi(bufs, li.l1_mask, li.signs, w.N, w.T, w.theta)
    q, pos = W.queries(w, steps=3)
    for s in range(3):
        qd, pd = torch.from_numpy(q[s]).cuda(), torch.from_numpy(pos[s]).cuda()
        sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
        out = torch.empty((w.B, w.Hq, 128), device="cuda")
        H.hsq_decode_step(ctx, cache, qd, pd, sel, out)
        assert H.hsq_sync_status(ctx) == 0
        gsel = sel.cpu().numpy().astype(np.int64)
        assert gsel.max() < G
        osel, oscores = O.route(gv, q[s], pos[s], w.beta)
        for b in range(w.B):
            for h in range(w.Hkv):
                assert sel_mismatch(gsel[b, h], osel[b, h], oscores[b, h], w.beta)[0] == 0
        err = rel_l2(out.cpu().numpy(), O.decode_attn(gv, q[s], pos[s], gsel))
        assert np.all(err <= 1e-3), f"step {s}: rel L2 {err.max():.3e}"
