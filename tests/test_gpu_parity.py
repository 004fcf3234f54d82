"""GPU parity: every call of the CUDA path against the float64 oracle on the
same seeded inputs (small and ragged workloads, every step).

Acceptance (per call):
  * packed codes (L1, L2, L3) bit-exact except coordinates within
    1e-5 * max(|tau_k|, 1/sqrt(d)) of a boundary (counted);
  * sel bit-exact except groups within 1e-5 * max(|s_beta|, rms(s)) of the
    beta-th score (counted);
  * fetched originals within 1e-5 relative per vector;
  * attention output within 1e-3 relative L2 per (b, query head), checked
    on the GPU's own cache and selection (conditional), and reported
    end to end.
"""

import numpy as np
import pytest

import oracle as O
import workloads as W
from hsq_harness import (abi_buffers, code_mismatch, ensure_built, gpu_encode, make_ctx, oracle_view,
                         rel_l2, sel_mismatch)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _rope(w):
    return lambda x, p: O.rope(x, p, w.theta)


def _workloads():
    tiny = W.get_workload("tiny_1k")
    return {
        "tiny_1k": tiny,
        "qwen3_0p6b_4k": W.get_workload("qwen3_0p6b_4k"),
        # ragged: T not a multiple of N or 32, B = 2, r = 5, N = 8
        "ragged_r5": tiny.with_(name="ragged_r5", B=2, Hq=10, Hkv=2, T=1001, N=8, beta=12, recent=40,
                                marked=17, storage="bf16", key_law="student_t", seed_tag=11),
        # r = 8, lowrank keys, N = 16, beta close to the number of groups
        "r8_lowrank": tiny.with_(name="r8_lowrank", B=1, Hq=16, Hkv=2, T=600, N=16, beta=30, recent=32,
                                 marked=6, storage="bf16", key_law="lowrank", seed_tag=12),
        # r = 1
        "r1": tiny.with_(name="r1", B=1, Hq=2, Hkv=2, T=512, N=16, beta=4, seed_tag=13),
    }


WL = _workloads()


class Layer:
    def __init__(self, name, l3_on_host=True, beta=None, n_splits=0):
        self.w = WL[name] if beta is None else WL[name].with_(beta=beta)
        self.li = W.layer_inputs(self.w, rope=_rope(self.w))
        self.ora = O.encode(self.li.K, self.li.V, self.li.l1_mask, self.li.signs, self.w.N, self.w.theta)
        self.ctx = make_ctx(self.w, n_splits=n_splits)
        self.cache = gpu_encode(self.ctx, self.w, self.li, l3_on_host=l3_on_host)
        self.bufs = abi_buffers(self.cache)
        self.gview = oracle_view(self.bufs, self.li, self.w)


_LAYERS = {}


def layer(name, **kw):
    key = (name, tuple(sorted(kw.items())))
    if key not in _LAYERS:
        _LAYERS[key] = Layer(name, **kw)
    return _LAYERS[key]


@pytest.mark.parametrize("name", list(WL))
def test_encode_parity(name):
    L = layer(name)
    w, ora, g = L.w, L.ora, L.gview
    np.testing.assert_array_equal(L.bufs["l1_count"], ora.l1_count)
    for b in range(w.B):
        c = ora.l1_count[b]
        np.testing.assert_array_equal(L.bufs["l1_pos"][b, :c], ora.l1_pos[b, :c])
    np.testing.assert_array_equal(g.l2_cnt, ora.l2_cnt)
    report = {}
    for tier, bits in (("l3_k", 4), ("l3_v", 4), ("l1_k", 4), ("l1_v", 4), ("l2_k", 3), ("l2_v", 3)):
        go, oo = getattr(g, tier), getattr(ora, tier)
        if tier.startswith("l1"):
            bad = tie_diff = ties = 0
            for b in range(w.B):
                n = int(ora.l1_count[b])
                r = code_mismatch(go.codes[b, :, :n], oo.codes[b, :, :n], oo.y[b, :, :n], bits, oo.norms[b, :, :n])
                bad, tie_diff, ties = bad + r[0], tie_diff + r[1], ties + r[2]
                np.testing.assert_allclose(go.norms[b, :, :n], oo.norms[b, :, :n], rtol=2e-6)
        else:
            bad, tie_diff, ties = code_mismatch(go.codes, oo.codes, oo.y, bits, oo.norms)
            np.testing.assert_allclose(go.norms, oo.norms, rtol=2e-6 if tier.startswith("l3") else 1e-5,
                                       atol=1e-30)
        report[tier] = (tie_diff, ties)
        assert bad == 0, f"{tier}: {bad} code mismatches outside the near-tie band"
    print(f"[{name}] near-tie coordinates (differing, total): {report}")
    # the ragged tail of the last L3 record holds the zero-vector encoding
    if w.T % w.N:
        rec = L.bufs["l3"][:, :, -1]
        tail = O.unpack_codes(rec[..., : w.N * 64].reshape(w.B, w.Hkv, w.N, 64), 4)[:, :, w.T % w.N:]
        assert np.all(tail == 7)


@pytest.mark.parametrize("name", list(WL))
def test_route_parity(name):
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    L = layer(name)
    w = L.w
    q, pos = W.queries(w, steps=4)
    for s in range(4):
        qd = torch.from_numpy(q[s]).cuda()
        pd = torch.from_numpy(pos[s]).cuda()
        sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
        scores = torch.empty((w.B, w.Hkv, L.cache.G), dtype=torch.float32, device="cuda")
        H.hsq_route(L.ctx, L.cache, qd, pd, sel, scores)
        assert H.hsq_sync_status(L.ctx) == 0
        osel, oscores = O.route(L.gview, q[s], pos[s], w.beta)
        gs = scores.cpu().numpy()
        fin = np.isfinite(oscores)
        np.testing.assert_array_equal(np.isfinite(gs), fin)
        scale = np.sqrt(np.mean(oscores[fin] ** 2))
        assert np.max(np.abs(gs[fin] - oscores[fin])) <= 1e-5 * scale
        gsel = sel.cpu().numpy()
        for b in range(w.B):
            for h in range(w.Hkv):
                row = gsel[b, h]
                valid = row[row >= 0]
                assert np.all(np.diff(valid) > 0) and np.all(row[len(valid):] == -1)
                bad, diff = sel_mismatch(row, osel[b, h], oscores[b, h], w.beta)  # band from the oracle's scores
                assert bad == 0, f"step {s} (b={b}, h={h}): selection differs beyond near-ties"


@pytest.mark.parametrize("name", ["tiny_1k", "ragged_r5", "r8_lowrank"])
@pytest.mark.parametrize("l3_on_host", [True, False])
def test_fetch_dequant_parity(name, l3_on_host):
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    L = layer(name, l3_on_host=l3_on_host)
    w = L.w
    q, pos = W.queries(w, steps=1)
    sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
    H.hsq_route(L.ctx, L.cache, torch.from_numpy(q[0]).cuda(), torch.from_numpy(pos[0]).cuda(), sel)
    shape = (w.B, w.Hkv, w.beta, w.N, 128)
    k = torch.full(shape, 7.0, device="cuda")
    v = torch.full(shape, 7.0, device="cuda")
    valid = torch.full(shape[:-1], 9, dtype=torch.uint8, device="cuda")
    H.hsq_fetch_dequant(L.ctx, L.cache, sel, k, v, valid)
    assert H.hsq_sync_status(L.ctx) == 0
    gsel = sel.cpu().numpy()
    ok, ov, ovalid = O.fetch_dequant(L.gview, gsel.astype(np.int64))
    np.testing.assert_array_equal(valid.cpu().numpy().astype(bool), ovalid)
    kk, vv = k.cpu().numpy(), v.cpu().numpy()
    nz = np.linalg.norm(ok, axis=-1) > 0
    assert np.all(rel_l2(kk, ok)[nz] <= 1e-5) and np.all(rel_l2(vv, ov)[nz] <= 1e-5)
    assert np.all(kk[~nz] == 0) and np.all(vv[~nz] == 0)
    # staging holds the raw records of the selected groups
    st = L.cache.view("staging").cpu().numpy()
    for b in range(w.B):
        for h in range(w.Hkv):
            for i, g in enumerate(gsel[b, h]):
                if g >= 0:
                    np.testing.assert_array_equal(st[b, h, i], L.bufs["l3"][b, h, g])


@pytest.mark.parametrize("name", list(WL))
def test_decode_attn_parity(name):
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    L = layer(name)
    w = L.w
    steps = 6
    q, pos = W.queries(w, steps=steps)
    worst, worst_e2e = 0.0, 0.0
    for s in range(steps):
        qd = torch.from_numpy(q[s]).cuda()
        pd = torch.from_numpy(pos[s]).cuda()
        sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
        out = torch.empty((w.B, w.Hq, 128), device="cuda")
        H.hsq_decode_step(L.ctx, L.cache, qd, pd, sel, out)
        assert H.hsq_sync_status(L.ctx) == 0
        # the fused step selects exactly what the routing call selects ...
        sel_r = torch.empty_like(sel)
        H.hsq_route(L.ctx, L.cache, qd, pd, sel_r)
        # ... and attends exactly like the attention call given that selection
        out_a = torch.empty_like(out)
        H.hsq_decode_attn(L.ctx, L.cache, qd, pd, sel_r, out_a)
        assert H.hsq_sync_status(L.ctx) == 0
        assert torch.equal(sel, sel_r)
        assert np.all(rel_l2(out.cpu().numpy(), out_a.cpu().numpy()) <= 1e-5)
        gsel = sel.cpu().numpy().astype(np.int64)
        ref = O.decode_attn(L.gview, q[s], pos[s], gsel)          # conditional: GPU cache + GPU sel
        err = rel_l2(out.cpu().numpy(), ref)
        worst = max(worst, float(err.max()))
        assert np.all(err <= 1e-3), f"step {s}: max rel L2 {err.max():.3e}"
        osel, _ = O.route(L.ora, q[s], pos[s], w.beta)             # independent end to end
        e2e = rel_l2(out.cpu().numpy(), O.decode_attn(L.ora, q[s], pos[s], osel))
        worst_e2e = max(worst_e2e, float(e2e.max()))
    print(f"[{name}] attention rel L2: conditional {worst:.2e}, end-to-end {worst_e2e:.2e}")


@pytest.mark.parametrize("n_splits", [1, 3, 16])
def test_decode_attn_split_counts_agree(n_splits):
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    L = layer("qwen3_0p6b_4k", n_splits=n_splits)
    w = L.w
    q, pos = W.queries(w, steps=1)
    qd, pd = torch.from_numpy(q[0]).cuda(), torch.from_numpy(pos[0]).cuda()
    sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
    out = torch.empty((w.B, w.Hq, 128), device="cuda")
    H.hsq_decode_step(L.ctx, L.cache, qd, pd, sel, out)
    ref = O.decode_attn(L.gview, q[0], pos[0], sel.cpu().numpy().astype(np.int64))
    assert np.all(rel_l2(out.cpu().numpy(), ref) <= 1e-3)


def test_staged_path_equals_fused_gather():
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    L = layer("ragged_r5")
    w = L.w
    q, pos = W.queries(w, steps=1)
    qd, pd = torch.from_numpy(q[0]).cuda(), torch.from_numpy(pos[0]).cuda()
    sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
    H.hsq_route(L.ctx, L.cache, qd, pd, sel)
    side = torch.cuda.Stream()
    ev = torch.cuda.Event()
    ev.record()
    with torch.cuda.stream(side):
        side.wait_event(ev)
        H.hsq_fetch_dequant(L.ctx, L.cache, sel, stream=side)
    done = torch.cuda.Event()
    done.record(side)
    torch.cuda.current_stream().wait_event(done)
    out_staged = torch.empty((w.B, w.Hq, 128), device="cuda")
    H.hsq_decode_attn(L.ctx, L.cache, qd, pd, sel, out_staged, flags=H.HSQ_ATTN_FROM_STAGING)
    out_fused = torch.empty_like(out_staged)
    H.hsq_decode_attn(L.ctx, L.cache, qd, pd, sel, out_fused)
    assert H.hsq_sync_status(L.ctx) == 0
    assert torch.equal(out_staged, out_fused)


def test_device_resident_l3_matches_pinned():
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    A = layer("tiny_1k")
    Bl = layer("tiny_1k", l3_on_host=False)
    np.testing.assert_array_equal(A.bufs["l3"], Bl.bufs["l3"])
    w = A.w
    q, pos = W.queries(w, steps=1)
    outs = []
    for L in (A, Bl):
        sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
        out = torch.empty((w.B, w.Hq, 128), device="cuda")
        H.hsq_decode_step(L.ctx, L.cache, torch.from_numpy(q[0]).cuda(), torch.from_numpy(pos[0]).cuda(), sel, out)
        outs.append(out)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])


# -- degenerate caches ------------------------------------------------------------------

def _degenerate(**kw):
    base = WL["tiny_1k"].with_(name="degenerate", seed_tag=21)
    return base.with_(**kw)


@pytest.mark.parametrize("kw", [
    dict(T=64, recent=60, marked=0, beta=3),            # every token in L1: all groups empty
    dict(T=128, recent=0, marked=0, sinks=0, beta=2),   # empty L1
    dict(T=80, recent=32, marked=0, beta=6),            # beta above the non-empty groups: -1 padding
    dict(T=17, recent=1, marked=0, sinks=1, beta=1, N=8),  # tiny ragged context
])
def test_degenerate_caches(kw):
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    w = _degenerate(**kw)
    li = W.layer_inputs(w)
    ctx = make_ctx(w)
    cache = gpu_encode(ctx, w, li)
    g = oracle_view(abi_buffers(cache), li, w)
    ora = O.encode(li.K, li.V, li.l1_mask, li.signs, w.N, w.theta)
    np.testing.assert_array_equal(g.l2_cnt, ora.l2_cnt)
    q, pos = W.queries(w, steps=2)
    for s in range(2):
        sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
        out = torch.empty((w.B, w.Hq, 128), device="cuda")
        H.hsq_decode_step(ctx, cache, torch.from_numpy(q[s]).cuda(), torch.from_numpy(pos[s]).cuda(), sel, out)
        assert H.hsq_sync_status(ctx) == 0
        gsel = sel.cpu().numpy().astype(np.int64)
        osel, _ = O.route(g, q[s], pos[s], w.beta)
        np.testing.assert_array_equal(gsel, osel)
        ref = O.decode_attn(g, q[s], pos[s], gsel)
        o = out.cpu().numpy()
        assert np.all(np.isfinite(o))
        assert np.all(rel_l2(o, ref) <= 1e-3)


def test_contexts_of_different_sizes_coexist():
    # a small context created after a large one (same head ratio) must not
    # shrink the large one's launch limits
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    big = layer("qwen3_0p6b_4k")
    small = WL["tiny_1k"].with_(Hq=16, Hkv=8, seed_tag=30)
    ctx_small = make_ctx(small)
    cache_small = gpu_encode(ctx_small, small, W.layer_inputs(small))
    w = big.w
    q, pos = W.queries(w, steps=1)
    sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
    out = torch.empty((w.B, w.Hq, 128), device="cuda")
    H.hsq_decode_step(big.ctx, big.cache, torch.from_numpy(q[0]).cuda(), torch.from_numpy(pos[0]).cuda(), sel, out)
    assert H.hsq_sync_status(big.ctx) == 0
    ref = O.decode_attn(big.gview, q[0], pos[0], sel.cpu().numpy().astype(np.int64))
    assert np.all(rel_l2(out.cpu().numpy(), ref) <= 1e-3)
    del cache_small
    ctx_small.close()


def test_invalid_selection_is_flagged_not_faulted():
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    L = layer("tiny_1k")
    w = L.w
    q, pos = W.queries(w, steps=1)
    bad = np.full((w.B, w.Hkv, w.beta), -1, np.int32)
    bad[:, :, 0] = 5
    bad[:, :, 1] = 3          # not ascending
    bad[:, :, 2] = 10 ** 6    # out of range
    out = torch.empty((w.B, w.Hq, 128), device="cuda")
    H.hsq_decode_attn(L.ctx, L.cache, torch.from_numpy(q[0]).cuda(), torch.from_numpy(pos[0]).cuda(),
                      torch.from_numpy(bad).cuda(), out)
    word = H.hsq_sync_status(L.ctx)
    assert word & H.HSQ_DEVERR_SEL
    assert np.all(np.isfinite(out.cpu().numpy()))
    # the context stays usable
    sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
    H.hsq_decode_step(L.ctx, L.cache, torch.from_numpy(q[0]).cuda(), torch.from_numpy(pos[0]).cuda(), sel, out)
    assert H.hsq_sync_status(L.ctx) == 0


def test_position_outside_tables_is_flagged():
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    L = layer("tiny_1k")
    w = L.w
    q, _ = W.queries(w, steps=1)
    sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
    out = torch.empty((w.B, w.Hq, 128), device="cuda")
    far = torch.full((w.B,), 10 ** 7, dtype=torch.int32, device="cuda")
    H.hsq_decode_step(L.ctx, L.cache, torch.from_numpy(q[0]).cuda(), far, sel, out)
    assert H.hsq_sync_status(L.ctx) & H.HSQ_DEVERR_POS


def test_injected_fetch_failure_returns_status():
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    L = layer("tiny_1k")
    w = L.w
    sel = torch.full((w.B, w.Hkv, w.beta), -1, dtype=torch.int32, device="cuda")
    H.hsq_debug_set_fault(H.HSQ_FAULT_FETCH)
    try:
        with pytest.raises(H.HSQError) as ei:
            H.hsq_fetch_dequant(L.ctx, L.cache, sel)
        assert ei.value.status == 2
    finally:
        H.hsq_debug_set_fault(0)
    H.hsq_fetch_dequant(L.ctx, L.cache, sel)
    assert H.hsq_sync_status(L.ctx) == 0


def test_l3_location_mismatch_rejected():
    import hierarchical_kv_cache_hsq_gb300 as H
    import torch
    w = WL["tiny_1k"]
    li = W.layer_inputs(w)
    ctx = make_ctx(w)
    cache = H.allocate_cache(ctx, w.B, w.T, l3_on_host=True)
    cache.l3_on_host = False   # lie about where L3 lives
    H.set_layer_inputs(cache, li.l1_mask, li.signs)
    K = torch.from_numpy(li.K).cuda()
    with pytest.raises(H.HSQError) as ei:
        H.hsq_encode(ctx, cache, K, K)
    assert ei.value.status == 1


def test_host_mapped_io_matches_device_io():
    # q, pos, sel and out in page-locked host memory are read and written in
    # place by the kernel; the step is the same as with device buffers
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    L = layer("qwen3_0p6b_4k")
    w = L.w
    q, pos = W.queries(w, steps=2)
    for s in range(2):
        qd, pd = torch.from_numpy(q[s]).cuda(), torch.from_numpy(pos[s]).cuda()
        sel_d = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
        out_d = torch.empty((w.B, w.Hq, 128), device="cuda")
        H.hsq_decode_step(L.ctx, L.cache, qd, pd, sel_d, out_d)
        qh, ph = torch.from_numpy(q[s]).pin_memory(), torch.from_numpy(pos[s]).pin_memory()
        sel_h = torch.full((w.B, w.Hkv, w.beta), 7, dtype=torch.int32).pin_memory()
        out_h = torch.full((w.B, w.Hq, 128), 7.0).pin_memory()
        H.hsq_decode_step(L.ctx, L.cache, qh, ph, sel_h, out_h)
        assert H.hsq_sync_status(L.ctx) == 0
        assert torch.equal(sel_h, sel_d.cpu())
        assert torch.equal(out_h, out_d.cpu())


def test_pageable_host_buffer_is_refused():
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    from hierarchical_kv_cache_hsq_gb300 import _binding as B
    L = layer("tiny_1k")
    w = L.w
    q, pos = W.queries(w, steps=1)
    qh = torch.from_numpy(q[0])  # ordinary (pageable) host memory
    pd = torch.from_numpy(pos[0]).cuda()
    sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
    out = torch.empty((w.B, w.Hq, 128), device="cuda")
    with pytest.raises(B.HSQError) as ei:
        H.hsq_decode_step(L.ctx, L.cache, qh, pd, sel, out)
    assert ei.value.status == B.HSQ_ERR_INVALID
    assert H.hsq_sync_status(L.ctx) == 0


@pytest.mark.parametrize("kw", [
    dict(T=16384, N=16, B=1, Hq=8, Hkv=2),   # G = 1024: the top half of the groups
    dict(T=5000, N=8, B=2, Hq=10, Hkv=2),    # G = 625, ragged, r = 5
])
def test_maximum_beta(kw):
    """beta = HSQ_MAX_BETA (512): the fused step selects what the routing call
    selects, that selection equals the oracle's up to near-ties of its
    beta-th score, and the attention over 512 fetched groups is within 1e-3
    of the oracle's on the GPU's cache and selection."""
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    w = WL["tiny_1k"].with_(name="beta_max", beta=512, recent=64, marked=40, storage="bf16", seed_tag=61, **kw)
    li = W.layer_inputs(w)
    ctx = make_ctx(w)
    cache = gpu_encode(ctx, w, li)
    g = oracle_view(abi_buffers(cache), li, w)
    q, pos = W.queries(w, steps=2)
    for s in range(2):
        qd, pd = torch.from_numpy(q[s]).cuda(), torch.from_numpy(pos[s]).cuda()
        sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
        out = torch.empty((w.B, w.Hq, 128), device="cuda")
        H.hsq_decode_step(ctx, cache, qd, pd, sel, out)
        sel_r = torch.empty_like(sel)
        H.hsq_route(ctx, cache, qd, pd, sel_r)
        assert H.hsq_sync_status(ctx) == 0
        assert torch.equal(sel, sel_r)
        gsel = sel.cpu().numpy().astype(np.int64)
        osel, oscores = O.route(g, q[s], pos[s], w.beta)
        for b in range(w.B):
            for h in range(w.Hkv):
                assert (gsel[b, h] >= 0).sum() == min(w.beta, int((g.l2_cnt[b] > 0).sum()))
                bad, _ = sel_mismatch(gsel[b, h], osel[b, h], oscores[b, h], w.beta)
                assert bad == 0, f"step {s} (b={b}, h={h}): {bad} selection differences outside the band"
        ref = O.decode_attn(g, q[s], pos[s], gsel)
        err = rel_l2(out.cpu().numpy(), ref)
        assert np.all(err <= 1e-3), f"step {s}: max rel L2 {err.max():.3e}"
    ctx.close()


def test_query_positions_up_to_max_pos():
    """max_pos = 2^24, the largest the configuration allows: the query's RoPE
    at positions near it (angle tables of 65536 + 256 rows combined by angle
    addition) routes and attends like the float64 oracle."""
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    w = WL["tiny_1k"].with_(name="far_positions", seed_tag=62)
    li = W.layer_inputs(w)
    cfg = H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, w.T, max(w.l1_size, 1), 1 << 24, w.theta)
    ctx = H.Context(cfg)
    cache = gpu_encode(ctx, w, li)
    g = oracle_view(abi_buffers(cache), li, w)
    q, _ = W.queries(w, steps=3)
    for s, p in enumerate(((1 << 24) - 1, (1 << 23) + 12345, 65536 * 255 + 17)):
        pos = np.full((w.B,), p, dtype=np.int32)
        sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
        out = torch.empty((w.B, w.Hq, 128), device="cuda")
        H.hsq_decode_step(ctx, cache, torch.from_numpy(q[s]).cuda(), torch.from_numpy(pos).cuda(), sel, out)
        assert H.hsq_sync_status(ctx) == 0
        gsel = sel.cpu().numpy().astype(np.int64)
        osel, oscores = O.route(g, q[s], pos, w.beta)
        for b in range(w.B):
            for h in range(w.Hkv):
                bad, _ = sel_mismatch(gsel[b, h], osel[b, h], oscores[b, h], w.beta)
                assert bad == 0, f"position {p} (b={b}, h={h})"
        err = rel_l2(out.cpu().numpy(), O.decode_attn(g, q[s], pos, gsel))
        assert np.all(err <= 1e-3), f"position {p}: max rel L2 {err.max():.3e}"
    ctx.close()
