"""The hot-group table of the fused decode step (hsq_config.hot_slots).

The table is a device copy of recently fetched L3 records per (sequence, KV
head), direct-mapped (group g in slot g mod slots).  It must not change any
result, and its state must follow its rule exactly.  Over sequences of
correlated decode steps (each step's queries share most of their direction
with the first step's, so consecutive selections overlap):
  * out and sel of every step are bit-identical to those of a context
    without the table, on the same encoded cache;
  * the table after a step is exactly what the rule gives from the table
    before it and the step's selection: a selected group that missed is in
    its slot (and its record equals its L3 record) iff no other selected
    group of that (b, h) maps to the slot; every other slot is unchanged;
  * selected groups hit the table (the correlated steps re-select groups);
  * hsq_encode empties the table; hsq_append drops the group it writes, and
    decoding continues bit-identical to the table-free cache.
Shapes: the 8B head layout (r = 4, N = 16), also at full size (the 8B/32K layer in the
benchmark's launch configuration); r = 5 with beta = 256 over four
splits (64 records per split: eight record batches per step) and a
1024-slot table; N = 8 with a 16-slot table (many slots shared within a
step) and L3 in device memory.
"""

import numpy as np
import pytest

import oracle as O
import workloads as W
from hsq_harness import ensure_built, oracle_view, rel_l2

pytestmark = pytest.mark.gpu

CASES = {
    "r4_n16_slots256": dict(B=1, Hq=32, Hkv=8, T=4096, N=16, beta=64, slots=256, n_splits=0, steps=10,
                            host=True),
    "r5_n16_beta256_s4_slots1024": dict(B=2, Hq=10, Hkv=2, T=8192, N=16, beta=256, slots=1024, n_splits=4,
                                        steps=6, host=True),
    "r2_n8_slots16_device_l3": dict(B=2, Hq=4, Hkv=2, T=2048, N=8, beta=48, slots=16, n_splits=0, steps=8,
                                    host=False),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _workload(name, c):
    base = W.get_workload("qwen3_8b_32k")
    return base.with_(name="hot_" + name, B=c["B"], Hq=c["Hq"], Hkv=c["Hkv"], T=c["T"], N=c["N"], beta=c["beta"],
                      recent=128, marked=c["T"] // 100, steps=c["steps"], needle=True, seed_tag=31 + len(name))


def _contexts(w, c, **extra):
    import hierarchical_kv_cache_hsq_gb300 as H
    ctxs = []
    for slots in (0, c["slots"]):
        cfg = H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, extra.get("max_ctx", w.T),
                            extra.get("max_l1", w.l1_size), extra.get("max_pos", w.T + w.steps + 1), w.theta,
                            c["n_splits"], sinks=extra.get("sinks", 0), recent=extra.get("recent", 0),
                            hot_slots=slots)
        ctxs.append(H.Context(cfg))
    return ctxs


def _table(cache):
    return cache.view("hot_tag").cpu().numpy().copy(), cache.view("hot_rec").cpu().numpy()


def _check_rule(tag0, tag1, rec1, l3, sel, slots):
    """The table after a step against the rule; returns the step's hits."""
    B, H = tag0.shape[:2]
    hits = 0
    want = tag0.copy()
    for b in range(B):
        for h in range(H):
            gs = [int(g) for g in sel[b, h] if g >= 0]
            slot_of = [g % slots for g in gs]
            counts = np.bincount(slot_of, minlength=slots)
            for g, sl in zip(gs, slot_of):
                if tag0[b, h, sl] == g:
                    hits += 1
                elif counts[sl] == 1:
                    want[b, h, sl] = g
    np.testing.assert_array_equal(tag1, want)
    for b, h, sl in zip(*np.nonzero(tag1 >= 0)):
        g = int(tag1[b, h, sl])
        assert g % slots == sl
        np.testing.assert_array_equal(rec1[b, h, sl], l3[b, h, g], err_msg=f"slot {sl} of ({b}, {h}) holds group {g}")
    return hits


@pytest.mark.parametrize("name", list(CASES))
def test_hot_table_is_invisible_and_follows_its_rule(name):
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    c = CASES[name]
    w = _workload(name, c)
    li = W.layer_inputs(w, rope=lambda x, p: O.rope(x, p, w.theta))
    q, pos = W.queries(w)
    ctx0, ctx1 = _contexts(w, c)
    dt = torch.bfloat16
    K = torch.from_numpy(np.ascontiguousarray(li.K, np.float32)).cuda().to(dt)
    V = torch.from_numpy(np.ascontiguousarray(li.V, np.float32)).cuda().to(dt)
    caches = []
    for ctx in (ctx0, ctx1):
        cache = H.allocate_cache(ctx, w.B, w.T, l3_on_host=c["host"], with_staging=False)
        H.set_layer_inputs(cache, li.l1_mask, li.signs)
        H.hsq_encode(ctx, cache, K, V)
        caches.append(cache)
    torch.cuda.synchronize()
    ref, hot = caches
    l3 = hot.view("l3").cpu().numpy()
    np.testing.assert_array_equal(l3, ref.view("l3").cpu().numpy())
    tag, _ = _table(hot)
    assert np.all(tag == -1)
    qd, pd = torch.from_numpy(q).cuda(), torch.from_numpy(pos).cuda()
    sel = [torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda") for _ in range(2)]
    out = [torch.empty((w.B, w.Hq, 128), device="cuda") for _ in range(2)]
    hits, selected = 0, 0
    for s in range(w.steps):
        tag0, _ = _table(hot)
        H.hsq_decode_step(ctx0, ref, qd[s], pd[s], sel[0], out[0])
        H.hsq_decode_step(ctx1, hot, qd[s], pd[s], sel[1], out[1])
        assert H.hsq_sync_status(ctx1) == 0
        np.testing.assert_array_equal(sel[1].cpu().numpy(), sel[0].cpu().numpy())
        np.testing.assert_array_equal(out[1].cpu().numpy(), out[0].cpu().numpy())
        tag1, rec1 = _table(hot)
        sl = sel[1].cpu().numpy()
        hits += _check_rule(tag0, tag1, rec1, l3, sl, c["slots"])
        selected += int(np.sum(sl >= 0))
    assert hits > 0, "correlated steps never hit the table"
    # one step of the table path against the oracle (its own selection)
    g = oracle_view({k: v for k, v in ((n, hot.view(n).cpu().numpy()) for n in (
        "l1_kc", "l1_vc", "l1_kn", "l1_vn", "l1_pos", "l1_count", "l2_kc", "l2_vc", "l2_kn", "l2_vn", "l2_cnt",
        "l3"))}, li, w)
    ref_out = O.decode_attn(g, q[w.steps - 1], pos[w.steps - 1], sel[1].cpu().numpy().astype(np.int64))
    assert float(np.max(rel_l2(out[1].cpu().numpy(), ref_out))) < 1e-3
    # encode empties the table
    H.hsq_encode(ctx1, hot, K, V)
    torch.cuda.synchronize()
    tag, _ = _table(hot)
    assert np.all(tag == -1)
    print(f"{name}: {hits} of {selected} selected groups hit the table")


def test_hot_table_with_growth():
    """Steps interleaved with hsq_append: the appended token's group leaves the
    table, and every step stays bit-identical to the table-free cache."""
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    c = dict(B=2, Hq=8, Hkv=2, T=1500, N=16, beta=24, slots=64, n_splits=0, steps=12)
    w = _workload("grow", c)
    T0, s = w.T, c["steps"]
    T1 = T0 + s
    sinks, recent = 4, 64
    wl = w.with_(T=T1, sinks=sinks, recent=recent, marked=20)
    li = W.layer_inputs(wl, rope=lambda x, p: O.rope(x, p, wl.theta))
    p = np.arange(T0)
    mask0 = (li.l1_mask[:, :T0] & (p >= sinks) & (p < T0 - recent)) | (p < sinks) | (p >= T0 - recent)
    ctx0, ctx1 = _contexts(w, c, max_ctx=T1, max_l1=sinks + 20 + recent, max_pos=T1 + 8, sinks=sinks,
                           recent=recent)
    K = torch.from_numpy(np.ascontiguousarray(li.K, np.float32)).cuda()
    V = torch.from_numpy(np.ascontiguousarray(li.V, np.float32)).cuda()
    caches = []
    for ctx in (ctx0, ctx1):
        cache = H.allocate_cache(ctx, w.B, T0, with_staging=False, t_cap=T1)
        H.set_layer_inputs(cache, mask0, li.signs)
        H.hsq_encode(ctx, cache, K[:, :, :T0].contiguous(), V[:, :, :T0].contiguous())
        caches.append(cache)
    ref, hot = caches
    q, _ = W.queries(w, steps=s)
    qd = torch.from_numpy(q).cuda()
    sel = [torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda") for _ in range(2)]
    out = [torch.empty((w.B, w.Hq, 128), device="cuda") for _ in range(2)]
    hits = 0
    for i in range(s):
        pd = torch.full((w.B,), hot.T, dtype=torch.int32, device="cuda")
        tag0, _ = _table(hot)
        H.hsq_decode_step(ctx0, ref, qd[i], pd, sel[0], out[0])
        H.hsq_decode_step(ctx1, hot, qd[i], pd, sel[1], out[1])
        assert H.hsq_sync_status(ctx1) == 0
        np.testing.assert_array_equal(sel[1].cpu().numpy(), sel[0].cpu().numpy())
        np.testing.assert_array_equal(out[1].cpu().numpy(), out[0].cpu().numpy())
        tag1, rec1 = _table(hot)
        hits += _check_rule(tag0, tag1, rec1, hot.view("l3").cpu().numpy(), sel[1].cpu().numpy(), c["slots"])
        # append: the group of the new token leaves the table if it is there
        t = hot.T
        for cache, ctx in ((ref, ctx0), (hot, ctx1)):
            H.hsq_append(ctx, cache, K[:, :, t].contiguous(), V[:, :, t].contiguous())
        tag2, rec2 = _table(hot)
        want = tag1.copy()
        sl = (t // w.N) % c["slots"]
        want[:, :, sl] = np.where(want[:, :, sl] == t // w.N, -1, want[:, :, sl])
        np.testing.assert_array_equal(tag2, want)
        l3 = hot.view("l3").cpu().numpy()
        for b, h, k in zip(*np.nonzero(tag2 >= 0)):
            np.testing.assert_array_equal(rec2[b, h, k], l3[b, h, tag2[b, h, k]])
    assert H.hsq_sync_status(ctx0) == 0 and H.hsq_sync_status(ctx1) == 0
    assert hits > 0


def test_hot_table_full_size_8b_32k():
    """The 8B/32K layer in the benchmark's launch configuration (B 1, Hkv 8, T 32768,
    N 16, beta 64, L3 in pinned host memory, 256 slots) over 8 correlated steps:
    out and sel bit-identical to the table-free step, the table following its rule."""
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    w = W.get_workload("qwen3_8b_32k").with_(steps=8)
    c = dict(slots=256, n_splits=0)
    li = W.layer_inputs(w, rope=lambda x, p: O.rope(x, p, w.theta))
    q, pos = W.queries(w)
    ctx0, ctx1 = _contexts(w, c)
    K = torch.from_numpy(np.ascontiguousarray(li.K, np.float32)).cuda().to(torch.bfloat16)
    V = torch.from_numpy(np.ascontiguousarray(li.V, np.float32)).cuda().to(torch.bfloat16)
    caches = []
    for ctx in (ctx0, ctx1):
        cache = H.allocate_cache(ctx, w.B, w.T, l3_on_host=True, with_staging=False)
        H.set_layer_inputs(cache, li.l1_mask, li.signs)
        H.hsq_encode(ctx, cache, K, V)
        caches.append(cache)
    torch.cuda.synchronize()
    ref, hot = caches
    l3 = hot.view("l3").cpu().numpy()
    qd, pd = torch.from_numpy(q).cuda(), torch.from_numpy(pos).cuda()
    sel = [torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda") for _ in range(2)]
    out = [torch.empty((w.B, w.Hq, 128), device="cuda") for _ in range(2)]
    hits = 0
    for s in range(w.steps):
        tag0, _ = _table(hot)
        H.hsq_decode_step(ctx0, ref, qd[s], pd[s], sel[0], out[0])
        H.hsq_decode_step(ctx1, hot, qd[s], pd[s], sel[1], out[1])
        assert H.hsq_sync_status(ctx1) == 0
        np.testing.assert_array_equal(sel[1].cpu().numpy(), sel[0].cpu().numpy())
        np.testing.assert_array_equal(out[1].cpu().numpy(), out[0].cpu().numpy())
        tag1, rec1 = _table(hot)
        hits += _check_rule(tag0, tag1, rec1, l3, sel[1].cpu().numpy(), c["slots"])
    assert hits > 0
    print(f"8B/32K: {hits} of {w.steps * w.Hkv * w.beta} selected groups hit the table")
