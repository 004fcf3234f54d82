"""Seeded random configurations across every mode the library offers, against
the oracle: head ratios {1, 2, 4, 5, 8}, 1-3 KV heads, N in {8, 16}, ragged
contexts, L1 sets from empty up, beta from 1 to past the number of groups,
the three key laws, f32 or bf16 input, both codecs, TQ-QKV, and the three
routings (sum, max, per query head), in the combinations the configuration
allows.  Per case and step: L3 codes within the near-tie band, routing
scores within 1e-5 of their rms and selections equal up to near-ties, the
fused step's selection equal to the routing call's, and attention within
1e-3 relative L2 of the oracle's on the GPU's cache and selection.
"""

import numpy as np
import pytest

import oracle as O
import workloads as W
from hsq_harness import abi_buffers, code_mismatch, ensure_built, rel_l2, sel_mismatch

pytestmark = pytest.mark.gpu

CASES = 40


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _case(k: int):
    rng = np.random.default_rng(7000 + k)
    r = int(rng.choice([1, 2, 4, 5, 8]))
    Hkv = int(rng.integers(1, 4))
    N = int(rng.choice([8, 16]))
    T = int(rng.integers(40, 900))
    sinks = int(rng.integers(0, 6))
    recent = int(rng.integers(0, min(64, T // 2)))
    marked = int(rng.integers(0, max(1, min(20, T - recent - sinks))))
    G = -(-T // N)
    beta = int(rng.integers(1, min(G + 3, 48)))
    codec = str(rng.choice(["tq", "plain"]))
    qjl = bool(codec == "tq" and rng.random() < 0.4)
    routing = str(rng.choice(["sum", "max", "head"]))
    w = W.get_workload("tiny_1k").with_(
        name=f"fuzz{k}", B=int(rng.integers(1, 3)), Hq=r * Hkv, Hkv=Hkv, T=T, N=N, beta=beta, sinks=sinks,
        recent=recent, marked=marked, storage=str(rng.choice(["f32", "bf16"])),
        key_law=str(rng.choice(["lognormal", "student_t", "lowrank"])), steps=2, seed_tag=300 + k)
    return w, codec, qjl, routing


@pytest.mark.parametrize("k", range(CASES))
def test_random_configuration(k):
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    w, codec, qjl, routing = _case(k)
    li = W.layer_inputs(w)
    cfg = H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, w.T, max(w.l1_size, 1), w.T + w.steps + 1, w.theta,
                        codec=codec, qjl=qjl, route_max=routing == "max", route_per_head=routing == "head")
    ctx = H.Context(cfg)
    cache = H.allocate_cache(ctx, w.B, w.T, l3_on_host=bool(k % 2 == 0))
    H.set_layer_inputs(cache, li.l1_mask, li.signs)
    S = W.qjl_matrix(w) if qjl else None
    if qjl:
        H.set_qjl_matrix(cache, S)
    dt = torch.bfloat16 if w.storage == "bf16" else torch.float32
    K = torch.from_numpy(np.ascontiguousarray(li.K, np.float32)).cuda().to(dt).contiguous()
    V = torch.from_numpy(np.ascontiguousarray(li.V, np.float32)).cuda().to(dt).contiguous()
    H.hsq_encode(ctx, cache, K, V)
    assert H.hsq_sync_status(ctx) == 0
    bufs = abi_buffers(cache)
    if qjl:
        for n in ("l1_qs", "l1_qn", "l3_qs", "l3_qn"):
            bufs[n] = cache.view(n).cpu().numpy()
        bufs["l1_qs"], bufs["l3_qs"] = bufs["l1_qs"].view(np.uint32), bufs["l3_qs"].view(np.uint32)
    view = O.cache_from_abi(bufs, li.l1_mask, li.signs, w.N, w.T, w.theta, codec=codec, qjl_S=S)
    ora = O.encode(li.K, li.V, li.l1_mask, li.signs, w.N, w.theta, codec=codec)
    for tier in ("l3_k", "l3_v"):
        bad, _, _ = code_mismatch(getattr(view, tier).codes, getattr(ora, tier).codes, getattr(ora, tier).y, 4,
                                  getattr(ora, tier).norms)
        assert bad == 0, f"{tier}: {bad} code mismatches outside the near-tie band"
    rows = w.Hq if routing == "head" else w.Hkv
    q, pos = W.queries(w, steps=2)
    for s in range(2):
        qd, pd = torch.from_numpy(q[s]).cuda(), torch.from_numpy(pos[s]).cuda()
        sel = torch.empty((w.B, rows, w.beta), dtype=torch.int32, device="cuda")
        scores = torch.empty((w.B, rows, cache.G), dtype=torch.float32, device="cuda")
        H.hsq_route(ctx, cache, qd, pd, sel, scores)
        out = torch.empty((w.B, w.Hq, 128), device="cuda")
        sel_s = torch.empty_like(sel)
        H.hsq_decode_step(ctx, cache, qd, pd, sel_s, out)
        assert H.hsq_sync_status(ctx) == 0
        assert torch.equal(sel_s, sel)
        osel, oscores = O.route(view, q[s], pos[s], w.beta, agg=routing)
        gs = scores.cpu().numpy()
        fin = np.isfinite(oscores)
        np.testing.assert_array_equal(np.isfinite(gs), fin)
        if fin.any():
            assert np.max(np.abs(gs[fin] - oscores[fin])) <= 1e-5 * np.sqrt(np.mean(oscores[fin] ** 2))
        gsel = sel.cpu().numpy()
        for b in range(w.B):
            for i in range(rows):
                bad, _ = sel_mismatch(gsel[b, i], osel[b, i], oscores[b, i], w.beta)
                assert bad == 0, f"step {s} (b={b}, row {i}): selection differs beyond near-ties"
        ref = O.decode_attn(view, q[s], pos[s], gsel.astype(np.int64))
        err = rel_l2(out.cpu().numpy(), ref)
        assert np.all(err <= 1e-3), f"step {s}: rel L2 {err.max():.3e} ({w}, {codec}, qjl={qjl}, {routing})"
    ctx.close()
