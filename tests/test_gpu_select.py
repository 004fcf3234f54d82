"""GPU top-beta selection: exact against a brute-force ranking of the GPU's
own fp32 routing scores.

hsq_route returns the fp32 scores it ranked, so its selection must be
exactly the beta largest of those scores (ties to the lower group,
ascending, -1 padded) -- no tie band is needed.  The fused decode step must
select the same groups bit for bit.  Besides the seeded workloads, the
summary keys of an encoded cache are overwritten to force the select's rare
paths: all scores equal, a few distinct values (crowded bins, equal keys at
the boundary), a dynamic range too wide for the first pass's fp32 bins, and
zero and negative scores.
"""

import numpy as np
import pytest

import oracle as O
import workloads as W
from hsq_harness import ensure_built, gpu_encode, make_ctx

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _check(ctx, cache, w, steps=2, G=None):
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    G = G or cache.G
    q, pos = W.queries(w, steps=steps)
    for s in range(steps):
        qd, pd = torch.from_numpy(q[s]).cuda(), torch.from_numpy(pos[s]).cuda()
        sel = torch.full((w.B, w.Hkv, w.beta), -7, dtype=torch.int32, device="cuda")
        scores = torch.empty((w.B, w.Hkv, G), dtype=torch.float32, device="cuda")
        H.hsq_route(ctx, cache, qd, pd, sel, scores)
        fsel = torch.full_like(sel, -7)
        out = torch.empty((w.B, w.Hq, 128), device="cuda")
        H.hsq_decode_step(ctx, cache, qd, pd, fsel, out)
        assert H.hsq_sync_status(ctx) == 0
        gs, gsel = scores.cpu().numpy(), sel.cpu().numpy()
        assert torch.equal(sel, fsel), "fused step and routing call select differently"
        for b in range(w.B):
            for h in range(w.Hkv):
                ref = O.select_top_beta(gs[b, h], np.isfinite(gs[b, h]), w.beta)
                np.testing.assert_array_equal(gsel[b, h], ref, err_msg=f"step {s} (b={b}, h={h})")


BASE = W.get_workload("tiny_1k")
SHAPES = {
    "g64": BASE,                                                          # 64 groups: one key per thread
    "g2048_n8": BASE.with_(name="g2048", T=16384, N=8, beta=64, seed_tag=41),   # 8 keys per thread
    "g4096_n8": BASE.with_(name="g4096", T=32768, N=8, beta=100, seed_tag=42, storage="bf16"),  # 16 per thread
    "beta_above_groups": BASE.with_(name="bbig", beta=70, seed_tag=43),   # beta > non-empty groups
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_select_is_exact_top_beta_of_gpu_scores(name):
    w = SHAPES[name]
    li = W.layer_inputs(w)
    ctx = make_ctx(w, steps=4)
    cache = gpu_encode(ctx, w, li)
    _check(ctx, cache, w)
    ctx.close()


def _overwrite(cache, mode, rng):
    """Rewrite the L2 summary keys (codes and norms) of every (b, h) in place."""
    import torch
    kc = cache.view("l2_kc")            # [B, H, G, 48] uint8
    kn = cache.view("l2_kn")            # [B, H, G] f32
    B, H, G, _ = kc.shape
    codes = kc.cpu().numpy()
    norms = kn.cpu().numpy()
    if mode == "all_equal":
        codes[:] = codes[:, :, :1]
        norms[:] = 1.0
    elif mode == "three_values":
        for g in range(G):
            codes[:, :, g] = codes[:, :, g % 3]
        norms[:] = 1.0
    elif mode == "crowded_boundary":
        # most groups share one summary; a few distinct ones above and below it
        base = codes[:, :, 5:6].copy()
        idx = rng.permutation(G)[: G - 12]
        codes[:, :, idx] = base
        norms[:, :, idx] = 1.0
    elif mode == "wide_range":
        norms[:] = (10.0 ** rng.uniform(-30, 30, size=norms.shape)).astype(np.float32)
    elif mode == "zeros_and_signs":
        norms[:] = rng.choice(np.array([0.0, -0.0, 1.0, 2.0], np.float32), size=norms.shape)
    kc.copy_(torch.from_numpy(codes))
    kn.copy_(torch.from_numpy(norms))


@pytest.mark.parametrize("shape", ["g64", "g2048_n8"])
@pytest.mark.parametrize("mode", ["all_equal", "three_values", "crowded_boundary", "wide_range", "zeros_and_signs"])
def test_select_rare_paths(shape, mode):
    w = SHAPES[shape].with_(beta=min(SHAPES[shape].beta, 40))
    li = W.layer_inputs(w)
    ctx = make_ctx(w, steps=4)
    cache = gpu_encode(ctx, w, li)
    _overwrite(cache, mode, np.random.default_rng(7))
    _check(ctx, cache, w)
    ctx.close()
