"""GPU parity of the prefill (hsq_prefill): the tensor-core causal attention
against the float64 oracle (prefill_attn) on the same bf16 inputs, within
1e-3 relative L2 per (sequence, query head, position); with a cache, the
encode written by the same pass equals hsq_encode's bit for bit.

Shapes: 128-multiple contexts (several query and key tiles), ragged contexts
(a partial last tile, key rows past T read as zeros), head ratios 1, 4 and 5,
two sequences."""

import numpy as np
import pytest

import oracle as O
import workloads as W
from hsq_harness import abi_buffers, ensure_built, make_ctx, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _bf16(x):
    return W.round_to_bf16(np.asarray(x, np.float32))


def _inputs(B, Hq, Hkv, T, seed):
    rng = np.random.default_rng(seed)
    Q = _bf16(rng.standard_normal((B, Hq, T, 128)))
    K = _bf16(rng.standard_normal((B, Hkv, T, 128)))
    V = _bf16(rng.standard_normal((B, Hkv, T, 128)))
    return Q, K, V


def _run(ctx, B, T, Q, K, V, cache=None):
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    ws = torch.empty(H.hsq_prefill_workspace_size(ctx, B, T), dtype=torch.uint8, device="cuda")
    tq, tk, tv = (torch.from_numpy(x).cuda().to(torch.bfloat16).contiguous() for x in (Q, K, V))
    out = torch.full((B, Q.shape[1], T, 128), float("nan"), device="cuda")
    H.hsq_prefill(ctx, cache, tq, tk, tv, out, ws)
    assert H.hsq_sync_status(ctx) == 0
    return out.cpu().numpy()


CASES = {
    "r4_t256": dict(B=1, Hq=4, Hkv=1, T=256),
    "r1_b2_t384": dict(B=2, Hq=2, Hkv=2, T=384),
    "r5_ragged_t200": dict(B=1, Hq=5, Hkv=1, T=200),
    "r4_ragged_t1001": dict(B=1, Hq=4, Hkv=1, T=1001),
    "r2_b2_tiny_t37": dict(B=2, Hq=4, Hkv=2, T=37),   # one query tile, one partial key tile
    "r8_t640": dict(B=1, Hq=8, Hkv=1, T=640),
}


@pytest.mark.parametrize("name", list(CASES))
def test_prefill_attention_matches_oracle(name):
    cs = CASES[name]
    B, Hq, Hkv, T = cs["B"], cs["Hq"], cs["Hkv"], cs["T"]
    w = W.get_workload("tiny_1k").with_(B=B, Hq=Hq, Hkv=Hkv, T=T, beta=4, recent=16, marked=3)
    ctx = make_ctx(w)
    Q, K, V = _inputs(B, Hq, Hkv, T, seed=len(name))
    got = _run(ctx, B, T, Q, K, V)
    ref = O.prefill_attn(Q, K, V, w.theta)
    err = rel_l2(got, ref)
    assert np.all(np.isfinite(got))
    assert err.max() <= 1e-3, f"worst relative L2 {err.max():.3e}"
    print(f"[{name}] prefill attention: worst rel L2 {err.max():.2e}, mean {err.mean():.2e}")
    ctx.close()


@pytest.mark.parametrize("name", ["tiny_1k", "ragged"])
def test_prefill_with_cache_encodes_like_hsq_encode(name):
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    w = W.get_workload("tiny_1k")
    if name == "ragged":
        w = w.with_(name="ragged_pf", T=1000, N=8, Hq=8, Hkv=2, storage="bf16", seed_tag=21)
    w = w.with_(storage="bf16")
    li = W.layer_inputs(w)
    ctx = make_ctx(w)
    rng = np.random.default_rng(5)
    Q = _bf16(rng.standard_normal((w.B, w.Hq, w.T, 128)))
    caches = []
    for fused in (True, False):
        cache = H.allocate_cache(ctx, w.B, w.T, l3_on_host=True)
        H.set_layer_inputs(cache, li.l1_mask, li.signs)
        if fused:
            got = _run(ctx, w.B, w.T, Q, li.K, li.V, cache=cache)
        else:
            H.hsq_encode(ctx, cache, torch.from_numpy(li.K).cuda().to(torch.bfloat16).contiguous(),
                         torch.from_numpy(li.V).cuda().to(torch.bfloat16).contiguous())
            torch.cuda.synchronize()
        caches.append(abi_buffers(cache))
    for k in caches[0]:
        np.testing.assert_array_equal(caches[0][k], caches[1][k], err_msg=k)
    ref = O.prefill_attn(Q, li.K, li.V, w.theta)
    err = rel_l2(got, ref)
    assert err.max() <= 1e-3, f"worst relative L2 {err.max():.3e}"
    # attention alone gives the same output as the fused call
    alone = _run(ctx, w.B, w.T, Q, li.K, li.V)
    np.testing.assert_array_equal(alone, got)
    ctx.close()


def test_prefill_full_size_8b_32k_sampled_rows():
    """The 8B-shaped 32K prompt (B1, Hq 32, Hkv 8) in the launch configuration the
    benchmark times: the first and the last 128 query rows of query heads 0-3 (KV
    head 0) and 28-31 (KV head 7) against the oracle (the last rows attend to all
    32768 keys)."""
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    B, Hq, Hkv, T = 1, 32, 8, 32768
    w = W.get_workload("qwen3_8b_32k")
    ctx = make_ctx(w)
    rng = np.random.default_rng(77)
    Q = _bf16(rng.standard_normal((B, Hq, T, 128), dtype=np.float32))
    K = _bf16(rng.standard_normal((B, Hkv, T, 128), dtype=np.float32))
    V = _bf16(rng.standard_normal((B, Hkv, T, 128), dtype=np.float32))
    got = _run(ctx, B, T, Q, K, V)
    assert np.all(np.isfinite(got))
    worst = 0.0
    for h in (0, 7):
        js = slice(4 * h, 4 * h + 4)
        for start in (0, T - 128):
            ref = O.prefill_attn(Q[:, js, start:start + 128], K[:, h:h + 1], V[:, h:h + 1], w.theta,
                                 q_start=start)
            err = rel_l2(got[:, js, start:start + 128], ref)
            worst = max(worst, float(err.max()))
            assert err.max() <= 1e-3, f"KV head {h}, rows from {start}: rel L2 {err.max():.3e}"
    print(f"[prefill 8B/32K] worst sampled rel L2 {worst:.2e}")
    ctx.close()


def test_prefill_with_tq_qkv_cache_sketches_like_hsq_encode():
    """With cfg.qjl the fused prefill also writes the key-residual sketches, and
    they equal hsq_encode's bit for bit (the same codes, the same sketch pass)."""
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    w = W.get_workload("tiny_1k").with_(name="ragged_pf_qjl", T=1000, N=8, Hq=8, Hkv=2, storage="bf16",
                                        seed_tag=22)
    li = W.layer_inputs(w)
    cfg = H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, w.T, max(w.l1_size, 1), w.T + w.steps + 1, w.theta,
                        qjl=True)
    ctx = H.Context(cfg)
    S = W.qjl_matrix(w)
    Q = _bf16(np.random.default_rng(6).standard_normal((w.B, w.Hq, w.T, 128)))
    got = []
    for fused in (True, False):
        cache = H.allocate_cache(ctx, w.B, w.T, l3_on_host=True)
        H.set_layer_inputs(cache, li.l1_mask, li.signs)
        H.set_qjl_matrix(cache, S)
        if fused:
            _run(ctx, w.B, w.T, Q, li.K, li.V, cache=cache)
        else:
            H.hsq_encode(ctx, cache, torch.from_numpy(li.K).cuda().to(torch.bfloat16).contiguous(),
                         torch.from_numpy(li.V).cuda().to(torch.bfloat16).contiguous())
            torch.cuda.synchronize()
        bufs = abi_buffers(cache)
        for n in ("l1_qs", "l1_qn", "l3_qs", "l3_qn"):
            bufs[n] = cache.view(n).cpu().numpy()
        got.append(bufs)
    assert H.hsq_sync_status(ctx) == 0
    for k in got[0]:
        np.testing.assert_array_equal(got[0][k], got[1][k], err_msg=k)
    ctx.close()
