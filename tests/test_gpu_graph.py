"""The decode step under CUDA graph capture: hsq_decode_step enqueues only
stream work once its launch plan exists, so a captured step (here three
layers back to back, on static query buffers) replays with the same bits as
direct calls, step after step with new queries copied into the buffers.
"""

import numpy as np
import pytest

import oracle as O
import workloads as W
from hsq_harness import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def test_captured_step_replays_like_direct_calls():
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    w = W.get_workload("qwen3_0p6b_4k").with_(steps=4)
    li = W.layer_inputs(w, rope=lambda x, p: O.rope(x, p, w.theta))
    ctx = H.Context(H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, w.T, w.l1_size, w.T + w.steps + 1, w.theta))
    K = torch.from_numpy(li.K).cuda().to(torch.bfloat16).contiguous()
    V = torch.from_numpy(li.V).cuda().to(torch.bfloat16).contiguous()
    layers = []
    for l in range(3):
        mask, signs = (li.l1_mask, li.signs) if l == 0 else W.layer_meta(w, l)
        c = H.allocate_cache(ctx, w.B, w.T, with_staging=False)
        H.set_layer_inputs(c, mask, signs)
        H.hsq_encode(ctx, c, K, V)
        layers.append(c)
    q, pos = W.queries(w, steps=w.steps)
    qd, pd = torch.from_numpy(q).cuda(), torch.from_numpy(pos).cuda()
    q_in, p_in = torch.empty_like(qd[0]), torch.empty_like(pd[0])
    sels = [torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda") for _ in layers]
    outs = [torch.empty((w.B, w.Hq, 128), device="cuda") for _ in layers]

    def step():
        for c, sel, out in zip(layers, sels, outs):
            H.hsq_decode_step(ctx, c, q_in, p_in, sel, out)

    q_in.copy_(qd[0])
    p_in.copy_(pd[0])
    step()  # makes and caches the launch plan outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for s in range(w.steps):
        q_in.copy_(qd[s])
        p_in.copy_(pd[s])
        g.replay()
        torch.cuda.synchronize()
        got = [(x.clone(), y.clone()) for x, y in zip(sels, outs)]
        step()
        assert H.hsq_sync_status(ctx) == 0
        for (gs, go), sel, out in zip(got, sels, outs):
            assert torch.equal(gs, sel) and torch.equal(go, out)
        assert np.isfinite(outs[0].cpu().numpy()).all()
