"""Pins for the oracle's encode, routing, fetch and union attention.

The checks reduce special cases to library routines (torch's scaled-dot-
product attention in float64), to brute force (rank counting for top-beta),
and to bookkeeping invariants (each token is counted exactly once).
"""

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W


def _small(T=256, N=16, B=2, Hq=4, Hkv=2, marked=10, recent=32, sinks=4, beta=4, law="lognormal",
           storage="f32"):
    return W.Workload(name="pin", B=B, Hq=Hq, Hkv=Hkv, T=T, N=N, beta=beta, sinks=sinks,
                      recent=recent, marked=marked, storage=storage, key_law=law, steps=3,
                      seed_tag=99)


def _setup(w, quantize=True):
    li = W.layer_inputs(w)
    cache = O.encode(li.K, li.V, li.l1_mask, li.signs, w.N, w.theta, quantize=quantize)
    q, pos = W.queries(w, steps=2)
    return li, cache, q, pos


def _sdpa(q, keys, vals, scale):
    qt = torch.from_numpy(np.ascontiguousarray(q))[None, None, None]
    kt = torch.from_numpy(np.ascontiguousarray(keys))[None, None]
    vt = torch.from_numpy(np.ascontiguousarray(vals))[None, None]
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)[0, 0, 0].numpy()


# -- top-beta ----------------------------------------------------------------------

def _brute_select(s32, ne, beta):
    idx = [g for g in range(len(s32)) if ne[g]]
    chosen = []
    for g in idx:
        rank = sum(1 for g2 in idx if s32[g2] > s32[g] or (s32[g2] == s32[g] and g2 < g))
        if rank < beta:
            chosen.append(g)
    out = np.full(beta, -1)
    out[: len(chosen)] = sorted(chosen)
    return out


def test_top_beta_matches_brute_force_with_ties():
    rng = np.random.default_rng(0)
    for trial in range(200):
        G = int(rng.integers(1, 17))
        s = rng.integers(-3, 4, G).astype(np.float32)  # many ties
        ne = rng.random(G) > 0.2
        for beta in range(1, G + 3):
            np.testing.assert_array_equal(O.select_top_beta(s, ne, beta), _brute_select(s, ne, beta))


def test_route_score_is_sum_of_head_dots():
    w = _small()
    li, cache, q, pos = _setup(w)
    sel, scores = O.route(cache, q[0], pos[0], w.beta)
    # rotated-frame form: s_g = n_g * (sum_j Pi q_r_j) . c3[codes]  (Pi orthonormal)
    c3, _ = O.codebook(3)
    Pi = cache.Pi
    qr = O.rope(q[0].astype(np.float64), pos[0][:, None])
    for b in range(w.B):
        for h in range(w.Hkv):
            gt = (qr[b, h * w.r:(h + 1) * w.r] @ Pi.T).sum(0)
            alt = cache.l2_k.norms[b, h] * (c3[cache.l2_k.codes[b, h]] @ gt)
            ne = cache.l2_cnt[b] > 0
            np.testing.assert_allclose(scores[b, h][ne], alt[ne], rtol=1e-10, atol=1e-10)
            assert np.all(np.isneginf(scores[b, h][~ne]))


# -- attention special cases ---------------------------------------------------------

def test_beta_all_equals_softmax_over_dequantised_tokens():
    w = _small(beta=64)
    li, cache, q, pos = _setup(w)
    sel, _ = O.route(cache, q[0], pos[0], cache.G)   # every non-empty group fetched
    out = O.decode_attn(cache, q[0], pos[0], sel)
    Pi = cache.Pi
    qr = O.rope(q[0].astype(np.float64), pos[0][:, None])
    l3k = O.tq_decode(cache.l3_k.codes, cache.l3_k.norms, 4, Pi)
    l3v = O.tq_decode(cache.l3_v.codes, cache.l3_v.norms, 4, Pi)
    l1k = O.tq_decode(cache.l1_k.codes, cache.l1_k.norms, 4, Pi)
    l1v = O.tq_decode(cache.l1_v.codes, cache.l1_v.norms, 4, Pi)
    for b in range(w.B):
        p1 = np.nonzero(li.l1_mask[b])[0]
        rest = np.nonzero(~li.l1_mask[b])[0]
        for h in range(w.Hkv):
            keys = np.concatenate([l1k[b, h, : len(p1)], O.rope(l3k[b, h, rest], rest)])
            vals = np.concatenate([l1v[b, h, : len(p1)], l3v[b, h, rest]])
            for j in range(h * w.r, (h + 1) * w.r):
                ref = _sdpa(qr[b, j], keys, vals, 1 / np.sqrt(128))
                np.testing.assert_allclose(out[b, j], ref, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("T,N", [(256, 16), (250, 8)])
def test_quantisation_off_beta_all_is_exact_attention(T, N):
    w = _small(T=T, N=N)
    li, cache, q, pos = _setup(w, quantize=False)
    sel, _ = O.route(cache, q[0], pos[0], cache.G)
    out = O.decode_attn(cache, q[0], pos[0], sel)
    # exact attention over RoPE(K), V with the GQA heads expanded
    qr = torch.from_numpy(O.rope(q[0].astype(np.float64), pos[0][:, None]))       # [B, Hq, d]
    Kr = torch.from_numpy(O.rope(li.K.astype(np.float64), np.arange(T)))          # [B, Hkv, T, d]
    V = torch.from_numpy(li.V.astype(np.float64))
    Kx = Kr.repeat_interleave(w.r, dim=1)
    Vx = V.repeat_interleave(w.r, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(qr[:, :, None], Kx, Vx)[:, :, 0]
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_quantisation_off_each_token_counted_once():
    w = _small(T=250, N=8, beta=5)
    li, cache, q, pos = _setup(w, quantize=False)
    sel, _ = O.route(cache, q[0], pos[0], w.beta)
    for b in range(w.B):
        for h in range(w.Hkv):
            _, _, prov = O.attention_entries(cache, sel, b, h)
            seen = np.zeros(w.T, int)
            for kind, i in prov:
                if kind == 1:
                    seen[cache.l1_pos[b, i]] += 1
                elif kind == 2:
                    t = np.arange(i * w.N, min((i + 1) * w.N, w.T))
                    seen[t[~li.l1_mask[b, t]]] += 1
                else:
                    seen[i] += 1
            assert np.all(seen == 1)
            # a summary is the exact mean of its members' rotated keys
            Kr = O.rope(li.K[b, h].astype(np.float64), np.arange(w.T))
            for g in range(cache.G):
                t = np.arange(g * w.N, min((g + 1) * w.N, w.T))
                m = t[~li.l1_mask[b, t]]
                if len(m):
                    np.testing.assert_allclose(cache.l2_k.exact[b, h, g], Kr[m].mean(0), atol=1e-14)


def test_fetch_dequant_recovers_originals_and_masks():
    w = _small(T=250, N=8, beta=40)
    li, cache, q, pos = _setup(w)
    sel, _ = O.route(cache, q[0], pos[0], w.beta)
    k, v, valid = O.fetch_dequant(cache, sel)
    Pi = cache.Pi
    for b in range(w.B):
        for h in range(w.Hkv):
            for i, g in enumerate(sel[b, h]):
                for n in range(w.N):
                    t = g * w.N + n
                    if g < 0 or t >= w.T:
                        assert not valid[b, h, i, n] and not np.any(k[b, h, i, n])
                        continue
                    assert valid[b, h, i, n] == (not li.l1_mask[b, t])
                    x = O.tq_decode(cache.l3_k.codes[b, h, t], cache.l3_k.norms[b, h, t], 4, Pi)
                    np.testing.assert_allclose(k[b, h, i, n], O.rope(x, t), atol=1e-12)


def test_padding_when_beta_exceeds_nonempty_groups():
    w = _small(T=64, N=16, recent=32, marked=0, beta=6)
    li, cache, q, pos = _setup(w)
    ne = int((cache.l2_cnt[0] > 0).sum())
    sel, scores = O.route(cache, q[0], pos[0], w.beta)
    assert ne == 2  # groups 0 and 1 only (sinks sit inside group 0), the rest is recent
    assert np.all(sel[:, :, ne:] == -1) and np.all(sel[:, :, :ne] >= 0)


def test_all_tokens_in_l1_leaves_no_groups():
    w = _small(T=64, N=16, recent=60, marked=0, beta=3)
    li, cache, q, pos = _setup(w)
    assert np.all(cache.l2_cnt == 0)
    sel, _ = O.route(cache, q[0], pos[0], w.beta)
    assert np.all(sel == -1)
    out = O.decode_attn(cache, q[0], pos[0], sel)
    # attention over L1 only (every token of the context)
    Pi = cache.Pi
    qr = O.rope(q[0].astype(np.float64), pos[0][:, None])
    l1k = O.tq_decode(cache.l1_k.codes, cache.l1_k.norms, 4, Pi)
    l1v = O.tq_decode(cache.l1_v.codes, cache.l1_v.norms, 4, Pi)
    ref = _sdpa(qr[0, 0], l1k[0, 0], l1v[0, 0], 1 / np.sqrt(128))
    np.testing.assert_allclose(out[0, 0], ref, rtol=1e-10)


def test_empty_l1_set():
    w = _small(T=128, N=16, recent=0, marked=0, sinks=0, beta=2)
    li, cache, q, pos = _setup(w)
    assert np.all(cache.l1_count == 0) and np.all(cache.l2_cnt == 16)
    sel, _ = O.route(cache, q[0], pos[0], w.beta)
    out = O.decode_attn(cache, q[0], pos[0], sel)
    assert np.all(np.isfinite(out))


def test_summary_codes_for_empty_groups():
    w = _small(T=64, N=16, recent=32, marked=0, beta=2)
    li, cache, q, pos = _setup(w)
    empty = cache.l2_cnt == 0
    assert np.all(cache.l2_k.codes[np.broadcast_to(empty[:, None], cache.l2_k.norms.shape)] == 3)
    assert np.all(cache.l2_k.norms[:, :, 2:] == 0)


def test_abi_layout_round_trip():
    w = _small(T=250, N=8)
    li, cache, q, pos = _setup(w)
    bufs = O.cache_to_abi(cache)
    assert bufs["l3"].shape == (w.B, w.Hkv, cache.G, O.record_bytes(w.N))
    back = O.cache_from_abi(bufs, li.l1_mask, li.signs, w.N, w.T)
    for name in ("l1_k", "l1_v", "l2_k", "l2_v", "l3_k", "l3_v"):
        a, b2 = getattr(cache, name), getattr(back, name)
        np.testing.assert_array_equal(a.codes, b2.codes)
        np.testing.assert_array_equal(a.norms, b2.norms)
    sel, _ = O.route(cache, q[1], pos[1], w.beta)
    np.testing.assert_array_equal(O.decode_attn(cache, q[1], pos[1], sel),
                                  O.decode_attn(back, q[1], pos[1], sel))
    # the ragged last record holds the zero-vector encoding past T
    last = bufs["l3"][0, 0, -1]
    tail = O.unpack_codes(last[: 8 * 64].reshape(8, 64), 4)[250 - 31 * 8:]
    assert np.all(tail == 7)


def test_needle_group_is_routed_first_step():
    # the 32K workload at reduced context keeps its needle construction
    w = W.get_workload("qwen3_8b_32k", T=4096, marked=40, Hkv=2, Hq=8)
    rope = lambda x, p: O.rope(x, p, w.theta)
    li = W.layer_inputs(w, rope=rope)
    cache = O.encode(li.K, li.V, li.l1_mask, li.signs, w.N, w.theta)
    q, pos = W.queries(w, steps=1)
    sel, scores = O.route(cache, q[0], pos[0], w.beta)
    for h in range(w.Hkv):
        g = li.needle_group[0, h]
        assert g in sel[0, h]
        assert scores[0, h, g] == np.max(scores[0, h])


# -- routing by the best query head (route_max) ------------------------------------

def test_max_routing_is_the_best_single_head():
    """A KV head's max score is, group by group, the largest of the scores its
    query heads get when each routes alone (one query head per KV head, where
    sum and max coincide)."""
    w = _small(Hq=8, Hkv=2)
    li, cache, q, pos = _setup(w)
    r = w.Hq // w.Hkv
    sel_max, s_max = O.route(cache, q[0], pos[0], w.beta, agg="max")
    singles = []
    for j in range(r):
        qj = q[0][:, [h * r + j for h in range(w.Hkv)]]      # head j of every KV head
        singles.append(O.route(cache, qj, pos[0], w.beta, agg="sum")[1])
    np.testing.assert_allclose(s_max, np.max(singles, axis=0), rtol=1e-12, atol=0)
    # and the selection is the top-beta of those scores
    for b in range(w.B):
        for h in range(w.Hkv):
            ne = cache.l2_cnt[b] > 0
            np.testing.assert_array_equal(sel_max[b, h], _brute_select(s_max[b, h].astype(np.float32), ne, w.beta))


def test_max_and_sum_routing_agree_with_one_query_head_per_kv_head():
    w = _small(Hq=2, Hkv=2)
    li, cache, q, pos = _setup(w)
    a = O.route(cache, q[0], pos[0], w.beta, agg="sum")
    b = O.route(cache, q[0], pos[0], w.beta, agg="max")
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_allclose(a[1], b[1], rtol=1e-15, atol=0)
    with pytest.raises(ValueError):
        O.route(cache, q[0], pos[0], w.beta, agg="mean")


# -- per-query-head routing (each query head selects and attends by itself) ---------

def test_per_head_routing_is_single_head_routing_of_each_query_head():
    """Query head j's scores and selection equal the default routing of a
    context with one query head per KV head made of head j alone, and its
    attention output equals that context's output for head j."""
    w = _small(Hq=8, Hkv=2)
    li, cache, q, pos = _setup(w)
    r = w.Hq // w.Hkv
    sel, scores = O.route(cache, q[0], pos[0], w.beta, agg="head")
    assert sel.shape == (w.B, w.Hq, w.beta) and scores.shape == (w.B, w.Hq, cache.G)
    out = O.decode_attn(cache, q[0], pos[0], sel)
    for j in range(r):
        heads = [h * r + j for h in range(w.Hkv)]
        s1, sc1 = O.route(cache, q[0][:, heads], pos[0], w.beta, agg="sum")
        np.testing.assert_array_equal(sel[:, heads], s1)
        np.testing.assert_allclose(scores[:, heads], sc1, rtol=1e-15, atol=0)
        o1 = O.decode_attn(cache, q[0][:, heads], pos[0], s1)
        np.testing.assert_allclose(out[:, heads], o1, rtol=1e-13, atol=1e-15)


def test_per_head_routing_of_identical_query_heads_is_the_shared_routing():
    """With the query heads of a KV head all equal (r a power of two, so the
    float32 scores scale exactly), every head selects what the sum selects
    and the outputs are the shared selection's outputs."""
    w = _small(Hq=8, Hkv=2)
    li, cache, q, pos = _setup(w)
    r = w.Hq // w.Hkv
    qs = np.repeat(q[0][:, ::r], r, axis=1)               # head h*r of each KV head, repeated
    shared, _ = O.route(cache, qs, pos[0], w.beta, agg="sum")
    per, _ = O.route(cache, qs, pos[0], w.beta, agg="head")
    np.testing.assert_array_equal(per, np.repeat(shared, r, axis=1))
    np.testing.assert_allclose(O.decode_attn(cache, qs, pos[0], per),
                               O.decode_attn(cache, qs, pos[0], shared), rtol=1e-13, atol=1e-15)


def test_per_head_selection_is_the_brute_force_top_beta_of_its_dots():
    w = _small(Hq=4, Hkv=2, T=200, N=8, beta=5)
    li, cache, q, pos = _setup(w)
    sel, scores = O.route(cache, q[0], pos[0], w.beta, agg="head")
    khat = cache.l2_k.vectors(cache.Pi)
    for b in range(w.B):
        for j in range(w.Hq):
            h = j // (w.Hq // w.Hkv)
            qr = O.rope(q[0][b, j].astype(np.float64), pos[0][b], w.theta)
            ne = cache.l2_cnt[b] > 0
            dots = np.array([sum(khat[b, h, g, i] * qr[i] for i in range(128)) for g in range(cache.G)])
            np.testing.assert_allclose(scores[b, j][ne], dots[ne], rtol=1e-12, atol=1e-12)
            assert np.all(np.isneginf(scores[b, j][~ne]))
            np.testing.assert_array_equal(sel[b, j], _brute_select(scores[b, j].astype(np.float32), ne, w.beta))


def test_per_head_routing_with_residual_sketches_is_single_head_attention():
    """TQ-QKV under per-query-head routing: each query head's output equals the
    shared-routing output of a one-head-per-KV-head context made of that head,
    sketch terms included (the sketches follow the KV head, not the row)."""
    w = _small(Hq=8, Hkv=2)
    li = W.layer_inputs(w)
    S = np.random.default_rng(3).standard_normal((128, 128))
    cache = O.encode(li.K, li.V, li.l1_mask, li.signs, w.N, w.theta, qjl_S=S)
    plain = O.encode(li.K, li.V, li.l1_mask, li.signs, w.N, w.theta)
    q, pos = W.queries(w, steps=1)
    r = w.Hq // w.Hkv
    sel, _ = O.route(cache, q[0], pos[0], w.beta, agg="head")
    out = O.decode_attn(cache, q[0], pos[0], sel)
    for j in range(r):
        heads = [h * r + j for h in range(w.Hkv)]
        o1 = O.decode_attn(cache, q[0][:, heads], pos[0], sel[:, heads])
        np.testing.assert_allclose(out[:, heads], o1, rtol=1e-13, atol=1e-15)
    # and the sketch terms are in: the same selection without them gives another output
    assert np.max(np.abs(out - O.decode_attn(plain, q[0], pos[0], sel))) > 1e-3
