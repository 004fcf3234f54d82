"""Pins for the oracle's prefill attention (dense causal softmax attention
over RoPE'd queries and keys, GQA).

Checked against torch's scaled_dot_product_attention (causal, float64) on
inputs rotated by a complex-number RoPE written here, against closed forms
(first row = the first value; zero keys = the running mean of the values),
against causality (later tokens do not move earlier outputs) and against the
GQA head mapping (equal to one-KV-head-per-query-head attention on expanded
K/V).
"""

import numpy as np
import pytest
import torch

import oracle as O


def _inputs(B=2, Hq=4, Hkv=2, T=37, d=128, seed=0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, Hq, T, d)), rng.standard_normal((B, Hkv, T, d)),
            rng.standard_normal((B, Hkv, T, d)))


def _rope_complex(x, theta=1.0e6):
    # rotate-half pairing (i, i + d/2) as the complex number x_i + j x_{i+d/2}
    # multiplied by exp(j t omega_i)
    d = x.shape[-1]
    h = d // 2
    t = np.arange(x.shape[-2])[:, None]
    w = theta ** (-np.arange(h) * 2.0 / d)
    z = (x[..., :h] + 1j * x[..., h:]) * np.exp(1j * t * w)
    return np.concatenate([z.real, z.imag], axis=-1)


def test_prefill_matches_torch_sdpa_causal():
    Q, K, V = _inputs()
    r = Q.shape[1] // K.shape[1]
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(_rope_complex(Q)),
        torch.from_numpy(np.repeat(_rope_complex(K), r, axis=1)),
        torch.from_numpy(np.repeat(V, r, axis=1)), is_causal=True).numpy()
    got = O.prefill_attn(Q, K, V)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_prefill_first_row_and_zero_keys():
    Q, K, V = _inputs(B=1, Hq=2, Hkv=1, T=20)
    got = O.prefill_attn(Q, K, V)
    np.testing.assert_allclose(got[:, :, 0], np.repeat(V[:, :, 0], 2, axis=1), rtol=0, atol=1e-14)
    # zero keys: uniform weights over 0..t, the running mean of the values
    got0 = O.prefill_attn(Q, np.zeros_like(K), V)
    run_mean = np.cumsum(V, axis=2) / np.arange(1, 21)[None, None, :, None]
    np.testing.assert_allclose(got0, np.repeat(run_mean, 2, axis=1), rtol=1e-13, atol=1e-13)


def test_prefill_is_causal():
    Q, K, V = _inputs(B=1, T=30)
    base = O.prefill_attn(Q, K, V)
    K2, V2 = K.copy(), V.copy()
    K2[:, :, 18:] += 5.0
    V2[:, :, 18:] *= -3.0
    moved = O.prefill_attn(Q, K2, V2)
    np.testing.assert_array_equal(moved[:, :, :18], base[:, :, :18])
    assert np.abs(moved[:, :, 18:] - base[:, :, 18:]).max() > 1e-3


def test_prefill_gqa_head_mapping():
    Q, K, V = _inputs(B=1, Hq=6, Hkv=2, T=25)
    got = O.prefill_attn(Q, K, V)
    exp = O.prefill_attn(Q, np.repeat(K, 3, axis=1), np.repeat(V, 3, axis=1))
    np.testing.assert_allclose(got, exp, rtol=0, atol=1e-15)
    # query heads 0-2 read KV head 0 and 3-5 KV head 1: swapping both halves
    # of the query heads and the two KV heads swaps the output halves
    swapped = O.prefill_attn(Q[:, [3, 4, 5, 0, 1, 2]], K[:, ::-1], V[:, ::-1])
    np.testing.assert_allclose(swapped[:, 3:], got[:, :3], rtol=0, atol=1e-15)
    np.testing.assert_allclose(swapped[:, :3], got[:, 3:], rtol=0, atol=1e-15)


def test_prefill_returns_the_encode_of_its_kv():
    Q, K, V = _inputs(B=1, Hq=2, Hkv=1, T=64)
    mask = np.zeros((1, 64), bool)
    mask[0, [0, 1, 40, 63]] = True
    signs = np.where(np.random.default_rng(3).random(128) < 0.5, -1, 1).astype(np.int8)
    o, cache = O.prefill(Q, K, V, mask, signs, 16)
    ref = O.encode(K, V, mask, signs, 16)
    np.testing.assert_array_equal(o, O.prefill_attn(Q, K, V))
    for tier in ("l1_k", "l1_v", "l2_k", "l2_v", "l3_k", "l3_v"):
        np.testing.assert_array_equal(getattr(cache, tier).codes, getattr(ref, tier).codes)


def test_prefill_query_rows_from_a_later_start():
    # rows a..b of the whole prompt's output equal the attention of those queries alone
    Q, K, V = _inputs(B=1, Hq=4, Hkv=2, T=40)
    full = O.prefill_attn(Q, K, V)
    part = O.prefill_attn(Q[:, :, 25:33], K[:, :, :33], V[:, :, :33], q_start=25)
    np.testing.assert_allclose(part, full[:, :, 25:33], rtol=1e-12, atol=1e-13)
    # against torch SDPA with an explicit mask for the shifted query positions
    r = 2
    tq, tk = np.arange(25, 33), np.arange(33)
    q = _rope_complex(np.concatenate([np.zeros((1, 4, 25, 128)), Q[:, :, 25:33]], axis=2))[:, :, 25:]
    mask = torch.from_numpy(tk[None, :] <= tq[:, None])
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(np.repeat(_rope_complex(K[:, :, :33]), r, axis=1)),
        torch.from_numpy(np.repeat(V[:, :, :33], r, axis=1)), attn_mask=mask).numpy()
    np.testing.assert_allclose(part, ref, rtol=1e-12, atol=1e-12)
    with pytest.raises(ValueError):
        O.prefill_attn(Q[:, :, 30:40], K[:, :, :35], V[:, :, :35], q_start=30)
