"""Pins for the oracle's codec variants and codec diagnostics.

Plain-KV ("Ablation, Statistical Inference, and Validation for KV-Cache
Compression", key contributions, item 1: scalar quantisation without the
rotation) against closed forms: an axis vector, permutation equivariance,
signs not applied, and -- on isotropic input, where both codecs see the
uniform law on the sphere -- the Lloyd-Max distortion of the codebook
integrated from the coordinate density.  The relMSE / cosine diagnostics
(same page, experimental setup, metrics) against hand-computed cases.
"""

import numpy as np
import pytest
from scipy import integrate

import oracle as O
import workloads as W

D = 128


def _signs(seed=5):
    rng = np.random.default_rng(seed)
    return np.where(rng.integers(0, 2, D) == 1, 1, -1).astype(np.int8)


def _roundtrip(x, bits, codec, signs):
    Pi = O.codec_rotation(signs, codec)
    codes, norms, _ = O.tq_encode(x, bits, Pi)
    return codes, norms, O.tq_decode(codes, norms, bits, Pi)


# -- codec diagnostics ----------------------------------------------------------

def test_codec_errors_closed_forms():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((50, D))
    e = O.codec_errors(x, x)
    assert e["relmse"] == 0.0 and abs(e["cosine"] - 1.0) < 1e-15
    e = O.codec_errors(x, 2.0 * x)  # |2x - x|^2 / |x|^2 = 1, same direction
    assert abs(e["relmse"] - 1.0) < 1e-14 and abs(e["cosine"] - 1.0) < 1e-14
    e = O.codec_errors(x, -x)       # |-2x|^2 / |x|^2 = 4, opposite direction
    assert abs(e["relmse"] - 4.0) < 1e-14 and abs(e["cosine"] + 1.0) < 1e-14
    # an orthogonal reconstruction of the same norm: relMSE 2, cosine 0
    x2 = np.zeros_like(x)
    x2[:, :2] = x[:, :2]
    y = np.zeros_like(x)
    y[:, 0], y[:, 1] = x[:, 1], -x[:, 0]
    e = O.codec_errors(x2, y)
    assert abs(e["relmse"] - 2.0) < 1e-14 and abs(e["cosine"]) < 1e-14
    # relMSE is a ratio of sums (vectors weigh by their energy), cosine a plain mean
    a = np.zeros((2, D)); a[0, 0] = 1.0; a[1, 0] = 3.0
    b = np.zeros((2, D)); b[0, 0] = 2.0; b[1, 0] = 3.0; b[1, 1] = 3.0
    e = O.codec_errors(a, b)
    assert abs(e["relmse"] - (1.0 + 9.0) / (1.0 + 9.0)) < 1e-15
    assert abs(e["cosine"] - (1.0 + 1.0 / np.sqrt(2.0)) / 2.0) < 1e-15
    # zero vectors count in relMSE's sums but not in the cosine mean
    e = O.codec_errors(np.vstack([a, np.zeros(D)]), np.vstack([b, np.ones(D)]))
    assert abs(e["relmse"] - (10.0 + D) / 10.0) < 1e-13
    assert abs(e["cosine"] - (1.0 + 1.0 / np.sqrt(2.0)) / 2.0) < 1e-15


# -- Plain-KV codec ---------------------------------------------------------------

@pytest.mark.parametrize("bits", [3, 4])
def test_plain_axis_vector_closed_form(bits):
    """x = n e_i: the unit vector is e_i itself.  Coordinate i lies above
    every boundary (top code); a zero coordinate lies above the L/2 - 1
    negative boundaries only (the middle boundary is 0), so it takes code
    L/2 - 1 and decodes to the negative centroid nearest zero."""
    c, tau = O.codebook(bits)
    L = 1 << bits
    assert tau[L // 2 - 1] == 0.0
    for i in (0, 37, 127):
        x = np.zeros(D)
        x[i] = 3.5
        codes, norms, xh = _roundtrip(x, bits, "plain", _signs())
        want = np.full(D, L // 2 - 1)
        want[i] = L - 1
        np.testing.assert_array_equal(codes, want)
        assert norms == np.float32(3.5)
        ref = np.full(D, 3.5 * c[L // 2 - 1])
        ref[i] = 3.5 * c[L - 1]
        np.testing.assert_allclose(xh, ref, rtol=0, atol=1e-15)


def test_tq_axis_vector_closed_form():
    """Under TurboQuant the same axis vector rotates to coordinates +-1/sqrt(d);
    the symmetric codebook maps them to +-c(1/sqrt(d)) and the inverse
    rotation returns n sqrt(d) c(1/sqrt(d)) e_i exactly along the axis."""
    c, tau = O.codebook(4)
    a = 1.0 / np.sqrt(D)
    ca = c[int(np.sum(np.float32(a) > tau.astype(np.float32)))]
    for i in (0, 37, 127):
        x = np.zeros(D)
        x[i] = 3.5
        _, _, xh = _roundtrip(x, 4, "tq", _signs())
        ref = np.zeros(D)
        ref[i] = 3.5 * np.sqrt(D) * ca
        np.testing.assert_allclose(xh, ref, rtol=0, atol=1e-13)


def test_plain_codes_are_permutation_equivariant_and_tq_codes_are_not():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((20, D))
    perm = rng.permutation(D)
    cp, _, _ = _roundtrip(x, 4, "plain", _signs())
    cq, _, _ = _roundtrip(x[:, perm], 4, "plain", _signs())
    np.testing.assert_array_equal(cq, cp[:, perm])
    tp, _, _ = _roundtrip(x, 4, "tq", _signs())
    tq_, _, _ = _roundtrip(x[:, perm], 4, "tq", _signs())
    assert np.mean(tq_ != tp[:, perm]) > 0.5


def test_plain_ignores_the_signs():
    rng = np.random.default_rng(8)
    x = np.abs(rng.standard_normal((20, D))) + 1e-3  # every coordinate positive
    a, _, xa = _roundtrip(x, 4, "plain", _signs(1))
    b, _, xb = _roundtrip(x, 4, "plain", _signs(2))
    np.testing.assert_array_equal(a, b)
    assert np.all(a >= 8)  # positive coordinates land in the upper half
    np.testing.assert_array_equal(xa, xb)


def _lloyd_max_distortion(bits):
    """E[(Y - Q(Y))^2] under the coordinate density, cell by cell."""
    c, tau = O.codebook(bits)
    edges = np.r_[-1.0, tau, 1.0]
    tot = 0.0
    for k in range(len(c)):
        val, _ = integrate.quad(lambda y: (y - c[k]) ** 2 * O.coordinate_pdf(y), edges[k], edges[k + 1],
                                epsabs=1e-14, epsrel=1e-12, limit=200)
        tot += val
    return tot


@pytest.mark.parametrize("bits", [3, 4])
def test_isotropic_distortion_matches_the_codebook_for_both_codecs(bits):
    """Gaussian x: x/|x| is uniform on the sphere before and after any
    orthogonal Pi, so both codecs' relMSE estimates d E[(Y - Q(Y))^2]."""
    rng = np.random.default_rng(11 + bits)
    x = rng.standard_normal((6000, D))
    want = D * _lloyd_max_distortion(bits)
    for codec in O.CODECS:
        _, norms, xh = _roundtrip(x, bits, codec, _signs())
        n = norms.astype(np.float64)
        per = np.sum((xh / n[:, None] - x / n[:, None]) ** 2, axis=1)  # |Q(y) - y|^2
        se = per.std(ddof=1) / np.sqrt(len(per))
        assert abs(per.mean() - want) <= 5 * se, (codec, per.mean(), want, se)
        rel = O.codec_errors(x, xh)["relmse"]
        assert abs(rel - want) <= 0.03 * want, (codec, rel, want)


def test_heavy_tailed_keys_favour_the_rotation():
    """Keys with a few large channels: without the rotation those channels
    saturate the codebook; with it their energy is spread over all
    coordinates (the page's finding for heavy-tailed data)."""
    w = W.get_workload("tiny_1k").with_(key_law="student_t", T=512, B=1, Hkv=1, Hq=4)
    K = W.layer_inputs(w).K[0, 0].astype(np.float64)
    errs = {codec: O.codec_errors(K, _roundtrip(K, 4, codec, _signs())[2]) for codec in O.CODECS}
    assert errs["plain"]["relmse"] > 3.0 * errs["tq"]["relmse"], errs
    assert errs["plain"]["cosine"] < errs["tq"]["cosine"], errs


def test_plain_encode_tiers_and_abi_round_trip():
    """encode(codec="plain") stores every tier unrotated; the packed ABI
    layout is codec-independent and reads back to the same vectors."""
    w = W.get_workload("tiny_1k").with_(T=300, B=1, Hkv=2, Hq=4, N=16)
    li = W.layer_inputs(w, rope=lambda x, p: O.rope(x, p, w.theta))
    ora = O.encode(li.K, li.V, li.l1_mask, li.signs, w.N, w.theta, codec="plain")
    assert ora.codec == "plain"
    np.testing.assert_array_equal(ora.Pi, np.eye(D))
    codes, norms, _ = O.tq_encode(li.V, 4, np.eye(D))
    np.testing.assert_array_equal(ora.l3_v.codes, codes)
    np.testing.assert_array_equal(ora.l3_v.norms, norms)
    back = O.cache_from_abi(O.cache_to_abi(ora), li.l1_mask, li.signs, w.N, w.T, w.theta, codec="plain")
    np.testing.assert_array_equal(back.l3_k.vectors(back.Pi), ora.l3_k.vectors(ora.Pi))
    np.testing.assert_array_equal(back.l2_k.vectors(back.Pi), ora.l2_k.vectors(ora.Pi))
    q, pos = W.queries(w, steps=1)
    sel, _ = O.route(ora, q[0], pos[0], w.beta)
    np.testing.assert_allclose(O.decode_attn(back, q[0], pos[0], sel), O.decode_attn(ora, q[0], pos[0], sel),
                               rtol=0, atol=1e-13)


# -- TQ-QKV: the 1-bit residual sketch of the keys --------------------------------

def test_qjl_estimator_is_unbiased_with_the_closed_form_variance():
    """For S with i.i.d. N(0, 1) entries, sqrt(pi/2)/m |rho| <S q, sign(S rho)>
    has mean q . rho and variance ((pi/2)|q|^2|rho|^2 - (q . rho)^2) / m."""
    rng = np.random.default_rng(21)
    q, rho = rng.standard_normal(D), rng.standard_normal(D)
    rho = 0.7 * q + rho           # correlated, so q . rho is far from 0
    m, draws = 128, 3000
    est = []
    for _ in range(draws // 500):
        S = rng.standard_normal((500, m, D))
        sk = O.Sketch(bits=np.einsum("kmd,d->km", S, rho) >= 0,
                      norm=np.full(500, np.linalg.norm(rho), np.float32))
        est.append(O.qjl_estimate(np.einsum("kmd,d->km", S, q), sk))
    est = np.concatenate(est)
    want = q @ rho
    var = ((np.pi / 2) * (q @ q) * (rho @ rho) - want ** 2) / m
    se = np.sqrt(var / draws)
    assert abs(est.mean() - want) <= 4 * se, (est.mean(), want, se)
    assert abs(est.var(ddof=1) / var - 1.0) <= 0.1, (est.var(ddof=1), var)
    # one draw through qjl_sketch itself: the bit convention and the stored norm
    S = rng.standard_normal((m, D))
    sk = O.qjl_sketch(rho, S)
    np.testing.assert_array_equal(sk.bits, S @ rho >= 0)
    assert sk.norm == np.float32(np.linalg.norm(rho))
    zero = O.qjl_sketch(np.zeros(D), S)
    assert zero.norm == 0 and O.qjl_estimate(S @ q, zero) == 0.0


def test_qjl_corrected_logits_are_unbiased_for_the_exact_logits():
    """Averaged over sketch matrices, a token entry's corrected dot equals the
    dot with the unquantised key (RoPE'd for fetched tokens) -- the residual is
    sketched in the frame its logit is taken in -- while the uncorrected dot
    keeps its fixed quantisation error."""
    w = W.get_workload("tiny_1k").with_(T=96, B=1, Hkv=1, Hq=1, N=16, beta=6, sinks=4, recent=16, marked=4)
    li = W.layer_inputs(w)
    q, pos = W.queries(w, steps=1)
    qr = O.rope(q[0][0, 0].astype(np.float64), pos[0][0], w.theta)
    sel = np.arange(6, dtype=np.int64)[None, None]          # every group (G = 6)
    rng = np.random.default_rng(5)
    exact = None
    diffs = []
    for _ in range(400):
        S = rng.standard_normal((128, D))
        c = O.encode(li.K, li.V, li.l1_mask, li.signs, w.N, w.theta, qjl_S=S)
        keys, _, prov = O.attention_entries(c, sel, 0, 0)
        sk = O.entry_sketches(c, sel, 0, 0)
        if exact is None:
            K = li.K[0, 0].astype(np.float64)
            exact = np.array([O.rope(K[idx if kind == 3 else c.l1_pos[0, idx]],
                                     idx if kind == 3 else c.l1_pos[0, idx], w.theta) @ qr
                              for kind, idx in prov])
            plain = keys @ qr
            tok = np.array([kind != 2 for kind, _ in prov])
            assert tok.sum() == 96 and np.all(sk.norm[~tok] == 0)
        diffs.append(keys @ qr + O.qjl_estimate(S @ (c.Pi @ qr), sk) - exact)
    diffs = np.array(diffs)[:, tok]
    se = diffs.std(axis=0, ddof=1) / np.sqrt(len(diffs))
    z = diffs.mean(axis=0) / se
    assert np.mean(np.abs(z) <= 3.5) >= 0.98, np.sort(np.abs(z))[-5:]
    # the uncorrected quantisation error is systematic: far outside the same band
    zq = (plain - exact)[tok] / se
    assert np.mean(np.abs(zq) > 3.5) >= 0.5


def test_qjl_sketch_words_round_trip():
    rng = np.random.default_rng(4)
    bits = rng.integers(0, 2, (3, 5, 128)).astype(bool)
    words = (bits.reshape(3, 5, 4, 32).astype(np.uint64) << np.arange(32, dtype=np.uint64)).sum(-1).astype(np.uint32)
    np.testing.assert_array_equal(O.unpack_sketch_words(words), bits)
    assert O.unpack_sketch_words(np.array([1, 0, 0, 0x80000000], np.uint32))[[0, 127]].all()
