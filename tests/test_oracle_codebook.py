"""Pins for the oracle's TurboQuant codebook (Beta Lloyd-Max, d = 128).

The codebook is checked against things other than itself: numerical
quadrature of the density (not the closed-form moment the oracle uses), the
empirical coordinate law of random unit vectors, brute-force nearest-centroid
search, and Max's 1960 Gaussian tables in the large-d limit.
"""

import numpy as np
import pytest
from scipy import integrate, stats

import oracle as O
from conftest import golden_path


def _golden_max():
    vals = {}
    with open(golden_path("max1960_gaussian_levels.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, *v = line.split()
            vals[k] = np.array([float(x) for x in v])
    return vals


def test_density_is_a_probability_law():
    tot, _ = integrate.quad(lambda y: O.coordinate_pdf(np.array([y]))[0], -1, 1, limit=200)
    assert abs(tot - 1.0) < 1e-12


@pytest.mark.parametrize("y", [-0.4, -0.1, 0.0, 0.03, 0.2, 0.5])
def test_cdf_matches_quadrature(y):
    ref, _ = integrate.quad(lambda t: O.coordinate_pdf(np.array([t]))[0], -1, y, limit=200)
    assert abs(O.coordinate_cdf(y) - ref) < 1e-12


def test_coordinate_law_matches_random_unit_vectors():
    # KS test: coordinates of x/|x| for Gaussian x follow the stated law.
    rng = np.random.default_rng(7)
    x = rng.standard_normal((4000, 128))
    y = (x / np.linalg.norm(x, axis=1, keepdims=True))[:, :3].ravel()
    res = stats.kstest(y, lambda t: O.coordinate_cdf(t))
    assert res.pvalue > 1e-3


@pytest.mark.parametrize("bits", [3, 4])
def test_centroid_condition_by_quadrature(bits):
    c, tau = O.codebook(bits)
    edges = np.concatenate([[-1.0], tau, [1.0]])
    pdf = lambda t: O.coordinate_pdf(np.array([t]))[0]
    for k in range(len(c)):
        m0, _ = integrate.quad(pdf, edges[k], edges[k + 1], limit=200, epsabs=1e-15, epsrel=1e-13)
        m1, _ = integrate.quad(lambda t: t * pdf(t), edges[k], edges[k + 1], limit=200,
                               epsabs=1e-16, epsrel=1e-13)
        assert abs(m1 / m0 - c[k]) < 1e-12


@pytest.mark.parametrize("bits", [3, 4])
def test_boundaries_symmetry_and_order(bits):
    c, tau = O.codebook(bits)
    L = 1 << bits
    assert len(c) == L and len(tau) == L - 1
    assert np.all(np.diff(c) > 0)
    np.testing.assert_array_equal(c, -c[::-1])
    np.testing.assert_allclose(tau, 0.5 * (c[:-1] + c[1:]), rtol=0, atol=1e-17)
    assert tau[L // 2 - 1] == 0.0
    assert np.all((tau > c[:-1]) & (tau < c[1:]))


def test_gaussian_limit_matches_max_1960():
    g = _golden_max()
    d = 1 << 16
    for bits, key in [(3, "levels8"), (4, "levels16")]:
        c, _ = O.lloyd_max_codebook(bits, d)
        pos = c[len(c) // 2:] * np.sqrt(d)
        np.testing.assert_allclose(pos, g[key], atol=2e-4)


def _distortion(bits, d):
    c, tau = O.codebook(bits, d) if d == O.D else O.lloyd_max_codebook(bits, d)
    edges = np.concatenate([[-1.0], tau, [1.0]])
    pdf = lambda t: O.coordinate_pdf(np.array([t]), d)[0]
    tot = 0.0
    for k in range(len(c)):
        v, _ = integrate.quad(lambda t: (t - c[k]) ** 2 * pdf(t), edges[k], edges[k + 1],
                              limit=200, epsabs=1e-16)
        tot += v
    return tot


def test_distortion_decreases_and_tends_to_gaussian():
    g = _golden_max()
    d3, d4 = _distortion(3, 128), _distortion(4, 128)
    assert d4 < d3
    # per-coordinate MSE times d approaches Max's unit-Gaussian MSE
    assert abs(d3 * 128 / g["mse8"][0] - 1) < 0.02
    assert abs(d4 * 128 / g["mse16"][0] - 1) < 0.02


@pytest.mark.parametrize("bits", [3, 4])
def test_boundary_count_equals_nearest_centroid(bits):
    # code = #{tau_k < y} must be the index of the nearest centroid
    c, _ = O.codebook(bits)
    rng = np.random.default_rng(bits)
    x = rng.standard_normal((500, 128))
    Pi = O.rotation_matrix(np.ones(128, np.int8))
    codes, _, y = O.tq_encode(x, bits, Pi)
    brute = np.argmin(np.abs(y[..., None] - c), axis=-1)
    far = ~O.near_boundary(y, bits, rel=1e-6)
    np.testing.assert_array_equal(codes[far], brute[far])


# The near-tie band of the acceptance rule: a coordinate within
# 1e-5 * max(|tau_k|, 1/sqrt(d)) of a boundary tau_k.  Its half-width at the
# zero boundary is 1e-5 / sqrt(128) = 8.8388e-7; at the outermost 4-bit
# boundary, about (2.0459 + 2.6889) / 2 / sqrt(128) = 0.20929 (the positive
# levels sqrt(d) c of the d = 128 codebook, computed independently of the
# oracle), it is 2.09e-6.  near_boundary takes coordinates of d = 128
# vectors (the last axis), so each probe value fills one such vector.
ZERO_BAND = 8.838834764831845e-07


def _nb(values, bits):
    y = np.repeat(np.asarray(values, np.float64)[:, None], 128, axis=1)
    got = O.near_boundary(y, bits)
    assert got.shape == y.shape and np.all(got == got[:, :1])
    return got[:, 0]


@pytest.mark.parametrize("bits", [3, 4])
def test_near_boundary_band_at_every_boundary(bits):
    _, tau = O.codebook(bits)
    for t in tau:
        tol = 1e-5 * max(abs(t), ZERO_BAND / 1e-5)
        inside = [t - 0.5 * tol, t, t + 0.5 * tol, t + 0.99 * tol, t - 0.99 * tol]
        outside = [t - 2 * tol, t + 2 * tol, t + 1.05 * tol, t - 1.05 * tol]
        assert np.all(_nb(inside, bits)), (bits, t)
        assert not np.any(_nb(outside, bits)), (bits, t)


@pytest.mark.parametrize("bits", [3, 4])
def test_near_boundary_is_relative_not_absolute(bits):
    _, tau = O.codebook(bits)
    assert tau[len(tau) // 2] == 0.0
    # the zero boundary: half-width 1e-5 / sqrt(128), not 1e-5
    assert _nb([0.9 * ZERO_BAND, -0.9 * ZERO_BAND], bits).all()
    assert not _nb([1.1 * ZERO_BAND, -1.1 * ZERO_BAND, 2e-6, 9e-6], bits).any()
    # the outermost boundary: half-width 1e-5 |tau|, wider than the zero boundary's
    t = tau[-1]
    assert t > 0.15
    assert _nb([t + 1.5 * ZERO_BAND, -t - 1.5 * ZERO_BAND], bits).all()
    assert not _nb([t + 1.2e-5 * t, -t - 1.2e-5 * t], bits).any()


def test_near_boundary_outermost_4bit_band_literal():
    # half-width at the outermost 4-bit boundary from the independently
    # computed levels above (0.20929 * 1e-5 = 2.093e-6)
    _, tau = O.codebook(4)
    assert abs(tau[-1] - (2.0459 + 2.6889) / 2 / np.sqrt(128)) < 1e-4
    assert _nb([tau[-1] + 2.07e-6, tau[-1] - 2.07e-6], 4).all()
    assert not _nb([tau[-1] + 2.12e-6, tau[-1] - 2.12e-6], 4).any()


@pytest.mark.parametrize("bits", [3, 4])
def test_near_boundary_far_values_and_shapes(bits):
    c, tau = O.codebook(bits)
    # centroids and the ends of the range lie far from every boundary
    assert not _nb(c, bits).any()
    assert not _nb([-1.0, 1.0, 0.5, -0.5], bits).any()
    # elementwise over any leading shape: a vector holding every boundary
    # and every centroid is flagged exactly at the boundaries
    y = np.zeros((2, 3, 128))
    y[:, :, : len(tau)] = tau
    y[:, :, len(tau): len(tau) + len(c)] = c
    y[:, :, len(tau) + len(c):] = 0.5
    got = O.near_boundary(y, bits)
    assert got.shape == (2, 3, 128)
    assert got[..., : len(tau)].all() and not got[..., len(tau):].any()
