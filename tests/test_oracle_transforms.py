"""Pins for the oracle's rotation, RoPE, quantiser round trip and packing."""

import numpy as np
import pytest
import scipy.linalg

import oracle as O
from conftest import golden_path


# -- Walsh-Hadamard rotation ---------------------------------------------------

def test_sylvester_matches_scipy():
    np.testing.assert_array_equal(O.sylvester_hadamard(128), scipy.linalg.hadamard(128))


def test_rotation_is_orthonormal_with_exact_inverse():
    rng = np.random.default_rng(1)
    s = np.where(rng.integers(0, 2, 128) == 1, 1, -1).astype(np.int8)
    Pi = O.rotation_matrix(s)
    np.testing.assert_allclose(Pi @ Pi.T, np.eye(128), atol=1e-15)
    x = rng.standard_normal((10, 128))
    y = x @ Pi.T
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-14)
    np.testing.assert_allclose(y @ Pi, x, atol=1e-14)
    # the sign vector is applied before H: Pi e_i = s_i * (column i of H) / sqrt(d)
    H = scipy.linalg.hadamard(128)
    for i in (0, 5, 127):
        e = np.zeros(128)
        e[i] = 1
        np.testing.assert_allclose(Pi @ e, s[i] * H[:, i] / np.sqrt(128), atol=1e-15)


def test_rotated_unit_coordinates_follow_the_codebook_law():
    from scipy import stats
    rng = np.random.default_rng(3)
    s = np.where(rng.integers(0, 2, 128) == 1, 1, -1)
    Pi = O.rotation_matrix(s)
    # isotropic input: x/|x| is uniform on the sphere and so is its rotation
    x = rng.standard_normal((3000, 128))
    y = (x / np.linalg.norm(x, axis=1, keepdims=True)) @ Pi.T
    res = stats.kstest(y[:, 17], lambda t: O.coordinate_cdf(t))
    assert res.pvalue > 1e-3


# -- RoPE ---------------------------------------------------------------------------

def test_rope_two_dim_is_plane_rotation():
    # d = 2: one pair (0, 1) with omega_0 = 1, so RoPE is rotation by angle p
    for p in (0, 1, 3, 1000):
        out = O.rope(np.array([1.0, 0.0]), p)
        np.testing.assert_allclose(out, [np.cos(p), np.sin(p)], atol=1e-12)
        out = O.rope(np.array([0.0, 1.0]), p)
        np.testing.assert_allclose(out, [-np.sin(p), np.cos(p)], atol=1e-12)


def test_rope_pairs_i_with_i_plus_half():
    # d = 4, theta = 100: pairs (0, 2) with omega 1 and (1, 3) with omega 0.1
    p = 7
    x = np.array([1.0, 0.0, 0.0, 0.0])
    np.testing.assert_allclose(O.rope(x, p, theta=100.0), [np.cos(7), 0, np.sin(7), 0], atol=1e-12)
    x = np.array([0.0, 1.0, 0.0, 0.0])
    np.testing.assert_allclose(O.rope(x, p, theta=100.0), [0, np.cos(0.7), 0, np.sin(0.7)], atol=1e-12)


def test_rope_matches_complex_multiplication():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((6, 128))
    pos = np.array([0, 1, 17, 4095, 32768, 33279])
    z = x[:, :64] + 1j * x[:, 64:]
    w = (1e6 ** (-np.arange(64) / 64.0))
    zr = z * np.exp(1j * pos[:, None] * w[None, :])
    np.testing.assert_allclose(O.rope(x, pos), np.concatenate([zr.real, zr.imag], 1), atol=1e-12)


def test_rope_invariants():
    rng = np.random.default_rng(6)
    q, k = rng.standard_normal((2, 128))
    np.testing.assert_array_equal(O.rope(q, 0), q)
    np.testing.assert_allclose(np.linalg.norm(O.rope(q, 12345)), np.linalg.norm(q), rtol=1e-14)
    a = O.rope(q, 40000) @ O.rope(k, 39000)
    b = O.rope(q, 1000) @ O.rope(k, 0)
    assert abs(a - b) < 1e-10
    np.testing.assert_allclose(O.rope(O.rope(q, 999), -999), q, atol=1e-13)


# -- quantiser -------------------------------------------------------------------------

@pytest.mark.parametrize("bits", [3, 4])
def test_zero_vector_encoding(bits):
    Pi = O.rotation_matrix(np.ones(128))
    codes, n, _ = O.tq_encode(np.zeros((2, 128)), bits, Pi)
    assert np.all(n == 0)
    assert np.all(codes == (1 << (bits - 1)) - 1)
    np.testing.assert_array_equal(O.tq_decode(codes, n, bits, Pi), 0.0)


@pytest.mark.parametrize("bits,expect", [(3, 0.0345), (4, 0.0095)])
def test_relative_mse_matches_distortion(bits, expect):
    rng = np.random.default_rng(20 + bits)
    s = np.where(rng.integers(0, 2, 128) == 1, 1, -1)
    Pi = O.rotation_matrix(s)
    x = rng.standard_normal((4000, 128)) * np.exp(0.5 * rng.standard_normal(128))
    codes, n, _ = O.tq_encode(x, bits, Pi)
    xh = O.tq_decode(codes, n, bits, Pi)
    rel = np.sum((xh - x) ** 2) / np.sum(x ** 2)
    assert abs(rel / expect - 1) < 0.05


# -- packing ---------------------------------------------------------------------------

def _golden_packing():
    rows = []
    with open(golden_path("packing_le_bitstream.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            b, codes, by = line.strip().split("|")
            rows.append((int(b), [int(c) for c in codes.split(",")], [int(x, 16) for x in by.split(",")]))
    return rows


def test_packing_worked_bytes():
    for bits, codes, expect in _golden_packing():
        got = O.pack_codes(np.array(codes, np.uint8), bits)
        assert list(got) == expect
        np.testing.assert_array_equal(O.unpack_codes(got, bits, len(codes)), codes)


@pytest.mark.parametrize("bits", [3, 4])
def test_packing_matches_integer_bitstring(bits):
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 1 << bits, (20, 128)).astype(np.uint8)
    packed = O.pack_codes(codes, bits)
    for row, pk in zip(codes, packed):
        v = 0
        for i, c in enumerate(row):
            v |= int(c) << (bits * i)
        assert bytes(pk) == v.to_bytes(128 * bits // 8, "little")
    np.testing.assert_array_equal(O.unpack_codes(packed, bits), codes)
