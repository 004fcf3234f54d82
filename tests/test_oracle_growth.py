"""The oracle's reading of decode-time growth: the grown L1 set
(oracle.grown_l1_mask) checked against its definition position by position,
and for the properties a sliding window must have (growing in two steps is
growing once; its size is constant once the window has passed the sinks;
growing by nothing changes nothing)."""

import numpy as np
import pytest

import oracle as O


def _mask(rng, B, T, sinks, recent, marked):
    m = np.zeros((B, T), bool)
    m[:, :sinks] = True
    m[:, max(T - recent, 0):] = True
    for b in range(B):
        lo, hi = sinks, max(T - recent, sinks)
        if hi > lo:
            m[b, lo + rng.choice(hi - lo, size=min(marked, hi - lo), replace=False)] = True
    return m


@pytest.mark.parametrize("T,grow,sinks,recent", [(100, 13, 4, 16), (64, 40, 2, 8), (20, 5, 4, 30), (50, 0, 3, 10)])
def test_grown_mask_position_by_position(T, grow, sinks, recent):
    rng = np.random.default_rng(7)
    m = _mask(rng, 3, T, sinks, recent, 6)
    g = O.grown_l1_mask(m, T + grow, sinks, recent)
    assert g.shape == (3, T + grow)
    for b in range(3):
        for x in range(T + grow):
            marked = x < T - recent and x < T and m[b, x]
            want = x < sinks or x >= T + grow - recent or marked
            assert g[b, x] == want, (b, x)


def test_growing_twice_is_growing_once():
    rng = np.random.default_rng(3)
    m = _mask(rng, 2, 300, 4, 32, 10)
    once = O.grown_l1_mask(m, 350, 4, 32)
    twice = O.grown_l1_mask(O.grown_l1_mask(m, 317, 4, 32), 350, 4, 32)
    np.testing.assert_array_equal(once, twice)
    one_by_one = m
    for T in range(301, 351):
        one_by_one = O.grown_l1_mask(one_by_one, T, 4, 32)
    np.testing.assert_array_equal(once, one_by_one)


def test_window_size_is_constant_and_growing_by_nothing_is_identity():
    rng = np.random.default_rng(5)
    m = _mask(rng, 2, 400, 4, 64, 20)
    for T in (400, 401, 417, 480, 1000):
        g = O.grown_l1_mask(m, T, 4, 64)
        np.testing.assert_array_equal(g.sum(axis=1), m.sum(axis=1))
        assert g[:, T - 64:].all() and not g[:, 400 - 64: T - 64].any()
    np.testing.assert_array_equal(O.grown_l1_mask(m, 400, 4, 64), m)
    with pytest.raises(ValueError):
        O.grown_l1_mask(m, 399, 4, 64)
