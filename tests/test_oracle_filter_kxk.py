"""Pins of the oracle's K x K filters.

The valid-region correlation follows the OpenCL convolution page §2 (filter
placed with its first row and column on the output position, products of
covered inputs and weights summed, no flip, output (W - K + 1) x (H - K + 1),
widths 8 to 64 in the page's sweep); it is checked against scipy's
correlate2d, shifted crops for delta filters, constants, and separable
filters applied as two 1-D passes.  The centred replicate-border form (the
fused epilogue for odd K) is checked against scipy.ndimage.correlate in
'nearest' mode, against the 3 x 3 oracle, and on deltas.
"""
import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("K", [1, 2, 3, 5, 8, 13, 16])
def test_valid_matches_scipy_correlate2d(K):
    from scipy import signal
    rng = np.random.default_rng(K)
    a = rng.random((K + 17, K + 23)) * 255
    w = rng.random((K, K)) - 0.3
    np.testing.assert_allclose(oracle.filter_valid(a, w), signal.correlate2d(a, w, mode="valid"),
                               rtol=0, atol=1e-9 * K * K)


@pytest.mark.parametrize("K", [8, 64])
def test_valid_wide_filters_match_scipy(K):
    from scipy import signal
    rng = np.random.default_rng(100 + K)
    a = rng.random((K + 9, K + 12)) * 255
    w = rng.random((K, K))
    w /= w.sum()
    np.testing.assert_allclose(oracle.filter_valid(a, w), signal.correlate2d(a, w, mode="valid"), rtol=0, atol=1e-9)


@pytest.mark.parametrize("K", [1, 4, 7])
def test_valid_delta_is_a_shifted_crop(K):
    rng = np.random.default_rng(3)
    a = rng.random((30, 41))
    for r0, c0 in [(0, 0), (K - 1, 0), (0, K - 1), (K // 2, K - 1)]:
        w = np.zeros((K, K))
        w[r0, c0] = 1.0
        want = a[r0:r0 + 30 - K + 1, c0:c0 + 41 - K + 1]
        np.testing.assert_array_equal(oracle.filter_valid(a, w), want)


def test_valid_constant_and_shape():
    a = np.full((12, 19), 7.0)
    w = np.arange(25, dtype=np.float64).reshape(5, 5)
    out = oracle.filter_valid(a, w)
    assert out.shape == (8, 15)
    np.testing.assert_allclose(out, 7.0 * w.sum(), rtol=1e-15)
    assert oracle.filter_valid(np.ones((4, 4)), np.ones((4, 4))).tolist() == [[16.0]]


def test_valid_separable_filter_is_two_passes():
    rng = np.random.default_rng(8)
    a = rng.random((40, 50))
    u, v = rng.random(6), rng.random(6)
    rows = np.stack([np.correlate(a[i], v, mode="valid") for i in range(a.shape[0])])
    both = np.stack([np.correlate(rows[:, j], u, mode="valid") for j in range(rows.shape[1])], 1)
    np.testing.assert_allclose(oracle.filter_valid(a, np.outer(u, v)), both, rtol=1e-12)


def test_valid_is_not_flipped():
    # a planted misreading (true convolution, the filter flipped) differs
    a = np.arange(36, dtype=np.float64).reshape(6, 6) ** 2
    w = np.array([[1.0, 2.0], [0.0, 0.0]])
    assert oracle.filter_valid(a, w)[0, 0] == a[0, 0] + 2 * a[0, 1]
    assert not np.allclose(oracle.filter_valid(a, w), oracle.filter_valid(a, w[::-1, ::-1]))


@pytest.mark.parametrize("K", [1, 3, 5, 7])
def test_centred_matches_scipy_nearest(K):
    from scipy import ndimage
    rng = np.random.default_rng(20 + K)
    r = rng.random((23, 31)) * 255
    w = rng.random((K, K))
    np.testing.assert_allclose(oracle.filter_centred(r, w), ndimage.correlate(r, w, mode="nearest"),
                               rtol=0, atol=1e-9)


def test_centred_three_agrees_with_the_3x3_oracle():
    rng = np.random.default_rng(4)
    r = rng.random((17, 9))
    w = rng.random(9)
    np.testing.assert_array_equal(oracle.filter_centred(r, w.reshape(3, 3)), oracle.filter3x3(r, w))


@pytest.mark.parametrize("K", [5, 7])
def test_centred_delta_is_a_replicated_shift(K):
    R = K // 2
    rng = np.random.default_rng(K)
    r = rng.random((12, 15))
    w = np.zeros((K, K))
    w[0, K - 1] = 1.0                  # reads r[y - R][x + R]
    want = np.pad(r, R, mode="edge")[0:12, 2 * R:2 * R + 15]
    np.testing.assert_array_equal(oracle.filter_centred(r, w), want)
