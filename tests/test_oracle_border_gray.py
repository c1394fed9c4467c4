"""Pins of the oracle's border rules and grayscale conversion.

Border rules (CUDA interpolation page §6.1: clamp, mirror, wrap) are checked
against numpy's padding modes and scipy's border-extended linear
interpolation, which implement the same rules independently, and against
closed forms on ramps and the cyclic-shift invariance that only the wrap rule
has.  The grayscale conversion (OpenCV object-tracking page §3.1.1, cvtColor
before resize; BT.601 luma weights) is checked against hand-worked values,
float64 evaluation away from ties, and exact rationals at ties.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle

CLAMP, MIRROR, WRAP = oracle.BORDER_CLAMP, oracle.BORDER_MIRROR, oracle.BORDER_WRAP
NP_PAD = {CLAMP: "edge", MIRROR: "reflect", WRAP: "wrap"}
SCIPY_MODE = {CLAMP: "nearest", MIRROR: "mirror", WRAP: "grid-wrap"}
BORDERS = [CLAMP, MIRROR, WRAP]


def half_pixel(n_in, n_out):
    return (np.arange(n_out) + 0.5) * n_in / n_out - 0.5


# ---------------------------------------------------------------- the index rules

def test_border_index_hand_sequences():
    ks = list(range(-3, 7))
    assert [oracle.border_index(k, 4, CLAMP) for k in ks] == [0, 0, 0, 0, 1, 2, 3, 3, 3, 3]
    assert [oracle.border_index(k, 4, MIRROR) for k in ks] == [3, 2, 1, 0, 1, 2, 3, 2, 1, 0]
    assert [oracle.border_index(k, 4, WRAP) for k in ks] == [1, 2, 3, 0, 1, 2, 3, 0, 1, 2]
    for b in BORDERS:
        assert all(oracle.border_index(k, 1, b) == 0 for k in ks)


@pytest.mark.parametrize("b", BORDERS)
@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_border_index_matches_numpy_pad(b, n):
    pad = 2 * n + 1
    want = np.pad(np.arange(n), pad, mode=NP_PAD[b])
    got = [oracle.border_index(k, n, b) for k in range(-pad, n + pad)]
    assert got == want.tolist()


# ---------------------------------------------------------------- bilinear with borders

GEOMS = [(5, 7, 13, 17), (4, 6, 8, 12), (3, 3, 10, 10), (1, 5, 4, 9), (6, 5, 3, 2), (2, 2, 7, 3), (5, 1, 9, 3),
         (7, 9, 7, 30)]


@pytest.mark.parametrize("b", BORDERS)
@pytest.mark.parametrize("geom", GEOMS)
def test_f32_border_matches_scipy_linear(b, geom):
    from scipy import ndimage
    H, W, OH, OW = geom
    img = (np.random.default_rng(H * 100 + W).random((H, W, 3)) * 255).astype(np.float32)
    got = oracle.linear_f32(img, OH, OW, b)
    yy, xx = np.meshgrid(half_pixel(H, OH), half_pixel(W, OW), indexing="ij")
    for c in range(3):
        ref = ndimage.map_coordinates(img[:, :, c].astype(np.float64), [yy, xx], order=1, mode=SCIPY_MODE[b])
        np.testing.assert_allclose(got[:, :, c], ref, rtol=0, atol=1e-9)


@pytest.mark.parametrize("b", BORDERS)
@pytest.mark.parametrize("geom", [(5, 7, 10, 14), (4, 6, 16, 24), (3, 8, 12, 16), (9, 2, 18, 8), (1, 4, 2, 8)])
def test_u8_border_matches_scipy_at_dyadic_ratios(b, geom):
    # at 2x and 4x every weight is a multiple of 1/8: the 11-bit weights are
    # exact, so the u8 result is the exact value rounded half-up
    from scipy import ndimage
    H, W, OH, OW = geom
    img = np.random.default_rng(7 + H + W).integers(0, 256, (H, W, 3), dtype=np.uint8)
    got = oracle.linear_u8(img, OH, OW, b)
    yy, xx = np.meshgrid(half_pixel(H, OH), half_pixel(W, OW), indexing="ij")
    for c in range(3):
        ref = ndimage.map_coordinates(img[:, :, c].astype(np.float64), [yy, xx], order=1, mode=SCIPY_MODE[b])
        np.testing.assert_array_equal(got[:, :, c], np.floor(ref + 0.5).astype(np.uint8))


@pytest.mark.parametrize("b", BORDERS)
@pytest.mark.parametrize("geom", [(720, 1280, 224, 224), (1080, 1920, 719, 1279), (37, 53, 23, 41),
                                  (13, 11, 29, 31), (100, 70, 31, 29), (8, 9, 3, 77)])
def test_u8_within_weight_quantisation_of_exact_bilinear(b, geom):
    # at ratios whose weights are not multiples of 2^-11 the u8 result is
    # pinned by a bound: each 11-bit weight is within 2^-12 of the exact
    # one, and the weights of an axis sum to one either way, so the weighted
    # sum moves by at most 255 * (2^-12 + 2^-12) from the exact bilinear
    # value; the result rounds that sum once
    from scipy import ndimage
    H, W, OH, OW = geom
    img = np.random.default_rng(H + 3 * W + b).integers(0, 256, (H, W, 3), dtype=np.uint8)
    got = oracle.linear_u8(img, OH, OW, b).astype(np.float64)
    yy, xx = np.meshgrid(half_pixel(H, OH), half_pixel(W, OW), indexing="ij")
    bound = 0.5 + 255 * 2 * 2.0 ** -12 + 1e-9
    for c in range(3):
        ref = ndimage.map_coordinates(img[:, :, c].astype(np.float64), [yy, xx], order=1, mode=SCIPY_MODE[b])
        assert np.abs(got[:, :, c] - ref).max() <= bound


@pytest.mark.parametrize("b", BORDERS)
@pytest.mark.parametrize("k", [2, 4])
def test_u8_border_is_clamp_resize_of_padded_image(b, k):
    # a k-times upscale samples x = d/k + (1-k)/(2k); padding the source by one
    # pixel (numpy's rule) and upscaling the padded image k times puts the same
    # positions, shifted by one pixel, at outputs k .. k(W+1)-1, all inside
    rng = np.random.default_rng(11 * k + b)
    H, W = 5, 7
    img = rng.integers(0, 256, (H, W, 3), dtype=np.uint8)
    pad = np.pad(img, ((1, 1), (1, 1), (0, 0)), mode=NP_PAD[b])
    want = oracle.linear_u8(pad, k * (H + 2), k * (W + 2), CLAMP)[k:k * (H + 1), k:k * (W + 1)]
    np.testing.assert_array_equal(oracle.linear_u8(img, k * H, k * W, b), want)


def test_ramp_closed_forms_2x():
    # src[x] = 4x, W = 64.  Output 0 samples x = -1/4, output 127 samples 63.25.
    # mirror: the even extension 4|x| gives 1 and 4 * 62.75 = 251;
    # wrap: the periodic extension gives 1/4 * 252 + 3/4 * 0 = 63 and
    #       3/4 * 252 + 1/4 * 0 = 189; clamp: 0 and 252
    src = (4 * np.arange(64)).astype(np.uint8)[None, :].repeat(3, 0)
    for b, first, last in [(CLAMP, 0, 252), (MIRROR, 1, 251), (WRAP, 63, 189)]:
        out = oracle.linear_u8(src, 6, 128, b)[:, :, 0]
        assert (out[:, 0] == first).all() and (out[:, 127] == last).all()
        assert (out[:, 1:127] == 2 * np.arange(1, 127) - 1).all()


@pytest.mark.parametrize("k", [2, 3, 4])
def test_wrap_commutes_with_cyclic_shift(k):
    img = np.random.default_rng(k).integers(0, 256, (6, 9, 3), dtype=np.uint8)
    out = oracle.linear_u8(img, k * 6, k * 9, WRAP)
    np.testing.assert_array_equal(oracle.linear_u8(np.roll(img, 1, axis=1), k * 6, k * 9, WRAP),
                                  np.roll(out, k, axis=1))
    np.testing.assert_array_equal(oracle.linear_u8(np.roll(img, 1, axis=0), k * 6, k * 9, WRAP),
                                  np.roll(out, k, axis=0))
    # the clamp rule does not have this invariance at the edges
    clamp = oracle.linear_u8(img, k * 6, k * 9, CLAMP)
    assert not np.array_equal(oracle.linear_u8(np.roll(img, 1, axis=1), k * 6, k * 9, CLAMP),
                              np.roll(clamp, k, axis=1))


@pytest.mark.parametrize("geom", [(9, 13, 4, 5), (20, 20, 20, 20), (1080, 1920, 540, 960), (7, 5, 7, 3)])
def test_downscales_never_reach_the_border(geom):
    H, W, OH, OW = geom
    img = np.random.default_rng(3).integers(0, 256, (H, W, 3), dtype=np.uint8)
    ref = oracle.linear_u8(img, OH, OW, CLAMP)
    for b in (MIRROR, WRAP):
        np.testing.assert_array_equal(oracle.linear_u8(img, OH, OW, b), ref)


def test_mirror_differs_from_edge_repeating_reflection():
    # a planted misreading (reflection that repeats the edge sample, numpy's
    # "symmetric") must not pass as the mirror rule: at a 2x upscale it
    # gives the clamp result, which the mirror rule does not
    img = np.random.default_rng(5).integers(0, 256, (5, 7, 3), dtype=np.uint8)
    pad = np.pad(img, ((1, 1), (1, 1), (0, 0)), mode="symmetric")
    wrong = oracle.linear_u8(pad, 14, 18, CLAMP)[2:12, 2:16]
    np.testing.assert_array_equal(wrong, oracle.linear_u8(img, 10, 14, CLAMP))
    assert not np.array_equal(wrong, oracle.linear_u8(img, 10, 14, MIRROR))


# ---------------------------------------------------------------- grayscale

def test_gray_hand_values():
    px = np.array([[[255, 0, 0], [0, 255, 0], [0, 0, 255], [255, 255, 255], [0, 0, 0], [0, 0, 250]]], np.uint8)
    # 76.245, 149.685, 29.07, 255, 0, and the tie 28.5 rounded up
    assert oracle.gray_u8(px).tolist() == [[76, 150, 29, 255, 0, 29]]


def test_gray_of_gray_is_identity_and_alpha_ignored():
    k = np.arange(256, dtype=np.uint8)
    px = np.stack([k, k, k, 255 - k], -1)[None]
    assert oracle.gray_u8(px[:, :, :3])[0].tolist() == k.tolist()
    assert oracle.gray_u8(px)[0].tolist() == k.tolist()


def test_gray_matches_float64_away_from_ties_and_exact_at_ties():
    rng = np.random.default_rng(0)
    rgb = rng.integers(0, 256, (512, 512, 3), dtype=np.uint8)
    got = oracle.gray_u8(rgb).astype(np.int64)
    v = 0.299 * rgb[..., 0] + 0.587 * rgb[..., 1] + 0.114 * rgb[..., 2]
    away = np.abs(v - np.floor(v) - 0.5) > 1e-6
    assert away.mean() > 0.99
    np.testing.assert_array_equal(got[away], np.floor(v[away] + 0.5).astype(np.int64))
    for y, x in zip(*np.nonzero(~away)):
        r, g, b = (int(t) for t in rgb[y, x])
        exact = Fraction(299 * r + 587 * g + 114 * b, 1000)
        assert got[y, x] == int(exact + Fraction(1, 2))  # floor of exact + 1/2: half-up


def test_gray_bgr_order_reverses_channels():
    img = np.random.default_rng(2).integers(0, 256, (17, 23, 3), dtype=np.uint8)
    np.testing.assert_array_equal(oracle.gray_u8(img, bgr=True), oracle.gray_u8(img[..., ::-1].copy()))
    assert not np.array_equal(oracle.gray_u8(img, bgr=True), oracle.gray_u8(img))


@pytest.mark.parametrize("b", BORDERS)
def test_row_band_equals_the_whole_resize(b):
    # the band form the benchmark times computes the same rows as the whole
    # resize (its rows are independent of one another)
    img = np.random.default_rng(23).integers(0, 256, (41, 37, 3), dtype=np.uint8)
    whole = oracle.linear_u8(img, 29, 53, b)
    for dy0, dy1 in [(0, 29), (0, 1), (5, 17), (28, 29), (10, 10)]:
        np.testing.assert_array_equal(oracle.linear_u8_rows(img, 29, 53, dy0, dy1, b), whole[dy0:dy1])
