"""Pins of the CPU oracle to facts the pages and the mathematics fix.

Each test checks the oracle against something other than its own code:
hand-worked examples, closed forms, invariants, brute force over exact
rationals, and library routines for the cases where they compute the same
thing (torch bilinear/nearest interpolation, scipy correlation).  A plausible
slip in the oracle (a dropped term, a wrong sign or index, a transposed
operand, a wrong rounding) fails at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from bilinear_image_resize_gb300 import synth
from conftest import GOLDEN


def exact_coord(d, n_in, n_out):
    """x = (d + 1/2) * n_in / n_out - 1/2 as an exact rational."""
    return Fraction(2 * d + 1, 2) * Fraction(n_in, n_out) - Fraction(1, 2)


# ---------------------------------------------------------------- mapping

@pytest.mark.parametrize("n_in", [1, 2, 3, 5, 7, 16, 31])
@pytest.mark.parametrize("n_out", [1, 2, 3, 4, 9, 17, 40])
def test_coord_matches_exact_rational(n_in, n_out):
    for d in range(n_out):
        x = exact_coord(d, n_in, n_out)
        i, r, den = oracle.linear_coord(n_in, n_out, d)
        assert i == math.floor(x)
        assert 0 <= r < den
        assert Fraction(r, den) == x - math.floor(x)


def test_weight_is_round_half_up_of_2048u():
    # exact ties: 2048 * r / 4096 = r / 2 for odd r; half-up gives (r + 1) / 2
    assert [oracle.weight_q11(r, 4096) for r in (1, 3, 5, 7, 4093, 4095)] == [1, 2, 3, 4, 2047, 2048]
    for den in (2, 6, 8, 10, 4096, 6144, 8192, 12000):
        for r in range(den):
            a1 = oracle.weight_q11(r, den)
            exact = Fraction(2048 * r, den)
            assert 0 <= a1 <= 2048
            assert exact - Fraction(1, 2) <= a1 <= exact + Fraction(1, 2)
            if exact.denominator == 2:   # a tie rounds up
                assert a1 == math.floor(exact) + 1
    # u just below 1 rounds up to the full weight, u = 0 gives 0
    assert oracle.weight_q11(0, 100) == 0
    assert oracle.weight_q11(8191, 8192) == 2048


# ---------------------------------------------------------------- golden, hand-worked

def test_golden_linear_2x2_to_4x4():
    with open(os.path.join(GOLDEN, "linear_2x2_to_4x4.json")) as f:
        g = json.load(f)
    src = np.array(g["src"], np.uint8)
    out = oracle.linear_u8(src, g["out_h"], g["out_w"])[:, :, 0]
    np.testing.assert_array_equal(out, np.array(g["u8"]))
    outf = oracle.linear_f32(src.astype(np.float32), g["out_h"], g["out_w"])[:, :, 0]
    np.testing.assert_allclose(outf, np.array(g["real"], np.float64), rtol=0, atol=1e-12)


def test_golden_filter3x3():
    with open(os.path.join(GOLDEN, "filter3x3_3x3.json")) as f:
        g = json.load(f)
    img = np.array(g["image"], np.float64)
    for case in g["cases"]:
        z = oracle.filter3x3(img, case["weights"])
        if "expected" in case:
            np.testing.assert_allclose(z, np.array(case["expected"], np.float64), atol=1e-12)
        else:
            np.testing.assert_allclose(z, np.array(case["sums_over_9"], np.float64) / 9.0, atol=1e-12)


# ---------------------------------------------------------------- identity and constants

@pytest.mark.parametrize("C", [1, 3, 4])
def test_identity_scale_one(C):
    src = synth.random_u8((13, 29, C), seed=C)
    np.testing.assert_array_equal(oracle.linear_u8(src, 13, 29), src)
    np.testing.assert_array_equal(oracle.nearest_u8(src, 13, 29), src)
    f = synth.random_f32((13, 29, C), seed=C)
    np.testing.assert_array_equal(oracle.linear_f32(f, 13, 29), f.astype(np.float64))
    np.testing.assert_array_equal(oracle.nearest_f32(f, 13, 29), f)


def test_identity_with_padded_pitch():
    big = synth.random_u8((10, 40, 3), seed=7)
    view = big[:, :17, :]          # rows keep the 120-byte pitch of the parent
    assert view.strides[0] == 120
    np.testing.assert_array_equal(oracle.linear_u8(view, 10, 17), np.ascontiguousarray(view))


@pytest.mark.parametrize("geom", [(5, 7, 13, 2), (48, 64, 96, 128), (9, 9, 1, 1), (1, 1, 7, 5), (30, 20, 11, 47),
                                  (2, 65536, 3, 65535), (65536, 1, 65535, 2), (1, 65535, 1, 65536)])
def test_constant_image_stays_constant(geom):
    H, W, OH, OW = geom
    for k in (0, 1, 77, 254, 255):
        src = np.full((H, W, 3), k, np.uint8)
        assert np.all(oracle.linear_u8(src, OH, OW) == k)
        f = np.full((H, W, 1), k + 0.25, np.float32)
        np.testing.assert_allclose(oracle.linear_f32(f, OH, OW), k + 0.25, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- ramps: closed forms

def test_exact_2x_ramp_upscale_u8():
    # src[y][x] = 4x on a 64-wide row: x(d) = d/2 - 1/4, so out = 2d - 1 inside,
    # 0 at d = 0 (clamped to x = 0) and 252 at d = 127 (clamped to x = 63)
    src = np.tile((4 * np.arange(64)).astype(np.uint8), (5, 1))
    out = oracle.linear_u8(src, 10, 128)[:, :, 0]
    expect = np.clip(2 * np.arange(128) - 1, 0, 252)
    for row in out:
        np.testing.assert_array_equal(row, expect)


def test_exact_2x_ramp_upscale_2d_u8():
    y, x = np.mgrid[0:16, 0:16]
    src = (4 * x + 4 * y).astype(np.uint8)
    out = oracle.linear_u8(src, 32, 32)[:, :, 0]
    d = np.clip(2 * np.arange(32) - 1, 0, 60)
    np.testing.assert_array_equal(out, d[:, None] + d[None, :])


@pytest.mark.parametrize("geom", [(8192, 5980), (1280, 224), (720, 224), (3, 4096), (97, 13), (13, 97), (64, 128),
                                  (65536, 65535), (65535, 65536), (65536, 3), (2, 65536)])
def test_affine_ramp_reproduced_f32(geom):
    # bilinear interpolation reproduces an affine function exactly at the mapped
    # point, clamped into the image: out = a*clamp(x) + b*clamp(y) + c
    n_in, n_out = geom
    a, b, c = 0.125, -0.0625, 3.0
    H = 3
    xs = np.arange(n_in, dtype=np.float64)
    ys = np.arange(H, dtype=np.float64)
    src = (a * xs[None, :] + b * ys[:, None] + c).astype(np.float32)
    out = oracle.linear_f32(src, 5, n_out)[:, :, 0]
    ex = np.array([float(min(max(exact_coord(d, n_in, n_out), 0), n_in - 1)) for d in range(n_out)])
    ey = np.array([float(min(max(exact_coord(d, H, 5), 0), H - 1)) for d in range(5)])
    expect = a * ex[None, :] + b * ey[:, None] + c
    np.testing.assert_allclose(out, expect, rtol=0, atol=1e-9)


# ---------------------------------------------------------------- integer ratios

@pytest.mark.parametrize("C", [1, 3])
def test_2x_downscale_is_rounded_box_mean(C):
    # x(d) = 2d + 1/2 on both axes: u = v = 1/2, weights 1024/1024
    src = synth.random_u8((40, 62, C), seed=11)
    out = oracle.linear_u8(src, 20, 31).astype(np.int64)
    s = src.astype(np.int64)
    box = s[0::2, 0::2] + s[0::2, 1::2] + s[1::2, 0::2] + s[1::2, 1::2]
    np.testing.assert_array_equal(out, (box + 2) >> 2)
    f = synth.random_f32((40, 62, C), seed=12).astype(np.float64)
    outf = oracle.linear_f32(f.astype(np.float32), 20, 31)
    mean = (f[0::2, 0::2] + f[0::2, 1::2] + f[1::2, 0::2] + f[1::2, 1::2]) / 4
    np.testing.assert_allclose(outf, mean, rtol=0, atol=1e-12)


def test_ratio_one_and_a_half_horizontal():
    # 6 -> 4 per period: x(2k) = 3k + 1/4, x(2k+1) = 3k + 7/4, weights 512 / 1536
    src = synth.random_u8((4, 48), seed=13)
    out = oracle.linear_u8(src, 4, 32)[:, :, 0].astype(np.int64)
    s = src.astype(np.int64)
    even = (3 * s[:, 0::3] + s[:, 1::3] + 2) >> 2
    odd = (s[:, 1::3] + 3 * s[:, 2::3] + 2) >> 2
    np.testing.assert_array_equal(out[:, 0::2], even)
    np.testing.assert_array_equal(out[:, 1::2], odd)


# ---------------------------------------------------------------- nearest

def test_nearest_brute_force_small():
    for n_in in range(1, 9):
        for n_out in range(1, 9):
            for d in range(n_out):
                # the largest s with s * n_out <= d * n_in
                s = max(k for k in range(n_in) if k * n_out <= d * n_in)
                assert oracle.nearest_index(n_in, n_out, d) == s


def test_nearest_4x4_images_brute_force():
    src = np.arange(16, dtype=np.uint8).reshape(4, 4) * 10
    for OH in range(1, 9):
        for OW in range(1, 9):
            out = oracle.nearest_u8(src, OH, OW)[:, :, 0]
            for dy in range(OH):
                sy = max(k for k in range(4) if k * OH <= dy * 4)
                for dx in range(OW):
                    sx = max(k for k in range(4) if k * OW <= dx * 4)
                    assert out[dy, dx] == src[sy, sx]


def test_nearest_tiny_gray_reads_even_pixels():
    src = synth.tiny_gray()
    out = oracle.nearest_u8(src, 24, 32)[:, :, 0]
    np.testing.assert_array_equal(out, src[0::2, 0::2])


def test_nearest_matches_torch_nearest():
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    for (H, W, OH, OW) in [(48, 64, 24, 32), (2160, 3840, 1080, 1920), (7, 5, 3, 11), (720, 1280, 224, 224)]:
        iota = np.arange(H * W, dtype=np.float64).reshape(H, W)
        t = F.interpolate(torch.from_numpy(iota)[None, None], size=(OH, OW), mode="nearest")[0, 0].numpy()
        f = oracle.nearest_f32(iota.astype(np.float32) if H * W < 2 ** 24 else iota.astype(np.float32), OH, OW)
        ours = np.array([[oracle.nearest_index(H, OH, dy) * W + oracle.nearest_index(W, OW, dx)
                          for dx in range(OW)] for dy in range(OH)]) if OH * OW < 5000 else None
        if ours is not None:
            np.testing.assert_array_equal(t, ours)
        if H * W < 2 ** 24:
            np.testing.assert_array_equal(f[:, :, 0], t.astype(np.float32))


# ---------------------------------------------------------------- invariants

def test_convexity_within_tap_window():
    src = synth.random_u8((9, 11, 3), seed=21)
    for (OH, OW) in [(4, 5), (17, 23), (9, 30)]:
        out = oracle.linear_u8(src, OH, OW)
        for dy in range(OH):
            j = math.floor(exact_coord(dy, 9, OH))
            rows = sorted({min(max(j, 0), 8), min(max(j + 1, 0), 8)})
            for dx in range(OW):
                i = math.floor(exact_coord(dx, 11, OW))
                cols = sorted({min(max(i, 0), 10), min(max(i + 1, 0), 10)})
                win = src[np.ix_(rows, cols)].reshape(-1, 3)
                assert np.all(out[dy, dx] >= win.min(0)) and np.all(out[dy, dx] <= win.max(0))


def _has_tie(n_in, n_out):
    return any((2048 * (exact_coord(d, n_in, n_out) % 1)).denominator == 2 for d in range(n_out))


@pytest.mark.parametrize("geom", [(48, 64, 96, 128), (1080, 1920, 720, 1280), (33, 47, 19, 71)])
def test_flip_symmetry(geom):
    H, W, OH, OW = geom
    src = synth.random_u8((H, W, 3), seed=31)
    f = src.astype(np.float32)
    a = oracle.linear_f32(f[::-1, ::-1], OH, OW)
    b = oracle.linear_f32(f, OH, OW)[::-1, ::-1]
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-9)
    if not _has_tie(W, OW) and not _has_tie(H, OH):
        np.testing.assert_array_equal(oracle.linear_u8(src[::-1, ::-1], OH, OW),
                                      oracle.linear_u8(src, OH, OW)[::-1, ::-1])


def test_graded_geometries_have_no_weight_ties():
    # with no tie, round-half-up and round-half-to-even give the same weights
    for n_in, n_out in [(64, 128), (48, 96), (1920, 960), (1080, 540), (1920, 1280), (1080, 720),
                        (3840, 1920), (2160, 1080), (1920, 3840), (1080, 2160), (1280, 224), (720, 224),
                        (8192, 5980)]:
        assert not _has_tie(n_in, n_out)


# ---------------------------------------------------------------- library special cases

@pytest.mark.parametrize("geom", [(48, 64, 96, 128), (1080, 1920, 540, 960), (1080, 1920, 720, 1280),
                                  (300, 301, 219, 219), (7, 9, 31, 2)])
def test_f32_matches_torch_bilinear_half_pixel(geom):
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    H, W, OH, OW = geom
    src = synth.random_f32((H, W, 3), seed=41)
    t = F.interpolate(torch.from_numpy(src.astype(np.float64)).permute(2, 0, 1)[None], size=(OH, OW),
                      mode="bilinear", align_corners=False, antialias=False)[0].permute(1, 2, 0).numpy()
    np.testing.assert_allclose(oracle.linear_f32(src, OH, OW), t, rtol=0, atol=1e-9)


def test_u8_within_one_of_torch_uint8_bilinear():
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    src = synth.smooth_rgb(1920, 1080, 2)
    t = torch.from_numpy(np.ascontiguousarray(src)).permute(2, 0, 1)[None]
    try:
        ref = F.interpolate(t, size=(720, 1280), mode="bilinear", align_corners=False,
                            antialias=False)[0].permute(1, 2, 0).numpy()
    except RuntimeError:
        pytest.skip("torch build has no uint8 bilinear")
    ours = oracle.linear_u8(src, 720, 1280)
    assert np.abs(ours.astype(np.int16) - ref.astype(np.int16)).max() <= 1


def test_filter_matches_scipy_correlate_nearest():
    ndimage = pytest.importorskip("scipy.ndimage")
    r = np.random.default_rng(3).random((37, 53)) * 255
    w = synth.filter_weights().astype(np.float64)
    ref = ndimage.correlate(r, w.reshape(3, 3), mode="nearest")
    np.testing.assert_allclose(oracle.filter3x3(r, w), ref, rtol=0, atol=1e-9)
    # an asymmetric filter pins the orientation (no flip)
    wa = np.arange(9, dtype=np.float64)
    np.testing.assert_allclose(oracle.filter3x3(r, wa), ndimage.correlate(r, wa.reshape(3, 3), mode="nearest"),
                               rtol=0, atol=1e-7)


def test_filter_delta_and_box():
    r = np.random.default_rng(4).random((6, 8))
    delta = np.zeros(9)
    delta[4] = 1.0
    np.testing.assert_array_equal(oracle.filter3x3(r, delta), r)
    box = np.full(9, 1.0 / 9.0)
    np.testing.assert_allclose(oracle.filter3x3(np.full((5, 5), 42.0), box), 42.0, atol=1e-12)


# ---------------------------------------------------------------- normalise

def test_normalize_closed_form_and_planes():
    mean, std = synth.NORM_MEAN, synth.NORM_STD
    q = np.zeros((3, 4, 3), np.uint8)
    q[:, :, 0], q[:, :, 1], q[:, :, 2] = 0, 255, 51
    out = oracle.normalize_nchw(q, mean, std)
    assert out.shape == (3, 3, 4)
    np.testing.assert_allclose(out[0], (0.0 - 0.485) / 0.229, atol=1e-12)
    np.testing.assert_allclose(out[1], (1.0 - 0.456) / 0.224, atol=1e-12)
    np.testing.assert_allclose(out[2], (0.2 - 0.406) / 0.225, atol=1e-12)


def test_fused_normalize_is_composition():
    src = synth.random_u8((30, 40, 3), seed=51)
    fused = oracle.linear_u8_normalize(src, 11, 13, synth.NORM_MEAN, synth.NORM_STD)
    q = oracle.linear_u8(src, 11, 13)
    np.testing.assert_array_equal(fused, oracle.normalize_nchw(q, synth.NORM_MEAN, synth.NORM_STD))
