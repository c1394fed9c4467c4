"""The closed forms the exact-ratio kernels compute, checked against the oracle.

At an exact 2x downscale every tap weight is 1024, so the fixed-point sum is
(t0 + t1 + b0 + b1 + 2) >> 2.  At an exact 2x upscale the weights are 512 and
1536, so the sum is (sum of b * a * t + 8) >> 4 with a, b in {1, 3} (the
9-3-3-1 filter), the outside tap at a border folded onto the edge pixel by
the plan being the same as repeating the edge pixel.  These identities are
what direct.cu relies on; here they are computed in numpy from their own
definition and compared with the oracle's general formula on random images.
"""
import numpy as np
import pytest

import oracle


def down2(img):
    t = img.astype(np.int64)
    return ((t[0::2, 0::2] + t[0::2, 1::2] + t[1::2, 0::2] + t[1::2, 1::2] + 2) >> 2).astype(np.uint8)


def up2(img):
    t = img.astype(np.int64)
    H, W = t.shape[:2]
    p = np.pad(t, ((1, 1), (1, 1), (0, 0)), mode="edge")   # edge repetition
    out = np.zeros((2 * H, 2 * W, t.shape[2]), np.int64)
    for j, (wy0, wy1, dy) in enumerate([(1, 3, 0), (3, 1, 1)]):   # rows (r-1, r) or (r, r+1)
        for i, (wx0, wx1, dx) in enumerate([(1, 3, 0), (3, 1, 1)]):
            v = (wy0 * wx0 * p[dy:dy + H, dx:dx + W] + wy0 * wx1 * p[dy:dy + H, dx + 1:dx + 1 + W] +
                 wy1 * wx0 * p[dy + 1:dy + 1 + H, dx:dx + W] + wy1 * wx1 * p[dy + 1:dy + 1 + H, dx + 1:dx + 1 + W])
            out[j::2, i::2] = (v + 8) >> 4
    return out.astype(np.uint8)


@pytest.mark.parametrize("C", [1, 3, 4])
def test_exact_2x_downscale_is_the_four_tap_mean(C):
    rng = np.random.default_rng(31 + C)
    for (H, W) in [(2, 2), (2, 18), (6, 34), (30, 46), (64, 62)]:
        img = rng.integers(0, 256, size=(H, W, C), dtype=np.uint8)
        np.testing.assert_array_equal(down2(img), oracle.linear_u8(img, H // 2, W // 2))


@pytest.mark.parametrize("C", [1, 3, 4])
def test_exact_2x_upscale_is_the_9331_filter(C):
    rng = np.random.default_rng(41 + C)
    for (H, W) in [(1, 1), (1, 5), (3, 2), (2, 9), (7, 13), (16, 16), (33, 70)]:
        img = rng.integers(0, 256, size=(H, W, C), dtype=np.uint8)
        np.testing.assert_array_equal(up2(img), oracle.linear_u8(img, 2 * H, 2 * W))


def test_the_identities_fail_on_a_planted_error():
    # a wrong weight pair would not pass: the comparison has teeth
    rng = np.random.default_rng(5)
    img = rng.integers(0, 256, size=(9, 11, 3), dtype=np.uint8)
    t = img.astype(np.int64)
    wrong = ((t[0::2, 0::2][:4, :5] * 3 + t[1::2, 1::2][:4, :5] + 2) >> 2).astype(np.uint8)
    assert not np.array_equal(wrong, oracle.linear_u8(img, 4, 5)[:4, :5])


def test_gray_split_weights_and_division_by_1000():
    # the gray kernels form 299 R + 587 G + 114 B + 500 as
    # 256 * (R + 2 G) + (43 R + 75 G + 114 B) + 500 (two byte dot products)
    # and take floor(s / 1000) as the high word of s * 4294968, exact for
    # every s the sum can reach (at most 255 * 1000 + 500); checked here
    # over all inputs against the oracle's conversion
    r, g, b = np.meshgrid(np.arange(256), np.arange(256), np.arange(256), indexing="ij")
    s = 256 * (r + 2 * g) + (43 * r + 75 * g + 114 * b) + 500
    y = (s.astype(np.uint64) * np.uint64(4294968)) >> np.uint64(32)
    rgb = np.stack([r, g, b], -1).astype(np.uint8).reshape(4096, 4096, 3)
    np.testing.assert_array_equal(y.reshape(4096, 4096).astype(np.uint8), oracle.gray_u8(rgb))
    t = np.arange(0, 255501, dtype=np.uint64)
    np.testing.assert_array_equal((t * np.uint64(4294968)) >> np.uint64(32), t // np.uint64(1000))


def down32(img):
    # exact 3:2 downscale: output 2m samples x = 3m + 1/4 (taps 3m, 3m+1 at
    # 3/4, 1/4), output 2m+1 samples 3m + 7/4 (taps 3m+1, 3m+2 at 1/4, 3/4);
    # the 11-bit weights are 1536 and 512, so the exact sum is the 9-3-3-1
    # filter (sum of b a t + 8) >> 4
    t = img.astype(np.int64)
    H, W = t.shape[:2]
    wts = [((0, 3), (1, 1)), ((1, 1), (2, 3))]     # (offset, weight) pairs for outputs 2m and 2m+1
    out = np.zeros((2 * H // 3, 2 * W // 3, t.shape[2]), np.int64)
    for j, ry in enumerate(wts):
        for i, rx in enumerate(wts):
            acc = 0
            for (oy, wy) in ry:
                for (ox, wx) in rx:
                    acc = acc + wy * wx * t[oy::3, ox::3][:H // 3, :W // 3]
            out[j::2, i::2] = (acc + 8) >> 4
    return out.astype(np.uint8)


@pytest.mark.parametrize("C", [1, 3, 4])
def test_exact_3_to_2_downscale_is_the_9331_filter(C):
    rng = np.random.default_rng(41 + C)
    for (H, W) in [(3, 3), (3, 12), (9, 24), (30, 45), (1080, 1920)]:
        img = rng.integers(0, 256, size=(H, W, C), dtype=np.uint8)
        np.testing.assert_array_equal(down32(img), oracle.linear_u8(img, 2 * H // 3, 2 * W // 3))
