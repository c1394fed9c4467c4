"""Extreme-valued images through every uint8 kernel family, bit-exact.

The integer kernels sum taps in packed lanes (two 16-bit lanes per 32-bit
word, byte dot products, the 1-3 and 3-1 sums of the exact 2x and 3:2
forms); a lane holds its largest value only where every tap of the sum is
255.  Uniform random images almost never put 255 under all the taps of one
output, so these cases take constant 0 and 255 images, 0/255 checkerboards,
channel and column stripes and random 0/255 images through the exact 2x
down, exact 2x up, exact 3:2, any-ratio and streaming upscale paths, under
every border rule, and through the fused gray conversion and the
many-geometry launch.  Every result must equal the oracle bit for bit.
"""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rz():
    import __graft_entry__
    __graft_entry__.build()
    import bilinear_image_resize_gb300 as m
    torch.cuda.set_device(0)
    return m


def patterns(H, W, C, seed):
    yy, xx = np.meshgrid(np.arange(H), np.arange(W), indexing="ij")
    cc = np.arange(C)
    checker = (((yy + xx) & 1) * 255).astype(np.uint8)
    stripes = ((xx & 1) * 255).astype(np.uint8)
    out = {
        "zeros": np.zeros((H, W, C), np.uint8),
        "full": np.full((H, W, C), 255, np.uint8),
        "checker": np.repeat(checker[:, :, None], C, axis=2),
        "column_stripes": np.repeat(stripes[:, :, None], C, axis=2),
        "channel_stripes": np.broadcast_to(((cc & 1) * 255).astype(np.uint8), (H, W, C)).copy(),
        "random_0_255": (np.random.default_rng(seed).integers(0, 2, (H, W, C)) * 255).astype(np.uint8),
    }
    return out


# (name, H, W, OH, OW): the kernel family each geometry selects
GEOMS = [("exact_2x_down", 64, 96, 32, 48), ("exact_2x_up", 24, 40, 48, 80), ("exact_3_2_down", 48, 96, 32, 64),
         ("any_ratio", 37, 53, 23, 41), ("any_ratio_up", 30, 20, 71, 53), ("streaming_up", 100, 150, 520, 700)]


@pytest.mark.parametrize("border", [0, 1, 2])
@pytest.mark.parametrize("C", [1, 3, 4])
@pytest.mark.parametrize("geom", GEOMS, ids=[g[0] for g in GEOMS])
def test_u8_extreme_images(rz, geom, C, border):
    _, H, W, OH, OW = geom
    with rz.resize_plan_create(H, W, OH, OW, rz.RZ_LINEAR, border=border) as plan:
        for name, img in patterns(H, W, C, seed=H + W + C).items():
            src = torch.from_numpy(img).cuda()
            dst = torch.full((OH, OW, C), 0xA5, dtype=torch.uint8, device="cuda")
            rz.resize_u8(plan, src, dst)
            torch.cuda.synchronize()
            want = oracle.linear_u8(img, OH, OW, border)
            got = dst.cpu().numpy()
            assert np.array_equal(got, want), (name, int((got != want).sum()))
        assert rz.resize_plan_status(plan) == rz.RZ_OK


@pytest.mark.parametrize("border", [0, 1, 2])
@pytest.mark.parametrize("C", [3, 4])
@pytest.mark.parametrize("geom", [GEOMS[0], GEOMS[3]], ids=["exact_2x_down", "any_ratio"])
def test_gray_extreme_images(rz, geom, C, border):
    _, H, W, OH, OW = geom
    with rz.resize_plan_create(H, W, OH, OW, rz.RZ_LINEAR, border=border) as plan:
        for name, img in patterns(H, W, C, seed=7 + C).items():
            src = torch.from_numpy(img).cuda()
            dst = torch.full((OH, OW), 0xA5, dtype=torch.uint8, device="cuda")
            rz.resize_fused(plan, src, dst, rz.make_epilogue(rz.RZ_EPI_GRAY_RGB))
            torch.cuda.synchronize()
            want = oracle.gray_resize_u8(img, OH, OW, border=border)
            assert np.array_equal(dst.cpu().numpy(), want), name


@pytest.mark.parametrize("C", [1, 3, 4])
def test_multi_extreme_images(rz, C):
    geoms = [(40, 64, 20, 32), (20, 32, 40, 64), (30, 45, 20, 30), (17, 23, 29, 31), (40, 320, 25, 640)]
    srcs, dsts, imgs = [], [], []
    for k, (H, W, OH, OW) in enumerate(geoms):
        for name, img in patterns(H, W, C, seed=k).items():
            imgs.append(img)
            srcs.append(torch.from_numpy(img).cuda())
            dsts.append(torch.full((OH, OW, C), 0xA5, dtype=torch.uint8, device="cuda"))
    jobs, CC = rz.make_jobs(srcs, dsts)
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    rz.resize_u8_multi(jobs, len(srcs), CC, rz.RZ_LINEAR, status)
    torch.cuda.synchronize()
    assert int(status.item()) == rz.RZ_OK
    for img, d in zip(imgs, dsts):
        np.testing.assert_array_equal(d.cpu().numpy(), oracle.linear_u8(img, *d.shape[:2]))
