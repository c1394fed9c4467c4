"""Parity of the border rules and the fused grayscale conversion (through the
C ABI) with the CPU oracle.

Border rules: clamp, mirror and wrap (CUDA interpolation page §6.1) on every
kernel that takes them: the exact 2x upscale, the direct-load kernels, the
streaming and staged kernels (mirror, which lives in the tables), the float32
direct kernel (wrap) and the fused epilogues.  Grayscale: BT.601 conversion
before the resize (OpenCV object-tracking page §3.1.1), both channel orders,
3 and 4 channels, both modes, every border, batches.  uint8 results are
bit-exact; float32 within 1e-4.
"""
import numpy as np
import pytest

import oracle
from bilinear_image_resize_gb300 import synth
from gpu_util import Canvas, device_image, max_abs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

F32_TOL = 1e-4
MIRROR, WRAP = 1, 2


@pytest.fixture(scope="module")
def rz():
    import __graft_entry__
    __graft_entry__.build()
    import bilinear_image_resize_gb300 as m
    torch.cuda.set_device(0)
    return m


def gpu_u8(rz, img, OH, OW, mode, border, src_pitch=None, src_off=0, dst_pad=0, opts=()):
    if img.ndim == 2:
        img = img[:, :, None]
    H, W, C = img.shape
    src, _keep = device_image(img, src_pitch, src_off)
    out = Canvas(OH, OW, C, torch.uint8, dst_pad)
    with rz.resize_plan_create(H, W, OH, OW, mode, border=border) as plan:
        for k, v in opts:
            rz.resize_plan_set_option(plan, k, v)
        rz.resize_u8(plan, src, out.view)
        torch.cuda.synchronize()
        assert rz.resize_plan_status(plan) == rz.RZ_OK
    out.check_canary()
    return out.result()


GEOMS_UP = [(48, 64, 96, 128), (37, 53, 100, 131), (5, 7, 13, 17), (1, 5, 4, 9), (2, 2, 7, 3), (9, 13, 30, 41),
            (3, 3, 10, 10), (5, 1, 9, 3), (31, 17, 62, 34), (40, 30, 41, 300)]
GEOMS_DOWN = [(90, 120, 37, 50), (64, 64, 32, 32), (33, 47, 11, 20)]


@pytest.mark.parametrize("border", [0, MIRROR, WRAP])
@pytest.mark.parametrize("C", [1, 3, 4])
@pytest.mark.parametrize("geom", GEOMS_UP + GEOMS_DOWN)
def test_u8_border_small(rz, border, C, geom):
    H, W, OH, OW = geom
    img = synth.random_u8((H, W, C), seed=H * 31 + W + C)
    np.testing.assert_array_equal(gpu_u8(rz, img, OH, OW, rz.RZ_LINEAR, border),
                                  oracle.linear_u8(img, OH, OW, border))


@pytest.mark.parametrize("border", [MIRROR, WRAP])
@pytest.mark.parametrize("C", [1, 3, 4])
def test_u8_border_unaligned_layouts(rz, border, C):
    # odd source offset and pitch, padded output rows: the byte paths
    for H, W, OH, OW in [(21, 30, 42, 60), (17, 23, 50, 61)]:
        img = synth.random_u8((H, W, C), seed=5 + C)
        got = gpu_u8(rz, img, OH, OW, rz.RZ_LINEAR, border, src_pitch=W * C + 3, src_off=1, dst_pad=5)
        np.testing.assert_array_equal(got, oracle.linear_u8(img, OH, OW, border))


@pytest.mark.parametrize("border", [0, MIRROR, WRAP])
def test_u8_border_1080p_to_4k(rz, border):
    img = synth.smooth_rgb(1920, 1080, 2)
    np.testing.assert_array_equal(gpu_u8(rz, img, 2160, 3840, rz.RZ_LINEAR, border),
                                  oracle.linear_u8(img, 2160, 3840, border))


@pytest.mark.parametrize("border", [MIRROR, WRAP])
def test_u8_border_large_upscale_not_2x(rz, border):
    # mirror: the streaming kernel (tables); wrap: the direct kernel
    img = synth.smooth_rgb(640, 360, 9)
    np.testing.assert_array_equal(gpu_u8(rz, img, 1000, 1700, rz.RZ_LINEAR, border),
                                  oracle.linear_u8(img, 1000, 1700, border))


@pytest.mark.parametrize("kernel", [1, 2, 3])
def test_u8_mirror_on_every_kernel(rz, kernel):
    for H, W, OH, OW in [(37, 53, 100, 131), (48, 64, 96, 128), (90, 120, 37, 50)]:
        img = synth.random_u8((H, W, 3), seed=kernel)
        got = gpu_u8(rz, img, OH, OW, rz.RZ_LINEAR, MIRROR, opts=[(rz.RZ_OPT_U8_KERNEL, kernel)])
        np.testing.assert_array_equal(got, oracle.linear_u8(img, OH, OW, MIRROR))


def test_u8_wrap_on_the_direct_kernels_only(rz):
    img = synth.random_u8((37, 53, 3), seed=1)
    got = gpu_u8(rz, img, 100, 131, rz.RZ_LINEAR, WRAP, opts=[(rz.RZ_OPT_U8_KERNEL, 3)])
    np.testing.assert_array_equal(got, oracle.linear_u8(img, 100, 131, WRAP))
    got = gpu_u8(rz, img, 74, 106, rz.RZ_LINEAR, WRAP, opts=[(rz.RZ_OPT_GENERIC_ONLY, 1)])
    np.testing.assert_array_equal(got, oracle.linear_u8(img, 74, 106, WRAP))
    for k in (1, 2):
        with pytest.raises(rz.ResizeError) as ei:
            gpu_u8(rz, img, 100, 131, rz.RZ_LINEAR, WRAP, opts=[(rz.RZ_OPT_U8_KERNEL, k)])
        assert ei.value.code == rz.RZ_ERR_UNSUPPORTED


@pytest.mark.parametrize("border", [MIRROR, WRAP])
def test_nearest_ignores_the_border(rz, border):
    img = synth.random_u8((33, 45, 3), seed=3)
    np.testing.assert_array_equal(gpu_u8(rz, img, 70, 100, rz.RZ_NEAREST, border),
                                  oracle.nearest_u8(img, 70, 100))


@pytest.mark.parametrize("border", [MIRROR, WRAP])
def test_u8_batch_border(rz, border):
    N, H, W, OH, OW = 5, 27, 41, 60, 95
    frames = np.stack([synth.random_u8((H, W, 3), seed=40 + n) for n in range(N)])
    src = torch.from_numpy(frames).cuda()
    dst = torch.zeros((N, OH, OW, 3), dtype=torch.uint8, device="cuda")
    with rz.resize_plan_create(H, W, OH, OW, rz.RZ_LINEAR, border=border) as plan:
        rz.resize_u8_batch(plan, src, dst)
        torch.cuda.synchronize()
    got = dst.cpu().numpy()
    for n in range(N):
        np.testing.assert_array_equal(got[n], oracle.linear_u8(frames[n], OH, OW, border))


# ---------------------------------------------------------------- float32

@pytest.mark.parametrize("border", [0, MIRROR, WRAP])
@pytest.mark.parametrize("C", [1, 3, 4])
@pytest.mark.parametrize("geom", [(37, 53, 100, 131), (5, 7, 13, 17), (1, 5, 4, 9), (90, 120, 37, 50),
                                  (256, 256, 512, 512)])
def test_f32_border(rz, border, C, geom):
    H, W, OH, OW = geom
    img = synth.random_f32((H, W, C), seed=H + W + C)
    src = torch.from_numpy(img).cuda()
    out = Canvas(OH, OW, C, torch.float32, 3)
    with rz.resize_plan_create(H, W, OH, OW, rz.RZ_LINEAR, border=border) as plan:
        rz.resize_f32(plan, src, out.view)
        torch.cuda.synchronize()
    out.check_canary()
    err = max_abs(out.result(), oracle.linear_f32(img, OH, OW, border))
    assert err <= F32_TOL, err


def test_f32_wrap_batch(rz):
    N, H, W, OH, OW = 3, 20, 30, 47, 70
    frames = np.stack([synth.random_f32((H, W, 3), seed=n) for n in range(N)])
    src = torch.from_numpy(frames).cuda()
    dst = torch.zeros((N, OH, OW, 3), dtype=torch.float32, device="cuda")
    with rz.resize_plan_create(H, W, OH, OW, rz.RZ_LINEAR, border=WRAP) as plan:
        rz.resize_f32_batch(plan, src, dst)
        torch.cuda.synchronize()
    for n in range(N):
        assert max_abs(dst[n].cpu().numpy(), oracle.linear_f32(frames[n], OH, OW, WRAP)) <= F32_TOL


# ---------------------------------------------------------------- epilogues

@pytest.mark.parametrize("border", [MIRROR, WRAP])
@pytest.mark.parametrize("kernel", [0, 1])
def test_normalize_border(rz, border, kernel):
    N, H, W, OH, OW = 4, 50, 70, 120, 160
    frames = np.stack([synth.random_u8((H, W, 3), seed=70 + n) for n in range(N)])
    src = torch.from_numpy(frames).cuda()
    dst = torch.zeros((N, 3, OH, OW), dtype=torch.float32, device="cuda")
    with rz.resize_plan_create(H, W, OH, OW, rz.RZ_LINEAR, border=border) as plan:
        rz.resize_plan_set_option(plan, rz.RZ_OPT_U8_KERNEL, kernel)
        e = rz.make_epilogue(rz.RZ_EPI_NORMALIZE_NCHW, mean=synth.NORM_MEAN, std=synth.NORM_STD)
        if border == WRAP and kernel == 1:
            with pytest.raises(rz.ResizeError) as ei:
                rz.resize_fused(plan, src, dst, e)
            assert ei.value.code == rz.RZ_ERR_UNSUPPORTED
            return
        rz.resize_fused(plan, src, dst, e)
        torch.cuda.synchronize()
    got = dst.cpu().numpy()
    for n in range(N):
        want = oracle.linear_u8_normalize(frames[n], OH, OW, synth.NORM_MEAN, synth.NORM_STD, border)
        assert max_abs(got[n], want) <= F32_TOL


def test_filter3x3_mirror_and_wrap(rz):
    H, W, OH, OW = 64, 80, 150, 170
    img = synth.random_f32((H, W), seed=9)
    w = synth.filter_weights()
    src = torch.from_numpy(img).cuda()
    dst = torch.zeros((OH, OW), dtype=torch.float32, device="cuda")
    with rz.resize_plan_create(H, W, OH, OW, rz.RZ_LINEAR, border=MIRROR) as plan:
        rz.resize_fused(plan, src, dst, rz.make_epilogue(rz.RZ_EPI_FILTER3X3, w3x3=w))
        torch.cuda.synchronize()
    want = oracle.filter3x3(oracle.linear_f32(img, OH, OW, MIRROR), w)
    assert max_abs(dst.cpu().numpy(), want) <= F32_TOL
    # wrap: the tile kernel (the streaming one takes monotone tables only)
    with rz.resize_plan_create(H, W, OH, OW, rz.RZ_LINEAR, border=WRAP) as plan:
        rz.resize_fused(plan, src, dst, rz.make_epilogue(rz.RZ_EPI_FILTER3X3, w3x3=w))
        torch.cuda.synchronize()
        want = oracle.filter3x3(oracle.linear_f32(img, OH, OW, WRAP), w)
        assert max_abs(dst.cpu().numpy(), want) <= F32_TOL
        rz.resize_plan_set_option(plan, rz.RZ_OPT_FILTER_KERNEL, 1)
        with pytest.raises(rz.ResizeError) as ei:
            rz.resize_fused(plan, src, dst, rz.make_epilogue(rz.RZ_EPI_FILTER3X3, w3x3=w))
        assert ei.value.code == rz.RZ_ERR_UNSUPPORTED


# ---------------------------------------------------------------- grayscale

def gpu_gray(rz, img, OH, OW, mode, border=0, bgr=False, src_pitch=None, src_off=0, dst_pad=0):
    H, W, C = img.shape
    src, _keep = device_image(img, src_pitch, src_off)
    out = Canvas(OH, OW, 1, torch.uint8, dst_pad)
    kind = rz.RZ_EPI_GRAY_BGR if bgr else rz.RZ_EPI_GRAY_RGB
    with rz.resize_plan_create(H, W, OH, OW, mode, border=border) as plan:
        rz.resize_fused(plan, src, out.view[:, :, 0], rz.make_epilogue(kind))
        torch.cuda.synchronize()
        assert rz.resize_plan_status(plan) == rz.RZ_OK
    out.check_canary()
    return out.result()[:, :, 0]


@pytest.mark.parametrize("C", [3, 4])
@pytest.mark.parametrize("bgr", [False, True])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("geom", [(48, 64, 96, 128), (37, 53, 100, 131), (90, 120, 37, 50), (64, 64, 32, 32),
                                  (1, 5, 4, 9), (33, 47, 33, 47), (20, 300, 7, 11), (46, 70, 23, 35),
                                  (2, 2, 1, 1), (6, 14, 3, 7)])
def test_gray_small(rz, C, bgr, mode, geom):
    H, W, OH, OW = geom
    img = synth.random_u8((H, W, C), seed=H + W + C + int(bgr))
    got = gpu_gray(rz, img, OH, OW, mode, bgr=bgr)
    np.testing.assert_array_equal(got, oracle.gray_resize_u8(img, OH, OW, linear=mode == 1, bgr=bgr))


@pytest.mark.parametrize("border", [MIRROR, WRAP])
@pytest.mark.parametrize("C", [3, 4])
def test_gray_border_and_unaligned(rz, border, C):
    for H, W, OH, OW in [(37, 53, 100, 131), (21, 30, 42, 60)]:
        img = synth.random_u8((H, W, C), seed=border + C)
        got = gpu_gray(rz, img, OH, OW, 1, border=border, src_pitch=W * C + 1, src_off=3, dst_pad=3)
        np.testing.assert_array_equal(got, oracle.gray_resize_u8(img, OH, OW, border=border))


@pytest.mark.parametrize("C", [3, 4])
@pytest.mark.parametrize("mode", [0, 1])
def test_gray_exact_2x_layouts(rz, C, mode):
    # vector loads only where the source and output layouts allow; an odd
    # source offset, an odd pitch or an odd output offset take the generic path
    img = synth.random_u8((30, 86, C), seed=C + 7 * mode)
    want = oracle.gray_resize_u8(img, 15, 43, linear=mode == 1)
    for kw in ({}, {"src_off": 1}, {"src_pitch": 86 * C + 8}, {"src_pitch": 86 * C + 3}, {"dst_pad": 1}):
        np.testing.assert_array_equal(gpu_gray(rz, img, 15, 43, mode, **kw), want)


@pytest.mark.parametrize("mode", [0, 1])
def test_gray_4k_to_1080p(rz, mode):
    img = synth.smooth_rgb(3840, 2160, 3)
    got = gpu_gray(rz, img, 1080, 1920, mode)
    np.testing.assert_array_equal(got, oracle.gray_resize_u8(img, 1080, 1920, linear=mode == 1))


def test_gray_batch(rz):
    N, H, W, OH, OW = 6, 45, 61, 30, 50
    frames = np.stack([synth.random_u8((H, W, 4), seed=90 + n) for n in range(N)])
    src = torch.from_numpy(frames).cuda()
    dst = torch.zeros((N, OH, OW), dtype=torch.uint8, device="cuda")
    with rz.resize_plan_create(H, W, OH, OW, rz.RZ_LINEAR) as plan:
        rz.resize_fused(plan, src, dst, rz.make_epilogue(rz.RZ_EPI_GRAY_BGR))
        torch.cuda.synchronize()
    got = dst.cpu().numpy()
    for n in range(N):
        np.testing.assert_array_equal(got[n], oracle.gray_resize_u8(frames[n], OH, OW, bgr=True))


def test_gray_argument_checks(rz):
    with rz.resize_plan_create(8, 8, 4, 4, rz.RZ_LINEAR) as plan:
        lib = rz._native.load()
        src = torch.zeros((8, 8, 3), dtype=torch.uint8, device="cuda")
        dst = torch.zeros((4, 4), dtype=torch.uint8, device="cuda")
        e = rz.make_epilogue(rz.RZ_EPI_GRAY_RGB)
        stream = torch.cuda.current_stream().cuda_stream
        import ctypes
        # one channel has no colour; float source is not a gray input
        assert lib.resize_fused(plan.handle, src.data_ptr(), rz.RZ_U8, 8, dst.data_ptr(), 4, 8, 8, 1, 4, 4,
                                rz.RZ_LINEAR, ctypes.byref(e), stream) == rz.RZ_ERR_ARG
        assert lib.resize_fused(plan.handle, src.data_ptr(), rz.RZ_F32, 96, dst.data_ptr(), 4, 8, 8, 3, 4, 4,
                                rz.RZ_LINEAR, ctypes.byref(e), stream) == rz.RZ_ERR_ARG
        # the output row is one channel wide: a pitch below out_w is rejected
        assert lib.resize_fused(plan.handle, src.data_ptr(), rz.RZ_U8, 24, dst.data_ptr(), 3, 8, 8, 3, 4, 4,
                                rz.RZ_LINEAR, ctypes.byref(e), stream) == rz.RZ_ERR_ARG
        assert lib.resize_fused(plan.handle, src.data_ptr(), rz.RZ_U8, 24, dst.data_ptr(), 4, 8, 8, 3, 4, 4,
                                rz.RZ_LINEAR, ctypes.byref(e), stream) == rz.RZ_OK
        torch.cuda.synchronize()
        with pytest.raises(rz.ResizeError):
            rz.resize_plan_set_tile(plan, 5, 1, 8)
