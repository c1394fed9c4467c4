"""The bounds-checked build (libgbresize_checked.so) on the resize kernels.

Built with -DRZ_CHECK_BOUNDS, the direct, staged and streaming kernels check
every global load and store against the source, output and table extents the
host declares, and every shared-memory copy and read window against the CTA's
dynamic shared memory; an access outside them is not made and RZ_ERR_ARG is
recorded in the status word (no trap, nothing faults).  Here:
  * a sweep of small and odd geometries, every channel count and mode, and
    every kernel family (direct loads, staged tiles, streaming, the exact
    2x / 3:2 kernels, float32, the fused epilogues, border rules, the no-alloc
    path) must run through the checked build with status RZ_OK and give the
    oracle's result;
  * with the declared extents shortened by one byte (the build's
    RZ_CHECK_SHRINK test hook; the buffers themselves stay whole, so a refused
    access would still have been valid memory), kernels that read the last
    source byte or write the last output byte must report RZ_ERR_ARG, and
    the next call without the hook is clean again.
Runs on the checked library by swapping it into the binding for this module.
"""
import os

import numpy as np
import pytest

import oracle
from bilinear_image_resize_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

F32_TOL = 1e-4


@pytest.fixture(scope="module")
def rz():
    import __graft_entry__
    __graft_entry__.build()
    from bilinear_image_resize_gb300 import _build, _native
    _build.build(checked=True)
    import bilinear_image_resize_gb300 as m
    torch.cuda.set_device(0)
    normal = _native.load()
    _native._lib = _native.load_checked()
    try:
        yield m
    finally:
        torch.cuda.synchronize()
        _native._lib = normal


def run_u8(rz, img, OH, OW, mode, border=0, opts=()):
    H, W = img.shape[:2]
    src = torch.from_numpy(np.ascontiguousarray(img)).cuda()
    dst = torch.full((OH, OW, img.shape[2]), 0x5A, dtype=torch.uint8, device="cuda")
    with rz.resize_plan_create(H, W, OH, OW, mode, border=border) as plan:
        for o, v in opts:
            rz.resize_plan_set_option(plan, o, v)
        rz.resize_u8(plan, src, dst)
        st = rz.resize_plan_status(plan)
    return dst.cpu().numpy(), st


def want_u8(img, OH, OW, mode, border=0):
    return oracle.linear_u8(img, OH, OW, border) if mode == 1 else oracle.nearest_u8(img, OH, OW)


@pytest.mark.parametrize("C", [1, 3, 4])
def test_checked_sweep_every_u8_kernel(rz, C):
    rng = np.random.default_rng(100 + C)
    for _ in range(10):
        H, W, OH, OW = (int(v) for v in rng.integers(1, 68, size=4))
        img = synth.random_u8((H, W, C), seed=H * 7 + W)
        for mode in (rz.RZ_LINEAR, rz.RZ_NEAREST):
            want = want_u8(img, OH, OW, mode)
            for opts in ((), ((rz.RZ_OPT_U8_KERNEL, 1),), ((rz.RZ_OPT_U8_KERNEL, 3),)):
                got, st = run_u8(rz, img, OH, OW, mode, opts=opts)
                assert st == rz.RZ_OK, (H, W, OH, OW, C, mode, opts)
                np.testing.assert_array_equal(got, want, err_msg=str((H, W, OH, OW, C, mode, opts)))


# exact 2x down / up, 3:2, generic up, on layouts that take the vector paths,
# and the streaming upscale (option 2)
EXACT = [(540, 976, 270, 488), (540, 960, 360, 640), (61, 50, 122, 100), (300, 480, 900, 700), (96, 64, 48, 32)]


@pytest.mark.parametrize("C", [1, 3, 4])
@pytest.mark.parametrize("geo", EXACT)
def test_checked_exact_ratio_and_streaming(rz, C, geo):
    H, W, OH, OW = geo
    img = synth.random_u8((H, W, C), seed=H + W + C)
    for mode in (rz.RZ_LINEAR, rz.RZ_NEAREST):
        want = want_u8(img, OH, OW, mode)
        for opts in ((), ((rz.RZ_OPT_U8_KERNEL, 2),)):
            got, st = run_u8(rz, img, OH, OW, mode, opts=opts)
            assert st == rz.RZ_OK, (geo, C, mode, opts)
            np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("border", [1, 2])
@pytest.mark.parametrize("C", [1, 3, 4])
def test_checked_border_rules(rz, border, C):
    for (H, W, OH, OW) in [(37, 41, 74, 82), (33, 20, 80, 50)]:
        img = synth.random_u8((H, W, C), seed=H + border)
        got, st = run_u8(rz, img, OH, OW, rz.RZ_LINEAR, border=border)
        assert st == rz.RZ_OK
        np.testing.assert_array_equal(got, oracle.linear_u8(img, OH, OW, border))


def test_checked_float32_and_epilogues(rz):
    img = synth.random_f32((97, 131), seed=3)
    src = torch.from_numpy(img).cuda()
    for (OH, OW, mode, opt) in [(61, 200, 1, 0), (61, 200, 1, 1), (150, 90, 0, 0)]:
        dst = torch.empty((OH, OW), dtype=torch.float32, device="cuda")
        with rz.resize_plan_create(97, 131, OH, OW, mode) as plan:
            rz.resize_plan_set_option(plan, rz.RZ_OPT_F32_KERNEL, opt)
            rz.resize_f32(plan, src, dst)
            assert rz.resize_plan_status(plan) == rz.RZ_OK
        want = (oracle.linear_f32(img, OH, OW) if mode == 1 else oracle.nearest_f32(img, OH, OW)).reshape(OH, OW)
        assert np.max(np.abs(dst.cpu().numpy().astype(np.float64) - want)) <= F32_TOL
    # fused 3x3 and 5x5 (streaming kernel), normalise (direct and staged)
    for K in (3, 5):
        w = synth.filter_weights() if K == 3 else synth.filter_weights_k(K)
        dst = torch.empty((70, 90), dtype=torch.float32, device="cuda")
        with rz.resize_plan_create(97, 131, 70, 90, rz.RZ_LINEAR) as plan:
            e = (rz.make_epilogue(rz.RZ_EPI_FILTER3X3, w3x3=w) if K == 3
                 else rz.make_epilogue(rz.RZ_EPI_FILTER, wk=w))
            rz.resize_fused(plan, src, dst, e)
            assert rz.resize_plan_status(plan) == rz.RZ_OK
        want = (oracle.linear_f32_filter3x3(img, 70, 90, w) if K == 3
                else oracle.linear_f32_filter(img, 70, 90, w)).reshape(70, 90)
        # the float32 bound of a K x K sum (K^2 products summed in float32)
        # on top of the resize's
        tol = F32_TOL * float(np.abs(w).sum()) + 2 * K * K * 2.0 ** -24 * 255.0
        assert np.max(np.abs(dst.cpu().numpy().astype(np.float64) - want)) <= tol
    frames = np.stack([synth.random_u8((90, 160, 3), seed=n) for n in range(2)])
    for kernel in (0, 1):
        dst = torch.empty((2, 3, 56, 56), dtype=torch.float32, device="cuda")
        with rz.resize_plan_create(90, 160, 56, 56, rz.RZ_LINEAR) as plan:
            rz.resize_plan_set_option(plan, rz.RZ_OPT_U8_KERNEL, kernel)
            rz.resize_fused(plan, torch.from_numpy(frames).cuda(), dst,
                            rz.make_epilogue(rz.RZ_EPI_NORMALIZE_NCHW, mean=synth.NORM_MEAN, std=synth.NORM_STD))
            assert rz.resize_plan_status(plan) == rz.RZ_OK
        for n in range(2):
            want = oracle.linear_u8_normalize(frames[n], 56, 56, synth.NORM_MEAN, synth.NORM_STD)
            assert np.max(np.abs(dst.cpu().numpy()[n].astype(np.float64) - want)) <= F32_TOL


def test_checked_gray_and_no_alloc(rz):
    img = synth.random_u8((120, 168, 3), seed=9)
    src = torch.from_numpy(img).cuda()
    for (OH, OW) in [(60, 84), (77, 50)]:
        dst = torch.zeros((OH, OW), dtype=torch.uint8, device="cuda")
        with rz.resize_plan_create(120, 168, OH, OW, rz.RZ_LINEAR) as plan:
            rz.resize_fused(plan, src, dst, rz.make_epilogue(rz.RZ_EPI_GRAY_RGB))
            assert rz.resize_plan_status(plan) == rz.RZ_OK
        np.testing.assert_array_equal(dst.cpu().numpy(), oracle.gray_resize_u8(img, OH, OW))
        out = torch.zeros((OH, OW, 3), dtype=torch.uint8, device="cuda")
        rz.resize_u8_noalloc(src, out)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.cpu().numpy(), oracle.linear_u8(img, OH, OW))


# kernels whose last source byte or last output byte is accessed: with the
# declared extents one byte short they must report and then recover
SHRINK_CASES = [
    ("exact 2x down, direct", (540, 976, 270, 488, 3), ()),
    ("any ratio, direct", (50, 70, 33, 91, 3), ()),
    ("exact 2x up, pixel lanes", (40, 64, 80, 128, 3), ()),
    ("staged tiles", (50, 70, 33, 91, 3), "staged"),
    ("streaming upscale", (40, 72, 200, 144, 1), "stream"),
]


@pytest.mark.parametrize("case", SHRINK_CASES, ids=[c[0] for c in SHRINK_CASES])
def test_checked_build_reports_an_access_past_the_declared_extent(rz, case):
    _, (H, W, OH, OW, C), which = case
    opts = {"staged": ((rz.RZ_OPT_U8_KERNEL, 1),), "stream": ((rz.RZ_OPT_U8_KERNEL, 2),)}.get(which, ())
    img = synth.random_u8((H, W, C), seed=5)
    os.environ["RZ_CHECK_SHRINK"] = "1"
    try:
        _, st = run_u8(rz, img, OH, OW, rz.RZ_LINEAR, opts=opts)
    finally:
        del os.environ["RZ_CHECK_SHRINK"]
    assert st == rz.RZ_ERR_ARG, st
    got, st = run_u8(rz, img, OH, OW, rz.RZ_LINEAR, opts=opts)
    assert st == rz.RZ_OK
    np.testing.assert_array_equal(got, oracle.linear_u8(img, OH, OW))
