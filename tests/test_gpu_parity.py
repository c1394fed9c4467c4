"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

uint8 results must be bit-exact; float32 results within 1e-4 absolute on
values in [0, 255] (the bound the float32 path is specified to); nearest is
a copy and must be exact for both types.  The five workloads run at full
size and are compared on every output element; a seeded sweep of small
geometries covers ragged tiles, every channel count, odd pitches, unaligned
pointers, extreme ratios and the degenerate sizes.
"""
import numpy as np
import pytest

import oracle
from bilinear_image_resize_gb300 import synth
from gpu_util import Canvas, device_image, max_abs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

F32_TOL = 1e-4


@pytest.fixture(scope="module")
def rz():
    import __graft_entry__
    __graft_entry__.build()
    import bilinear_image_resize_gb300 as m
    torch.cuda.set_device(0)
    return m


def gpu_u8(rz, img, OH, OW, mode, src_pitch=None, src_off=0, dst_pad=0, dst_off=0, tile=None, stream=None, opts=()):
    if img.ndim == 2:
        img = img[:, :, None]
    H, W, C = img.shape
    src, _keep = device_image(img, src_pitch, src_off)
    out = Canvas(OH, OW, C, torch.uint8, dst_pad, dst_off)
    with rz.resize_plan_create(H, W, OH, OW, mode) as plan:
        for k, v in opts:
            rz.resize_plan_set_option(plan, k, v)
        if tile:
            rz.resize_plan_set_tile(plan, rz.KIND_U8, *tile)
        rz.resize_u8(plan, src, out.view, stream=stream)
        torch.cuda.synchronize()
        assert rz.resize_plan_status(plan) == rz.RZ_OK
    out.check_canary()
    return out.result()


def gpu_f32(rz, img, OH, OW, mode, src_pitch=None, src_off=0, dst_pad=0, dst_off=0, tile=None):
    if img.ndim == 2:
        img = img[:, :, None]
    H, W, C = img.shape
    src, _keep = device_image(img, src_pitch, src_off)
    out = Canvas(OH, OW, C, torch.float32, dst_pad, dst_off)
    with rz.resize_plan_create(H, W, OH, OW, mode) as plan:
        if tile:
            rz.resize_plan_set_tile(plan, rz.KIND_F32, *tile)
        rz.resize_f32(plan, src, out.view)
        torch.cuda.synchronize()
        assert rz.resize_plan_status(plan) == rz.RZ_OK
    out.check_canary()
    return out.result()


def check_u8(rz, img, OH, OW, mode, **kw):
    got = gpu_u8(rz, img, OH, OW, mode, **kw)
    want = (oracle.linear_u8 if mode == rz.RZ_LINEAR else oracle.nearest_u8)(img, OH, OW)
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        raise AssertionError(f"{len(bad)} u8 mismatches, first at {bad[0].tolist()}: "
                             f"gpu {got[tuple(bad[0])]} oracle {want[tuple(bad[0])]}")


def check_f32(rz, img, OH, OW, mode, **kw):
    got = gpu_f32(rz, img, OH, OW, mode, **kw)
    if mode == rz.RZ_LINEAR:
        err = max_abs(got, oracle.linear_f32(img, OH, OW))
        assert err <= F32_TOL, err
        return err
    np.testing.assert_array_equal(got, oracle.nearest_f32(img, OH, OW))
    return 0.0


# ------------------------------------------------------------------ the five workloads, full size

@pytest.mark.parametrize("C", [1, 3, 4])
@pytest.mark.parametrize("geom", [(24, 48, 16, 32), (33, 45, 22, 30), (9, 3, 6, 2), (150, 603, 100, 402),
                                  (3, 1563, 2, 1042)])
def test_exact_three_halves_downscale(rz, C, geom):
    # the exact 3:2 kernel (lane words for three and four channels): whole
    # eight-pixel groups, ragged row ends and rows of the tail alone, every
    # channel count; 4-byte aligned layouts take the kernel, an odd start the
    # generic one
    H, W, OH, OW = geom
    img = synth.random_u8((H, W, C), seed=H + W + C)
    sp = W * C + (-W * C) % 4
    dp = (-OW * C) % 4
    for kw in ({"src_pitch": sp, "dst_pad": dp}, {"src_pitch": sp + 8, "dst_pad": dp + 8},
               {"src_off": 1, "dst_off": 3}):
        check_u8(rz, img, OH, OW, rz.RZ_LINEAR, **kw)


def test_tiny_gray_64x48(rz):
    img = synth.tiny_gray()
    check_u8(rz, img, 96, 128, rz.RZ_LINEAR)
    check_u8(rz, img, 24, 32, rz.RZ_NEAREST)


def test_smooth_rgb_1080p(rz):
    img = synth.smooth_rgb(1920, 1080, 2)
    check_u8(rz, img, 540, 960, rz.RZ_LINEAR)
    check_u8(rz, img, 720, 1280, rz.RZ_LINEAR)


def test_smooth_rgb_4k(rz):
    img4k = synth.smooth_rgb(3840, 2160, 3)
    check_u8(rz, img4k, 1080, 1920, rz.RZ_LINEAR)
    check_u8(rz, img4k, 1080, 1920, rz.RZ_NEAREST)
    img1080 = synth.smooth_rgb(1920, 1080, 2)
    check_u8(rz, img1080, 2160, 3840, rz.RZ_LINEAR)


def test_batch_normalize_nchw(rz):
    frames = synth.frames_rgb()                       # (64, 720, 1280, 3)
    src = torch.from_numpy(frames).cuda()
    dst = torch.full((64, 3, 224, 224), -7.0, dtype=torch.float32, device="cuda")
    with rz.resize_plan_create(720, 1280, 224, 224, rz.RZ_LINEAR) as plan:
        rz.resize_fused(plan, src, dst, rz.make_epilogue(rz.RZ_EPI_NORMALIZE_NCHW, mean=synth.NORM_MEAN,
                                                         std=synth.NORM_STD))
        torch.cuda.synchronize()
        assert rz.resize_plan_status(plan) == rz.RZ_OK
    got = dst.cpu().numpy()
    worst = 0.0
    for n in range(64):
        want = oracle.linear_u8_normalize(frames[n], 224, 224, synth.NORM_MEAN, synth.NORM_STD)
        worst = max(worst, max_abs(got[n], want))
    assert worst <= F32_TOL, worst


def test_float_gray_8192_filter3x3(rz):
    img = synth.float_gray()                          # 8192 x 8192 f32
    w = synth.filter_weights()
    OH = OW = int(8192 * 0.73)
    assert OH == 5980
    src = torch.from_numpy(img).cuda()
    dst = torch.empty((OH, OW), dtype=torch.float32, device="cuda")
    with rz.resize_plan_create(8192, 8192, OH, OW, rz.RZ_LINEAR) as plan:
        rz.resize_fused(plan, src, dst, rz.make_epilogue(rz.RZ_EPI_FILTER3X3, w3x3=w))
        torch.cuda.synchronize()
        assert rz.resize_plan_status(plan) == rz.RZ_OK
    want = oracle.linear_f32_filter3x3(img, OH, OW, w)
    err = max_abs(dst.cpu().numpy(), want)
    assert err <= F32_TOL, err


def test_float_gray_8192_plain_bilinear(rz):
    img = synth.float_gray()
    check_f32(rz, img, 5980, 5980, rz.RZ_LINEAR)


# ------------------------------------------------------------------ seeded sweeps

def sweep_cases(seed, n):
    rng = np.random.default_rng(seed)
    for _ in range(n):
        H, W = int(rng.integers(1, 68)), int(rng.integers(1, 68))
        OH, OW = int(rng.integers(1, 68)), int(rng.integers(1, 68))
        C = int(rng.choice([1, 3, 4]))
        pad = int(rng.choice([0, 0, 1, 3, 16, 29]))
        off = int(rng.choice([0, 0, 1, 5, 16]))
        yield H, W, OH, OW, C, pad, off


@pytest.mark.parametrize("seed", range(4))
def test_sweep_u8(rz, seed):
    for (H, W, OH, OW, C, pad, off) in sweep_cases(100 + seed, 40):
        img = synth.random_u8((H, W, C), seed=H * 1000 + W)
        for mode in (rz.RZ_LINEAR, rz.RZ_NEAREST):
            check_u8(rz, img, OH, OW, mode, src_pitch=W * C + pad, src_off=off, dst_pad=pad, dst_off=off)


@pytest.mark.parametrize("seed", range(2))
def test_sweep_u8_staged_tiles(rz, seed):
    # the staged-tile kernel forced on every geometry (the default takes
    # direct loads or streaming)
    for (H, W, OH, OW, C, pad, off) in sweep_cases(800 + seed, 40):
        img = synth.random_u8((H, W, C), seed=H * 1000 + W + 9)
        for mode in (rz.RZ_LINEAR, rz.RZ_NEAREST):
            check_u8(rz, img, OH, OW, mode, src_pitch=W * C + pad, src_off=off, dst_pad=pad, dst_off=off,
                     opts=[(rz.RZ_OPT_U8_KERNEL, 1)])


@pytest.mark.parametrize("seed", range(2))
def test_sweep_u8_direct(rz, seed):
    # direct loads forced on every geometry, upscales too
    for (H, W, OH, OW, C, pad, off) in sweep_cases(900 + seed, 40):
        img = synth.random_u8((H, W, C), seed=H * 1000 + W + 11)
        for mode in (rz.RZ_LINEAR, rz.RZ_NEAREST):
            check_u8(rz, img, OH, OW, mode, src_pitch=W * C + pad, src_off=off, dst_pad=pad, dst_off=off,
                     opts=[(rz.RZ_OPT_U8_KERNEL, 3)])


@pytest.mark.parametrize("seed", range(3))
def test_sweep_u8_streaming(rz, seed):
    # the row-separable streaming form forced on every geometry (downscales
    # too), with odd pitches and unaligned pointers
    for (H, W, OH, OW, C, pad, off) in sweep_cases(700 + seed, 40):
        img = synth.random_u8((H, W, C), seed=H * 1000 + W + 7)
        check_u8(rz, img, OH, OW, rz.RZ_LINEAR, src_pitch=W * C + pad, src_off=off, dst_pad=pad, dst_off=off,
                 opts=[(rz.RZ_OPT_U8_KERNEL, 2)])


_STREAM_GEOMS = [(1080, 1920, 3, 2160, 3840), (300, 410, 3, 611, 797), (97, 130, 4, 260, 333),
                 (64, 75, 1, 190, 201), (500, 700, 3, 333, 401), (33, 2000, 1, 70, 4100)]
_stream_want = {}


def stream_case(rz, geom):
    H, W, C, OH, OW = geom
    if geom not in _stream_want:
        img = synth.smooth_rgb(W, H, 2) if C == 3 and W >= 1920 else synth.random_u8((H, W, C), seed=H + W + C)
        _stream_want[geom] = (img, oracle.linear_u8(img, OH, OW))
    return _stream_want[geom]


@pytest.mark.parametrize("ring", [2, 3, 5, 0])
@pytest.mark.parametrize("ctas", [1, 0, "per_unit"])
def test_u8_stream_ring_and_grid_do_not_change_results(rz, ring, ctas):
    # rings of two or three rows wrap every few rows and one CTA per SM makes
    # each CTA walk many units; "per_unit" launches one CTA per unit
    opts = [(rz.RZ_OPT_U8_KERNEL, 2), (rz.RZ_OPT_RING_ROWS, ring)]
    if ctas == "per_unit":
        opts += [(rz.RZ_OPT_GRID_MODE, 1), (rz.RZ_OPT_PDL, 0)]
    else:
        opts += [(rz.RZ_OPT_CTAS_PER_SM, ctas)]
    for geom in _STREAM_GEOMS:
        img, want = stream_case(rz, geom)
        got = gpu_u8(rz, img, geom[3], geom[4], rz.RZ_LINEAR, opts=opts)
        np.testing.assert_array_equal(got, want, err_msg=str(geom))


@pytest.mark.parametrize("tile", [(1, 32), (7, 64), (40, 1024), (3, 100), (2160, 96), (16, 1)])
def test_u8_stream_unit_shapes(rz, tile):
    for geom in _STREAM_GEOMS[:3]:
        img, want = stream_case(rz, geom)
        got = gpu_u8(rz, img, geom[3], geom[4], rz.RZ_LINEAR, tile=tile, opts=[(rz.RZ_OPT_U8_KERNEL, 2)])
        np.testing.assert_array_equal(got, want, err_msg=str((geom, tile)))


@pytest.mark.parametrize("rows", [1, 2, 3, 8, 31, 2160])
def test_u8_direct_rows_per_thread(rz, rows):
    # the row-walking direct kernel on upscales: any rows per thread (the
    # tile override's row count), ragged segments and odd layouts
    for geom in _STREAM_GEOMS[:4]:
        img, want = stream_case(rz, geom)
        got = gpu_u8(rz, img, geom[3], geom[4], rz.RZ_LINEAR, tile=(rows, 64), opts=[(rz.RZ_OPT_U8_KERNEL, 3)])
        np.testing.assert_array_equal(got, want, err_msg=str((geom, rows)))
    img, want = stream_case(rz, _STREAM_GEOMS[1])
    H, W, C = img.shape
    got = gpu_u8(rz, img, 611, 797, rz.RZ_LINEAR, src_pitch=W * C + 3, src_off=1, dst_pad=5, dst_off=2,
                 tile=(rows, 64), opts=[(rz.RZ_OPT_U8_KERNEL, 3)])
    np.testing.assert_array_equal(got, want)


def test_u8_stream_and_staged_tiles_agree(rz):
    # both uint8 kernels on the same upscale: identical bytes
    img, want = stream_case(rz, _STREAM_GEOMS[1])
    a = gpu_u8(rz, img, 611, 797, rz.RZ_LINEAR, opts=[(rz.RZ_OPT_U8_KERNEL, 1)])
    b = gpu_u8(rz, img, 611, 797, rz.RZ_LINEAR, opts=[(rz.RZ_OPT_U8_KERNEL, 2)])
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(a, want)


@pytest.mark.parametrize("seed", range(3))
def test_sweep_f32(rz, seed):
    for (H, W, OH, OW, C, pad, off) in sweep_cases(200 + seed, 30):
        img = synth.random_f32((H, W, C), seed=H * 1000 + W)
        for mode in (rz.RZ_LINEAR, rz.RZ_NEAREST):
            check_f32(rz, img, OH, OW, mode, src_pitch=W * C + pad, src_off=off, dst_pad=pad, dst_off=off)


@pytest.mark.parametrize("seed", range(3))
def test_sweep_fused_filter(rz, seed):
    rng = np.random.default_rng(300 + seed)
    for _ in range(12):
        H, W, OH, OW = (int(v) for v in rng.integers(1, 90, size=4))
        C = int(rng.choice([1, 3, 4]))
        N = int(rng.integers(1, 4))
        img = synth.random_f32((N, H, W, C), seed=H * 7 + W)
        w = (rng.random(9) - 0.3).astype(np.float32)
        src = torch.from_numpy(img).cuda()
        dst = torch.empty((N, OH, OW, C), dtype=torch.float32, device="cuda")
        with rz.resize_plan_create(H, W, OH, OW, rz.RZ_LINEAR) as plan:
            rz.resize_fused(plan, src, dst, rz.make_epilogue(rz.RZ_EPI_FILTER3X3, w3x3=w))
            torch.cuda.synchronize()
        got = dst.cpu().numpy()
        for n in range(N):
            for c in range(C):
                want = oracle.filter3x3(oracle.linear_f32(img[n][:, :, c:c + 1].copy(), OH, OW), w)
                err = max_abs(got[n, :, :, c], want)
                assert err <= F32_TOL * np.abs(w).sum(), (H, W, OH, OW, C, n, c, err)


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("kernel", [0, 1])
def test_sweep_fused_normalize(rz, seed, kernel):
    # kernel 0: automatic (direct loads); 1: staged tiles
    rng = np.random.default_rng(400 + seed)
    for _ in range(12):
        H, W, OH, OW = (int(v) for v in rng.integers(1, 90, size=4))
        C = int(rng.choice([1, 3, 4]))
        N = int(rng.integers(1, 5))
        frames = synth.random_u8((N, H, W, C), seed=H * 13 + W)
        mean = rng.random(4) * 0.8
        std = 0.1 + rng.random(4) * 0.5
        src = torch.from_numpy(frames).cuda()
        dst = torch.empty((N, C, OH, OW), dtype=torch.float32, device="cuda")
        with rz.resize_plan_create(H, W, OH, OW, rz.RZ_LINEAR) as plan:
            rz.resize_plan_set_option(plan, rz.RZ_OPT_U8_KERNEL, kernel)
            e = rz.make_epilogue(rz.RZ_EPI_NORMALIZE_NCHW, mean=np.float32(mean), std=np.float32(std))
            rz.resize_fused(plan, src, dst, e)
            torch.cuda.synchronize()
        got = dst.cpu().numpy()
        for n in range(N):
            want = oracle.linear_u8_normalize(frames[n], OH, OW, np.float32(mean).astype(np.float64),
                                              np.float32(std).astype(np.float64))
            err = max_abs(got[n], want)
            assert err <= F32_TOL, (H, W, OH, OW, C, err)


# ------------------------------------------------------------------ edge cases

@pytest.mark.parametrize("geom", [(1, 1, 1, 1), (1, 1, 7, 5), (7, 5, 1, 1), (1, 64, 3, 1), (64, 1, 1, 3),
                                  (2, 3, 2, 4096), (2, 4096, 3, 2), (4096, 2, 2, 3), (3, 2, 4096, 2),
                                  (2, 65536, 2, 5), (1, 65536, 1, 65536), (9, 9, 9, 9)])
def test_degenerate_and_extreme_geometries(rz, geom):
    H, W, OH, OW = geom
    for C in (1, 3):
        img = synth.random_u8((H, W, C), seed=OH + OW)
        check_u8(rz, img, OH, OW, rz.RZ_LINEAR)
        check_u8(rz, img, OH, OW, rz.RZ_NEAREST)
    check_f32(rz, synth.random_f32((H, W, 1), seed=3), OH, OW, rz.RZ_LINEAR)


def test_identity_is_a_copy(rz):
    img = synth.random_u8((33, 47, 3), seed=9)
    np.testing.assert_array_equal(gpu_u8(rz, img, 33, 47, rz.RZ_LINEAR), img)
    f = synth.random_f32((33, 47, 4), seed=9)
    np.testing.assert_array_equal(gpu_f32(rz, f, 33, 47, rz.RZ_LINEAR), f)


def test_empty_output_is_a_no_op(rz):
    img = synth.random_u8((8, 8, 3), seed=1)
    src, _k = device_image(img)
    with rz.resize_plan_create(8, 8, 0, 5, rz.RZ_LINEAR) as plan:
        dst = torch.empty((0, 5, 3), dtype=torch.uint8, device="cuda")
        rz.resize_u8(plan, src, dst)
    torch.cuda.synchronize()


@pytest.mark.parametrize("tile", [(1, 1), (1, 16), (3, 7), (5, 64), (16, 128), (64, 4096), (2, 33)])
def test_tile_shapes_do_not_change_results(rz, tile):
    img = synth.random_u8((97, 131, 3), seed=77)
    for (OH, OW) in [(41, 59), (200, 263), (97, 131)]:
        check_u8(rz, img, OH, OW, rz.RZ_LINEAR, tile=tile)
        check_u8(rz, img, OH, OW, rz.RZ_NEAREST, tile=tile)
    f = synth.random_f32((97, 131, 1), seed=78)
    check_f32(rz, f, 53, 211, rz.RZ_LINEAR, tile=tile)


def test_filter_tile_shapes_do_not_change_results(rz):
    img = synth.random_f32((150, 170), seed=79)
    w = synth.filter_weights()
    want = oracle.linear_f32_filter3x3(img, 109, 124, w)
    src = torch.from_numpy(img).cuda()
    for tile in [(1, 1), (2, 3), (7, 16), (32, 128), (40, 124), (13, 200)]:
        dst = torch.empty((109, 124), dtype=torch.float32, device="cuda")
        with rz.resize_plan_create(150, 170, 109, 124, rz.RZ_LINEAR) as plan:
            rz.resize_plan_set_tile(plan, rz.KIND_FILTER3X3, *tile)
            rz.resize_fused(plan, src, dst, rz.make_epilogue(rz.RZ_EPI_FILTER3X3, w3x3=w))
            torch.cuda.synchronize()
        assert max_abs(dst.cpu().numpy(), want) <= F32_TOL, tile


def run_filter(rz, img, OH, OW, w, opts=(), tile=None, src_pitch=None, src_off=0):
    H, W, C = img.shape
    src, _keep = device_image(img, src_pitch, src_off)
    out = Canvas(OH, OW, C, torch.float32)
    with rz.resize_plan_create(H, W, OH, OW, rz.RZ_LINEAR) as plan:
        for k, v in opts:
            rz.resize_plan_set_option(plan, k, v)
        if tile:
            rz.resize_plan_set_tile(plan, rz.KIND_FILTER3X3, *tile)
        rz.resize_fused(plan, src, out.view, rz.make_epilogue(rz.RZ_EPI_FILTER3X3, w3x3=w))
        torch.cuda.synchronize()
        assert rz.resize_plan_status(plan) == rz.RZ_OK
    out.check_canary()
    return out.result()


def want_filter(img, OH, OW, w):
    return np.stack([oracle.filter3x3(oracle.linear_f32(img[:, :, c:c + 1].copy(), OH, OW), w)
                     for c in range(img.shape[2])], axis=-1)


@pytest.mark.parametrize("ring", [2, 3, 5, 0])
@pytest.mark.parametrize("ctas", [1, 0, "per_unit"])
def test_filter_ring_and_grid_do_not_change_results(rz, ring, ctas):
    # rings of two or three rows wrap every few rows and one CTA per SM makes
    # each CTA walk many units, carrying ring slots and barrier phases across
    # them; "per_unit" launches one CTA per unit
    w = synth.filter_weights()
    opts = [(rz.RZ_OPT_RING_ROWS, ring)]
    if ctas == "per_unit":
        opts += [(rz.RZ_OPT_GRID_MODE, 1), (rz.RZ_OPT_PDL, 0)]
    else:
        opts += [(rz.RZ_OPT_CTAS_PER_SM, ctas)]
    for (H, W, C, OH, OW, tile) in [(300, 410, 1, 211, 173, None), (300, 410, 1, 211, 173, (7, 30)),
                                    (97, 130, 3, 260, 333, (19, 64)), (640, 480, 4, 150, 170, (5, 240)),
                                    (1500, 1200, 1, 1099, 877, None)]:
        img = synth.random_f32((H, W, C), seed=H + W + C)
        got = run_filter(rz, img, OH, OW, w, opts, tile)
        err = max_abs(got, want_filter(img, OH, OW, w))
        assert err <= F32_TOL * np.abs(w).sum(), (H, W, C, OH, OW, tile, err)


def test_filter_unaligned_source_rows(rz):
    # a source that is not 16-byte aligned (start or pitch) is copied by the
    # producer warp's lanes instead of bulk copies
    w = synth.filter_weights()
    for (H, W, C, OH, OW, pitch, off) in [(120, 97, 1, 80, 61, 101, 1), (64, 75, 3, 99, 140, 75 * 3, 3),
                                          (50, 33, 4, 40, 29, 33 * 4 + 2, 2)]:
        img = synth.random_f32((H, W, C), seed=H * 3 + W)
        for ring in (2, 0):
            got = run_filter(rz, img, OH, OW, w, [(rz.RZ_OPT_RING_ROWS, ring), (rz.RZ_OPT_CTAS_PER_SM, 1)],
                             src_pitch=pitch, src_off=off)
            err = max_abs(got, want_filter(img, OH, OW, w))
            assert err <= F32_TOL * np.abs(w).sum(), (H, W, C, OH, OW, ring, err)


def batch_canvas(N, H, W, C, dtype, pitch, bstride, off=0):
    """An (N, H, W, C) view with the given row pitch, batch stride and start offset (elements)."""
    flat = torch.zeros(off + (N - 1) * bstride + (H - 1) * pitch + W * C + 64, dtype=dtype, device="cuda")
    return torch.as_strided(flat, (N, H, W, C), (bstride, pitch, C, 1), off), flat


@pytest.mark.parametrize("kind", ["u8", "f32"])
@pytest.mark.parametrize("layout", ["packed", "padded", "unaligned"])
def test_batch_matches_per_image_oracle(rz, kind, layout):
    # one launch over N images equals N single-image resizes; padding between
    # rows and images, and unaligned strides (plain copies), change nothing
    N, H, W, C, OH, OW = 3, 270, 480, 3, 181, 317
    rng = np.random.default_rng(91)
    if kind == "u8":
        imgs = rng.integers(0, 256, size=(N, H, W, C), dtype=np.uint8)
        dt, fn = torch.uint8, rz.resize_u8_batch
    else:
        imgs = (rng.random((N, H, W, C)) * 255).astype(np.float32)
        dt, fn = torch.float32, rz.resize_f32_batch
    pad, opad, off = {"packed": (0, 0, 0), "padded": (16, 32, 0), "unaligned": (5, 7, 3)}[layout]
    if kind == "f32" and layout == "unaligned":
        pad, opad, off = 1, 3, 1
    sp = W * C + pad
    src, _ks = batch_canvas(N, H, W, C, dt, sp, H * sp + opad, off)
    src.copy_(torch.from_numpy(imgs).cuda())
    dp = OW * C + pad
    dst, dflat = batch_canvas(N, OH, OW, C, dt, dp, OH * dp + opad, off)
    for mode in (rz.RZ_LINEAR, rz.RZ_NEAREST):
        dflat.fill_(0)
        with rz.resize_plan_create(H, W, OH, OW, mode) as plan:
            fn(plan, src, dst)
            torch.cuda.synchronize()
            assert rz.resize_plan_status(plan) == rz.RZ_OK
        got = dst.cpu().numpy()
        for n in range(N):
            if kind == "u8":
                want = (oracle.linear_u8 if mode == rz.RZ_LINEAR else oracle.nearest_u8)(imgs[n], OH, OW)
                np.testing.assert_array_equal(got[n], want, err_msg=f"image {n}")
            else:
                want = (oracle.linear_f32 if mode == rz.RZ_LINEAR else oracle.nearest_f32)(imgs[n], OH, OW)
                assert max_abs(got[n], want) <= F32_TOL, n


def test_batch_of_4k_frames_is_bit_exact(rz):
    # the exact 2x path over a batch of frames, as the bench runs it
    N = 3
    frames = np.stack([synth.smooth_rgb(3840, 2160, 10 + n) for n in range(N)])
    src = torch.from_numpy(frames).cuda()
    dst = torch.empty((N, 1080, 1920, 3), dtype=torch.uint8, device="cuda")
    with rz.resize_plan_create(2160, 3840, 1080, 1920, rz.RZ_LINEAR) as plan:
        rz.resize_u8_batch(plan, src, dst)
        torch.cuda.synchronize()
    got = dst.cpu().numpy()
    for n in range(N):
        np.testing.assert_array_equal(got[n], oracle.linear_u8(frames[n], 1080, 1920))


def test_batch_argument_checks(rz):
    with rz.resize_plan_create(8, 8, 4, 4, rz.RZ_LINEAR) as plan:
        lib = rz._native.load()
        src = torch.zeros((2, 8, 8, 3), dtype=torch.uint8, device="cuda")
        dst = torch.zeros((2, 4, 4, 3), dtype=torch.uint8, device="cuda")
        s, d = src.data_ptr(), dst.data_ptr()
        # batch stride smaller than an image
        assert lib.resize_u8_batch(plan.handle, s, 24, 100, d, 12, 48, 2, 8, 8, 3, 4, 4, 1, None) == rz.RZ_ERR_ARG
        assert lib.resize_u8_batch(plan.handle, s, 24, 192, d, 12, 40, 2, 8, 8, 3, 4, 4, 1, None) == rz.RZ_ERR_ARG
        # negative batch; zero is a no-op
        assert lib.resize_u8_batch(plan.handle, s, 24, 192, d, 12, 48, -1, 8, 8, 3, 4, 4, 1, None) == rz.RZ_ERR_ARG
        assert lib.resize_u8_batch(plan.handle, s, 24, 192, d, 12, 48, 0, 8, 8, 3, 4, 4, 1, None) == rz.RZ_OK
        # a destination image overlapping a source image
        assert lib.resize_u8_batch(plan.handle, s, 24, 192, s + 192, 12, 48, 2, 8, 8, 3, 4, 4, 1,
                                   None) == rz.RZ_ERR_ARG
        # float32 batch strides must be multiples of 4
        f = torch.zeros((2 * 8 * 8 * 3 + 8,), dtype=torch.float32, device="cuda")
        g = torch.zeros((2 * 4 * 4 * 3 + 8,), dtype=torch.float32, device="cuda")
        assert lib.resize_f32_batch(plan.handle, f.data_ptr(), 96, 770, g.data_ptr(), 48, 192, 2, 8, 8, 3, 4, 4, 1,
                                    None) == rz.RZ_ERR_ARG
        torch.cuda.synchronize()
        assert not dst.any()


def test_non_default_stream(rz):
    img = synth.smooth_rgb(1920, 1080, 2)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        got = gpu_u8(rz, img, 540, 960, rz.RZ_LINEAR, stream=s)
    np.testing.assert_array_equal(got, oracle.linear_u8(img, 540, 960))


def test_host_buffers_entry_point(rz):
    img = synth.smooth_rgb(1920, 1080, 2)
    hsrc = torch.from_numpy(np.ascontiguousarray(img)).pin_memory()
    hdst = torch.empty((540, 960, 3), dtype=torch.uint8).pin_memory()
    dsrc = torch.empty((1080, 1920, 3), dtype=torch.uint8, device="cuda")
    ddst = torch.empty((540, 960, 3), dtype=torch.uint8, device="cuda")
    with rz.resize_plan_create(1080, 1920, 540, 960, rz.RZ_LINEAR) as plan:
        rz.resize_u8_host(plan, hsrc, hdst, dsrc, ddst)
        torch.cuda.synchronize()
    np.testing.assert_array_equal(hdst.numpy(), oracle.linear_u8(img, 540, 960))


def test_invalid_calls_raise(rz):
    img = synth.random_u8((8, 8, 3), seed=1)
    src, _k = device_image(img)
    with rz.resize_plan_create(8, 8, 4, 4, rz.RZ_LINEAR) as plan:
        dst = torch.empty((4, 4, 3), dtype=torch.uint8, device="cuda")
        with pytest.raises(rz.ResizeError):          # wrong geometry
            rz.resize_u8(plan, src, torch.empty((5, 4, 3), dtype=torch.uint8, device="cuda"))
        with pytest.raises(rz.ResizeError):          # wrong mode for this plan
            rz.resize_u8(plan, src, dst, mode=rz.RZ_NEAREST)
        with pytest.raises(rz.ResizeError):          # C = 2
            rz.resize_u8(plan, torch.zeros((8, 8, 2), dtype=torch.uint8, device="cuda"),
                         torch.zeros((4, 4, 2), dtype=torch.uint8, device="cuda"))
        flat = torch.zeros(4096, dtype=torch.uint8, device="cuda")
        a = torch.as_strided(flat, (8, 8, 3), (24, 3, 1), 0)
        b = torch.as_strided(flat, (4, 4, 3), (12, 3, 1), 100)
        with pytest.raises(rz.ResizeError):          # overlapping source and destination
            rz.resize_u8(plan, a, b)
        assert rz.resize_plan_status(plan) == rz.RZ_OK


# ------------------------------------------------------------------ pipeline depth and the exact 2x path

def run_u8_opts(rz, img, OH, OW, mode, opts, tile=None):
    H, W, C = img.shape
    src, _k = device_image(img)
    out = Canvas(OH, OW, C, torch.uint8)
    with rz.resize_plan_create(H, W, OH, OW, mode) as plan:
        for k, v in opts.items():
            rz.resize_plan_set_option(plan, k, v)
        if tile:
            rz.resize_plan_set_tile(plan, rz.KIND_U8, *tile)
        rz.resize_u8(plan, src, out.view)
        torch.cuda.synchronize()
        assert rz.resize_plan_status(plan) == rz.RZ_OK
    out.check_canary()
    return out.result()


@pytest.mark.parametrize("stages", [1, 2, 3, 4])
@pytest.mark.parametrize("ctas", [1, 2, 0, "per_tile"])
def test_ring_depth_and_grid_do_not_change_results(rz, stages, ctas):
    # one or two CTAs per SM make every CTA walk many tiles, so each stage's
    # barrier goes through many phases; "per_tile" launches one CTA per tile
    img = synth.smooth_rgb(1920, 1080, 2)
    # staged tiles everywhere (the options shape that kernel)
    if ctas == "per_tile":
        opts = {rz.RZ_OPT_STAGES: stages, rz.RZ_OPT_GRID_MODE: 1, rz.RZ_OPT_PDL: 0, rz.RZ_OPT_U8_KERNEL: 1}
    else:
        opts = {rz.RZ_OPT_STAGES: stages, rz.RZ_OPT_CTAS_PER_SM: ctas, rz.RZ_OPT_U8_KERNEL: 1}
    for (OH, OW) in [(540, 960), (720, 1280), (2160, 3840)]:
        got = run_u8_opts(rz, img, OH, OW, rz.RZ_LINEAR, opts)
        np.testing.assert_array_equal(got, oracle.linear_u8(img, OH, OW))
    got = run_u8_opts(rz, img, 270, 480, rz.RZ_NEAREST, opts)
    np.testing.assert_array_equal(got, oracle.nearest_u8(img, 270, 480))


@pytest.mark.parametrize("C", [1, 3, 4])
@pytest.mark.parametrize("geom", [(2160, 3840), (48, 64), (2, 2), (6, 34), (1080, 1922), (30, 18)])
def test_exact_2x_path_is_bit_identical_to_generic(rz, C, geom):
    H, W = geom
    img = synth.random_u8((H, W, C), seed=H + W + C)
    direct = run_u8_opts(rz, img, H // 2, W // 2, rz.RZ_LINEAR, {})
    staged = run_u8_opts(rz, img, H // 2, W // 2, rz.RZ_LINEAR, {rz.RZ_OPT_U8_KERNEL: 1})
    slow = run_u8_opts(rz, img, H // 2, W // 2, rz.RZ_LINEAR, {rz.RZ_OPT_GENERIC_ONLY: 1})
    np.testing.assert_array_equal(direct, slow)
    np.testing.assert_array_equal(staged, slow)
    np.testing.assert_array_equal(direct, oracle.linear_u8(img, H // 2, W // 2))


@pytest.mark.parametrize("C", [1, 3, 4])
def test_exact_2x_direct_loads(rz, C):
    # the direct-load kernel: ragged widths (a row's last pixels fewer than a
    # group), a one-pixel output, unaligned layouts (which take the staged
    # kernel) and both paths against the oracle
    for (H, W) in [(2, 2), (2, 18), (6, 34), (30, 46), (64, 64), (200, 1002), (1080, 1926)]:
        img = synth.random_u8((H, W, C), seed=H * 7 + W + C)
        for mode, fn in ((rz.RZ_LINEAR, oracle.linear_u8), (rz.RZ_NEAREST, oracle.nearest_u8)):
            want = fn(img, H // 2, W // 2)
            for pad, off in [(0, 0), (16, 0), (3, 1), (8, 4)]:
                got = gpu_u8(rz, img, H // 2, W // 2, mode, src_pitch=W * C + pad, src_off=off, dst_pad=pad,
                             dst_off=off, opts=[(rz.RZ_OPT_U8_KERNEL, 3)])
                np.testing.assert_array_equal(got, want, err_msg=str((mode, H, W, pad, off)))


@pytest.mark.parametrize("C", [1, 3, 4])
def test_exact_2x_upscale(rz, C):
    # the 1-3 weight kernel: tiny and odd sizes (edge groups take the byte
    # path), unaligned layouts, and agreement with the streaming and staged
    # kernels
    for (H, W) in [(1, 1), (1, 5), (3, 2), (2, 9), (7, 13), (16, 16), (33, 70), (540, 961), (1080, 1920)]:
        img = synth.random_u8((H, W, C), seed=H * 11 + W + C)
        want = oracle.linear_u8(img, 2 * H, 2 * W)
        for pad, off in [(0, 0), (16, 0), (3, 1), (5, 2)]:
            got = gpu_u8(rz, img, 2 * H, 2 * W, rz.RZ_LINEAR, src_pitch=W * C + pad, src_off=off, dst_pad=pad,
                         dst_off=off)
            np.testing.assert_array_equal(got, want, err_msg=str((H, W, pad, off)))
    img = synth.random_u8((97, 130, C), seed=5)
    a = gpu_u8(rz, img, 194, 260, rz.RZ_LINEAR)
    for k in (1, 2):
        np.testing.assert_array_equal(a, gpu_u8(rz, img, 194, 260, rz.RZ_LINEAR, opts=[(rz.RZ_OPT_U8_KERNEL, k)]))


def test_exact_2x_upscale_batch(rz):
    N = 3
    frames = np.stack([synth.random_u8((135, 240, 3), seed=70 + n) for n in range(N)])
    src = torch.from_numpy(frames).cuda()
    dst = torch.empty((N, 270, 480, 3), dtype=torch.uint8, device="cuda")
    with rz.resize_plan_create(135, 240, 270, 480, rz.RZ_LINEAR) as plan:
        rz.resize_u8_batch(plan, src, dst)
        torch.cuda.synchronize()
    got = dst.cpu().numpy()
    for n in range(N):
        np.testing.assert_array_equal(got[n], oracle.linear_u8(frames[n], 270, 480))


def test_exact_2x_direct_batch_and_pdl_chain(rz):
    # a batch through the direct kernel, then a second resize of its output
    # queued right after it (the dependent launch must wait for the first)
    N = 4
    frames = np.stack([synth.random_u8((540, 960, 3), seed=60 + n) for n in range(N)])
    src = torch.from_numpy(frames).cuda()
    mid = torch.empty((N, 270, 480, 3), dtype=torch.uint8, device="cuda")
    out = torch.empty((N, 135, 240, 3), dtype=torch.uint8, device="cuda")
    with rz.resize_plan_create(540, 960, 270, 480, rz.RZ_LINEAR) as p1, \
            rz.resize_plan_create(270, 480, 135, 240, rz.RZ_LINEAR) as p2:
        for _ in range(3):
            rz.resize_u8_batch(p1, src, mid)
            rz.resize_u8_batch(p2, mid, out)
        torch.cuda.synchronize()
    got = out.cpu().numpy()
    for n in range(N):
        np.testing.assert_array_equal(got[n], oracle.linear_u8(oracle.linear_u8(frames[n], 270, 480), 135, 240))


@pytest.mark.parametrize("tile", [(1, 8), (1, 16), (2, 24), (3, 64), (1, 960), (4, 1920)])
def test_exact_2x_path_tiles(rz, tile):
    img = synth.smooth_rgb(3840, 2160, 3)
    got = run_u8_opts(rz, img, 1080, 1920, rz.RZ_LINEAR, {rz.RZ_OPT_STAGES: 2, rz.RZ_OPT_U8_KERNEL: 1}, tile=tile)
    np.testing.assert_array_equal(got, oracle.linear_u8(img, 1080, 1920))


def test_options_reject_bad_values(rz):
    with rz.resize_plan_create(8, 8, 4, 4, rz.RZ_LINEAR) as plan:
        for opt, val in [(rz.RZ_OPT_STAGES, 5), (rz.RZ_OPT_STAGES, -1), (rz.RZ_OPT_GENERIC_ONLY, 2),
                         (rz.RZ_OPT_CTAS_PER_SM, 33), (rz.RZ_OPT_GRID_MODE, 2), (rz.RZ_OPT_PDL, 3),
                         (rz.RZ_OPT_RING_ROWS, 1), (rz.RZ_OPT_RING_ROWS, 129), (rz.RZ_OPT_U8_KERNEL, 4),
                         (rz.RZ_OPT_U8_KERNEL, -1), (rz.RZ_OPT_F32_KERNEL, 2), (rz.RZ_OPT_F32_KERNEL, -1),
                         (99, 0)]:
            with pytest.raises(rz.ResizeError):
                rz.resize_plan_set_option(plan, opt, val)


def test_bounded_wait_reports_timeout(rz):
    # the barrier waits in the staged and streaming kernels give up after a
    # limit and report RZ_ERR_TIMEOUT; here a wait on a barrier nothing
    # completes must end within its limit, report, and leave the context usable
    import time
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rz.resize_wait_selftest(status, 2000)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == rz.RZ_ERR_TIMEOUT
    assert 0.002 <= elapsed < 1.0
    for bad in (0, -5, 1000001):
        with pytest.raises(rz.ResizeError):
            rz.resize_wait_selftest(status, bad)
    img = synth.smooth_rgb(96, 64, 3)
    np.testing.assert_array_equal(gpu_u8(rz, img, 40, 70, rz.RZ_LINEAR), oracle.linear_u8(img, 40, 70))


def test_back_to_back_dependent_resizes(rz):
    # a chain where each resize reads the previous one's output, queued with
    # programmatic dependent launches: every link must see its input complete
    img = synth.smooth_rgb(1920, 1080, 2)
    a = torch.from_numpy(np.ascontiguousarray(img)).cuda()
    b = torch.empty((540, 960, 3), dtype=torch.uint8, device="cuda")
    c = torch.empty((270, 480, 3), dtype=torch.uint8, device="cuda")
    d = torch.empty((540, 960, 3), dtype=torch.uint8, device="cuda")
    p1 = rz.resize_plan_create(1080, 1920, 540, 960, rz.RZ_LINEAR)
    p2 = rz.resize_plan_create(540, 960, 270, 480, rz.RZ_LINEAR)
    p3 = rz.resize_plan_create(270, 480, 540, 960, rz.RZ_LINEAR)
    torch.cuda.synchronize()
    for _ in range(3):
        rz.resize_u8(p1, a, b)
        rz.resize_u8(p2, b, c)
        rz.resize_u8(p3, c, d)
    torch.cuda.synchronize()
    e1 = oracle.linear_u8(img, 540, 960)
    e2 = oracle.linear_u8(e1, 270, 480)
    np.testing.assert_array_equal(d.cpu().numpy(), oracle.linear_u8(e2, 540, 960))
    for p in (p1, p2, p3):
        assert rz.resize_plan_status(p) == rz.RZ_OK
        p.destroy()


def test_one_plan_on_two_streams_at_once(rz):
    # the plan's tables are read-only on the device: calls on different
    # streams may share a plan and run concurrently
    img_a = synth.smooth_rgb(1920, 1080, 2)
    img_b = synth.random_u8((1080, 1920, 3), seed=8)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    a = torch.from_numpy(img_a).cuda()
    b = torch.from_numpy(img_b).cuda()
    oa = torch.zeros((720, 1280, 3), dtype=torch.uint8, device="cuda")
    ob = torch.zeros((720, 1280, 3), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    with rz.resize_plan_create(1080, 1920, 720, 1280, rz.RZ_LINEAR) as plan:
        for _ in range(20):
            rz.resize_u8(plan, a, oa, stream=sa)
            rz.resize_u8(plan, b, ob, stream=sb)
        torch.cuda.synchronize()
        assert rz.resize_plan_status(plan) == rz.RZ_OK
    np.testing.assert_array_equal(oa.cpu().numpy(), oracle.linear_u8(img_a, 720, 1280))
    np.testing.assert_array_equal(ob.cpu().numpy(), oracle.linear_u8(img_b, 720, 1280))


def test_plans_on_many_streams(rz):
    # independent plans of different geometries on their own streams
    img = synth.random_u8((200, 300, 3), seed=12)
    src = torch.from_numpy(img).cuda()
    geoms = [(100, 150), (400, 600), (133, 77), (200, 300), (37, 512)]
    streams = [torch.cuda.Stream() for _ in geoms]
    outs = [torch.zeros((h, w, 3), dtype=torch.uint8, device="cuda") for h, w in geoms]
    plans = [rz.resize_plan_create(200, 300, h, w, rz.RZ_LINEAR) for h, w in geoms]
    torch.cuda.synchronize()
    for _ in range(5):
        for p, o, s in zip(plans, outs, streams):
            rz.resize_u8(p, src, o, stream=s)
    torch.cuda.synchronize()
    for (h, w), o, p in zip(geoms, outs, plans):
        np.testing.assert_array_equal(o.cpu().numpy(), oracle.linear_u8(img, h, w))
        p.destroy()


@pytest.mark.parametrize("C", [1, 3, 4])
@pytest.mark.parametrize("kernel", [0, 1])
def test_f32_streaming_and_staged_kernels(rz, C, kernel):
    # the plain float32 bilinear resize on the streaming kernel (K = 1
    # filter, the default) and on staged tiles, over up- and downscales,
    # ragged strips, padded and unaligned layouts, batches
    for (H, W, OH, OW) in [(150, 170, 333, 201), (64, 700, 97, 1500), (300, 40, 130, 19), (1, 9, 5, 4),
                           (512, 512, 373, 600)]:
        img = synth.random_f32((H, W, C), seed=H + C)
        for pitch, off in [(None, 0), (W * C + 3, 1)]:
            src, _keep = device_image(img, pitch, off)
            out = Canvas(OH, OW, C, torch.float32, 2)
            with rz.resize_plan_create(H, W, OH, OW, rz.RZ_LINEAR) as plan:
                rz.resize_plan_set_option(plan, rz.RZ_OPT_F32_KERNEL, kernel)
                rz.resize_f32(plan, src, out.view)
                torch.cuda.synchronize()
                assert rz.resize_plan_status(plan) == rz.RZ_OK
            out.check_canary()
            assert max_abs(out.result(), oracle.linear_f32(img, OH, OW)) <= F32_TOL
    frames = np.stack([synth.random_f32((40, 60, C), seed=n) for n in range(5)])
    dst = torch.zeros((5, 70, 33, C), dtype=torch.float32, device="cuda")
    with rz.resize_plan_create(40, 60, 70, 33, rz.RZ_LINEAR, border=1) as plan:
        rz.resize_plan_set_option(plan, rz.RZ_OPT_F32_KERNEL, kernel)
        rz.resize_f32_batch(plan, torch.from_numpy(frames).cuda(), dst)
        torch.cuda.synchronize()
    for n in range(5):
        assert max_abs(dst[n].cpu().numpy(), oracle.linear_f32(frames[n], 70, 33, 1)) <= F32_TOL


@pytest.mark.parametrize("C", [1, 3, 4])
def test_exact_3_to_2_downscale(rz, C):
    # the exact 3:2 kernel (eight outputs by two rows per thread), its ragged
    # row ends, layouts that send it to the generic kernel, and batches
    for (H, W) in [(3, 3), (3, 12), (9, 24), (30, 45), (33, 57), (48, 96), (1080, 1920)]:
        img = synth.random_u8((H, W, C), seed=H + W + C)
        OH, OW = 2 * H // 3, 2 * W // 3
        want = oracle.linear_u8(img, OH, OW)
        np.testing.assert_array_equal(gpu_u8(rz, img, OH, OW, rz.RZ_LINEAR), want)
        np.testing.assert_array_equal(gpu_u8(rz, img, OH, OW, rz.RZ_LINEAR, src_pitch=W * C + 1, src_off=3,
                                             dst_pad=1), want)
        np.testing.assert_array_equal(gpu_u8(rz, img, OH, OW, rz.RZ_LINEAR, opts=[(rz.RZ_OPT_GENERIC_ONLY, 1)]),
                                      want)
    frames = np.stack([synth.random_u8((45, 60, C), seed=n) for n in range(7)])
    dst = torch.zeros((7, 30, 40, C), dtype=torch.uint8, device="cuda")
    with rz.resize_plan_create(45, 60, 30, 40, rz.RZ_LINEAR) as plan:
        rz.resize_u8_batch(plan, torch.from_numpy(frames).cuda(), dst)
        torch.cuda.synchronize()
    for n in range(7):
        np.testing.assert_array_equal(dst[n].cpu().numpy(), oracle.linear_u8(frames[n], 30, 40))
