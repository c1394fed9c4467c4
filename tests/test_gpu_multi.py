"""Parity of resize_u8_multi (many geometries in one launch) with the oracle.

Every job's output must equal the oracle's resize of its own image bit for
bit (and so resize_u8 with a plan of that geometry), whatever the mix: up-
and downscales, identity, one-pixel and empty outputs, padded pitches,
unaligned starts, both modes, every channel count; invalid jobs are skipped
and flagged while the others still run.  Exact 2x bilinear jobs take their
own forms inside the launch (the 2 x 2 mean; the 9-3-3-1 upscale on pixel
lanes), so their ragged groups, one-pixel images, wide rows, row runs that
end inside a unit, and the layouts that send them back to the generic form
are checked as well.
"""
import numpy as np
import pytest

import oracle
from bilinear_image_resize_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rz():
    import __graft_entry__
    __graft_entry__.build()
    import bilinear_image_resize_gb300 as m
    torch.cuda.set_device(0)
    return m


def run_jobs(rz, geoms, C, mode, seed=0, pad=0, off=0):
    rng = np.random.default_rng(seed)
    imgs, srcs, dsts, keep = [], [], [], []
    for (H, W, OH, OW) in geoms:
        img = rng.integers(0, 256, (H, W, C), dtype=np.uint8)
        flat = torch.zeros(off + H * (W * C + pad) + 8, dtype=torch.uint8, device="cuda")
        s = torch.as_strided(flat, (H, W, C), (W * C + pad, C, 1), off)
        s.copy_(torch.from_numpy(img).cuda())
        d = torch.full((OH, OW, C), 0xA5, dtype=torch.uint8, device="cuda")
        imgs.append(img); srcs.append(s); dsts.append(d); keep.append(flat)
    jobs, CC = rz.make_jobs(srcs, dsts)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rz.resize_u8_multi(jobs, len(geoms), C, mode, status)
    torch.cuda.synchronize()
    return imgs, [d.cpu().numpy() for d in dsts], int(status.item())


def want(img, OH, OW, mode):
    return oracle.linear_u8(img, OH, OW) if mode == 1 else oracle.nearest_u8(img, OH, OW)


MIX = [(48, 64, 96, 128), (37, 53, 100, 131), (90, 120, 37, 50), (33, 47, 33, 47), (1, 1, 1, 1), (1, 5, 4, 9),
       (5, 1, 9, 3), (64, 64, 32, 32), (20, 300, 7, 11), (7, 3, 0, 5), (3, 7, 4, 0), (200, 150, 61, 1030),
       # rows cut into 32-quad slices: whole, ragged last slice, ragged last quad
       (40, 320, 25, 640), (30, 200, 71, 530), (50, 101, 33, 371)]


@pytest.mark.parametrize("C", [1, 3, 4])
@pytest.mark.parametrize("mode", [0, 1])
def test_multi_mixed_geometries(rz, C, mode):
    imgs, got, st = run_jobs(rz, MIX, C, mode, seed=C + 10 * mode)
    assert st == rz.RZ_OK
    for img, g, (H, W, OH, OW) in zip(imgs, got, MIX):
        np.testing.assert_array_equal(g, want(img, OH, OW, mode))


@pytest.mark.parametrize("C", [1, 3])
def test_multi_padded_and_unaligned(rz, C):
    imgs, got, st = run_jobs(rz, MIX[:6], C, 1, seed=5, pad=3, off=1)
    assert st == rz.RZ_OK
    for img, g, (H, W, OH, OW) in zip(imgs, got, MIX[:6]):
        np.testing.assert_array_equal(g, want(img, OH, OW, 1))


# exact 2x down- and upscales: ragged last groups, one-row and one-column
# images, rows of 256 groups and more, row counts that end inside a unit
EXACT2X = [(26, 42, 13, 21), (2, 2, 1, 1), (2, 14, 1, 7), (18, 2, 9, 1), (64, 2080, 32, 1040), (22, 18, 11, 9),
           (40, 34, 20, 17), (13, 21, 26, 42), (1, 1, 2, 2), (1, 7, 2, 14), (9, 1, 18, 2), (4, 4, 8, 8),
           (30, 1100, 60, 2200), (7, 6, 14, 12), (17, 1025, 34, 2050)]


@pytest.mark.parametrize("C", [1, 3, 4])
@pytest.mark.parametrize("pad,off", [(0, 0), (8, 0), (3, 1), (4, 4)])
def test_multi_exact_2x_forms(rz, C, pad, off):
    imgs, got, st = run_jobs(rz, EXACT2X, C, 1, seed=C + pad + off, pad=pad, off=off)
    assert st == rz.RZ_OK
    for img, g, (H, W, OH, OW) in zip(imgs, got, EXACT2X):
        np.testing.assert_array_equal(g, want(img, OH, OW, 1), err_msg=str((H, W, OH, OW)))


# exact 3:2 downscales (the generic form: weights 1536 and 512 from the
# stepped positions), including cfg2's 1080p -> 720p
EXACT32 = [(24, 48, 16, 32), (33, 45, 22, 30), (9, 3, 6, 2), (150, 603, 100, 402), (3, 1563, 2, 1042),
           (1080, 1920, 720, 1280)]


@pytest.mark.parametrize("C", [1, 3, 4])
@pytest.mark.parametrize("pad,off", [(0, 0), (4, 0), (3, 1)])
def test_multi_exact_three_halves_form(rz, C, pad, off):
    imgs, got, st = run_jobs(rz, EXACT32, C, 1, seed=3 * C + pad + off, pad=pad, off=off)
    assert st == rz.RZ_OK
    for img, g, (H, W, OH, OW) in zip(imgs, got, EXACT32):
        np.testing.assert_array_equal(g, want(img, OH, OW, 1), err_msg=str((H, W, OH, OW)))


@pytest.mark.parametrize("n", [64, 256])
def test_multi_long_row_runs(rz, n):
    # the benchmark's mix of geometries (every form: 2x down, 2x up, and two
    # generic ratios) at a quarter of its job count and at its full count
    geoms = [[(480, 640, 240, 320), (720, 1280, 224, 224), (240, 320, 480, 640), (600, 800, 300, 300)][k % 4]
             for k in range(n)]
    imgs, got, st = run_jobs(rz, geoms, 3, 1, seed=n)
    assert st == rz.RZ_OK
    for img, g, (H, W, OH, OW) in zip(imgs, got, geoms):
        np.testing.assert_array_equal(g, want(img, OH, OW, 1))


def test_multi_many_jobs(rz):
    rng = np.random.default_rng(9)
    geoms = [tuple(int(v) for v in rng.integers(1, 40, 4)) for _ in range(600)]
    imgs, got, st = run_jobs(rz, geoms, 3, 1, seed=9)
    assert st == rz.RZ_OK
    for img, g, (H, W, OH, OW) in zip(imgs, got, geoms):
        np.testing.assert_array_equal(g, want(img, OH, OW, 1))


def test_multi_matches_plan_path_at_full_size(rz):
    img = synth.smooth_rgb(1920, 1080, 2)
    geoms = [(1080, 1920, 720, 1280), (1080, 1920, 540, 960), (1080, 1920, 224, 224)]
    srcs = [torch.from_numpy(img).cuda() for _ in geoms]
    dsts = [torch.zeros((g[2], g[3], 3), dtype=torch.uint8, device="cuda") for g in geoms]
    jobs, C = rz.make_jobs(srcs, dsts)
    rz.resize_u8_multi(jobs, len(geoms), C, rz.RZ_LINEAR)
    for (H, W, OH, OW), d in zip(geoms, dsts):
        ref = torch.zeros_like(d)
        with rz.resize_plan_create(H, W, OH, OW, rz.RZ_LINEAR) as plan:
            rz.resize_u8(plan, srcs[0], ref)
        torch.cuda.synchronize()
        assert torch.equal(d, ref)


def test_multi_invalid_jobs_are_skipped_and_flagged(rz):
    img = synth.random_u8((20, 30, 3), seed=1)
    src = torch.from_numpy(img).cuda()
    good = torch.zeros((40, 60, 3), dtype=torch.uint8, device="cuda")
    bad_dst = torch.full((10, 10, 3), 7, dtype=torch.uint8, device="cuda")
    arr = (rz.RzJob * 3)()
    arr[0] = rz.RzJob(src.data_ptr(), good.data_ptr(), 90, 180, 20, 30, 40, 60)
    arr[1] = rz.RzJob(src.data_ptr(), bad_dst.data_ptr(), 10, 30, 20, 30, 10, 10)     # source pitch too small
    arr[2] = rz.RzJob(0, bad_dst.data_ptr(), 90, 30, 20, 30, 10, 10)                   # null source
    import ctypes
    jobs = torch.frombuffer(bytearray(bytes(memoryview(arr))), dtype=torch.uint8).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rz.resize_u8_multi(jobs, 3, 3, rz.RZ_LINEAR, status)
    torch.cuda.synchronize()
    assert int(status.item()) == rz.RZ_ERR_ARG
    np.testing.assert_array_equal(good.cpu().numpy(), oracle.linear_u8(img, 40, 60))
    assert bool((bad_dst == 7).all())
    lib = rz._native.load()
    assert lib.resize_u8_multi(jobs.data_ptr(), rz.RZ_MULTI_MAX_JOBS + 1, 3, 1, None, None) == rz.RZ_ERR_ARG
    assert lib.resize_u8_multi(jobs.data_ptr(), 1, 2, 1, None, None) == rz.RZ_ERR_UNSUPPORTED
    assert lib.resize_u8_multi(jobs.data_ptr(), 1, 3, 5, None, None) == rz.RZ_ERR_ARG
    assert lib.resize_u8_multi(None, 0, 3, 1, None, None) == rz.RZ_OK
    assert lib.resize_u8_multi(None, 1, 3, 1, None, None) == rz.RZ_ERR_ARG
    assert ctypes.sizeof(rz.RzJob) == 48
