"""resize_u8_noalloc: the uint8 resize for callers that may not allocate device
memory (a plugin living inside another framework's memory pool, a real-time
pipeline that forbids allocation once running).  It keeps its sampling tables
in the library's static device array instead of a plan.

Its output must equal the plan-based resize_u8 output (uint8 results are
bit-exact, the tolerance every uint8 test here uses), for two calls in a row,
since the second call finds the first call's tables in the shared array.  The
file is named to be collected last and works alone in a fresh process.
"""
import numpy as np
import pytest

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


def with_plan(rz, src, OH, OW, mode):
    H, W = src.shape[:2]
    C = src.shape[2] if src.dim() == 3 else 1
    dst = torch.empty((OH, OW, C) if src.dim() == 3 else (OH, OW), dtype=torch.uint8, device="cuda")
    with rz.resize_plan_create(H, W, OH, OW, mode) as plan:
        rz.resize_u8(plan, src, dst)
        torch.cuda.synchronize()
    return dst


def test_no_alloc_matches_plan_path_two_calls_in_a_row(rz):
    img = synth.smooth_rgb(3840, 2160, 3)
    src = torch.from_numpy(np.ascontiguousarray(img)).cuda()
    # two different geometries back to back, then the first again: each call
    # must rebuild the shared tables it needs
    for (OH, OW, mode) in [(1080, 1920, rz.RZ_LINEAR), (720, 1280, rz.RZ_LINEAR), (1080, 1920, rz.RZ_LINEAR),
                           (540, 960, rz.RZ_NEAREST)]:
        want = with_plan(rz, src, OH, OW, mode)
        out1 = torch.full((OH, OW, 3), 7, dtype=torch.uint8, device="cuda")
        out2 = torch.full((OH, OW, 3), 9, dtype=torch.uint8, device="cuda")
        rz.resize_u8_noalloc(src, out1, mode)
        rz.resize_u8_noalloc(src, out2, mode)
        torch.cuda.synchronize()
        assert torch.equal(out1, want)
        assert torch.equal(out2, want)


@pytest.mark.parametrize("C", [1, 3, 4])
def test_no_alloc_small_and_odd_geometries(rz, C):
    rng = np.random.default_rng(C)
    for _ in range(12):
        H, W, OH, OW = (int(v) for v in rng.integers(1, 200, size=4))
        img = synth.random_u8((H, W, C), seed=H + W)
        src = torch.from_numpy(img).cuda()
        for mode in (rz.RZ_LINEAR, rz.RZ_NEAREST):
            want = with_plan(rz, src, OH, OW, mode)
            got = torch.empty_like(want)
            rz.resize_u8_noalloc(src, got, mode)
            rz.resize_u8_noalloc(src, got, mode)
            torch.cuda.synchronize()
            assert torch.equal(got, want), (H, W, OH, OW, C, mode)


def test_no_alloc_rejects_sizes_beyond_its_array(rz):
    src = torch.zeros((16, 16, 3), dtype=torch.uint8, device="cuda")
    big = torch.empty((4, rz.RZ_NOALLOC_MAX_DIM + 1, 3), dtype=torch.uint8, device="cuda")
    with pytest.raises(rz.ResizeError) as e:
        rz.resize_u8_noalloc(src, big)
    assert e.value.code == rz.RZ_ERR_UNSUPPORTED


# Wide outputs that the no-alloc tile loop cuts into strips: a generic
# 8192-wide output, an exact 2x whose strips are narrower than the output,
# and a heavy downscale whose one-strip source span is over 16 KB; every
# channel count and both modes, two calls in a row, against the plan path.
@pytest.mark.parametrize("C", [1, 3, 4])
@pytest.mark.parametrize("geo", [(64, 12000, 32, 8192), (8, 16384, 4, 8192), (4, 65536, 2, 100)])
def test_no_alloc_wide_outputs_and_strips(rz, C, geo):
    H, W, OH, OW = geo
    img = synth.random_u8((H, W, C), seed=W + C)
    src = torch.from_numpy(img).cuda()
    for mode in (rz.RZ_LINEAR, rz.RZ_NEAREST):
        want = with_plan(rz, src, OH, OW, mode)
        got = torch.full_like(want, 3)
        rz.resize_u8_noalloc(src, got, mode)
        rz.resize_u8_noalloc(src, got, mode)
        torch.cuda.synchronize()
        assert torch.equal(got, want), (geo, C, mode)


def test_no_alloc_rejects_a_stream_of_another_device(rz):
    # only one device may be present: then a stream of the current device is
    # accepted and the check cannot be exercised further here
    src = torch.zeros((16, 16, 3), dtype=torch.uint8, device="cuda")
    dst = torch.empty((8, 8, 3), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    rz.resize_u8_noalloc(src, dst, stream=s)
    torch.cuda.synchronize()
    if torch.cuda.device_count() < 2:
        return
    with torch.cuda.device(1):
        other = torch.cuda.Stream()
    with pytest.raises(rz.ResizeError) as e:
        rz.resize_u8_noalloc(src, dst, stream=other)
    assert e.value.code == rz.RZ_ERR_ARG
