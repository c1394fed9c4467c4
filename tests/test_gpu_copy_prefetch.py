"""The 1:1 copy baseline and the exact-ratio kernels' pre-wait L2 prefetch.

resize_copy_baseline must copy every byte and nothing else, under every
launch flag; it rejects misaligned, ragged, overlapping and unknown-flag
calls.  The prefetch is a hint: every exact-ratio kernel gives the same
bytes with RZ_OPT_L2_PREFETCH on and off, equal to the oracle, including
when the resize reads a frame that the kernel queued right before it is
still writing (the prefetch is issued before the dependency wait).
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


FLAG_SETS = [0, 1, 2, 3]


@pytest.mark.parametrize("nbytes", [16, 4096, 4112, 65536 + 48, 15_552_000])
@pytest.mark.parametrize("flags", FLAG_SETS)
def test_copy_baseline_copies_exactly(rz, nbytes, flags):
    g = torch.Generator(device="cuda").manual_seed(nbytes + flags)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device="cuda", generator=g)
    guard = 4096
    buf = torch.full((nbytes + 2 * guard,), 0xA5, dtype=torch.uint8, device="cuda")
    dst = buf[guard:guard + nbytes]
    rz.resize_copy_baseline(src, dst, flags)
    torch.cuda.synchronize()
    assert torch.equal(dst, src)
    assert bool((buf[:guard] == 0xA5).all()) and bool((buf[guard + nbytes:] == 0xA5).all())


def test_copy_baseline_back_to_back_chain(rz):
    # each copy reads the previous copy's output, queued as dependent launches
    n = 1 << 22
    bufs = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(4)]
    bufs[0].copy_(torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda"))
    for _ in range(3):
        for k in range(3):
            rz.resize_copy_baseline(bufs[k], bufs[k + 1], rz.RZ_COPY_PDL | rz.RZ_COPY_L2_PREFETCH)
    torch.cuda.synchronize()
    assert torch.equal(bufs[3], bufs[0])


def test_copy_baseline_rejects_bad_calls(rz):
    lib = rz._native.load()
    a = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    b = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert lib.resize_copy_baseline(a.data_ptr(), b.data_ptr(), 0, 3, s) == rz.RZ_OK
    assert lib.resize_copy_baseline(a.data_ptr() + 1, b.data_ptr(), 64, 3, s) == rz.RZ_ERR_ARG
    assert lib.resize_copy_baseline(a.data_ptr(), b.data_ptr() + 8, 64, 3, s) == rz.RZ_ERR_ARG
    assert lib.resize_copy_baseline(a.data_ptr(), b.data_ptr(), 40, 3, s) == rz.RZ_ERR_ARG
    assert lib.resize_copy_baseline(a.data_ptr(), a.data_ptr() + 64, 128, 3, s) == rz.RZ_ERR_ARG
    assert lib.resize_copy_baseline(a.data_ptr(), b.data_ptr(), 64, 4, s) == rz.RZ_ERR_ARG
    assert lib.resize_copy_baseline(None, b.data_ptr(), 64, 3, s) == rz.RZ_ERR_ARG
    torch.cuda.synchronize()


def _run(rz, img, OH, OW, mode, prefetch, border=0, epi=None):
    H, W = img.shape[:2]
    C = img.shape[2] if img.ndim == 3 else 1
    src = torch.from_numpy(np.ascontiguousarray(img)).cuda()
    with rz.resize_plan_create(H, W, OH, OW, mode, border=border) as plan:
        rz.resize_plan_set_option(plan, rz.RZ_OPT_L2_PREFETCH, prefetch)
        if epi is not None:
            dst = torch.full((OH, OW), 7, dtype=torch.uint8, device="cuda")
            rz.resize_fused(plan, src, dst, epi)
        else:
            dst = torch.full((OH, OW, C) if img.ndim == 3 else (OH, OW), 7, dtype=torch.uint8, device="cuda")
            rz.resize_u8(plan, src, dst)
        torch.cuda.synchronize()
        assert rz.resize_plan_status(plan) == rz.RZ_OK
    return dst.cpu().numpy()


# (H, W, OH, OW, C, mode, border): the exact 2x down (bilinear, nearest),
# 3:2 down and 2x up kernels (layouts that take their vector paths), every
# channel count, the border rules of the upscale, odd sizes; then the any-ratio
# direct kernel (spans from the plan's tables: wide and narrow rows, CTAs
# that cover several output rows, both modes, the wrap rule's far tap)
EXACT_CASES = [
    (2160, 3840, 1080, 1920, 3, 1, 0), (2160, 3840, 1080, 1920, 3, 0, 0), (540, 976, 270, 488, 1, 1, 0),
    (540, 968, 270, 484, 4, 0, 0), (1080, 1920, 720, 1280, 3, 1, 0), (333, 1047, 222, 698, 4, 1, 0),
    (90, 132, 60, 88, 1, 1, 0), (1080, 1920, 2160, 3840, 3, 1, 0), (77, 131, 154, 262, 4, 1, 1),
    (77, 131, 154, 262, 1, 1, 2), (61, 50, 122, 100, 3, 1, 1),
    (2160, 3840, 768, 1366, 3, 1, 0), (1080, 1920, 600, 1000, 4, 1, 0), (720, 1280, 224, 224, 3, 1, 0),
    (300, 500, 77, 31, 1, 1, 0), (1080, 1920, 600, 1000, 3, 0, 0), (303, 405, 101, 135, 3, 1, 2),
    (303, 405, 101, 135, 4, 1, 1),
]


@pytest.mark.parametrize("case", EXACT_CASES)
def test_prefetch_on_and_off_match_oracle(rz, case):
    H, W, OH, OW, C, mode, border = case
    img = synth.random_u8((H, W, C), seed=H + W + C)
    want = oracle.linear_u8(img, OH, OW, border) if mode == 1 else oracle.nearest_u8(img, OH, OW)
    for prefetch in (1, 0):
        np.testing.assert_array_equal(_run(rz, img, OH, OW, mode, prefetch, border), want)


@pytest.mark.parametrize("C", [3, 4])
def test_prefetch_gray_exact_2x(rz, C):
    img = synth.random_u8((540, 968, C), seed=C)
    want = oracle.gray_resize_u8(img, 270, 484)
    for prefetch in (1, 0):
        got = _run(rz, img, 270, 484, rz.RZ_LINEAR, prefetch, epi=rz.make_epilogue(rz.RZ_EPI_GRAY_RGB))
        np.testing.assert_array_equal(got, want)


def test_prefetch_with_batches(rz):
    N = 5
    frames = np.stack([synth.random_u8((270, 480, 3), seed=70 + n) for n in range(N)])
    src = torch.from_numpy(frames).cuda()
    for prefetch in (1, 0):
        dst = torch.zeros((N, 135, 240, 3), dtype=torch.uint8, device="cuda")
        with rz.resize_plan_create(270, 480, 135, 240, rz.RZ_LINEAR) as plan:
            rz.resize_plan_set_option(plan, rz.RZ_OPT_L2_PREFETCH, prefetch)
            rz.resize_u8_batch(plan, src, dst)
            torch.cuda.synchronize()
        got = dst.cpu().numpy()
        for n in range(N):
            np.testing.assert_array_equal(got[n], oracle.linear_u8(frames[n], 135, 240))


def test_prefetch_reads_frame_the_previous_kernel_writes(rz):
    # the 4K frame X is written by a 2x upscale and read by the 2x downscale
    # queued right after it; the downscale's CTAs prefetch X before waiting
    # for the upscale, while X still holds the previous round's content (or
    # the initial 0xEE fill), so every round must still see the new frame
    rounds = 4
    srcs = [synth.random_u8((1080, 1920, 3), seed=80 + k) for k in range(rounds)]
    a = [torch.from_numpy(s).cuda() for s in srcs]
    x = torch.full((2160, 3840, 3), 0xEE, dtype=torch.uint8, device="cuda")
    outs = [torch.empty((1080, 1920, 3), dtype=torch.uint8, device="cuda") for _ in range(rounds)]
    up = rz.resize_plan_create(1080, 1920, 2160, 3840, rz.RZ_LINEAR)
    down = rz.resize_plan_create(2160, 3840, 1080, 1920, rz.RZ_LINEAR)
    torch.cuda.synchronize()
    for k in range(rounds):
        rz.resize_u8(up, a[k], x)
        rz.resize_u8(down, x, outs[k])
    torch.cuda.synchronize()
    for k in range(rounds):
        want = oracle.linear_u8(oracle.linear_u8(srcs[k], 2160, 3840), 1080, 1920)
        np.testing.assert_array_equal(outs[k].cpu().numpy(), want)
    up.destroy()
    down.destroy()


def test_prefetch_option_rejects_bad_values(rz):
    with rz.resize_plan_create(8, 8, 4, 4, rz.RZ_LINEAR) as plan:
        for val in (-1, 2):
            with pytest.raises(rz.ResizeError):
                rz.resize_plan_set_option(plan, rz.RZ_OPT_L2_PREFETCH, val)
        rz.resize_plan_set_option(plan, rz.RZ_OPT_L2_PREFETCH, 0)
        rz.resize_plan_set_option(plan, rz.RZ_OPT_L2_PREFETCH, 1)
