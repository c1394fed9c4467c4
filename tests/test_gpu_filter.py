"""Parity of the K x K filters (through the C ABI) with the CPU oracle.

Standalone: the valid-region correlation of the OpenCL convolution page §2
for widths 1 to 64 (the page sweeps 8 to 64), ragged tiles, padded pitches,
unaligned outputs, degenerate and invalid calls.  Fused: the bilinear resize
followed by the centred odd K x K filter with replicate on the output grid,
K in 1, 3, 5, 7, every channel count and border rule, batches, full size.

Tolerances follow from the float32 arithmetic: a sum of n products carries
at most about n roundings of its partial sums, so the valid-region result is
within 2 K^2 2^-24 sum|w| max|x| of the exact sum; the fused result adds
sum|w| times the resize's 1e-4 to the filter's own bound.
"""
import numpy as np
import pytest

import oracle
from bilinear_image_resize_gb300 import synth
from gpu_util import Canvas, max_abs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rz():
    import __graft_entry__
    __graft_entry__.build()
    import bilinear_image_resize_gb300 as m
    torch.cuda.set_device(0)
    return m


def valid_tol(w, xmax):
    K = w.shape[0]
    return 2.0 * K * K * 2.0 ** -24 * float(np.abs(w).sum()) * xmax + 1e-6


def gpu_valid(rz, img, w, dst_pad=0, src_pad=0, dst_off=0):
    H, W = img.shape
    K = w.shape[0]
    OH, OW = max(H - K + 1, 0), max(W - K + 1, 0)
    sbuf = torch.zeros((H, W + src_pad), dtype=torch.float32, device="cuda")
    sbuf[:, :W] = torch.from_numpy(img).cuda()
    src = sbuf[:, :W]
    flat = torch.full(((OH + 2) * (OW + dst_pad) + dst_off + 8,), -777.0, dtype=torch.float32, device="cuda")
    dst = torch.as_strided(flat, (OH, OW), (OW + dst_pad, 1), dst_off + (OW + dst_pad))
    wt = torch.from_numpy(np.ascontiguousarray(w)).cuda()
    rz.filter2d_valid_f32(src, wt, dst)
    torch.cuda.synchronize()
    # nothing written outside the output
    mask = torch.ones_like(flat, dtype=torch.bool)
    if OH and OW:
        idx = (dst_off + (OW + dst_pad) + torch.arange(OH, device="cuda")[:, None] * (OW + dst_pad)
               + torch.arange(OW, device="cuda")[None, :]).flatten()
        mask[idx] = False
    assert bool((flat[mask] == -777.0).all())
    return dst.cpu().numpy()


@pytest.mark.parametrize("K", [1, 2, 3, 5, 7, 8, 13, 16, 31, 32, 33, 64])
def test_valid_widths(rz, K):
    H, W = K + 37, K + 300
    img = synth.random_f32((H, W), seed=K)
    w = (np.random.default_rng(K).random((K, K)) - 0.25).astype(np.float32)
    got = gpu_valid(rz, img, w)
    want = oracle.filter_valid(img, w)
    assert got.shape == want.shape
    assert max_abs(got, want) <= valid_tol(w, 255.0), (max_abs(got, want), valid_tol(w, 255.0))


@pytest.mark.parametrize("K", [8, 64])
def test_valid_larger_image(rz, K):
    img = synth.random_f32((520, 700), seed=100 + K)
    w = synth.filter_weights_k(K)
    got = gpu_valid(rz, img, w)
    assert max_abs(got, oracle.filter_valid(img, w)) <= valid_tol(w, 255.0)


@pytest.mark.parametrize("K", [3, 16])
def test_valid_layouts(rz, K):
    img = synth.random_f32((K + 20, K + 45), seed=7)
    w = synth.filter_weights_k(K)
    want = oracle.filter_valid(img, w)
    for kw in ({"src_pad": 3}, {"dst_pad": 5}, {"dst_off": 1}, {"src_pad": 1, "dst_pad": 2, "dst_off": 3}):
        assert max_abs(gpu_valid(rz, img, w, **kw), want) <= valid_tol(w, 255.0)


def test_valid_delta_is_exact(rz):
    img = synth.random_f32((40, 333), seed=2)
    for K, (r0, c0) in [(5, (4, 0)), (9, (2, 7)), (64, (63, 63))]:
        if img.shape[0] < K:
            img = synth.random_f32((K + 10, 333), seed=2)
        w = np.zeros((K, K), np.float32)
        w[r0, c0] = 1.0
        got = gpu_valid(rz, img, w)
        np.testing.assert_array_equal(got, img[r0:r0 + got.shape[0], c0:c0 + got.shape[1]])


def test_valid_degenerate_and_invalid(rz):
    import ctypes
    lib = rz._native.load()
    s = torch.zeros((8, 8), dtype=torch.float32, device="cuda")
    d = torch.zeros((8, 8), dtype=torch.float32, device="cuda")
    w = torch.ones((9, 9), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    # smaller than the filter: empty output, nothing launched
    assert lib.filter2d_valid_f32(s.data_ptr(), 32, 8, 8, w.data_ptr(), 9, d.data_ptr(), 32, st) == rz.RZ_OK
    assert lib.filter2d_valid_f32(s.data_ptr(), 32, 8, 8, w.data_ptr(), 0, d.data_ptr(), 32, st) == rz.RZ_ERR_ARG
    assert lib.filter2d_valid_f32(s.data_ptr(), 32, 8, 8, w.data_ptr(), 65, d.data_ptr(), 32,
                                  st) == rz.RZ_ERR_UNSUPPORTED
    assert lib.filter2d_valid_f32(s.data_ptr(), 16, 8, 8, w.data_ptr(), 3, d.data_ptr(), 32, st) == rz.RZ_ERR_ARG
    assert lib.filter2d_valid_f32(s.data_ptr(), 32, 8, 8, w.data_ptr(), 3, d.data_ptr(), 18, st) == rz.RZ_ERR_ARG
    assert lib.filter2d_valid_f32(s.data_ptr(), 32, 8, 8, None, 3, d.data_ptr(), 32, st) == rz.RZ_ERR_ARG
    # in place
    assert lib.filter2d_valid_f32(s.data_ptr(), 32, 8, 8, w.data_ptr(), 3, s.data_ptr(), 32, st) == rz.RZ_ERR_ARG
    assert lib.filter2d_valid_f32(s.data_ptr(), 32, 8, 8, w.data_ptr(), 8, d.data_ptr(), 4, st) == rz.RZ_OK
    torch.cuda.synchronize()


# ---------------------------------------------------------------- fused K x K

def fused_tol(w):
    # the resized values are within 1e-4 each (the float32 resize bound), so
    # the filter carries sum|w| * 1e-4 of it, plus its own sum's roundings
    K = w.shape[0]
    sw = float(np.abs(w).sum())
    return sw * 1e-4 + 2.0 * K * K * 2.0 ** -24 * sw * 255.0


def gpu_fused(rz, img, OH, OW, w, border=0, opts=(), batch=None):
    H, W, C = img.shape[-3:]
    src = torch.from_numpy(np.ascontiguousarray(img)).cuda()
    shape = (OH, OW, C) if batch is None else (batch, OH, OW, C)
    out = torch.full(shape, -99.0, dtype=torch.float32, device="cuda")
    with rz.resize_plan_create(H, W, OH, OW, rz.RZ_LINEAR, border=border) as plan:
        for k, v in opts:
            rz.resize_plan_set_option(plan, k, v)
        rz.resize_fused(plan, src, out, rz.make_epilogue(rz.RZ_EPI_FILTER, wk=w))
        torch.cuda.synchronize()
        assert rz.resize_plan_status(plan) == rz.RZ_OK
    return out.cpu().numpy()


def want_fused(img, OH, OW, w, border=0):
    r = oracle.linear_f32(img, OH, OW, border)
    return np.stack([oracle.filter_centred(r[:, :, c], w) for c in range(r.shape[2])], -1)


@pytest.mark.parametrize("K", [1, 3, 5, 7])
@pytest.mark.parametrize("C", [1, 3, 4])
@pytest.mark.parametrize("border", [0, 1, 2])
@pytest.mark.parametrize("geom", [(37, 53, 100, 131), (90, 120, 37, 50), (5, 7, 13, 17), (1, 5, 4, 9),
                                  (70, 64, 70, 64)])
def test_fused_kxk(rz, K, C, border, geom):
    H, W, OH, OW = geom
    img = synth.random_f32((H, W, C), seed=K + C + H)
    w = (np.random.default_rng(K).random((K, K)) - 0.2).astype(np.float32)
    got = gpu_fused(rz, img, OH, OW, w, border)
    assert max_abs(got, want_fused(img, OH, OW, w, border)) <= fused_tol(w)


@pytest.mark.parametrize("kernel", [1, 2])
@pytest.mark.parametrize("K", [3, 5, 7])
@pytest.mark.parametrize("C", [1, 3, 4])
def test_fused_on_both_kernels(rz, kernel, K, C):
    # the streaming kernel (1) and the tile kernel (2), ragged strips and
    # segments at several output sizes
    for (H, W, OH, OW) in [(150, 170, 333, 201), (64, 700, 97, 1500), (300, 40, 130, 19)]:
        img = synth.random_f32((H, W, C), seed=3 + K)
        w = synth.filter_weights_k(K)
        got = gpu_fused(rz, img, OH, OW, w, opts=[(rz.RZ_OPT_FILTER_KERNEL, kernel)])
        assert max_abs(got, want_fused(img, OH, OW, w)) <= fused_tol(w)


@pytest.mark.parametrize("K", [3, 5, 7])
def test_fused_streaming_tiles_and_rings(rz, K):
    # explicit strips and ring depths on the streaming kernel
    img = synth.random_f32((200, 260, 1), seed=K)
    w = synth.filter_weights_k(K)
    want = want_fused(img, 310, 390, w)
    for tile, ring in [((5, 40), 0), ((64, 100), 16), ((1, 17), 2), ((300, 478), 0)]:
        with rz.resize_plan_create(200, 260, 310, 390, rz.RZ_LINEAR) as plan:
            rz.resize_plan_set_tile(plan, rz.KIND_FILTER3X3, *tile)
            if ring:
                rz.resize_plan_set_option(plan, rz.RZ_OPT_RING_ROWS, ring)
            src = torch.from_numpy(img).cuda()
            out = torch.full((310, 390, 1), -99.0, dtype=torch.float32, device="cuda")
            rz.resize_fused(plan, src, out, rz.make_epilogue(rz.RZ_EPI_FILTER, wk=w))
            torch.cuda.synchronize()
            assert rz.resize_plan_status(plan) == rz.RZ_OK
        assert max_abs(out.cpu().numpy(), want) <= fused_tol(w), (tile, ring)


@pytest.mark.parametrize("K", [3, 5, 7])
def test_fused_widest_strips(rz, K):
    # one-channel strips as wide as the kernel takes (every lane's four
    # column slots in use, neighbours taken across the slot boundaries), and
    # a strip width one column short of it
    img = synth.random_f32((64, 1400, 1), seed=40 + K)
    w = synth.filter_weights_k(K)
    want = want_fused(img, 70, 1290, w)
    widest = 8 * (32 * 4 - 2 * (K // 2))
    for tile in [(16, 4096), (9, widest - 1), None]:
        with rz.resize_plan_create(64, 1400, 70, 1290, rz.RZ_LINEAR) as plan:
            if tile:
                rz.resize_plan_set_tile(plan, rz.KIND_FILTER3X3, *tile)
            src = torch.from_numpy(img).cuda()
            out = torch.full((70, 1290, 1), -99.0, dtype=torch.float32, device="cuda")
            rz.resize_fused(plan, src, out, rz.make_epilogue(rz.RZ_EPI_FILTER, wk=w))
            torch.cuda.synchronize()
            assert rz.resize_plan_status(plan) == rz.RZ_OK
        assert max_abs(out.cpu().numpy(), want) <= fused_tol(w), tile


def test_fused_batch(rz):
    N, H, W, OH, OW = 3, 40, 50, 77, 33
    frames = np.stack([synth.random_f32((H, W, 3), seed=n) for n in range(N)])
    w = synth.filter_weights_k(5)
    got = gpu_fused(rz, frames, OH, OW, w, batch=N)
    for n in range(N):
        assert max_abs(got[n], want_fused(frames[n], OH, OW, w)) <= fused_tol(w)


@pytest.mark.parametrize("K", [5, 7])
def test_fused_full_size(rz, K):
    img = synth.float_gray()                          # 8192 x 8192
    w = synth.filter_weights_k(K)
    got = gpu_fused(rz, img[:, :, None], 5980, 5980, w)[:, :, 0]
    want = oracle.filter_centred(oracle.linear_f32(img, 5980, 5980), w)
    assert max_abs(got, want) <= fused_tol(w)


def test_fused_argument_checks(rz):
    import ctypes
    lib = rz._native.load()
    src = torch.zeros((8, 8), dtype=torch.float32, device="cuda")
    dst = torch.zeros((16, 16), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    with rz.resize_plan_create(8, 8, 16, 16, rz.RZ_LINEAR) as plan:
        for K, code in [(2, rz.RZ_ERR_ARG), (0, rz.RZ_ERR_ARG), (-3, rz.RZ_ERR_ARG), (9, rz.RZ_ERR_UNSUPPORTED)]:
            e = rz.make_epilogue(rz.RZ_EPI_FILTER)
            e.ksize = K
            assert lib.resize_fused(plan.handle, src.data_ptr(), rz.RZ_F32, 32, dst.data_ptr(), 64, 8, 8, 1, 16, 16,
                                    rz.RZ_LINEAR, ctypes.byref(e), st) == code
        e = rz.make_epilogue(rz.RZ_EPI_FILTER, wk=np.ones((5, 5)))
        assert lib.resize_fused(plan.handle, src.data_ptr(), rz.RZ_U8, 32, dst.data_ptr(), 64, 8, 8, 1, 16, 16,
                                rz.RZ_LINEAR, ctypes.byref(e), st) == rz.RZ_ERR_ARG
        rz.resize_plan_set_option(plan, rz.RZ_OPT_FILTER_KERNEL, 1)
        e1 = rz.make_epilogue(rz.RZ_EPI_FILTER, wk=np.ones((1, 1)))
        assert lib.resize_fused(plan.handle, src.data_ptr(), rz.RZ_F32, 32, dst.data_ptr(), 64, 8, 8, 1, 16, 16,
                                rz.RZ_LINEAR, ctypes.byref(e1), st) == rz.RZ_ERR_UNSUPPORTED
        with pytest.raises(rz.ResizeError):
            rz.resize_plan_set_option(plan, rz.RZ_OPT_FILTER_KERNEL, 3)
    torch.cuda.synchronize()
