"""The standalone K x K correlation on the tensor cores (filter2d_valid_f32_ex
with RZ_FILTER_TENSOR), against the CPU oracle.

The kernel forms each output tile as a sum over filter rows of one TF32
matrix product per row (the input tile shifted down r rows times the banded
Toeplitz matrix of filter row r), each float split into a TF32 high part and
the remainder with three products per tap pair.  Its results must stay within
the float32 bound the FP32 kernel is held to (2 K^2 2^-24 sum|w| max|x|, the
"OpenCL image convolution" page's correlation over the valid region) for
every width it takes (16 <= K <= 64), tile-ragged sizes, padded pitches and
unaligned outputs; the automatic choice must equal the kernel it picks bit
for bit; layouts it cannot take must be refused; and at the benchmark's size
sampled row bands must match the oracle.
"""
import numpy as np
import pytest

import oracle
from bilinear_image_resize_gb300 import synth
from gpu_util import max_abs

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


def run(rz, img, w, kernel, src_pad=0, dst_pad=0, dst_off=0):
    H, W = img.shape
    K = w.shape[0]
    OH, OW = H - K + 1, W - K + 1
    sbuf = torch.zeros((H, W + src_pad), dtype=torch.float32, device="cuda")
    sbuf[:, :W] = torch.from_numpy(img).cuda()
    flat = torch.full(((OH + 2) * (OW + dst_pad) + dst_off + 8,), -777.0, dtype=torch.float32, device="cuda")
    dst = torch.as_strided(flat, (OH, OW), (OW + dst_pad, 1), dst_off + (OW + dst_pad))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rz.filter2d_valid_f32(sbuf[:, :W], torch.from_numpy(np.ascontiguousarray(w)).cuda(), dst, kernel=kernel,
                          status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == rz.RZ_OK
    mask = torch.ones_like(flat, dtype=torch.bool)
    idx = (dst_off + (OW + dst_pad) + torch.arange(OH, device="cuda")[:, None] * (OW + dst_pad)
           + torch.arange(OW, device="cuda")[None, :]).flatten()
    mask[idx] = False
    assert bool((flat[mask] == -777.0).all()), "written outside the output"
    return dst.cpu().numpy()


@pytest.mark.parametrize("K", [16, 17, 31, 33, 48, 63, 64])
def test_tensor_widths_against_oracle(rz, K):
    img = synth.random_f32((300, 296), seed=K)
    w = synth.filter_weights_k(K)
    got = run(rz, img, w, rz.RZ_FILTER_TENSOR)
    want = oracle.filter_valid(img, w)
    assert max_abs(got, want) <= valid_tol(w, 255.0), (K, max_abs(got, want), valid_tol(w, 255.0))


@pytest.mark.parametrize("shape,K", [((129, 160), 16), ((128 + 63, 96), 64), ((600, 100), 16), ((64, 64), 64),
                                     ((130, 4096), 48), ((4100, 36), 16), ((257, 332), 40)])
def test_tensor_ragged_tiles(rz, shape, K):
    img = synth.random_f32(shape, seed=shape[0] + K)
    w = synth.filter_weights_k(K)
    assert max_abs(run(rz, img, w, rz.RZ_FILTER_TENSOR), oracle.filter_valid(img, w)) <= valid_tol(w, 255.0)


def test_tensor_signed_weights_and_layouts(rz):
    # weights of both signs (sum|w| > 1), padded source and output rows, an
    # output start that is not 16-byte aligned
    rng = np.random.default_rng(4)
    img = synth.random_f32((200, 244), seed=9)
    w = (rng.random((24, 24)) - 0.5).astype(np.float32)
    want = oracle.filter_valid(img, w)
    for kw in ({}, {"src_pad": 12}, {"dst_pad": 3}, {"dst_off": 1}):
        assert max_abs(run(rz, img, w, rz.RZ_FILTER_TENSOR, **kw), want) <= valid_tol(w, 255.0), kw


def test_auto_choice_equals_the_kernel_it_picks(rz):
    img = synth.random_f32((400, 400), seed=2)
    for K, picked in ((64, "tensor"), (48, "tensor"), (32, "fp32"), (8, "fp32")):
        w = synth.filter_weights_k(K)
        auto = run(rz, img, w, rz.RZ_FILTER_AUTO)
        tensor = run(rz, img, w, rz.RZ_FILTER_TENSOR) if K >= 16 else None
        fp32 = run(rz, img, w, rz.RZ_FILTER_FP32)
        assert np.array_equal(auto, tensor if picked == "tensor" else fp32), K
        assert max_abs(auto, oracle.filter_valid(img, w)) <= valid_tol(w, 255.0)


def test_tensor_refuses_what_it_cannot_take(rz):
    img = synth.random_f32((100, 101), seed=1)   # 404-byte rows: not a multiple of 16
    w = synth.filter_weights_k(20)
    with pytest.raises(rz.ResizeError) as e:
        run(rz, img, w, rz.RZ_FILTER_TENSOR)
    assert e.value.code == rz.RZ_ERR_UNSUPPORTED
    # the automatic choice falls back to the FP32 kernel on that layout
    assert max_abs(run(rz, img, w, rz.RZ_FILTER_AUTO), oracle.filter_valid(img, w)) <= valid_tol(w, 255.0)
    img2 = synth.random_f32((100, 100), seed=1)
    with pytest.raises(rz.ResizeError) as e:
        run(rz, img2, synth.filter_weights_k(8), rz.RZ_FILTER_TENSOR)
    assert e.value.code == rz.RZ_ERR_UNSUPPORTED
    with pytest.raises(rz.ResizeError) as e:
        run(rz, img2, synth.filter_weights_k(8), 7)
    assert e.value.code == rz.RZ_ERR_ARG


@pytest.mark.parametrize("K", [16, 64])
def test_tensor_full_size_row_bands(rz, K):
    # the benchmark's 4096^2 image: row bands at the top, middle and bottom
    # computed by the oracle one band at a time
    img = synth.float_gray(4096, 4096, 5)
    w = synth.filter_weights_k(K)
    OH = 4097 - K
    src = torch.from_numpy(img).cuda()
    dst = torch.empty((OH, OH), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rz.filter2d_valid_f32(src, torch.from_numpy(w).cuda(), dst, kernel=rz.RZ_FILTER_TENSOR, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == rz.RZ_OK
    got = dst.cpu().numpy()
    for y0 in (0, 1977, OH - 6):
        want = oracle.filter_valid(img[y0:y0 + 6 + K - 1], w)
        assert max_abs(got[y0:y0 + 6], want) <= valid_tol(w, 255.0), y0


def test_tensor_back_to_back_dependent_calls(rz):
    # the second correlation reads the first one's output, queued as a
    # dependent launch
    img = synth.random_f32((512, 512), seed=3)
    w1, w2 = synth.filter_weights_k(16), synth.filter_weights_k(17)
    a = torch.from_numpy(img).cuda()
    # 497-float rows are not 16-byte multiples: the intermediate has padded rows
    bpad = torch.zeros((497, 500), dtype=torch.float32, device="cuda")
    c = torch.empty((481, 481), dtype=torch.float32, device="cuda")
    for _ in range(2):
        rz.filter2d_valid_f32(a, torch.from_numpy(w1).cuda(), bpad[:, :497], kernel=rz.RZ_FILTER_TENSOR)
        rz.filter2d_valid_f32(bpad[:, :497], torch.from_numpy(w2).cuda(), c, kernel=rz.RZ_FILTER_TENSOR)
    torch.cuda.synchronize()
    mid = oracle.filter_valid(img, w1).astype(np.float32)
    want = oracle.filter_valid(mid, w2)
    assert max_abs(c.cpu().numpy(), want) <= valid_tol(w2, 255.0) + valid_tol(w1, 255.0)
