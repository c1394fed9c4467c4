"""The hardware-filtered (texture) bilinear path, measured against the oracle.

It is a comparison path (Volcanic resize page, *Naive resize with linear
sampling*; CUDA interpolation page §4.1): the texture unit's weights carry
about 8 fractional bits, so it is not bit-exact.  The tests bound its error
against the exact oracle (the weights' quantisation moves a value by at most
255 * 2 * 2^-9 < 1, plus the final rounding: at most 2 units) and check that
most outputs are exact, plus the handle's argument checks.
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


def tex_resize(rz, img, OH, OW):
    H, W, C = img.shape
    src = torch.from_numpy(np.ascontiguousarray(img)).cuda()
    dst = torch.zeros((OH, OW, C), dtype=torch.uint8, device="cuda")
    with rz.resize_texture_create(src) as t:
        t.resize(dst)
        torch.cuda.synchronize()
    return dst.cpu().numpy()


@pytest.mark.parametrize("C", [1, 4])
@pytest.mark.parametrize("geom", [(64, 64, 128, 128), (96, 128, 37, 50), (32, 64, 100, 131), (64, 32, 64, 32)])
def test_texture_error_is_bounded(rz, C, geom):
    H, W, OH, OW = geom
    img = synth.random_u8((H, W, C), seed=H + W + C)
    got = tex_resize(rz, img, OH, OW).astype(np.int64)
    want = oracle.linear_u8(img, OH, OW).astype(np.int64)
    err = np.abs(got - want)
    assert err.max() <= 2, err.max()
    if (H, W) == (OH, OW):
        assert err.max() == 0          # identity: every sample at a texel centre
    assert (err == 0).mean() > 0.5


def test_texture_4k_to_1080p_rgba(rz):
    img = np.concatenate([synth.smooth_rgb(3840, 2160, 3), np.full((2160, 3840, 1), 255, np.uint8)], -1)
    got = tex_resize(rz, img, 1080, 1920).astype(np.int64)
    want = oracle.linear_u8(img, 1080, 1920).astype(np.int64)
    err = np.abs(got - want)
    assert err.max() <= 2
    assert (err == 0).mean() > 0.5


def test_texture_argument_checks(rz):
    import ctypes
    lib = rz._native.load()
    buf = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    h = ctypes.c_void_p()
    dev = torch.cuda.current_device()
    assert lib.resize_texture_create(ctypes.byref(h), buf.data_ptr(), 256, 16, 64, 3) == rz.RZ_ERR_UNSUPPORTED
    assert lib.resize_texture_create(ctypes.byref(h), buf.data_ptr(), 256, 16, 64, 2) == rz.RZ_ERR_UNSUPPORTED
    assert lib.resize_texture_create(ctypes.byref(h), buf.data_ptr(), 100, 16, 64, 4) == rz.RZ_ERR_ARG
    assert lib.resize_texture_create(ctypes.byref(h), buf.data_ptr() + 1, 256, 16, 64, 4) == rz.RZ_ERR_ARG
    assert lib.resize_texture_create(ctypes.byref(h), buf.data_ptr(), 257, 16, 64, 4) == rz.RZ_ERR_ARG
    assert lib.resize_texture_create(None, buf.data_ptr(), 256, 16, 64, 4) == rz.RZ_ERR_ARG
    assert lib.resize_texture_create(ctypes.byref(h), buf.data_ptr(), 256, 16, 64, 4) == rz.RZ_OK
    assert lib.resize_texture_u8(h, buf.data_ptr() + 65536, 10, 8, 32, None) == rz.RZ_ERR_ARG
    assert lib.resize_texture_u8(h, buf.data_ptr() + 65536, 128, 0, 32, None) == rz.RZ_OK
    assert lib.resize_texture_destroy(h) == rz.RZ_OK
    assert lib.resize_texture_destroy(None) == rz.RZ_OK
    assert dev == torch.cuda.current_device()
