"""CPU oracle for image resize — TEST INFRASTRUCTURE ONLY.

This package wraps the plain single-threaded C oracle in ``oracle.c`` with
ctypes.  Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import it; the library under
``bilinear_image_resize_gb300/`` never does, and it shares no code with it.

Every function takes numpy arrays and returns numpy arrays.  Pitches are in
bytes.  See ``oracle.c`` for the definitions and the passages they follow.
"""
from __future__ import annotations

import ctypes

import numpy as np

from ._build import build

_lib = None

_i64 = ctypes.c_int64
_int = ctypes.c_int
_p = ctypes.c_void_p


def _load():
    global _lib
    if _lib is not None:
        return _lib
    path = build()          # compiles only when oracle.c is newer than the library
    lib = ctypes.CDLL(path)
    lib.oracle_linear_coord.argtypes = [_i64, _i64, _i64, ctypes.POINTER(_i64),
                                        ctypes.POINTER(_i64), ctypes.POINTER(_i64)]
    lib.oracle_linear_coord.restype = None
    lib.oracle_weight_q11.argtypes = [_i64, _i64]
    lib.oracle_weight_q11.restype = _i64
    lib.oracle_nearest_index.argtypes = [_i64, _i64, _i64]
    lib.oracle_nearest_index.restype = _i64
    lib.oracle_border_index.argtypes = [_i64, _i64, _int]
    lib.oracle_border_index.restype = _i64
    lib.oracle_nearest_u8.argtypes = [_p, _i64, _int, _int, _int, _p, _i64, _int, _int]
    lib.oracle_nearest_u8.restype = None
    lib.oracle_linear_u8.argtypes = [_p, _i64, _int, _int, _int, _p, _i64, _int, _int, _int]
    lib.oracle_linear_u8.restype = None
    lib.oracle_linear_u8_rows.argtypes = [_p, _i64, _int, _int, _int, _p, _i64, _int, _int, _int, _int]
    lib.oracle_linear_u8_rows.restype = None
    lib.oracle_linear_u8_border_rows.argtypes = [_p, _i64, _int, _int, _int, _p, _i64, _int, _int, _int, _int,
                                                 _int]
    lib.oracle_linear_u8_border_rows.restype = None
    lib.oracle_linear_f32.argtypes = [_p, _i64, _int, _int, _int, _p, _int, _int, _int]
    lib.oracle_linear_f32.restype = None
    lib.oracle_gray_u8.argtypes = [_p, _i64, _int, _int, _int, _int, _p, _i64]
    lib.oracle_gray_u8.restype = None
    lib.oracle_filter_valid.argtypes = [_p, _int, _int, _p, _int, _p]
    lib.oracle_filter_valid.restype = None
    lib.oracle_filter_centred.argtypes = [_p, _int, _int, _p, _int, _p]
    lib.oracle_filter_centred.restype = None
    lib.oracle_nearest_f32.argtypes = [_p, _i64, _int, _int, _int, _p, _int, _int]
    lib.oracle_nearest_f32.restype = None
    lib.oracle_normalize_nchw.argtypes = [_p, _int, _int, _int, _p, _p, _p]
    lib.oracle_normalize_nchw.restype = None
    lib.oracle_filter3x3.argtypes = [_p, _int, _int, _p, _p]
    lib.oracle_filter3x3.restype = None
    _lib = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _as_hwc(img: np.ndarray) -> np.ndarray:
    if img.ndim == 2:
        img = img[:, :, None]
    if img.ndim != 3:
        raise ValueError("image must be HxW or HxWxC")
    # rows may be padded (a pitch wider than W*C) but pixels must be packed
    if img.strides[2] != img.itemsize or img.strides[1] != img.shape[2] * img.itemsize:
        img = np.ascontiguousarray(img)
    return img


def linear_coord(n_in: int, n_out: int, d: int):
    """(i, r, den) with x = i + r/den the sampling position of output index d."""
    i, r, den = _i64(), _i64(), _i64()
    _load().oracle_linear_coord(n_in, n_out, d, ctypes.byref(i), ctypes.byref(r), ctypes.byref(den))
    return i.value, r.value, den.value


def weight_q11(r: int, den: int) -> int:
    """round-half-up(2048 * r / den)."""
    return _load().oracle_weight_q11(r, den)


def nearest_index(n_in: int, n_out: int, d: int) -> int:
    return _load().oracle_nearest_index(n_in, n_out, d)


# border rules (CUDA interpolation page §6.1)
BORDER_CLAMP, BORDER_MIRROR, BORDER_WRAP = 0, 1, 2


def border_index(k: int, n: int, border: int) -> int:
    """Index k of an axis of n samples mapped inside by the border rule."""
    return _load().oracle_border_index(k, n, border)


def linear_u8(src: np.ndarray, out_h: int, out_w: int, border: int = BORDER_CLAMP) -> np.ndarray:
    """u8 bilinear resize of an HxW or HxWxC image; returns (out_h, out_w, C) u8."""
    s = _as_hwc(np.asarray(src))
    assert s.dtype == np.uint8 and border in (0, 1, 2)
    H, W, C = s.shape
    dst = np.empty((out_h, out_w, C), np.uint8)
    _load().oracle_linear_u8(_ptr(s), s.strides[0], H, W, C, _ptr(dst), dst.strides[0], out_h, out_w, border)
    return dst


def linear_u8_rows(src: np.ndarray, out_h: int, out_w: int, dy0: int, dy1: int,
                   border: int = BORDER_CLAMP) -> np.ndarray:
    """Output rows [dy0, dy1) of the u8 bilinear resize to (out_h, out_w); shape (dy1-dy0, out_w, C)."""
    s = _as_hwc(np.asarray(src))
    assert s.dtype == np.uint8 and 0 <= dy0 <= dy1 <= out_h and border in (0, 1, 2)
    H, W, C = s.shape
    full = np.empty((dy1 - dy0, out_w, C), np.uint8)
    # rows dy0.. land at the start of `full`: shift the destination base back by dy0 rows
    base = full.ctypes.data - dy0 * full.strides[0]
    _load().oracle_linear_u8_border_rows(_ptr(s), s.strides[0], H, W, C, base, full.strides[0], out_h, out_w,
                                         border, dy0, dy1)
    return full


def nearest_u8(src: np.ndarray, out_h: int, out_w: int) -> np.ndarray:
    s = _as_hwc(np.asarray(src))
    assert s.dtype == np.uint8
    H, W, C = s.shape
    dst = np.empty((out_h, out_w, C), np.uint8)
    _load().oracle_nearest_u8(_ptr(s), s.strides[0], H, W, C, _ptr(dst), dst.strides[0], out_h, out_w)
    return dst


def linear_f32(src: np.ndarray, out_h: int, out_w: int, border: int = BORDER_CLAMP) -> np.ndarray:
    """f32 bilinear resize evaluated in double; returns (out_h, out_w, C) float64."""
    s = _as_hwc(np.asarray(src))
    assert s.dtype == np.float32 and border in (0, 1, 2)
    H, W, C = s.shape
    dst = np.empty((out_h, out_w, C), np.float64)
    _load().oracle_linear_f32(_ptr(s), s.strides[0], H, W, C, _ptr(dst), out_h, out_w, border)
    return dst


def nearest_f32(src: np.ndarray, out_h: int, out_w: int) -> np.ndarray:
    s = _as_hwc(np.asarray(src))
    assert s.dtype == np.float32
    H, W, C = s.shape
    dst = np.empty((out_h, out_w, C), np.float32)
    _load().oracle_nearest_f32(_ptr(s), s.strides[0], H, W, C, _ptr(dst), out_h, out_w)
    return dst


def normalize_nchw(q: np.ndarray, mean, std) -> np.ndarray:
    """(q/255 - mean[c]) / std[c] of a dense HxWxC u8 image, as (C, H, W) float64."""
    q = np.ascontiguousarray(q)
    if q.ndim == 2:
        q = q[:, :, None]
    OH, OW, C = q.shape
    m = np.ascontiguousarray(np.asarray(mean, np.float64)[:C])
    sd = np.ascontiguousarray(np.asarray(std, np.float64)[:C])
    out = np.empty((C, OH, OW), np.float64)
    _load().oracle_normalize_nchw(_ptr(q), OH, OW, C, _ptr(m), _ptr(sd), _ptr(out))
    return out


def filter3x3(r: np.ndarray, w) -> np.ndarray:
    """3x3 replicate-border correlation of a single-channel float64 image."""
    r = np.ascontiguousarray(np.asarray(r, np.float64))
    if r.ndim == 3:
        assert r.shape[2] == 1
        r = r[:, :, 0]
    OH, OW = r.shape
    wd = np.ascontiguousarray(np.asarray(w, np.float64).reshape(9))
    z = np.empty((OH, OW), np.float64)
    _load().oracle_filter3x3(_ptr(r), OH, OW, _ptr(wd), _ptr(z))
    return z


def linear_f32_filter3x3(src: np.ndarray, out_h: int, out_w: int, w) -> np.ndarray:
    """The fused op's definition: filter3x3(linear_f32(src)), all in double."""
    return filter3x3(linear_f32(src, out_h, out_w), w)


def linear_u8_normalize(src: np.ndarray, out_h: int, out_w: int, mean, std,
                        border: int = BORDER_CLAMP) -> np.ndarray:
    """The fused op's definition: normalize_nchw(linear_u8(src))."""
    return normalize_nchw(linear_u8(src, out_h, out_w, border), mean, std)


def gray_u8(src: np.ndarray, bgr: bool = False) -> np.ndarray:
    """Grayscale (H, W) u8 of an HxWxC u8 image, C >= 3 (channel order RGB, or BGR)."""
    s = _as_hwc(np.asarray(src))
    assert s.dtype == np.uint8 and s.shape[2] >= 3
    H, W, C = s.shape
    dst = np.empty((H, W), np.uint8)
    _load().oracle_gray_u8(_ptr(s), s.strides[0], H, W, C, int(bool(bgr)), _ptr(dst), dst.strides[0])
    return dst


def gray_resize_u8(src: np.ndarray, out_h: int, out_w: int, linear: bool = True, bgr: bool = False,
                   border: int = BORDER_CLAMP) -> np.ndarray:
    """The fused op's definition: resize(gray_u8(src)), shape (out_h, out_w) u8."""
    g = gray_u8(src, bgr)
    if linear:
        return linear_u8(g, out_h, out_w, border)[:, :, 0]
    return nearest_u8(g, out_h, out_w)[:, :, 0]


def filter_valid(img: np.ndarray, w) -> np.ndarray:
    """K x K correlation over the valid region of a single-channel image, in
    double; shape (H - K + 1, W - K + 1)."""
    a = np.ascontiguousarray(np.asarray(img, np.float64))
    if a.ndim == 3:
        assert a.shape[2] == 1
        a = np.ascontiguousarray(a[:, :, 0])
    wk = np.ascontiguousarray(np.asarray(w, np.float64))
    K = wk.shape[0]
    assert wk.shape == (K, K) and a.shape[0] >= K and a.shape[1] >= K
    H, W = a.shape
    out = np.empty((H - K + 1, W - K + 1), np.float64)
    _load().oracle_filter_valid(_ptr(a), H, W, _ptr(wk), K, _ptr(out))
    return out


def filter_centred(r: np.ndarray, w) -> np.ndarray:
    """Odd K x K replicate-border correlation of a single-channel image, in double."""
    a = np.ascontiguousarray(np.asarray(r, np.float64))
    if a.ndim == 3:
        assert a.shape[2] == 1
        a = np.ascontiguousarray(a[:, :, 0])
    wk = np.ascontiguousarray(np.asarray(w, np.float64))
    K = wk.shape[0]
    assert wk.shape == (K, K) and K % 2 == 1
    OH, OW = a.shape
    z = np.empty((OH, OW), np.float64)
    _load().oracle_filter_centred(_ptr(a), OH, OW, _ptr(wk), K, _ptr(z))
    return z


def linear_f32_filter(src: np.ndarray, out_h: int, out_w: int, w, border: int = BORDER_CLAMP) -> np.ndarray:
    """The fused K x K op's definition: filter_centred(linear_f32(src)), all in double."""
    return filter_centred(linear_f32(src, out_h, out_w, border), w)
