"""ctypes declarations of the C ABI in include/gbresize.h.

Loading fails loudly (``RuntimeError``) when ``libgbresize.so`` has not been
built; there is no other implementation to fall back on.
"""
from __future__ import annotations

import ctypes
import os

from ._build import library_path

RZ_NEAREST = 0
RZ_LINEAR = 1
RZ_U8 = 0
RZ_F32 = 1
RZ_EPI_NORMALIZE_NCHW = 1
RZ_EPI_FILTER3X3 = 2
RZ_EPI_GRAY_RGB = 3
RZ_EPI_GRAY_BGR = 4
RZ_EPI_FILTER = 5
RZ_BORDER_CLAMP = 0
RZ_BORDER_MIRROR = 1
RZ_BORDER_WRAP = 2
RZ_OK = 0
RZ_ERR_ARG = 1
RZ_ERR_UNSUPPORTED = 2
RZ_ERR_CUDA = 3
RZ_ERR_NOMEM = 4
RZ_ERR_TIMEOUT = 5
RZ_MAX_DIM = 65536
RZ_NOALLOC_MAX_DIM = 8192

RZ_OPT_STAGES = 1
RZ_OPT_GENERIC_ONLY = 2
RZ_OPT_CTAS_PER_SM = 3
RZ_OPT_GRID_MODE = 4
RZ_OPT_PDL = 5
RZ_OPT_RING_ROWS = 6
RZ_OPT_U8_KERNEL = 7
RZ_OPT_FILTER_KERNEL = 8
RZ_OPT_F32_KERNEL = 9
RZ_OPT_L2_PREFETCH = 10

RZ_FILTER_AUTO = 0
RZ_FILTER_FP32 = 1
RZ_FILTER_TENSOR = 2

RZ_COPY_PDL = 1
RZ_COPY_L2_PREFETCH = 2

# kernel families for resize_plan_set_tile
KIND_U8 = 0
KIND_F32 = 1
KIND_NORMALIZE = 2 + RZ_EPI_NORMALIZE_NCHW
KIND_FILTER3X3 = 2 + RZ_EPI_FILTER3X3


class RzEpilogue(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int),
        ("batch", ctypes.c_int),
        ("src_batch_stride", ctypes.c_size_t),
        ("dst_batch_stride", ctypes.c_size_t),
        ("mean", ctypes.c_float * 4),
        ("std", ctypes.c_float * 4),
        ("w3x3", ctypes.c_float * 9),
        ("ksize", ctypes.c_int),
        ("wk", ctypes.c_float * 49),
    ]


_p = ctypes.c_void_p
_sz = ctypes.c_size_t
_i = ctypes.c_int


class RzJob(ctypes.Structure):
    _fields_ = [
        ("src", ctypes.c_void_p),
        ("dst", ctypes.c_void_p),
        ("src_pitch", ctypes.c_size_t),
        ("dst_pitch", ctypes.c_size_t),
        ("H", ctypes.c_int),
        ("W", ctypes.c_int),
        ("out_h", ctypes.c_int),
        ("out_w", ctypes.c_int),
    ]


RZ_MULTI_MAX_JOBS = 2048

# name -> (restype, argtypes); every symbol include/gbresize.h declares
SIGNATURES = {
    "resize_plan_create": (_i, [ctypes.POINTER(_p), _i, _i, _i, _i, _i, _p]),
    "resize_plan_create_border": (_i, [ctypes.POINTER(_p), _i, _i, _i, _i, _i, _i, _p]),
    "resize_plan_destroy": (_i, [_p]),
    "resize_plan_status": (_i, [_p, ctypes.POINTER(_i)]),
    "resize_plan_set_tile": (_i, [_p, _i, _i, _i]),
    "resize_plan_set_option": (_i, [_p, _i, _i]),
    "resize_u8": (_i, [_p, _p, _sz, _p, _sz, _i, _i, _i, _i, _i, _i, _p]),
    "resize_f32": (_i, [_p, _p, _sz, _p, _sz, _i, _i, _i, _i, _i, _i, _p]),
    "resize_u8_batch": (_i, [_p, _p, _sz, _sz, _p, _sz, _sz, _i, _i, _i, _i, _i, _i, _i, _p]),
    "resize_wait_selftest": (_i, [_p, _i, _p]),
    "resize_f32_batch": (_i, [_p, _p, _sz, _sz, _p, _sz, _sz, _i, _i, _i, _i, _i, _i, _i, _p]),
    "resize_fused": (_i, [_p, _p, _i, _sz, _p, _sz, _i, _i, _i, _i, _i, _i, ctypes.POINTER(RzEpilogue), _p]),
    "resize_u8_host": (_i, [_p, _p, _sz, _p, _sz, _p, _sz, _p, _sz, _i, _i, _i, _i, _i, _i, _p]),
    "filter2d_valid_f32": (_i, [_p, _sz, _i, _i, _p, _i, _p, _sz, _p]),
    "filter2d_valid_f32_ex": (_i, [_p, _sz, _i, _i, _p, _i, _p, _sz, _i, _p, _p]),
    "resize_u8_multi": (_i, [_p, _i, _i, _i, _p, _p]),
    "resize_texture_create": (_i, [ctypes.POINTER(_p), _p, _sz, _i, _i, _i]),
    "resize_texture_u8": (_i, [_p, _p, _sz, _i, _i, _p]),
    "resize_texture_destroy": (_i, [_p]),
    "resize_axis_table": (_i, [_i, _i, _i, _p, _p, _p]),
    "resize_axis_table_border": (_i, [_i, _i, _i, _i, _p, _p, _p]),
    "resize_strerror": (ctypes.c_char_p, [_i]),
    "resize_last_cuda_error": (_i, []),
    "resize_u8_noalloc": (_i, [_p, _sz, _p, _sz, _i, _i, _i, _i, _i, _i, _p]),
    "resize_copy_baseline": (_i, [_p, _p, _sz, _i, _p]),
}

_lib = None
_lib_checked = None


def load() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def load_checked() -> ctypes.CDLL:
    """The bounds-checked variant of the library (libgbresize_checked.so, built
    by _build.build(checked=True)), with the same signatures: a test tool,
    not used by the package's functions."""
    global _lib_checked
    if _lib_checked is not None:
        return _lib_checked
    path = library_path(checked=True)
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with _build.build(checked=True)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib_checked = lib
    return lib
