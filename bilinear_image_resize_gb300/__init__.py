"""GB300-native image resize: Python binding of the C ABI (include/gbresize.h).

Every function here only marshals arguments (torch tensors -> device pointers,
byte pitches, the current CUDA stream) and calls the C entry point of the
same name; all computation runs in the library's CUDA kernels.  A non-zero
status raises ``ResizeError``.

Images are torch tensors laid out HWC (or HW for one channel) with the last
two dimensions packed; the row pitch is taken from ``stride(0)``, so row
padding (a view into a wider buffer) is allowed.
"""
from __future__ import annotations

import ctypes

from . import _native
from ._native import (KIND_F32, KIND_FILTER3X3, KIND_NORMALIZE, KIND_U8, RZ_BORDER_CLAMP, RZ_BORDER_MIRROR,
                      RZ_BORDER_WRAP, RZ_EPI_FILTER, RZ_EPI_FILTER3X3, RZ_EPI_GRAY_BGR, RZ_EPI_GRAY_RGB, RZ_EPI_NORMALIZE_NCHW, RZ_ERR_ARG, RZ_ERR_CUDA, RZ_ERR_NOMEM, RZ_ERR_TIMEOUT,
                      RZ_ERR_UNSUPPORTED, RZ_F32, RZ_LINEAR, RZ_MAX_DIM, RZ_NEAREST, RZ_NOALLOC_MAX_DIM, RZ_OK,
                      RZ_OPT_CTAS_PER_SM, RZ_OPT_GENERIC_ONLY, RZ_OPT_GRID_MODE, RZ_OPT_PDL, RZ_OPT_RING_ROWS,
                      RZ_MULTI_MAX_JOBS, RZ_OPT_F32_KERNEL, RZ_OPT_FILTER_KERNEL, RZ_OPT_L2_PREFETCH, RZ_COPY_PDL, RZ_COPY_L2_PREFETCH, RZ_FILTER_AUTO, RZ_FILTER_FP32, RZ_FILTER_TENSOR, RZ_OPT_STAGES, RZ_OPT_U8_KERNEL, RZ_U8,
                      RzEpilogue, RzJob)

__all__ = [
    "ResizeError", "Plan", "resize_plan_create", "resize_plan_destroy", "resize_plan_status",
    "resize_plan_set_tile", "resize_plan_set_option", "resize_u8", "resize_f32", "resize_u8_batch",
    "resize_f32_batch", "resize_fused", "resize_u8_host", "resize_wait_selftest",
    "resize_axis_table", "resize_strerror", "resize_last_cuda_error", "make_epilogue", "resize_u8_noalloc",
    "RZ_NOALLOC_MAX_DIM",
    "RZ_LINEAR", "RZ_NEAREST", "RZ_U8", "RZ_F32", "RZ_EPI_NORMALIZE_NCHW", "RZ_EPI_FILTER3X3",
    "RZ_EPI_GRAY_RGB", "RZ_EPI_GRAY_BGR", "RZ_BORDER_CLAMP", "RZ_BORDER_MIRROR", "RZ_BORDER_WRAP",
    "resize_plan_create_border", "resize_axis_table_border", "RZ_EPI_FILTER", "RZ_OPT_FILTER_KERNEL", "RZ_OPT_F32_KERNEL",
    "filter2d_valid_f32", "Texture", "resize_texture_create", "make_jobs", "resize_u8_multi",
    "RZ_MULTI_MAX_JOBS",
    "RZ_OK", "RZ_ERR_ARG", "RZ_ERR_UNSUPPORTED", "RZ_ERR_CUDA", "RZ_ERR_NOMEM", "RZ_ERR_TIMEOUT",
    "RZ_MAX_DIM", "KIND_U8", "KIND_F32", "KIND_NORMALIZE", "KIND_FILTER3X3",
    "RZ_OPT_STAGES", "RZ_OPT_GENERIC_ONLY", "RZ_OPT_CTAS_PER_SM", "RZ_OPT_GRID_MODE", "RZ_OPT_PDL",
    "RZ_OPT_RING_ROWS", "RZ_OPT_U8_KERNEL", "RZ_OPT_L2_PREFETCH",
    "resize_copy_baseline", "RZ_COPY_PDL", "RZ_COPY_L2_PREFETCH",
    "RZ_FILTER_AUTO", "RZ_FILTER_FP32", "RZ_FILTER_TENSOR",
]


class ResizeError(RuntimeError):
    def __init__(self, code: int, where: str):
        lib = _native.load()
        msg = lib.resize_strerror(code).decode()
        if code == RZ_ERR_CUDA:
            msg += f" (cudaError {lib.resize_last_cuda_error()})"
        super().__init__(f"{where}: {msg} [status {code}]")
        self.code = code


def _check(code: int, where: str) -> None:
    if code != RZ_OK:
        raise ResizeError(code, where)


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Plan:
    """Owns an ``rz_plan`` handle; freed by ``resize_plan_destroy`` or on collection."""

    def __init__(self, handle: int, in_h: int, in_w: int, out_h: int, out_w: int, mode: int,
                 border: int = RZ_BORDER_CLAMP):
        self.handle = handle
        self.in_h, self.in_w, self.out_h, self.out_w, self.mode = in_h, in_w, out_h, out_w, mode
        self.border = border

    def destroy(self) -> None:
        if self.handle:
            h, self.handle = self.handle, None
            _check(_native.load().resize_plan_destroy(h), "resize_plan_destroy")

    def __del__(self):
        try:
            if self.handle:
                _native.load().resize_plan_destroy(self.handle)
                self.handle = None
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.destroy()


def resize_plan_create(in_h: int, in_w: int, out_h: int, out_w: int, mode: int = RZ_LINEAR, stream=None,
                       border: int = RZ_BORDER_CLAMP) -> Plan:
    if border != RZ_BORDER_CLAMP:
        return resize_plan_create_border(in_h, in_w, out_h, out_w, mode, border, stream)
    h = ctypes.c_void_p()
    _check(_native.load().resize_plan_create(ctypes.byref(h), in_h, in_w, out_h, out_w, mode, _stream(stream)),
           "resize_plan_create")
    return Plan(h.value, in_h, in_w, out_h, out_w, mode)


def resize_plan_create_border(in_h: int, in_w: int, out_h: int, out_w: int, mode: int, border: int,
                              stream=None) -> Plan:
    h = ctypes.c_void_p()
    _check(_native.load().resize_plan_create_border(ctypes.byref(h), in_h, in_w, out_h, out_w, mode, border,
                                                    _stream(stream)), "resize_plan_create_border")
    return Plan(h.value, in_h, in_w, out_h, out_w, mode, border)


def resize_plan_destroy(plan: Plan) -> None:
    plan.destroy()


def resize_plan_status(plan: Plan) -> int:
    st = ctypes.c_int(-1)
    _check(_native.load().resize_plan_status(plan.handle, ctypes.byref(st)), "resize_plan_status")
    return st.value


def resize_plan_set_tile(plan: Plan, kind: int, tile_rows: int, tile_cols: int) -> None:
    _check(_native.load().resize_plan_set_tile(plan.handle, kind, tile_rows, tile_cols), "resize_plan_set_tile")


def resize_plan_set_option(plan: Plan, option: int, value: int) -> None:
    _check(_native.load().resize_plan_set_option(plan.handle, option, value), "resize_plan_set_option")


def _hwc(t, name):
    """(H, W, C, pitch_bytes) of an HWC/HW tensor whose pixels are packed."""
    if t.dim() == 2:
        H, W = t.shape
        C = 1
        if t.stride(1) != 1:
            raise ValueError(f"{name}: columns must be contiguous")
    elif t.dim() == 3:
        H, W, C = t.shape
        if (C > 1 and t.stride(2) != 1) or t.stride(1) != C:
            raise ValueError(f"{name}: pixels must be packed (stride(1) == C, stride(2) == 1)")
    else:
        raise ValueError(f"{name}: expected HxW or HxWxC, got shape {tuple(t.shape)}")
    return H, W, C, t.stride(0) * t.element_size()


def resize_u8(plan: Plan, src, dst, mode: int | None = None, stream=None) -> None:
    """dst[:] = resize(src) for uint8 tensors (H, W[, C]) -> (OH, OW[, C])."""
    H, W, C, sp = _hwc(src, "src")
    OH, OW, C2, dp = _hwc(dst, "dst")
    if C2 != C:
        raise ValueError("src and dst channel counts differ")
    _check(_native.load().resize_u8(plan.handle, src.data_ptr(), sp, dst.data_ptr(), dp, H, W, C, OH, OW,
                                    plan.mode if mode is None else mode, _stream(stream)), "resize_u8")


def resize_u8_noalloc(src, dst, mode: int = RZ_LINEAR, stream=None) -> None:
    """dst[:] = resize(src) for uint8 tensors without a plan and without any
    device allocation (tables in the library's static device array; see
    include/gbresize.h for the size limit and the sharing rules)."""
    H, W, C, sp = _hwc(src, "src")
    OH, OW, C2, dp = _hwc(dst, "dst")
    if C2 != C:
        raise ValueError("src and dst channel counts differ")
    _check(_native.load().resize_u8_noalloc(src.data_ptr(), sp, dst.data_ptr(), dp, H, W, C, OH, OW, mode,
                                            _stream(stream)), "resize_u8_noalloc")


def resize_f32(plan: Plan, src, dst, mode: int | None = None, stream=None) -> None:
    """dst[:] = resize(src) for float32 tensors (H, W[, C]) -> (OH, OW[, C])."""
    H, W, C, sp = _hwc(src, "src")
    OH, OW, C2, dp = _hwc(dst, "dst")
    if C2 != C:
        raise ValueError("src and dst channel counts differ")
    _check(_native.load().resize_f32(plan.handle, src.data_ptr(), sp, dst.data_ptr(), dp, H, W, C, OH, OW,
                                     plan.mode if mode is None else mode, _stream(stream)), "resize_f32")


def _nhwc(t, name):
    """(N, H, W, C, pitch_bytes, batch_stride_bytes) of an NHWC tensor whose pixels are packed."""
    if t.dim() != 4:
        raise ValueError(f"{name}: expected NxHxWxC, got shape {tuple(t.shape)}")
    N, H, W, C = t.shape
    if (C > 1 and t.stride(3) != 1) or t.stride(2) != C:
        raise ValueError(f"{name}: pixels must be packed (stride(2) == C, stride(3) == 1)")
    es = t.element_size()
    return N, H, W, C, t.stride(1) * es, t.stride(0) * es


def _batch(fn_name, plan, src, dst, mode, stream):
    N, H, W, C, sp, sb = _nhwc(src, "src")
    N2, OH, OW, C2, dp, db = _nhwc(dst, "dst")
    if N2 != N or C2 != C:
        raise ValueError("src and dst batch or channel counts differ")
    _check(getattr(_native.load(), fn_name)(plan.handle, src.data_ptr(), sp, sb, dst.data_ptr(), dp, db, N, H, W, C,
                                            OH, OW, plan.mode if mode is None else mode, _stream(stream)), fn_name)


def resize_u8_batch(plan: Plan, src, dst, mode: int | None = None, stream=None) -> None:
    """dst[n] = resize(src[n]) for uint8 tensors (N, H, W, C) -> (N, OH, OW, C), one launch."""
    _batch("resize_u8_batch", plan, src, dst, mode, stream)


def resize_f32_batch(plan: Plan, src, dst, mode: int | None = None, stream=None) -> None:
    """dst[n] = resize(src[n]) for float32 tensors (N, H, W, C) -> (N, OH, OW, C), one launch."""
    _batch("resize_f32_batch", plan, src, dst, mode, stream)


def resize_wait_selftest(dev_status, limit_us: int, stream=None) -> None:
    """Launch the bounded-wait self-test: dev_status (a one-element int32 CUDA
    tensor) receives RZ_ERR_TIMEOUT when the wait gives up after limit_us."""
    _check(_native.load().resize_wait_selftest(dev_status.data_ptr(), limit_us, _stream(stream)),
           "resize_wait_selftest")


def make_epilogue(kind: int, batch: int = 1, src_batch_stride: int = 0, dst_batch_stride: int = 0,
                  mean=(0.0, 0.0, 0.0, 0.0), std=(1.0, 1.0, 1.0, 1.0), w3x3=None, wk=None) -> RzEpilogue:
    """An rz_epilogue; wk is a K x K weight array (odd K <= 7) for RZ_EPI_FILTER."""
    e = RzEpilogue()
    e.kind, e.batch = kind, batch
    e.src_batch_stride, e.dst_batch_stride = src_batch_stride, dst_batch_stride
    for i in range(4):
        e.mean[i] = float(mean[i]) if i < len(mean) else 0.0
        e.std[i] = float(std[i]) if i < len(std) else 1.0
    if w3x3 is not None:
        for i in range(9):
            e.w3x3[i] = float(w3x3[i])
    if wk is not None:
        rows = [list(r) for r in wk]
        e.ksize = len(rows)
        flat = [float(v) for r in rows for v in r]
        if len(flat) != e.ksize * e.ksize or e.ksize > 7:
            raise ValueError("wk must be a square array of at most 7 x 7 weights")
        for i, v in enumerate(flat):
            e.wk[i] = v
    return e


def resize_fused(plan: Plan, src, dst, epilogue: RzEpilogue, stream=None) -> None:
    """Resize with a fused epilogue.

    RZ_EPI_NORMALIZE_NCHW: src uint8 (N, H, W, C) or (H, W, C); dst float32
    (N, C, OH, OW) or (C, OH, OW).  RZ_EPI_FILTER3X3: src and dst float32
    (N, H, W, C) / (H, W, C) / (H, W).  RZ_EPI_GRAY_RGB / RZ_EPI_GRAY_BGR:
    src uint8 (N, H, W, C) or (H, W, C) with C = 3 or 4, dst uint8 (N, OH, OW)
    or (OH, OW), in the plan's mode.  The epilogue's batch and batch strides
    are filled in from the tensors.
    """
    import torch
    e = RzEpilogue.from_buffer_copy(epilogue)
    batched = src.dim() == 4
    s = src if batched else src.unsqueeze(0)
    mode = RZ_LINEAR
    if e.kind in (RZ_EPI_GRAY_RGB, RZ_EPI_GRAY_BGR):
        d = dst if dst.dim() == 3 else dst.unsqueeze(0)
        N, OH, OW = d.shape
        C = s.shape[3]
        if d.stride(2) != 1:
            raise ValueError("dst rows must be contiguous")
        dp = d.stride(1)
        dtype_code = RZ_U8
        mode = plan.mode
        if s.dtype != torch.uint8 or d.dtype != torch.uint8:
            raise ValueError("gray epilogue takes uint8 src and dst")
    elif e.kind == RZ_EPI_NORMALIZE_NCHW:
        d = dst if dst.dim() == 4 else dst.unsqueeze(0)
        N, C, OH, OW = d.shape
        if d.stride(3) != 1 or d.stride(1) != OH * d.stride(2):
            raise ValueError("dst planes must be rows of contiguous floats with planes stacked by rows")
        dp = d.stride(2) * 4
        dtype_code = RZ_U8
        if s.dtype != torch.uint8 or d.dtype != torch.float32:
            raise ValueError("normalise epilogue takes uint8 src and float32 dst")
    elif e.kind in (RZ_EPI_FILTER3X3, RZ_EPI_FILTER):
        if not batched and src.dim() == 2:
            s = src.unsqueeze(0).unsqueeze(-1)
            d = dst.unsqueeze(0).unsqueeze(-1)
        else:
            d = dst if dst.dim() == 4 else dst.unsqueeze(0)
        N, OH, OW, C = d.shape
        dp = d.stride(1) * 4
        dtype_code = RZ_F32
        if s.dtype != torch.float32 or d.dtype != torch.float32:
            raise ValueError("filter epilogues take float32 src and dst")
    else:
        raise ValueError(f"unknown epilogue kind {e.kind}")
    Nb, H, W, Cs = s.shape
    if Nb != N or Cs != C:
        raise ValueError("src and dst batch or channel counts differ")
    if (C > 1 and s.stride(3) != 1) or s.stride(2) != C:
        raise ValueError("src pixels must be packed")
    e.batch = N
    e.src_batch_stride = s.stride(0) * s.element_size()
    e.dst_batch_stride = d.stride(0) * d.element_size()
    _check(_native.load().resize_fused(plan.handle, s.data_ptr(), dtype_code, s.stride(1) * s.element_size(),
                                       d.data_ptr(), dp, H, W, C, OH, OW, mode, ctypes.byref(e),
                                       _stream(stream)), "resize_fused")


def filter2d_valid_f32(src, weights, dst, stream=None, kernel: int = RZ_FILTER_AUTO, status=None) -> None:
    """dst[:] = the K x K correlation of src over its valid region.

    src: float32 CUDA tensor (H, W) with contiguous rows; weights: float32
    CUDA tensor (K, K); dst: float32 CUDA tensor (H - K + 1, W - K + 1).
    kernel: RZ_FILTER_AUTO, RZ_FILTER_FP32 or RZ_FILTER_TENSOR; status:
    optional int32 CUDA tensor for the tensor-core kernel's time-outs.
    """
    if src.dim() != 2 or dst.dim() != 2 or src.stride(1) != 1 or dst.stride(1) != 1:
        raise ValueError("src and dst must be 2-D with contiguous rows")
    K = weights.shape[0]
    if weights.dim() != 2 or weights.shape[1] != K or not weights.is_contiguous():
        raise ValueError("weights must be a contiguous K x K tensor")
    H, W = src.shape
    _check(_native.load().filter2d_valid_f32_ex(src.data_ptr(), src.stride(0) * 4, H, W, weights.data_ptr(), K,
                                                dst.data_ptr(), dst.stride(0) * 4, kernel,
                                                status.data_ptr() if status is not None else None, _stream(stream)),
           "filter2d_valid_f32")


def resize_copy_baseline(src, dst, flags: int = RZ_COPY_PDL | RZ_COPY_L2_PREFETCH, stream=None) -> None:
    """dst[:] = src, bytes moved by the library's 1:1 copy baseline kernel.

    src, dst: contiguous CUDA tensors of the same byte size (a multiple of
    16), 16-byte aligned, not overlapping.
    """
    if not (src.is_contiguous() and dst.is_contiguous()):
        raise ValueError("src and dst must be contiguous")
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("src and dst differ in byte size")
    _check(_native.load().resize_copy_baseline(src.data_ptr(), dst.data_ptr(), nbytes, flags, _stream(stream)),
           "resize_copy_baseline")


def make_jobs(srcs, dsts, device=None):
    """A device array of rz_job descriptors for resize_u8_multi from lists of
    uint8 HWC (or HW) CUDA tensors; returns (jobs tensor, C)."""
    import torch
    if len(srcs) != len(dsts):
        raise ValueError("srcs and dsts differ in length")
    arr = (_native.RzJob * max(1, len(srcs)))()
    C = None
    for k, (s, d) in enumerate(zip(srcs, dsts)):
        H, W, cs, sp = _hwc(s, "src")
        OH, OW, cd, dp = _hwc(d, "dst")
        if cs != cd or (C is not None and cs != C):
            raise ValueError("every job must have the same channel count")
        C = cs
        arr[k] = _native.RzJob(s.data_ptr(), d.data_ptr(), sp, dp, H, W, OH, OW)
    raw = bytes(memoryview(arr))[:ctypes.sizeof(_native.RzJob) * len(srcs)]
    dev = device if device is not None else (srcs[0].device if srcs else "cuda")
    jobs = torch.frombuffer(bytearray(raw), dtype=torch.uint8).to(dev) if raw else torch.empty(
        0, dtype=torch.uint8, device=dev)
    return jobs, (C or 1)


def resize_u8_multi(jobs, njobs: int, C: int, mode: int = RZ_LINEAR, status=None, stream=None) -> None:
    """Launch the jobs of a device job array (make_jobs) in one kernel;
    status: optional one-element int32 CUDA tensor receiving RZ_ERR_ARG when
    a job is invalid."""
    _check(_native.load().resize_u8_multi(jobs.data_ptr() if njobs else None, njobs, C, mode,
                                          status.data_ptr() if status is not None else None, _stream(stream)),
           "resize_u8_multi")


class Texture:
    """Owns an ``rz_tex`` handle (a texture object over a uint8 image); the
    image tensor is kept alive with it."""

    def __init__(self, src):
        H, W, C, pitch = _hwc(src, "src")
        h = ctypes.c_void_p()
        _check(_native.load().resize_texture_create(ctypes.byref(h), src.data_ptr(), pitch, H, W, C),
               "resize_texture_create")
        self.handle, self.src, self.C = h.value, src, C

    def resize(self, dst, stream=None) -> None:
        """dst[:] = the hardware-filtered bilinear resize of the image."""
        OH, OW, C, pitch = _hwc(dst, "dst")
        if C != self.C:
            raise ValueError("dst channels differ from the image's")
        _check(_native.load().resize_texture_u8(self.handle, dst.data_ptr(), pitch, OH, OW, _stream(stream)),
               "resize_texture_u8")

    def destroy(self) -> None:
        if self.handle:
            h, self.handle = self.handle, None
            _check(_native.load().resize_texture_destroy(h), "resize_texture_destroy")

    def __del__(self):
        try:
            if self.handle:
                _native.load().resize_texture_destroy(self.handle)
                self.handle = None
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.destroy()


def resize_texture_create(src) -> Texture:
    return Texture(src)


def resize_u8_host(plan: Plan, host_src, host_dst, dev_src, dev_dst, stream=None) -> None:
    """Host -> device copy, resize, device -> host copy, queued on one stream.

    host_src/host_dst are CPU tensors (page-locked for asynchronous copies);
    dev_src/dev_dst are the caller's device buffers of the same shapes.
    """
    H, W, C, hsp = _hwc(host_src, "host_src")
    OH, OW, _, hdp = _hwc(host_dst, "host_dst")
    _, _, _, dsp = _hwc(dev_src, "dev_src")
    _, _, _, ddp = _hwc(dev_dst, "dev_dst")
    _check(_native.load().resize_u8_host(plan.handle, host_src.data_ptr(), hsp, host_dst.data_ptr(), hdp,
                                         dev_src.data_ptr(), dsp, dev_dst.data_ptr(), ddp, H, W, C, OH, OW,
                                         plan.mode, _stream(stream)), "resize_u8_host")


def resize_axis_table(n_in: int, n_out: int, mode: int = RZ_LINEAR):
    """Host-only sampling table of one axis: (ofs int32, w_q11 int32, u float32) numpy arrays."""
    import numpy as np
    ofs = np.zeros(n_out, np.int32)
    w = np.zeros(n_out, np.int32)
    u = np.zeros(n_out, np.float32)
    _check(_native.load().resize_axis_table(n_in, n_out, mode, ofs.ctypes.data, w.ctypes.data, u.ctypes.data),
           "resize_axis_table")
    return ofs, w, u


def resize_axis_table_border(n_in: int, n_out: int, mode: int, border: int):
    """resize_axis_table under a border rule."""
    import numpy as np
    ofs = np.zeros(n_out, np.int32)
    w = np.zeros(n_out, np.int32)
    u = np.zeros(n_out, np.float32)
    _check(_native.load().resize_axis_table_border(n_in, n_out, mode, border, ofs.ctypes.data, w.ctypes.data,
                                                   u.ctypes.data), "resize_axis_table_border")
    return ofs, w, u


def resize_strerror(code: int) -> str:
    return _native.load().resize_strerror(code).decode()


def resize_last_cuda_error() -> int:
    return _native.load().resize_last_cuda_error()
