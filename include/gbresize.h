/*
 * gbresize — image resize for NVIDIA GB300 (sm_103a), C ABI.
 *
 * Operations (the method these calls implement):
 *  - bilinear resize, OpenCV INTER_LINEAR style: output pixel (dx, dy) samples
 *    the input at x = (dx + 1/2) * W / OW - 1/2, y = (dy + 1/2) * H / OH - 1/2
 *    ("From Prototype to Performance: Optimizing OpenCV Resize on Volcanic
 *    GPUs", section "Naive resize with linear sampling": the output coordinate
 *    plus 0.5 times the inverse scale, fed to a linear sampler whose texel
 *    centres sit at +0.5), with weights (1-u)(1-v), u(1-v), (1-u)v, uv on the
 *    four neighbours (CUDA interpolation page, hnwysp.cn/news/129086, §2.2)
 *    and neighbour indices clamped into the image (same page, §6.1);
 *  - nearest resize, OpenCV INTER_NEAREST: source index floor(dx * W / OW)
 *    (CUDA interpolation page §2.1, read as OpenCV's floor rule);
 *  - border rules for bilinear taps outside the source: clamp, mirror, wrap
 *    (same page, §6.1; resize_plan_create_border);
 *  - epilogues fused into the resize (CUDA interpolation page §4.2, operator
 *    fusion): per-channel normalisation to float32 planar (NCHW); an odd K x K
 *    float filter, 3x3 included (correlation, replicate border on the output
 *    grid; "OpenCL image convolution", §2); grayscale conversion before the
 *    resize ("Performance Optimization of Object Tracking Algorithms in
 *    OpenCV on GPUs", §3.1.1);
 *  - beside the method: the standalone K x K correlation over the valid
 *    region, many geometries in one launch, a texture-unit comparison path
 *    and an allocation-free uint8 entry.
 *
 * Numerics:
 *  - uint8 bilinear is exact integer arithmetic: 11-bit weights
 *    A1 = round-half-up(2048 u), A0 = 2048 - A1 (and B0/B1 for v), the four
 *    products summed in int32 and rounded half-up once, (sum + 2^21) >> 22
 *    (CUDA interpolation page §6.2, fixed point).  The result is bit-exact
 *    and independent of evaluation order.
 *  - float32 bilinear uses weights u = r / den computed exactly in double on
 *    the host and rounded once to float; max abs error about 5e-5 on values
 *    in [0, 255].
 *  - nearest is a copy (bit-exact for both types).
 *
 * Layout: images are row-major, interleaved HWC, with an explicit row pitch in
 * BYTES (pitch >= W * C * sizeof(element); any value, odd pitches included).
 * C is 1, 3 or 4.  All image pointers are DEVICE pointers unless a call says
 * otherwise; the caller owns them.  Sizes follow OpenCV's dsize convention
 * only in spirit: every call takes heights and widths separately.
 *
 * Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 * default stream).  Every resize call is asynchronous on that stream, does
 * not allocate, and does not synchronise the host.
 *
 * Errors: every call returns an RZ_* status.  Arguments are validated before
 * anything is launched; a rejected call has no effect.  RZ_ERR_CUDA means a
 * CUDA runtime call failed; resize_last_cuda_error() gives its cudaError_t
 * (per host thread).  The library never aborts, prints or throws.
 *
 * Threads: a plan may be used from several host threads and streams at once;
 * calls on different streams that write the same output race, as any CUDA
 * work would.
 */
#ifndef GBRESIZE_H
#define GBRESIZE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Symbols of the C ABI keep default visibility; everything else in the
 * library is hidden. */
#if defined(__GNUC__)
#define RZ_API __attribute__((visibility("default")))
#else
#define RZ_API
#endif

#define RZ_NEAREST 0
#define RZ_LINEAR 1

#define RZ_U8 0
#define RZ_F32 1

#define RZ_EPI_NORMALIZE_NCHW 1
#define RZ_EPI_FILTER3X3 2
#define RZ_EPI_GRAY_RGB 3
#define RZ_EPI_GRAY_BGR 4
#define RZ_EPI_FILTER 5

/* Border rules for taps outside the source (CUDA interpolation page §6.1). */
#define RZ_BORDER_CLAMP 0   /* the edge sample repeats                          */
#define RZ_BORDER_MIRROR 1  /* reflection about the edge samples: index -1 reads
                               sample 1, index n reads sample n-2              */
#define RZ_BORDER_WRAP 2    /* the image repeats: index -1 reads n-1, n reads 0 */

#define RZ_OK 0
#define RZ_ERR_ARG 1          /* bad pointer, size, pitch, mode or overlap     */
#define RZ_ERR_UNSUPPORTED 2  /* valid but not implemented (e.g. C = 2)        */
#define RZ_ERR_CUDA 3         /* a CUDA runtime call failed                    */
#define RZ_ERR_NOMEM 4        /* host or device allocation failed (plans only) */
#define RZ_ERR_TIMEOUT 5      /* a kernel gave up waiting on a bulk copy       */

/* Largest accepted height or width, input or output. */
#define RZ_MAX_DIM 65536

/* Opaque plan: per-column and per-row sampling tables for one geometry
 * (H x W -> OH x OW) and one mode, resident in device memory. */
typedef struct rz_plan_s *rz_plan;

/*
 * Build the sampling tables of one geometry and mode.
 *
 * For RZ_LINEAR, per output column dx:  num = (2dx + 1) W - OW,  den = 2 OW,
 * xofs = floor(num / den),  r = num - xofs * den,  u = r / den; the uint8
 * weight a1 = round-half-up(2048 r / den); columns whose left tap falls left
 * of 0 or whose right tap falls right of W-1 are folded onto one clamped tap
 * (a1 = 0, u = 0), which gives exactly the values of clamping both taps.
 * The same per output row (yofs, b1, v).  For RZ_NEAREST, xn = floor(dx W / OW)
 * and yn = floor(dy H / OH).  Sampling position: Volcanic resize page,
 * "Naive resize with linear sampling"; weights: CUDA interpolation page §2.2
 * and §6.2; nearest: §2.1; output size int(in * scale) is the caller's
 * choice (Volcanic page, "Step 2").
 *
 * in_h, in_w >= 1; out_h, out_w >= 0; all <= RZ_MAX_DIM; mode RZ_LINEAR or
 * RZ_NEAREST.  Allocates device memory for the tables and a status word and
 * copies them on `stream` (asynchronously); the plan may be used on any stream
 * once that copy has completed (synchronise `stream` first, or use the same
 * stream).  On success *out receives the plan; on failure *out is NULL.
 */
RZ_API int resize_plan_create(rz_plan *out, int in_h, int in_w, int out_h, int out_w, int mode, void *stream);

/*
 * resize_plan_create with a border rule for bilinear taps outside the source
 * (RZ_BORDER_CLAMP, RZ_BORDER_MIRROR or RZ_BORDER_WRAP; CUDA interpolation
 * page §6.1).  Each tap's integer index is mapped by the rule; the weights
 * stay those of the unmapped position.  Only upscaled axes sample outside
 * (the sampled position lies in [-1/2, n - 1/2]), so the rule changes
 * nothing on downscales, and nothing for RZ_NEAREST (indices are always
 * inside).  A one-sample axis reads its sample under every rule.
 *
 * Table forms (resize_axis_table_border): under MIRROR the two taps stay
 * adjacent, so an edge column is stored as that adjacent pair (xofs 0 or
 * n - 2, a1 = 2048 - the unmapped a1, u = 1 - the unmapped u); under WRAP an
 * edge column is stored as xofs = n - 1 with its unmapped weight and the far
 * tap is index 0.  WRAP plans run on the direct-load kernels only: the 3x3
 * filter epilogue, and RZ_OPT_U8_KERNEL values 1 and 2, return
 * RZ_ERR_UNSUPPORTED for them.
 */
RZ_API int resize_plan_create_border(rz_plan *out, int in_h, int in_w, int out_h, int out_w, int mode, int border,
                                     void *stream);

/* Free a plan (NULL is accepted).  Synchronises the device first so that no
 * queued kernel still reads the tables. */
RZ_API int resize_plan_destroy(rz_plan p);

/*
 * Read and clear the plan's device status word (RZ_OK, or RZ_ERR_TIMEOUT if a
 * kernel using this plan gave up waiting on a bulk copy).  Synchronises the
 * device.  *status may be NULL.
 */
RZ_API int resize_plan_status(rz_plan p, int *status);

/*
 * uint8 resize of one interleaved image.
 *   src, dst: device pointers; src_pitch, dst_pitch: bytes between rows.
 *   H, W, out_h, out_w and mode must equal the plan's; C in {1, 3, 4}.
 *   src_pitch >= W*C, dst_pitch >= out_w*C; the source and destination byte
 *   ranges must not overlap.
 * Output (dx, dy, c) is written at dst + dy*dst_pitch + dx*C + c; bytes of a
 * row beyond out_w*C are not touched.  Bilinear is bit-exact with the
 * definition above; nearest is a byte copy.
 */
RZ_API int resize_u8(rz_plan p, const uint8_t *src, size_t src_pitch, uint8_t *dst, size_t dst_pitch,
              int H, int W, int C, int out_h, int out_w, int mode, void *stream);

/* float32 resize; as resize_u8 with 4-byte elements (pitches still in bytes,
 * multiples of 4). */
RZ_API int resize_f32(rz_plan p, const float *src, size_t src_pitch, float *dst, size_t dst_pitch,
               int H, int W, int C, int out_h, int out_w, int mode, void *stream);

/*
 * Batched forms: `batch` images of the plan's geometry in one launch (one
 * kernel walks the tiles of all of them, so a stream of frames pays the
 * launch's fixed start-up and drain once per batch instead of once per
 * frame).  Image n starts at src + n*src_batch_stride and
 * dst + n*dst_batch_stride (bytes); with batch > 1 the strides must cover an
 * image (src_batch_stride >= (H-1)*src_pitch + W*C*element size, likewise
 * dst) and the float32 strides must be multiples of 4.  No source image may
 * overlap any destination image.  batch = 0 does nothing; batch = 1 is the
 * single-image call (strides ignored).  Results per image equal the
 * single-image call's.
 */
RZ_API int resize_u8_batch(rz_plan p, const uint8_t *src, size_t src_pitch, size_t src_batch_stride, uint8_t *dst,
                           size_t dst_pitch, size_t dst_batch_stride, int batch, int H, int W, int C, int out_h,
                           int out_w, int mode, void *stream);
RZ_API int resize_f32_batch(rz_plan p, const float *src, size_t src_pitch, size_t src_batch_stride, float *dst,
                            size_t dst_pitch, size_t dst_batch_stride, int batch, int H, int W, int C, int out_h,
                            int out_w, int mode, void *stream);

/*
 * Epilogue fused into the bilinear kernel (CUDA interpolation page §4.2;
 * kernel merging leaves results unchanged, "Performance Optimization of Object
 * Tracking Algorithms in OpenCV on GPUs", §4.2 and Table 10).
 *
 * RZ_EPI_NORMALIZE_NCHW: src uint8 HWC, dst float32 planar.  The uint8
 *   bilinear result q is computed exactly as resize_u8 does and written as
 *   y = (q / 255 - mean[c]) / std[c], evaluated in float32 as
 *   fmaf(q, 1 / (255 std[c]), -mean[c] / std[c]) with both constants rounded
 *   once from double on the host.  Element (c, dy, dx) of image n lands at
 *   dst + n*dst_batch_stride + c*out_h*dst_pitch + dy*dst_pitch + dx*4, so
 *   dst_pitch is the byte pitch of one plane row (>= out_w*4, multiple of 4).
 *   Images are `batch` frames src + n*src_batch_stride.
 * RZ_EPI_FILTER3X3: src and dst float32 HWC.  z = sum_{a,b in -1..1}
 *   w3x3[(a+1)*3 + (b+1)] * r[clamp(dy+a)][clamp(dx+b)] where r is the float32
 *   bilinear result on the output grid and clamp keeps rows in [0, out_h-1]
 *   and columns in [0, out_w-1] (replicate border).  Each channel is filtered
 *   on its own.  Batch as above (plane layout is HWC here).
 * RZ_EPI_GRAY_RGB / RZ_EPI_GRAY_BGR: src uint8 HWC with C = 3 or 4 channels
 *   (R, G, B in that order, or B, G, R; a fourth channel is ignored), dst
 *   uint8 single-channel (dst_pitch >= out_w).  The conversion to grayscale
 *   that precedes the resize in OpenCV's detection preprocessing ("Performance
 *   Optimization of Object Tracking Algorithms in OpenCV on GPUs", §3.1.1):
 *   each source pixel's gray value Y = floor((299 R + 587 G + 114 B + 500) /
 *   1000), i.e. the BT.601 weights 0.299, 0.587, 0.114 rounded half-up
 *   exactly, then the uint8 resize of the gray image (bilinear or nearest,
 *   the plan's mode and border), so the result equals resize_u8 of the
 *   converted image bit for bit.  Batch as above.
 * RZ_EPI_FILTER: the 3x3 rule for any odd ksize K in 1..7: src and dst
 *   float32 HWC, z = sum_{a,b in -K/2..K/2} wk[(a+K/2)*K + (b+K/2)] *
 *   r[clamp(dy+a)][clamp(dx+b)], each channel on its own, replicate border
 *   on the output grid.  K = 3 gives RZ_EPI_FILTER3X3's result.  Any border
 *   rule of the plan.
 *
 * batch >= 0 (0 is a no-op); batch strides are bytes and must keep the frames
 * from overlapping when batch > 1.
 */
typedef struct {
    int kind;
    int batch;
    size_t src_batch_stride;
    size_t dst_batch_stride;
    float mean[4];
    float std[4];
    float w3x3[9];
    int ksize;        /* RZ_EPI_FILTER: K (odd, 1..7) */
    float wk[49];     /* RZ_EPI_FILTER: K x K weights, row-major */
} rz_epilogue;

/*
 * Resize with an epilogue.  src_dtype is RZ_U8 for RZ_EPI_NORMALIZE_NCHW and
 * the gray kinds, RZ_F32 for RZ_EPI_FILTER3X3 and RZ_EPI_FILTER; mode must be RZ_LINEAR except
 * for the gray kinds (either mode).  Other arguments as resize_u8/resize_f32.
 * std[c] must be non-zero and finite.
 */
RZ_API int resize_fused(rz_plan p, const void *src, int src_dtype, size_t src_pitch, void *dst, size_t dst_pitch,
                 int H, int W, int C, int out_h, int out_w, int mode, const rz_epilogue *e, void *stream);

/*
 * Many independent uint8 resizes of different geometries in ONE launch, for
 * small frames whose own launches would each cost more than their work
 * (kernel-call overhead: "Performance Optimization of Object Tracking
 * Algorithms in OpenCV on GPUs" §4.2; batching launches: CUDA interpolation
 * page §8.1).  Each job resizes src (H x W x C interleaved, src_pitch bytes
 * per row) into dst (out_h x out_w x C, dst_pitch bytes per row) exactly as
 * resize_u8 with a clamp-border plan of that geometry does (bit-identical);
 * no plan is needed: sampling positions and weights are computed in the
 * kernel.  All jobs share C (1, 3 or 4) and mode.
 *
 * dev_jobs: DEVICE array of njobs descriptors (caller-owned, read by the
 * kernel; fill it once and the launch can be captured and replayed in a
 * graph).  0 <= njobs <= RZ_MULTI_MAX_JOBS.  A job whose fields are invalid
 * (null pointers, sizes outside 1..RZ_MAX_DIM for the source or 0..RZ_MAX_DIM
 * for the output, pitches below the row bytes; an empty output's pointers
 * and pitches are not checked) is skipped and RZ_ERR_ARG is
 * written to *dev_status (a caller-owned device int, may be NULL); the other
 * jobs still run.  Jobs must not overlap one another's outputs or write
 * their own inputs.  Asynchronous on `stream`; no allocation.
 */
typedef struct {
    const uint8_t *src;
    uint8_t *dst;
    size_t src_pitch;
    size_t dst_pitch;
    int H, W, out_h, out_w;
} rz_job;
#define RZ_MULTI_MAX_JOBS 2048
RZ_API int resize_u8_multi(const rz_job *dev_jobs, int njobs, int C, int mode, int *dev_status, void *stream);

/*
 * Hardware-filtered bilinear resize, a comparison path: the texture unit's
 * linear filtering sampled at (dst + 0.5) * in / out with clamped addressing
 * ("From Prototype to Performance: Optimizing OpenCV Resize on Volcanic
 * GPUs", *Naive resize with linear sampling*; CUDA interpolation page §4.1).
 * Its weights have about 8 fractional bits, so results may differ from
 * resize_u8 (and the oracle) by a unit or so; resize_u8 is the exact path.
 *
 * resize_texture_create binds a texture object to the caller's uint8 image
 * (device memory, C = 1 or 4 interleaved channels; C = 3 has no texture
 * format: RZ_ERR_UNSUPPORTED).  The base must be aligned to the device's
 * texture alignment and src_pitch a multiple of its texture pitch alignment
 * (cudaDevAttrTextureAlignment / cudaDevAttrTexturePitchAlignment);
 * otherwise RZ_ERR_ARG.  The image must stay allocated
 * while the handle lives.  resize_texture_u8 resizes it into dst (out_w * C
 * bytes per row at dst_pitch), asynchronously on `stream`, no allocation.
 * resize_texture_destroy synchronises the device and frees the handle.
 */
typedef struct rz_tex_s *rz_tex;
RZ_API int resize_texture_create(rz_tex *out, const uint8_t *src, size_t src_pitch, int H, int W, int C);
RZ_API int resize_texture_u8(rz_tex t, uint8_t *dst, size_t dst_pitch, int out_h, int out_w, void *stream);
RZ_API int resize_texture_destroy(rz_tex t);

/*
 * K x K correlation over the valid region ("OpenCL image convolution" §2):
 *   dst[y][x] = sum_{r, c in [0, K)} w[r*K + c] * src[y + r][x + c]
 * for 0 <= y <= H - K, 0 <= x <= W - K (the filter's first row and column on
 * the output position; no flip).  float32, one channel; src and dst rows at
 * byte pitches (multiples of 4, src_pitch >= W*4, dst_pitch >= (W-K+1)*4);
 * weights: DEVICE pointer to K*K floats, row-major, read during the call's
 * kernel.  1 <= K <= 64 (RZ_ERR_UNSUPPORTED above); H, W <= RZ_MAX_DIM.
 * H < K or W < K gives an
 * empty output (RZ_OK, nothing launched).  Asynchronous on `stream`; no
 * allocation; src and dst must not overlap.  Results are float32 sums in an
 * order of the kernel's choosing (within K*K float32 roundings of the exact
 * sum).
 */
RZ_API int filter2d_valid_f32(const float *src, size_t src_pitch, int H, int W, const float *weights, int K,
                              float *dst, size_t dst_pitch, void *stream);

/*
 * filter2d_valid_f32 with the kernel chosen by the caller (for tests and
 * measurements; filter2d_valid_f32 is kernel = RZ_FILTER_AUTO, dev_status =
 * NULL).  RZ_FILTER_FP32: the FP32 FMA kernel (any layout of the arguments
 * above).  RZ_FILTER_TENSOR: the tensor-core kernel (tcgen05 MMAs on TF32
 * operands, each float split into a TF32 high part and the remainder, three
 * products per tap pair summed in float32: the float32 result within the
 * bound stated above); it needs src 16-byte aligned and src_pitch a multiple
 * of 16, and 16 <= K (RZ_ERR_UNSUPPORTED otherwise).  RZ_FILTER_AUTO: the tensor cores
 * for K >= 48 where their layout conditions hold, FP32 otherwise.
 * dev_status: optional caller-owned device int; the tensor-core kernel's
 * bounded waits (1 s) write RZ_ERR_TIMEOUT there when one gives up (the
 * word is not cleared by the call).  Unknown kernel values: RZ_ERR_ARG.
 */
#define RZ_FILTER_AUTO 0
#define RZ_FILTER_FP32 1
#define RZ_FILTER_TENSOR 2
RZ_API int filter2d_valid_f32_ex(const float *src, size_t src_pitch, int H, int W, const float *weights, int K,
                                 float *dst, size_t dst_pitch, int kernel, int *dev_status, void *stream);

/*
 * End-to-end uint8 resize from HOST memory: copies the image from
 * host_src (pitch host_src_pitch) into the caller's device buffer dev_src
 * (pitch dev_src_pitch), resizes it into dev_dst (pitch dev_dst_pitch) and
 * copies the result back to host_dst (pitch host_dst_pitch), all queued on
 * `stream` (asynchronous; page-locked host memory makes the copies overlap
 * other work).  Allocates nothing; the caller provides both device buffers.
 * The host buffers must stay valid until the stream reaches the end of the
 * call's work.
 */
RZ_API int resize_u8_host(rz_plan p, const uint8_t *host_src, size_t host_src_pitch, uint8_t *host_dst,
                   size_t host_dst_pitch, uint8_t *dev_src, size_t dev_src_pitch, uint8_t *dev_dst,
                   size_t dev_dst_pitch, int H, int W, int C, int out_h, int out_w, int mode, void *stream);

/*
 * Host-only: fill the tables resize_plan_create would upload, for tests and
 * tools.  Any output pointer may be NULL.  For RZ_LINEAR: ofs[n_out] (int32),
 * w_q11[n_out] (int32, 0..2048), u[n_out] (float).  For RZ_NEAREST only ofs is
 * written.  n_in >= 1, 0 <= n_out, both <= RZ_MAX_DIM.  No CUDA call is made.
 */
RZ_API int resize_axis_table(int n_in, int n_out, int mode, int32_t *ofs, int32_t *w_q11, float *u);

/* resize_axis_table under a border rule (the table forms described at
 * resize_plan_create_border). */
RZ_API int resize_axis_table_border(int n_in, int n_out, int mode, int border, int32_t *ofs, int32_t *w_q11,
                                    float *u);

/*
 * Self-test of the bounded waits the staged and streaming kernels use on
 * their shared-memory barriers: launches one CTA whose thread waits on a
 * barrier that nothing completes, for at most limit_us microseconds
 * (1..1000000), and writes RZ_ERR_TIMEOUT to *dev_status (caller-owned
 * device memory; RZ_OK is written first) when the wait gives up.
 * Asynchronous on `stream`.  It makes failure reporting testable without
 * faulting or hanging a GPU; the pages have no counterpart.
 */
RZ_API int resize_wait_selftest(int *dev_status, int limit_us, void *stream);

/*
 * The 1:1 copy baseline (Volcanic page, "From Prototype to Performance:
 * Optimizing OpenCV Resize on Volcanic GPUs", *Kernel evolution -> Baseline:
 * simple 1:1 copy behavior*): copies `bytes` bytes from src to dst (device
 * memory) with no resize arithmetic, in the launch shape of the exact-ratio
 * resize kernels (256-thread CTAs, one 16-byte load and store per thread),
 * so that a resize's time can be set against what a launch moving the same
 * bytes reaches on this GPU.  flags: RZ_COPY_PDL launches it as a
 * programmatic dependent launch (as the resizes are by default);
 * RZ_COPY_L2_PREFETCH makes each CTA prefetch its source span into L2 before
 * waiting for the previous kernel (as RZ_OPT_L2_PREFETCH does for the
 * resizes).  src and dst 16-byte aligned, bytes a multiple of 16, the ranges
 * disjoint, unknown flag bits unset: otherwise RZ_ERR_ARG.  bytes = 0 is a
 * no-op.  Asynchronous on `stream`; no allocation.
 */
#define RZ_COPY_PDL 1
#define RZ_COPY_L2_PREFETCH 2
RZ_API int resize_copy_baseline(const void *src, void *dst, size_t bytes, int flags, void *stream);

/* Human-readable name of a status code (static string). */
RZ_API const char *resize_strerror(int code);

/* cudaError_t of the last RZ_ERR_CUDA returned on this host thread (0 if none). */
RZ_API int resize_last_cuda_error(void);

/*
 * Tile override for tuning (0 = automatic): output rows and output columns
 * per CTA for kernel family `kind` (RZ_U8, RZ_F32, or 2 + RZ_EPI_* for the
 * normalise and filter kernels) of this plan.  Results do not depend on it; only speed does.
 * For the streaming kernels (the filter family, uint8 bilinear upscales)
 * a tile is one streamed unit: tile_rows output rows of a strip of tile_cols
 * output columns (at most the kernel's widest strip).  A tile that does not
 * fit in shared memory makes the next call of that family fail with
 * RZ_ERR_ARG (RZ_ERR_UNSUPPORTED for the filter family).
 */
RZ_API int resize_plan_set_tile(rz_plan p, int kind, int tile_rows, int tile_cols);

/*
 * Tuning and testing options of a plan (results never depend on them):
 *   RZ_OPT_STAGES       value 0 (automatic) or 1..4: source tiles each CTA
 *                       keeps in flight ahead of the one it computes (all
 *                       families but the filters, which stream rows);
 *   RZ_OPT_GENERIC_ONLY value 0 or 1: 1 disables the exact-ratio fast path
 *                       (uint8 2x downscale, used only when every table entry
 *                       is the 2x pattern, where it is bit-identical);
 *   RZ_OPT_CTAS_PER_SM  value 0 (as many as fit) or 1..32: caps the resident
 *                       CTAs per SM of the persistent grid;
 *   RZ_OPT_GRID_MODE    value 0 (persistent CTAs, the default) or 1 (one CTA
 *                       per output tile);
 *   RZ_OPT_PDL          value 1 (default) or 0: launch as a programmatic
 *                       dependent launch, so that a resize queued right after
 *                       another kernel on the same stream starts its set-up
 *                       while that kernel finishes (it still reads and writes
 *                       memory only after that kernel has completed);
 *   RZ_OPT_RING_ROWS    value 0 (automatic) or 2..128: source rows in the
 *                       shared-memory ring through which each CTA of a
 *                       streaming kernel (the filter family; uint8
 *                       bilinear upscales) streams its strip;
 *   RZ_OPT_U8_KERNEL    value 0 (automatic), 1, 2 or 3: which kernel runs
 *                       uint8-source resizes (plain, and the normalise
 *                       epilogue).  0: vertical bilinear upscales to at
 *                       least 2^18 output pixels streamed (each source row's
 *                       horizontal sums computed once, kept in registers),
 *                       everything else with direct
 *                       loads (each thread reads its own taps; the exact 2x
 *                       case with vector loads when the source base, pitch
 *                       and batch stride are multiples of 16 bytes, 8 for
 *                       three channels, and the output ones of 8, 4 for three
 *                       channels); 1: staged tiles always; 2: streamed
 *                       whenever a strip's source span fits (not the exact 2x
 *                       case or the normalise epilogue); 3: direct loads
 *                       always (upscales with each thread walking output
 *                       rows, tile_rows of resize_plan_set_tile per thread).
 *                       Bit-exact whichever runs;
 *   RZ_OPT_FILTER_KERNEL value 0 (automatic), 1 or 2: which kernel runs the
 *                       filter epilogues (RZ_EPI_FILTER3X3, RZ_EPI_FILTER).
 *                       0: streaming for K = 3, 5, 7, the tile kernel for
 *                       K = 1 and under RZ_BORDER_WRAP; 1: streaming
 *                       (RZ_ERR_UNSUPPORTED for K = 1 or under wrap); 2: the
 *                       tile kernel.  Equal within float32 rounding;
 *   RZ_OPT_F32_KERNEL   value 0 (automatic) or 1: which kernel runs the plain
 *                       float32 bilinear resize under the clamp and mirror
 *                       rules.  0: the streaming kernel (source rows streamed
 *                       once through shared memory), unless a float32 tile
 *                       override is set; 1: staged tiles.  Same arithmetic;
 *   RZ_OPT_L2_PREFETCH  value 1 (default) or 0: the exact-ratio uint8 kernels
 *                       (2x down, bilinear, nearest and gray; 3:2 down; 2x
 *                       up) and the any-ratio direct-load one ask for the
 *                       source rows each CTA reads to be
 *                       moved into L2 as soon as the CTA is resident, before
 *                       it waits for the previous kernel in the stream (with
 *                       RZ_OPT_PDL, while that kernel finishes).  A prefetch
 *                       is a hint and changes no result.
 * Returns RZ_ERR_ARG for an unknown option or value.
 */
#define RZ_OPT_STAGES 1
#define RZ_OPT_GENERIC_ONLY 2
#define RZ_OPT_CTAS_PER_SM 3
#define RZ_OPT_GRID_MODE 4
#define RZ_OPT_PDL 5
#define RZ_OPT_RING_ROWS 6
#define RZ_OPT_U8_KERNEL 7
#define RZ_OPT_FILTER_KERNEL 8
#define RZ_OPT_F32_KERNEL 9
#define RZ_OPT_L2_PREFETCH 10
RZ_API int resize_plan_set_option(rz_plan p, int option, int value);

/*
 * uint8 resize that allocates nothing, for callers that may not allocate
 * device memory themselves: a plugin whose device memory belongs to its host
 * framework's pooling allocator (a stray cudaMalloc there can fail under a
 * tight budget or wait on the device), or a real-time pipeline that forbids
 * allocation once it runs.  The pages have no counterpart; it is an addition
 * to the resize_plan_create / resize_u8 pair.
 *
 * Arguments, layout and results are those of resize_u8 (bit-identical
 * output), without a plan: src and dst are the caller's device buffers.  The
 * sampling tables and the kernel's status word live in one static device
 * array of about 128 KB that every GPU loading the library keeps until the
 * process exits; a small kernel rebuilds the tables on the device at the
 * start of each call.  No cudaMalloc, cudaFree or other allocating routine
 * is called.
 *   - out_h and out_w must not exceed RZ_NOALLOC_MAX_DIM: larger sizes return
 *     RZ_ERR_UNSUPPORTED before anything is queued.
 *   - All calls share the array.  Calls queued on one stream are ordered and
 *     safe; calls that overlap on the GPU (different streams running at the
 *     same time) race on the tables and may produce wrong results.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - `stream` must belong to the current device (RZ_ERR_ARG otherwise).
 *   - Kernel time-outs are not reported (there is no plan to hold a status).
 */
#define RZ_NOALLOC_MAX_DIM 8192
RZ_API int resize_u8_noalloc(const uint8_t *src, size_t src_pitch, uint8_t *dst, size_t dst_pitch, int H, int W,
                             int C, int out_h, int out_w, int mode, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GBRESIZE_H */
