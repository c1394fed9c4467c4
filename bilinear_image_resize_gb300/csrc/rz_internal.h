// Internal declarations shared by the host API (api.cu) and the kernels
// (kernels.cu).  Nothing here is part of the C ABI.
#pragma once

#include <cuda.h>   // CUtensorMap (a plain struct; no driver library is linked)

#include <cstddef>
#include <cstdint>

#include "gbresize.h"

namespace rz {

constexpr int kConsumers = 256;         // compute threads per CTA (warps 0..7)
constexpr int kThreads = kConsumers + 32;  // plus one producer warp that stages tiles
// Bounds-checked build (compiled with -DRZ_CHECK_BOUNDS into a separate
// library, for tests): the kernels check their global and shared-memory
// accesses against the extents in KArgs and record RZ_ERR_ARG in the status
// word instead of making an access outside them.
#ifdef RZ_CHECK_BOUNDS
constexpr bool kCheckBounds = true;
#else
constexpr bool kCheckBounds = false;
#endif

// opt-in dynamic shared memory per CTA on sm_103a (the checked build keeps
// 256 bytes back for its static per-CTA bounds record)
constexpr int kMaxSmem = 227 * 1024 - (kCheckBounds ? 256 : 0);
constexpr int kMaxStages = 4;           // staged-tile ring depth limit
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // bounded mbarrier waits: 1 s

// Kernel families.  The numbering matches resize_plan_set_tile's `kind`
// (the gray family runs on direct-load kernels only and takes no tile).
enum Family { FAM_U8 = 0, FAM_F32 = 1, FAM_NORM = 3, FAM_FILT = 4, FAM_GRAY = 5, FAM_COUNT = 6 };

// Compute variants of the uint8 bilinear family.
enum Variant { VAR_GENERIC = 0, VAR_DOWN2 = 1 };

__host__ __device__ constexpr int align_up(int v, int a) { return (v + a - 1) / a * a; }

__host__ __device__ constexpr int fam_in_es(int fam) { return (fam == FAM_U8 || fam == FAM_NORM || fam == FAM_GRAY) ? 1 : 4; }
__host__ __device__ constexpr int fam_out_es(int fam) { return (fam == FAM_U8 || fam == FAM_GRAY) ? 1 : 4; }
__host__ __device__ constexpr int fam_halo(int fam) { return fam == FAM_FILT ? 1 : 0; }
// Families whose producer also stages the tile's sampling-table entries.
__host__ __device__ constexpr bool fam_tables_in_stage(int fam) { return fam == FAM_NORM; }
// Staged table entries: a tile's x (y) entries are copied in one bulk copy
// that starts on an even entry, so one entry of slack at each end.
__host__ __device__ constexpr int tab_x_entries(int TW) { return align_up(TW + 8, 2); }
__host__ __device__ constexpr int tab_y_entries(int TR) { return align_up(TR + 4, 2); }
// Entries before and after each of the plan's device tables that repeat the
// first and last entry, so that a tile's range of entries widened to even
// bounds (one bulk copy) stays inside the allocation and reads as the clamp.
constexpr int kTabPad = 8;

// Padding after each staged row: the uint8 bilinear tap reads are 32-bit
// words and may pass the end of a row's span by up to 11 bytes.
__host__ __device__ constexpr int fam_slot_pad(int fam) { return (fam == FAM_U8 || fam == FAM_NORM) ? 16 : 0; }

// Byte offsets of the pieces of a CTA's dynamic shared memory.  Host and
// device compute them with this one function.
//
//   [0, 128)                      per stage: a "full" and an "empty" mbarrier
//   (stages + 1) x plan_bytes     tile plans: header {nrows, b_lo, nbytes, tile, image,
//                                 table ranges}, int rows[max_rows], int map[2 * output rows]
//   stages x stage_bytes          staged tiles: table entries (normalise family), then
//                                 max_rows staged row segments of slot_bytes
//   2 x out_bytes                 double-buffered output tile
// The plan ring has one entry more than the stage ring, so the producer can
// plan the next tile while every stage is still in use.
struct SmemLayout {
    int plan_off, plan_bytes;
    int rows_off, map_off;       // within a plan
    int stage_off, stage_bytes;
    int tab_off, slots_off;      // within a stage
    int out_off, out_bytes, out_row_bytes;
    int total;
};

__host__ __device__ inline SmemLayout smem_layout(int fam, int C, int TR, int TW, int max_rows, int slot_bytes,
                                                  int stages)
{
    SmemLayout L;
    L.plan_off = 128;
    L.rows_off = 64;
    L.map_off = align_up(L.rows_off + 4 * max_rows, 16);
    L.plan_bytes = align_up(L.map_off + 8 * TR, 16);
    L.stage_off = align_up(L.plan_off + (stages + 1) * L.plan_bytes, 128);
    // the normalise family stages the tile's table entries too: x entries
    // for its columns (+ slack), then y entries for its rows
    const int tab = fam_tables_in_stage(fam) ? 8 * (tab_x_entries(TW) + tab_y_entries(TR)) : 0;
    L.tab_off = 0;
    L.slots_off = align_up(tab, 128);
    L.stage_bytes = align_up(L.slots_off + max_rows * slot_bytes, 128);
    L.out_off = L.stage_off + stages * L.stage_bytes;
    if (fam == FAM_NORM) {
        L.out_row_bytes = align_up(TW * 4, 16);
        L.out_bytes = align_up(C * TR * L.out_row_bytes, 128);
    } else {
        L.out_row_bytes = align_up(TW * C * fam_out_es(fam), 16);
        L.out_bytes = align_up(TR * L.out_row_bytes, 128);
    }
    L.total = L.out_off + 2 * L.out_bytes;
    return L;
}

// Streaming kernels (stream.cu): the K x K filter family and the uint8
// bilinear resize in row-separable form.  Units of TW output columns by TR
// output rows, whose source rows stream through a ring of chunks.  A chunk
// holds up to chunk_rows rows; each row's span is cut into chunk_boxes blocks
// of box_bytes (<= 2048, a multiple of 16), stored block-major: block k of
// row i at k * block_bytes + i * box_bytes, block_bytes = chunk_rows *
// box_bytes rounded up to 128.  Shared memory: ring_chunks "full" and
// ring_chunks "empty" mbarriers, the producer's list window, then the chunks.
enum StreamOp { STREAM_FILTER = 0, STREAM_U8 = 1 };
constexpr int kStreamChunkRows = 8;     // rows per chunk (a power of two)
constexpr int kStreamRingMax = 128;     // ring rows (chunks x rows per chunk)
constexpr int kStreamListWindow = 128;  // listed rows the producer keeps (ints)
// K x K filter: resized columns per consumer lane (four for one channel, else
// one); widest strip = eight consumer warps x (32 x lane columns - 2 K/2)
// outputs
__host__ __device__ constexpr int filter_lane_cols(int C) { return C == 1 ? 4 : 1; }
__host__ __device__ constexpr int filter_strip(int C, int R = 1) { return 8 * (32 * filter_lane_cols(C) - 2 * R); }
// uint8 bilinear: consecutive output pixels per consumer lane; widest strip
__host__ __device__ constexpr int stream_u8_run(int C) { return C == 4 ? 2 : 4; }
__host__ __device__ constexpr int stream_u8_strip(int C) { return 8 * 32 * stream_u8_run(C); }
__host__ __device__ constexpr int stream_block_bytes(int rows, int box_bytes) { return align_up(rows * box_bytes, 128); }
__host__ __device__ constexpr int stream_chunks_off(int chunks) { return align_up(16 * chunks + 4 * kStreamListWindow, 128); }
__host__ __device__ constexpr int stream_smem(int chunks, int rows, int boxes, int box_bytes)
{
    return stream_chunks_off(chunks) + chunks * boxes * stream_block_bytes(rows, box_bytes);
}

// Everything a resize kernel reads, passed by value in the parameter bank.
struct KArgs {
    const uint8_t *src;
    long long src_pitch;    // bytes between source rows
    long long src_bstride;  // bytes between source images of a batch
    uint8_t *dst;
    long long dst_pitch;    // bytes between output rows (plane rows for NCHW)
    long long dst_bstride;  // bytes between outputs of a batch
    long long dst_plane;    // bytes between planes (NCHW only)
    int H, W, OH, OW, C;
    int TR, TW;             // output rows / columns per tile
    int tiles_x, tiles_y;   // tiles per image
    int batch;              // images
    int max_rows;           // staged source rows reserved per tile
    int slot_bytes;         // bytes reserved per staged row
    int stages;             // depth of the staged-tile ring (1..kMaxStages)
    int tma_in, tma_out;    // bulk copies allowed for loads / stores
    int tensor_in;          // stage each tile with one tensor-map copy (box below)
    int box_words;          // box width in 8-byte words
    int box_rows;           // box height in rows
    int ring_chunks;        // streaming kernels: chunks in the ring (>= 2)
    int chunk_rows;         // streaming kernels: rows per chunk (1, 2, 4 or 8)
    int chunk_boxes;        // streaming kernels: blocks per row span
    int box_bytes;          // streaming kernels: bytes per block of a row
    const int2 *xt;         // per output column {source column, weight}; kTabPad clamped entries either side
    const int2 *yt;         // per output row    {source row, weight}; kTabPad clamped entries either side
    int *status;            // device status word (RZ_OK or RZ_ERR_TIMEOUT)
    int border;             // RZ_BORDER_*: the plan's rule for taps outside the source
    int bgr;                // gray epilogue: channels in B, G, R order
    float scale[4], shift[4];  // normalise epilogue: y = q * scale[c] + shift[c]
    float w[49];               // K x K epilogue weights (K <= 7), row-major
    int ksize;                 // K of the filter epilogue (3 for the 3x3 kind)
    int l2_prefetch;           // exact-ratio direct kernels: prefetch the CTA's source span into L2 before the dependency wait
    // extents for the bounds-checked build: bytes readable from src, bytes
    // writable from dst, the table block [tab, tab + tab_bytes)
    long long src_extent, dst_extent;
    const uint8_t *tab;
    long long tab_bytes;
};

// Record a cudaError_t for resize_last_cuda_error (this host thread).
void record_cuda_error(int e);

// Kernel entry for (family, mode, variant, C); nullptr if none.
const void *kernel_for(int fam, int mode, int variant, int C);

// The streaming kernel for (StreamOp, mode, C, filter halo R = K / 2);
// nullptr if none.
const void *stream_kernel_for(int op, int mode, int C, int R = 1);

// Launch it on grid x grid_y CTAs of `threads` (asynchronous), optionally as
// a programmatic dependent launch.  `tmap` describes the source when
// a.tensor_in is set (otherwise its contents are ignored).  Returns a
// cudaError_t value.
int launch_resize(const void *fn, const KArgs &a, const CUtensorMap &tmap, int grid, size_t smem, bool pdl,
                  void *stream, int threads = kThreads, int grid_y = 1);

// Exact 2x uint8 downscale: output pixels per group, 8 (C = 1), 4 (C = 3),
// 2 (C = 4), i.e. 8, 12, 8 output bytes from 16, 24, 16 source bytes of each
// of two rows.
__host__ __device__ constexpr int down2_px(int C) { return C == 1 ? 8 : (C == 3 ? 4 : 2); }

// One CTA waiting on a barrier nothing completes, at most limit_ns; writes
// RZ_ERR_TIMEOUT to *status when the wait gives up.  Returns a cudaError_t.
int launch_wait_selftest(int *status, unsigned long long limit_ns, void *stream);

// K x K filters (filter.cu).  Fused: odd K <= 7 after the float32 bilinear
// resize, output tiles of kFTW x kFTH with a K / 2 halo of resized values in
// shared memory.  Standalone: the valid-region correlation, 1 <= K <= 64,
// output tiles of kVTW columns by two rows per warp (eight columns a lane).
constexpr int kFilterThreads = 256;
constexpr int kFTW = 64, kFTH = 32;
constexpr int kVTW = 256;
constexpr int kMaxFilterK = 64;
__host__ __device__ constexpr int valid_threads(int K) { return K > 32 ? 512 : 256; }
__host__ __device__ constexpr int valid_tile_rows(int threads) { return 2 * threads / 32; }
__host__ __device__ constexpr int filter_valid_row_floats(int K) { return kVTW + ((K + 7) & ~7) + 8; }
__host__ __device__ constexpr int filter_valid_smem(int K, int threads)
{
    return 4 * ((valid_tile_rows(threads) + K - 1) * filter_valid_row_floats(K) + K * ((K + 7) & ~7));
}
const void *resize_filter_kernel_for(int C, int K, bool wrap);
int launch_filter_valid(const float *src, long long src_pitch, int H, int W, const float *w, int K, float *dst,
                        long long dst_pitch, bool pdl, void *stream);

// Many geometries in one launch (multi.cu): a persistent grid over the jobs'
// output row segments.  Returns a cudaError_t.
constexpr int kMultiMaxJobs = RZ_MULTI_MAX_JOBS;
int launch_multi(const rz_job *jobs, int njobs, int C, int mode, int *status, bool pdl, void *stream);

// Direct-load kernels (direct.cu): a thread per output group, no staging.
constexpr int kDirectThreads = 256;
// The exact 2x uint8 downscale (bilinear or nearest) for C channels; nullptr
// if none.
const void *direct_down2_kernel_for(int mode, int C);
// Any ratio, uint8 source: DIRECT_U8 (uint8 out) or DIRECT_NORM (normalise
// epilogue, float32 planes) for (mode, C); nullptr if none.
enum DirectOp { DIRECT_U8 = 0, DIRECT_NORM = 1 };
constexpr int kDirectRun = 4;   // output pixels per thread
constexpr int kNormRun = 1;     // normalise: output pixels per lane (interleaved by 32)
// WRAP: the plan's border rule is RZ_BORDER_WRAP (a far tap past the last
// sample reads sample 0).
const void *direct_kernel_for(int op, int mode, int C, bool wrap = false);
// Grayscale conversion then uint8 resize, C = 3 or 4 source channels; the
// exact 2x downscale form (four outputs per thread, vector loads).
const void *direct_gray_kernel_for(int mode, int C, bool wrap);
const void *direct_down2_gray_kernel_for(int mode, int C, bool bgr);
// float32 bilinear, a thread per output pixel (used for WRAP plans).
const void *direct_f32_kernel_for(int C, bool wrap);
// The exact 2x uint8 bilinear upscale (thread per 4 source columns of a
// source row: 8 x 2 outputs); nullptr if none.
constexpr int kUp2Cols = 4;
const void *direct_up2_kernel_for(int C, int border);
// The exact 2x upscale with pixel lanes, each thread walking a.TR source rows
// (three and four channels; nullptr otherwise).
const void *direct_up2_rows_kernel_for(int C, int border);
// The exact 3:2 uint8 bilinear downscale (thread per 8 outputs of a row from
// 12 x 2 source pixels); nullptr if none.
const void *direct_down32_kernel_for(int C);
// uint8 bilinear with each thread walking a.TR output rows (vertical
// upscales); nullptr if none.
const void *direct_rows_kernel_for(int C);

}  // namespace rz
