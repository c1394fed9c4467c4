// Internal declarations shared by the host API (api.cu) and the kernels
// (kernels.cu).  Nothing here is part of the C ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include "gbresize.h"

namespace rz {

constexpr int kThreads = 256;           // threads per CTA, every kernel
constexpr int kMaxSmem = 227 * 1024;    // opt-in dynamic shared memory per CTA on sm_103a
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // bounded mbarrier waits: 1 s

// Kernel families.  The numbering matches resize_plan_set_tile's `kind`.
enum Family { FAM_U8 = 0, FAM_F32 = 1, FAM_NORM = 3, FAM_FILT = 4, FAM_COUNT = 5 };

__host__ __device__ inline int align_up(int v, int a) { return (v + a - 1) / a * a; }

__host__ __device__ inline int fam_in_es(int fam) { return (fam == FAM_U8 || fam == FAM_NORM) ? 1 : 4; }
__host__ __device__ inline int fam_out_es(int fam) { return fam == FAM_U8 ? 1 : 4; }
__host__ __device__ inline int fam_halo(int fam) { return fam == FAM_FILT ? 1 : 0; }

// Byte offsets of the pieces of a CTA's dynamic shared memory.  Host and
// device compute them with this one function.
struct SmemLayout {
    int off_rows;   // int[max_rows]: staged source row indices
    int off_map;    // int[2 * computed rows]: slot of the top / bottom tap row
    int off_slots;  // max_rows staged row segments of slot_bytes each
    int off_mid;    // float[(TR+2) * (TW+2) * C]: resized values incl. halo (3x3 only)
    int off_out;    // output tile, rows of out_row_bytes (planes for NCHW)
    int out_row_bytes;
    int total;
};
// header at offset 0: u64 mbarrier, then int nrows, int b_lo, int nbytes
constexpr int kHdrBytes = 32;

__host__ __device__ inline SmemLayout smem_layout(int fam, int C, int TR, int TW, int max_rows, int slot_bytes)
{
    SmemLayout L;
    const int halo = fam_halo(fam);
    const int nrc = TR + 2 * halo;
    L.off_rows = kHdrBytes;
    L.off_map = align_up(L.off_rows + 4 * max_rows, 16);
    L.off_slots = align_up(L.off_map + 8 * nrc, 128);
    L.off_mid = L.off_slots + max_rows * slot_bytes;
    const int mid = halo ? (TR + 2) * (TW + 2) * C * 4 : 0;
    L.off_out = align_up(L.off_mid + mid, 128);
    if (fam == FAM_NORM) {
        L.out_row_bytes = align_up(TW * 4, 16);
        L.total = L.off_out + C * TR * L.out_row_bytes;
    } else {
        L.out_row_bytes = align_up(TW * C * fam_out_es(fam), 16);
        L.total = L.off_out + TR * L.out_row_bytes;
    }
    return L;
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
    int max_rows;           // staged source rows reserved per tile
    int slot_bytes;         // bytes reserved per staged row
    int tma_in, tma_out;    // bulk copies allowed for loads / stores
    const int2 *xt;         // per output column {source column, weight}
    const int2 *yt;         // per output row    {source row, weight}
    int *status;            // device status word (RZ_OK or RZ_ERR_TIMEOUT)
    float scale[4], shift[4];  // normalise epilogue: y = q * scale[c] + shift[c]
    float w[9];                // 3x3 epilogue weights, row-major
};

// Launch one resize kernel (asynchronous).  Returns a cudaError_t value.
int launch_resize(int fam, int mode, const KArgs &a, int batch, size_t smem, void *stream);

}  // namespace rz
