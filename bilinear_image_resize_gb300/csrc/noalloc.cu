// resize_u8_noalloc: the uint8 resize for callers that may not allocate
// device memory.
//
// resize_u8 reads its per-column and per-row sampling tables from memory a
// plan allocated with cudaMalloc.  This entry point needs no plan: the tables
// (and the status word the kernel reports time-outs in) live in one
// file-scope __device__ array, NoAllocScratch, filled on the device by a small
// kernel at the start of every call.  Nothing here calls cudaMalloc,
// cudaFree, operator new or any other allocating routine, on the host or the
// device.
//
// Limits and sharing: out_w and out_h are at most kNoAllocMaxDim.  Every GPU
// that loads the library holds one copy of the array (about 128 KB) until the
// process exits.  All calls share it and it keeps the last call's contents,
// so calls that overlap on the GPU (queued on different streams and running
// at the same time) race on it; calls on one stream are ordered and safe.
// The first call on a device looks up the array's device address
// (cudaGetSymbolAddress) with that device current; make that first call
// before any stream capture.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "gbresize.h"
#include "rz_internal.h"

namespace {

constexpr int kNoAllocMaxDim = RZ_NOALLOC_MAX_DIM;
constexpr int kMaxDevices = 64;

struct NoAllocScratch {
    // per output column {source column, 11-bit weight}; a staged tile's
    // paired table loads may read up to three entries past xt[out_w - 1],
    // which at out_w = kNoAllocMaxDim land in yt below (inside this struct;
    // the values are not used)
    int2 xt[kNoAllocMaxDim];
    int2 yt[kNoAllocMaxDim];   // per output row    {source row, 11-bit weight}
    int status;                // kernel status word (RZ_OK / RZ_ERR_TIMEOUT)
    int pad[63];
};

static __device__ __align__(256) NoAllocScratch g_noalloc_scratch;

// Table entry of output index d on an axis of n_in -> n_out samples, the
// same values the plan builds on the host: bilinear samples
// x = ((2d+1) n_in - n_out) / (2 n_out), left tap floor(x), far-tap weight
// round-half-up(2048 frac(x)), taps outside the image folded onto one clamped
// tap with weight 0; nearest takes floor(d n_in / n_out).
__device__ int2 table_entry(int n_in, int n_out, int d, bool linear)
{
    if (!linear) {
        long long s = static_cast<long long>(d) * n_in / n_out;
        if (s > n_in - 1) s = n_in - 1;
        return make_int2(static_cast<int>(s), 0);
    }
    const long long num = (2LL * d + 1) * n_in - n_out;
    const long long den = 2LL * n_out;
    long long s = num / den;
    if (num % den != 0 && num < 0) s -= 1;
    const long long r = num - s * den;
    long long w = (4096 * r + den) / (2 * den);
    if (s < 0) {
        s = 0;
        w = 0;
    } else if (s >= n_in - 1) {
        s = n_in - 1;
        w = 0;
    }
    return make_int2(static_cast<int>(s), static_cast<int>(w));
}

__global__ void k_noalloc_tables(NoAllocScratch *sc, int H, int W, int OH, int OW, int linear)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i == 0)
        sc->status = RZ_OK;   // the array keeps the previous call's contents
    if (i < OW)
        sc->xt[i] = table_entry(W, OW, i, linear != 0);
    else if (i - OW < OH)
        sc->yt[i - OW] = table_entry(H, OH, i - OW, linear != 0);
}

// Host copy of table_entry's source index (exact, no tables kept).
int host_index(int n_in, int n_out, int d, bool linear)
{
    if (!linear)
        return static_cast<int>(std::min<long long>(static_cast<long long>(d) * n_in / n_out, n_in - 1));
    const long long num = (2LL * d + 1) * n_in - n_out;
    const long long den = 2LL * n_out;
    long long s = num / den;
    if (num % den != 0 && num < 0) s -= 1;
    return static_cast<int>(std::clamp<long long>(s, 0, n_in - 1));
}

std::mutex g_mu;
NoAllocScratch *g_addr[kMaxDevices] = {};
const void *g_attr_fn[kMaxDevices][16] = {};

int fail(cudaError_t e)
{
    rz::record_cuda_error(static_cast<int>(e));   // read back by resize_last_cuda_error
    return RZ_ERR_CUDA;
}

}  // namespace

extern "C" int resize_u8_noalloc(const uint8_t *src, size_t src_pitch, uint8_t *dst, size_t dst_pitch, int H, int W,
                                 int C, int out_h, int out_w, int mode, void *stream)
{
    if (H < 1 || W < 1 || out_h < 0 || out_w < 0 || H > RZ_MAX_DIM || W > RZ_MAX_DIM) return RZ_ERR_ARG;
    if (mode != RZ_LINEAR && mode != RZ_NEAREST) return RZ_ERR_ARG;
    if (out_h > kNoAllocMaxDim || out_w > kNoAllocMaxDim) return RZ_ERR_UNSUPPORTED;
    if (C <= 0) return RZ_ERR_ARG;
    if (C != 1 && C != 3 && C != 4) return RZ_ERR_UNSUPPORTED;
    if (out_h == 0 || out_w == 0) return RZ_OK;
    if (!src || !dst) return RZ_ERR_ARG;
    const size_t in_row = static_cast<size_t>(W) * C, out_row = static_cast<size_t>(out_w) * C;
    if (src_pitch < in_row || dst_pitch < out_row) return RZ_ERR_ARG;
    const size_t src_bytes = (H - 1) * src_pitch + in_row, dst_bytes = (out_h - 1) * dst_pitch + out_row;
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), d0 = reinterpret_cast<uintptr_t>(dst);
    if (s0 < d0 + dst_bytes && d0 < s0 + src_bytes) return RZ_ERR_ARG;
    const bool linear = mode == RZ_LINEAR;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(e);
    if (dev < 0 || dev >= kMaxDevices) return RZ_ERR_UNSUPPORTED;
    // the array's address, the kernel attributes and the SM count are those
    // of the current device, so the stream must belong to it
    int stream_dev = dev;
    e = cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &stream_dev);
    if (e != cudaSuccess) return fail(e);
    if (stream_dev != dev) return RZ_ERR_ARG;

    // exact 2x on both axes (W = 2 out_w, H = 2 out_h make x = 2d + 1/2)
    const bool exact2 = linear && W == 2 * out_w && H == 2 * out_h;
    // tile: one output row, as wide as the output or the widest power-of-two
    // strip whose staged source row stays within 16 KB; two staged tiles per CTA
    int TW = 1, slot_bytes = 16;
    for (int k = 0; k <= 13; k++) {
        const int w = k == 0 ? out_w : (8192 >> k);      // out_w, 4096, 2048, ..., 1
        if (k > 0 && w >= out_w) continue;
        if (w < out_w && ((w * C) % 16 != 0 || (exact2 && w % 8 != 0)) && w > 1) continue;
        int span = 0;
        for (int dx0 = 0; dx0 < out_w; dx0 += w) {
            const int dx1 = std::min(dx0 + w, out_w);
            const int xs0 = host_index(W, out_w, dx0, linear);
            int xs1 = host_index(W, out_w, dx1 - 1, linear);
            if (linear) xs1 = std::min(xs1 + 1, W - 1);
            span = std::max(span, (((xs1 + 1) * C + 15) & ~15) - ((xs0 * C) & ~15));
        }
        TW = w;
        slot_bytes = span + rz::fam_slot_pad(rz::FAM_U8);
        if (span <= 16384 && w * C <= 16384) break;
    }
    // the kernel: the exact 2x path when every table entry is the 2x pattern
    // and each strip starts on a 16-byte boundary of the staged rows
    const bool down2 = exact2 && (TW == out_w || TW % 8 == 0);
    const void *fn = rz::kernel_for(rz::FAM_U8, mode, down2 ? rz::VAR_DOWN2 : rz::VAR_GENERIC, C);
    if (!fn) return RZ_ERR_UNSUPPORTED;
    const int fn_slot = (C == 1 ? 0 : (C == 3 ? 1 : 2)) * 3 + (down2 ? 2 : (linear ? 1 : 0));

    // one-time set-up per device, with that device current
    NoAllocScratch *sc = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_addr[dev]) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess) return fail(e);
            g_addr[dev] = static_cast<NoAllocScratch *>(p);
        }
        sc = g_addr[dev];
        if (g_attr_fn[dev][fn_slot] != fn) {
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, rz::kMaxSmem);
            if (e != cudaSuccess) return fail(e);
            g_attr_fn[dev][fn_slot] = fn;
        }
    }

    const int max_rows = linear ? 2 : 1;
    const int stages = 2;
    const rz::SmemLayout L = rz::smem_layout(rz::FAM_U8, C, 1, TW, max_rows, slot_bytes, stages);
    if (L.total > rz::kMaxSmem) return RZ_ERR_UNSUPPORTED;
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, rz::kThreads, static_cast<size_t>(L.total));
    if (e != cudaSuccess) return fail(e);
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(e);
    if (per_sm < 1) return RZ_ERR_UNSUPPORTED;

    rz::KArgs a = {};
    a.src = src;
    a.src_pitch = static_cast<long long>(src_pitch);
    a.dst = dst;
    a.dst_pitch = static_cast<long long>(dst_pitch);
    a.H = H; a.W = W; a.OH = out_h; a.OW = out_w; a.C = C;
    a.TR = 1; a.TW = TW;
    a.tiles_x = (out_w + TW - 1) / TW;
    a.tiles_y = out_h;
    a.batch = 1;
    a.max_rows = max_rows;
    a.slot_bytes = slot_bytes;
    a.stages = stages;
    a.tma_in = (s0 % 16 == 0) && (src_pitch % 16 == 0) && (in_row % 16 == 0);
    a.tma_out = (d0 % 16 == 0) && (dst_pitch % 16 == 0) && (a.tiles_x == 1 || (TW * C) % 16 == 0);
    a.xt = sc->xt;
    a.yt = sc->yt;
    a.status = &sc->status;
    a.src_extent = static_cast<long long>(src_bytes);
    a.dst_extent = static_cast<long long>(dst_bytes);
    a.tab = reinterpret_cast<const uint8_t *>(sc);
    a.tab_bytes = static_cast<long long>(sizeof(NoAllocScratch));
    const long long ntiles = static_cast<long long>(a.tiles_x) * a.tiles_y;
    const int grid = static_cast<int>(std::min<long long>(ntiles, static_cast<long long>(per_sm) * sms));

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int n = out_w + out_h;
    k_noalloc_tables<<<(n + 255) / 256, 256, 0, s>>>(sc, H, W, out_h, out_w, linear ? 1 : 0);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(e);
    CUtensorMap unused;   // row copies only: the kernel ignores the map
    for (size_t i = 0; i < sizeof(unused.opaque) / sizeof(unused.opaque[0]); i++) unused.opaque[i] = 0;
    const int le = rz::launch_resize(fn, a, unused, grid, static_cast<size_t>(L.total), true, stream);
    if (le != 0) return fail(static_cast<cudaError_t>(le));
    return RZ_OK;
}
