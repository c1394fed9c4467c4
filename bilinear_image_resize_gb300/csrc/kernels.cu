// Resize kernels for sm_103a.
//
// One CTA owns a tile of TR output rows x TW output columns.  It
//   1. lists the distinct source rows its output rows sample (two per row for
//      bilinear, one for nearest, plus a one-row halo for the 3x3 epilogue),
//   2. stages the needed column span of each of those rows in shared memory
//      with one bulk (TMA) copy per row, completing on an mbarrier (plain
//      loads when the addresses are not 16-byte aligned),
//   3. computes its outputs from shared memory (bilinear as the exact 11-bit
//      fixed-point sum for uint8, as two lerps for float32), applies the
//      fused epilogue, and writes the tile into shared memory,
//   4. stores each output row with one bulk (TMA) copy.
// HBM is touched once per needed source byte and once per output byte; the
// staged rows are reused by every output row and column of the tile that
// samples them.
//
// Sampling: CUDA interpolation page (hnwysp.cn/news/129086) §2.1 nearest,
// §2.2 bilinear weights, §6.1 clamp, §6.2 fixed point, §4.2 fused epilogue;
// half-pixel mapping: "From Prototype to Performance: Optimizing OpenCV Resize
// on Volcanic GPUs", "Naive resize with linear sampling".  The per-column and
// per-row tables come from the plan (api.cu), where they are computed exactly.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "rz_internal.h"

namespace rz {
namespace {

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of the barrier, at most kWaitLimitNs.  On time-out
// the status word records RZ_ERR_TIMEOUT and false is returned.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, int *status)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > kWaitLimitNs) {
            if (status)
                atomicExch(status, RZ_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// Bulk copy global -> this CTA's shared memory, completing on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void *sdst, const void *gsrc, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(sdst)),
        "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Bulk copy shared -> global (bulk-group completion).
__device__ __forceinline__ void bulk_store(void *gdst, const void *ssrc, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_addr(ssrc)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Make this thread's generic-proxy shared-memory writes visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

__device__ __forceinline__ int ceil_log2(int v)
{
    return v <= 1 ? 0 : 32 - __clz(v - 1);
}

// ------------------------------------------------------------------ tile set-up

struct Tile {
    int b;              // image index within the batch
    int dy0, dy1;       // output rows [dy0, dy1)
    int dx0, dx1;       // output columns [dx0, dx1)
    const uint8_t *src; // this image's first source row
    uint8_t *dst;       // this image's output base
};

__device__ __forceinline__ Tile decode_tile(const KArgs &a)
{
    Tile t;
    const int per_img = a.tiles_x * a.tiles_y;
    const int bid = blockIdx.x;
    t.b = bid / per_img;
    const int r = bid - t.b * per_img;
    const int ty = r / a.tiles_x;
    const int tx = r - ty * a.tiles_x;
    t.dy0 = ty * a.TR;
    t.dy1 = min(t.dy0 + a.TR, a.OH);
    t.dx0 = tx * a.TW;
    t.dx1 = min(t.dx0 + a.TW, a.OW);
    t.src = a.src + (long long)t.b * a.src_bstride;
    t.dst = a.dst + (long long)t.b * a.dst_bstride;
    return t;
}

// Stage the source rows of the tile.  Thread 0 builds the list of distinct
// source rows for the computed rows dy0-halo .. dy1-1+halo (clamped into the
// image; rows are non-decreasing in dy, so a row already listed is one of the
// last two entries), records for each computed row the slots of its two tap
// rows, and issues one bulk copy per listed row.  Returns false if the copies
// did not arrive in time (status word set) — the caller then leaves the tile.
template <int LINEAR>
__device__ bool stage_rows(const KArgs &a, const Tile &t, int halo, int in_es, uint8_t *smem, const SmemLayout &L)
{
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    int *hdr = reinterpret_cast<int *>(smem + 8);
    int *rows = reinterpret_cast<int *>(smem + L.off_rows);
    int *map = reinterpret_cast<int *>(smem + L.off_map);
    uint8_t *slots = smem + L.off_slots;

    if (threadIdx.x == 0) {
        // column span of the computed columns, in bytes of a source row
        const int cx0 = clampi(t.dx0 - halo, 0, a.OW - 1);
        const int cx1 = clampi(t.dx1 - 1 + halo, 0, a.OW - 1);
        const int xs0 = a.xt[cx0].x;
        const int xs1 = LINEAR ? min(a.xt[cx1].x + 1, a.W - 1) : a.xt[cx1].x;
        int b_lo = xs0 * a.C * in_es;
        int b_hi = (xs1 + 1) * a.C * in_es;
        if (a.tma_in) {
            b_lo &= ~15;
            b_hi = (b_hi + 15) & ~15;
        }
        const int nbytes = b_hi - b_lo;

        int n = 0;
        bool overflow = nbytes > a.slot_bytes;
        const int nrc = (t.dy1 - t.dy0) + 2 * halo;
        for (int k = 0; k < nrc && !overflow; k++) {
            const int dy = clampi(t.dy0 - halo + k, 0, a.OH - 1);
            const int r0 = a.yt[dy].x;
            const int r1 = LINEAR ? min(r0 + 1, a.H - 1) : r0;
            int s0, s1;
            if (n > 0 && rows[n - 1] == r0)
                s0 = n - 1;
            else if (n > 1 && rows[n - 2] == r0)
                s0 = n - 2;
            else {
                if (n == a.max_rows) { overflow = true; break; }
                rows[n] = r0;
                s0 = n++;
            }
            if (rows[n - 1] == r1)
                s1 = n - 1;
            else {
                if (n == a.max_rows) { overflow = true; break; }
                rows[n] = r1;
                s1 = n++;
            }
            map[2 * k] = s0;
            map[2 * k + 1] = s1;
        }
        if (overflow) {
            // the host sizes max_rows and slot_bytes from the same tables, so
            // this is unreachable; it guards shared memory all the same
            atomicExch(a.status, RZ_ERR_ARG);
            n = -1;
        }
        hdr[0] = n;
        hdr[1] = b_lo;
        hdr[2] = nbytes;
        if (n > 0 && a.tma_in) {
            mbar_init(bar, 1);
            fence_mbar_init();
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n * nbytes));
            for (int s = 0; s < n; s++)
                bulk_load(slots + s * a.slot_bytes, t.src + (long long)rows[s] * a.src_pitch + b_lo,
                          static_cast<uint32_t>(nbytes), bar);
        }
    }
    __syncthreads();
    const int n = hdr[0];
    if (n < 0)
        return false;
    if (a.tma_in) {
        const bool ok = mbar_wait_bounded(bar, 0, a.status);
        // every thread leaves together if any timed out, so no barrier below
        // is left waiting for threads that returned
        if (__syncthreads_or(!ok)) {
            // give copies still in flight a second bounded wait before leaving
            if (!ok)
                mbar_wait_bounded(bar, 0, nullptr);
            return false;
        }
    } else {
        const int b_lo = hdr[1], nbytes = hdr[2];
        for (int s = 0; s < n; s++) {
            const uint8_t *g = t.src + (long long)rows[s] * a.src_pitch + b_lo;
            uint8_t *d = slots + s * a.slot_bytes;
            for (int k = threadIdx.x; k < nbytes; k += kThreads)
                d[k] = __ldg(g + k);
        }
        __syncthreads();
    }
    return true;
}

// Write the output tile from shared memory: `nrow` rows of `row_bytes` bytes,
// row i from obuf + i*obuf_pitch to gdst + i*gpitch.  Bulk copies when
// allowed (16-byte aligned start and pitch); the ragged tail of each row,
// under 16 bytes, and the whole row otherwise, by plain stores.
__device__ __forceinline__ void store_rows(const KArgs &a, uint8_t *gdst, long long gpitch, const uint8_t *obuf,
                                           int obuf_pitch, int nrow, int row_bytes)
{
    const int bulk = a.tma_out ? (row_bytes & ~15) : 0;
    if (bulk > 0) {
        fence_proxy_async_smem();
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int i = 0; i < nrow; i++)
                bulk_store(gdst + i * gpitch, obuf + i * obuf_pitch, static_cast<uint32_t>(bulk));
            bulk_commit();
        }
    } else {
        __syncthreads();
    }
    const int tail = row_bytes - bulk;
    if (tail > 0) {
        for (int i = 0; i < nrow; i++)
            for (int k = threadIdx.x; k < tail; k += kThreads)
                gdst[i * gpitch + bulk + k] = obuf[i * obuf_pitch + bulk + k];
    }
    if (bulk > 0 && threadIdx.x == 0)
        bulk_wait_read_all();
}

// ------------------------------------------------------------------ plain resize

template <typename T, int C, int LINEAR>
__global__ void __launch_bounds__(kThreads) k_resize(const KArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int ES = sizeof(T);
    constexpr int FAM = (ES == 1) ? FAM_U8 : FAM_F32;
    const Tile t = decode_tile(a);
    const SmemLayout L = smem_layout(FAM, C, a.TR, a.TW, a.max_rows, a.slot_bytes);
    if (!stage_rows<LINEAR>(a, t, 0, ES, smem, L))
        return;

    const int *hdr = reinterpret_cast<const int *>(smem + 8);
    const int *map = reinterpret_cast<const int *>(smem + L.off_map);
    const T *slots = reinterpret_cast<const T *>(smem + L.off_slots);
    T *obuf = reinterpret_cast<T *>(smem + L.off_out);
    const int lo = hdr[1] / ES;              // element index of slot element 0
    const int slot_el = a.slot_bytes / ES;
    const int orow_el = L.out_row_bytes / ES;

    const int nr = t.dy1 - t.dy0, nc = t.dx1 - t.dx0;
    const int lg = min(8, ceil_log2(nc));
    const int tpr = 1 << lg, rpp = kThreads >> lg;
    for (int rl = threadIdx.x >> lg; rl < nr; rl += rpp) {
        const int dy = t.dy0 + rl;
        const int2 yw = a.yt[dy];
        const T *top = slots + map[2 * rl] * slot_el - lo;
        const T *bot = slots + map[2 * rl + 1] * slot_el - lo;
        T *orow = obuf + rl * orow_el;
        for (int cl = threadIdx.x & (tpr - 1); cl < nc; cl += tpr) {
            const int2 xw = __ldg(&a.xt[t.dx0 + cl]);
            const int o0 = xw.x * C;
            if (!LINEAR) {
#pragma unroll
                for (int c = 0; c < C; c++)
                    orow[cl * C + c] = top[o0 + c];
            } else {
                const int o1 = min(xw.x + 1, a.W - 1) * C;
                if constexpr (ES == 1) {
                    const int A1 = xw.y, A0 = 2048 - A1;
                    const int B1 = yw.y, B0 = 2048 - B1;
#pragma unroll
                    for (int c = 0; c < C; c++) {
                        const int hT = A0 * top[o0 + c] + A1 * top[o1 + c];
                        const int hB = A0 * bot[o0 + c] + A1 * bot[o1 + c];
                        orow[cl * C + c] = static_cast<T>((B0 * hT + B1 * hB + (1 << 21)) >> 22);
                    }
                } else {
                    const float u = __int_as_float(xw.y), v = __int_as_float(yw.y);
#pragma unroll
                    for (int c = 0; c < C; c++) {
                        const float t0 = top[o0 + c], t1 = top[o1 + c];
                        const float b0 = bot[o0 + c], b1 = bot[o1 + c];
                        const float hT = fmaf(u, t1 - t0, t0);
                        const float hB = fmaf(u, b1 - b0, b0);
                        orow[cl * C + c] = fmaf(v, hB - hT, hT);
                    }
                }
            }
        }
    }
    uint8_t *gdst = t.dst + (long long)t.dy0 * a.dst_pitch + (long long)t.dx0 * C * ES;
    store_rows(a, gdst, a.dst_pitch, reinterpret_cast<const uint8_t *>(obuf), L.out_row_bytes, nr, nc * C * ES);
}

// ------------------------------------------------------------------ bilinear + normalise (u8 HWC -> f32 NCHW)

template <int C>
__global__ void __launch_bounds__(kThreads) k_resize_normalize(const KArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const Tile t = decode_tile(a);
    const SmemLayout L = smem_layout(FAM_NORM, C, a.TR, a.TW, a.max_rows, a.slot_bytes);
    if (!stage_rows<1>(a, t, 0, 1, smem, L))
        return;

    const int *hdr = reinterpret_cast<const int *>(smem + 8);
    const int *map = reinterpret_cast<const int *>(smem + L.off_map);
    const uint8_t *slots = smem + L.off_slots;
    float *obuf = reinterpret_cast<float *>(smem + L.off_out);
    const int lo = hdr[1];
    const int orow_el = L.out_row_bytes / 4;
    const int plane_el = a.TR * orow_el;

    const int nr = t.dy1 - t.dy0, nc = t.dx1 - t.dx0;
    const int lg = min(8, ceil_log2(nc));
    const int tpr = 1 << lg, rpp = kThreads >> lg;
    for (int rl = threadIdx.x >> lg; rl < nr; rl += rpp) {
        const int2 yw = a.yt[t.dy0 + rl];
        const int B1 = yw.y, B0 = 2048 - B1;
        const uint8_t *top = slots + map[2 * rl] * a.slot_bytes - lo;
        const uint8_t *bot = slots + map[2 * rl + 1] * a.slot_bytes - lo;
        for (int cl = threadIdx.x & (tpr - 1); cl < nc; cl += tpr) {
            const int2 xw = __ldg(&a.xt[t.dx0 + cl]);
            const int o0 = xw.x * C, o1 = min(xw.x + 1, a.W - 1) * C;
            const int A1 = xw.y, A0 = 2048 - A1;
#pragma unroll
            for (int c = 0; c < C; c++) {
                const int hT = A0 * top[o0 + c] + A1 * top[o1 + c];
                const int hB = A0 * bot[o0 + c] + A1 * bot[o1 + c];
                const int q = (B0 * hT + B1 * hB + (1 << 21)) >> 22;
                obuf[c * plane_el + rl * orow_el + cl] = fmaf(static_cast<float>(q), a.scale[c], a.shift[c]);
            }
        }
    }
    // one bulk store per (plane, row): plane c of image b at dst + c*dst_plane
    const int row_bytes = nc * 4;
    const int bulk = a.tma_out ? (row_bytes & ~15) : 0;
    uint8_t *gbase = t.dst + (long long)t.dy0 * a.dst_pitch + (long long)t.dx0 * 4;
    const uint8_t *ob = reinterpret_cast<const uint8_t *>(obuf);
    if (bulk > 0) {
        fence_proxy_async_smem();
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int c = 0; c < C; c++)
                for (int i = 0; i < nr; i++)
                    bulk_store(gbase + c * a.dst_plane + i * a.dst_pitch,
                               ob + (c * plane_el + i * orow_el) * 4, static_cast<uint32_t>(bulk));
            bulk_commit();
        }
    } else {
        __syncthreads();
    }
    const int tail = row_bytes - bulk;
    if (tail > 0)
        for (int c = 0; c < C; c++)
            for (int i = 0; i < nr; i++)
                for (int k = threadIdx.x; k < tail; k += kThreads)
                    gbase[c * a.dst_plane + i * a.dst_pitch + bulk + k] = ob[(c * plane_el + i * orow_el) * 4 + bulk + k];
    if (bulk > 0 && threadIdx.x == 0)
        bulk_wait_read_all();
}

// ------------------------------------------------------------------ bilinear + 3x3 filter (f32)

template <int C>
__global__ void __launch_bounds__(kThreads) k_resize_filter3x3(const KArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const Tile t = decode_tile(a);
    const SmemLayout L = smem_layout(FAM_FILT, C, a.TR, a.TW, a.max_rows, a.slot_bytes);
    if (!stage_rows<1>(a, t, 1, 4, smem, L))
        return;

    const int *hdr = reinterpret_cast<const int *>(smem + 8);
    const int *map = reinterpret_cast<const int *>(smem + L.off_map);
    const float *slots = reinterpret_cast<const float *>(smem + L.off_slots);
    float *mid = reinterpret_cast<float *>(smem + L.off_mid);
    float *obuf = reinterpret_cast<float *>(smem + L.off_out);
    const int lo = hdr[1] / 4;
    const int slot_el = a.slot_bytes / 4;
    const int orow_el = L.out_row_bytes / 4;
    const int mid_w = a.TW + 2;  // row pitch of mid, in pixels

    const int nr = t.dy1 - t.dy0, nc = t.dx1 - t.dx0;
    // 1. resized values on the tile plus a one-pixel ring, rows and columns
    //    clamped into the output grid (replicate border)
    {
        const int hr = nr + 2, hc = nc + 2;
        const int lg = min(8, ceil_log2(hc));
        const int tpr = 1 << lg, rpp = kThreads >> lg;
        for (int k = threadIdx.x >> lg; k < hr; k += rpp) {
            const int dy = clampi(t.dy0 - 1 + k, 0, a.OH - 1);
            const float v = __int_as_float(a.yt[dy].y);
            const float *top = slots + map[2 * k] * slot_el - lo;
            const float *bot = slots + map[2 * k + 1] * slot_el - lo;
            for (int j = threadIdx.x & (tpr - 1); j < hc; j += tpr) {
                const int dx = clampi(t.dx0 - 1 + j, 0, a.OW - 1);
                const int2 xw = __ldg(&a.xt[dx]);
                const float u = __int_as_float(xw.y);
                const int o0 = xw.x * C, o1 = min(xw.x + 1, a.W - 1) * C;
#pragma unroll
                for (int c = 0; c < C; c++) {
                    const float t0 = top[o0 + c], t1 = top[o1 + c];
                    const float b0 = bot[o0 + c], b1 = bot[o1 + c];
                    const float hT = fmaf(u, t1 - t0, t0);
                    const float hB = fmaf(u, b1 - b0, b0);
                    mid[(k * mid_w + j) * C + c] = fmaf(v, hB - hT, hT);
                }
            }
        }
    }
    __syncthreads();
    // 2. 3x3 correlation over the ring-extended tile
    {
        const int lg = min(8, ceil_log2(nc));
        const int tpr = 1 << lg, rpp = kThreads >> lg;
        for (int rl = threadIdx.x >> lg; rl < nr; rl += rpp) {
            for (int cl = threadIdx.x & (tpr - 1); cl < nc; cl += tpr) {
#pragma unroll
                for (int c = 0; c < C; c++) {
                    float z = 0.0f;
#pragma unroll
                    for (int i = 0; i < 3; i++)
#pragma unroll
                        for (int j = 0; j < 3; j++)
                            z = fmaf(a.w[i * 3 + j], mid[((rl + i) * mid_w + (cl + j)) * C + c], z);
                    obuf[rl * orow_el + cl * C + c] = z;
                }
            }
        }
    }
    uint8_t *gdst = t.dst + (long long)t.dy0 * a.dst_pitch + (long long)t.dx0 * C * 4;
    store_rows(a, gdst, a.dst_pitch, reinterpret_cast<const uint8_t *>(obuf), L.out_row_bytes, nr, nc * C * 4);
}

// ------------------------------------------------------------------ dispatch

using KernelFn = void (*)(const KArgs);

KernelFn pick(int fam, int mode, int C)
{
    const int ci = (C == 1) ? 0 : (C == 3 ? 1 : (C == 4 ? 2 : -1));
    if (ci < 0)
        return nullptr;
    static const KernelFn u8[2][3] = {
        {k_resize<uint8_t, 1, 0>, k_resize<uint8_t, 3, 0>, k_resize<uint8_t, 4, 0>},
        {k_resize<uint8_t, 1, 1>, k_resize<uint8_t, 3, 1>, k_resize<uint8_t, 4, 1>}};
    static const KernelFn f32[2][3] = {
        {k_resize<float, 1, 0>, k_resize<float, 3, 0>, k_resize<float, 4, 0>},
        {k_resize<float, 1, 1>, k_resize<float, 3, 1>, k_resize<float, 4, 1>}};
    static const KernelFn norm[3] = {k_resize_normalize<1>, k_resize_normalize<3>, k_resize_normalize<4>};
    static const KernelFn filt[3] = {k_resize_filter3x3<1>, k_resize_filter3x3<3>, k_resize_filter3x3<4>};
    const int m = mode == RZ_LINEAR ? 1 : 0;
    switch (fam) {
    case FAM_U8: return u8[m][ci];
    case FAM_F32: return f32[m][ci];
    case FAM_NORM: return m ? norm[ci] : nullptr;
    case FAM_FILT: return m ? filt[ci] : nullptr;
    default: return nullptr;
    }
}

}  // namespace

int launch_resize(int fam, int mode, const KArgs &a, int batch, size_t smem, void *stream)
{
    KernelFn fn = pick(fam, mode, a.C);
    if (!fn)
        return static_cast<int>(cudaErrorInvalidValue);
    // opt every kernel in to the full shared-memory carve-out once per process
    // (per device the attribute is applied lazily by the runtime)
    static std::mutex mu;
    static int done_dev[64][FAM_COUNT * 2 * 3] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return static_cast<int>(e);
    const int ci = (a.C == 1) ? 0 : (a.C == 3 ? 1 : 2);
    const int slot = (fam * 2 + (mode == RZ_LINEAR ? 1 : 0)) * 3 + ci;
    if (dev >= 0 && dev < 64) {
        std::lock_guard<std::mutex> lk(mu);
        if (!done_dev[dev][slot]) {
            e = cudaFuncSetAttribute(reinterpret_cast<const void *>(fn), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kMaxSmem);
            if (e != cudaSuccess)
                return static_cast<int>(e);
            done_dev[dev][slot] = 1;
        }
    }
    const long long nblk = (long long)batch * a.tiles_x * a.tiles_y;
    if (nblk <= 0)
        return 0;
    if (nblk > 0x7fffffffLL)
        return static_cast<int>(cudaErrorInvalidConfiguration);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nblk), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    e = cudaLaunchKernelEx(&cfg, fn, a);
    return static_cast<int>(e);
}

}  // namespace rz
