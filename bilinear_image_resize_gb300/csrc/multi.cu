// Many independent uint8 resizes of different geometries in one launch, for
// small frames whose own launches would each cost more than their work (the
// kernel-call overhead of the object-tracking page, §4.2; CUDA interpolation
// page §8.1 on batching launches).
//
// The jobs sit in a device array the caller fills (so a graph can replay the
// launch).  A persistent grid takes the work in units sized to the job.  Each
// job has a form, fixed by its geometry and layout alone:
//  - generic: a thread forms four consecutive output columns (a quad) on
//    kMultiRows rows, sampling indices and 11-bit weights computed on the fly
//    from the exact rational position (no tables; the columns' once per
//    unit, then stepped by exact remainder arithmetic), the taps read as
//    two 8-byte loads (three channels, 8-byte aligned rows) or 32-bit words
//    (hsum_u8) where the layout allows and as bytes otherwise, the sum
//    (B0 (A0 t0 + A1 t1) + B1 (A0 b0 + A1 b1) + 2^21) >> 22 (CUDA
//    interpolation page §2.2, §6.2), clamp border (§6.1); nearest takes
//    floor(d n_in / n_out) (§2.1);
//  - exact 2x downscale (bilinear, W = 2 out_w and H = 2 out_h, source and
//    output aligned to the group loads and stores): a thread forms one group
//    of down2_px(C) output pixels on kMultiRows rows, each the rounded mean
//    of its 2 x 2 block, the value the general sum takes at weights 1024;
//  - exact 2x upscale (bilinear, three or four channels, out_w = 2 W and
//    out_h = 2 H): a thread takes four source columns of kUp2Rows
//    consecutive source rows (eight output columns of 2 kUp2Rows rows), the
//    9-3-3-1 sums on pixel lane words, each source row loaded and unpacked
//    once per thread, the value the general sum takes at weights 1536 and
//    512.
// The exact 2x forms run a fraction of the generic form's instructions per
// pixel.  A unit is kMultiRows output rows (kUp2Rows source rows for the
// upscale) of 256 items for rows of 256 items or more, else P
// row lanes side by side, each its own rows, so that narrow frames still
// keep the CTA busy: either P = 256 / items-per-row whole rows, or, where
// that leaves more threads idle, eight lanes of 32-item slices of the row (a
// 640-pixel row of quads: five slices, every thread busy, where one whole
// row per unit would idle 96 of the 256).  Every CTA scans the jobs' unit
// counts into shared memory, then walks units grid-stride, finding each
// unit's job by a binary search.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "rz_device.h"
#include "rz_internal.h"

namespace rz {
namespace {

using namespace dev;

constexpr int kMultiThreads = 256;
constexpr int kMultiRows = 8;   // output rows per thread in a unit
constexpr int kUp2Rows = 8;     // source rows per thread in a unit of the 2x upscale form

// Form of a job (the launch's C and mode fixed): the per-pixel path or one of
// the exact 2x paths.
enum : int { kFormGeneric = 0, kFormDown2 = 1, kFormUp2 = 2 };

struct JobForm {
    int form;
    int ipr;    // items per row: quads; down2_px(C)-pixel output groups; four-column source groups
    int rows;   // rows the items repeat over: output rows; source rows for the upscale
    int rpl;    // rows per row lane in a unit
};

template <int C, int LINEAR>
__device__ __forceinline__ JobForm job_form(const rz_job &j)
{
    if constexpr (LINEAR) {
        if (j.W == 2 * j.out_w && j.H == 2 * j.out_h) {
            // the group's loads (8 bytes for three channels, else 16) and
            // stores (4, else 8)
            constexpr uintptr_t LW = C == 3 ? 8 : 16, SW = C == 3 ? 4 : 8;
            constexpr int PX = down2_px(C);
            if (((reinterpret_cast<uintptr_t>(j.src) | static_cast<uintptr_t>(j.src_pitch)) % LW) == 0 &&
                ((reinterpret_cast<uintptr_t>(j.dst) | static_cast<uintptr_t>(j.dst_pitch)) % SW) == 0)
                return {kFormDown2, (j.out_w + PX - 1) / PX, j.out_h, kMultiRows};
        }
        if (C != 1 && j.out_w == 2 * j.W && j.out_h == 2 * j.H)
            return {kFormUp2, (j.W + 3) / 4, j.H, kUp2Rows};
    }
    return {kFormGeneric, (j.out_w + 3) / 4, j.out_h, kMultiRows};
}

// Unit shape for ipr items per row: items per row lane, row lanes side by
// side, column units (thread t takes item cu qw + t % qw of row lane t / qw).
struct UnitShape {
    int qw, P, col_units;
};

__device__ __forceinline__ UnitShape unit_shape(int ipr)
{
    if (ipr >= kMultiThreads)
        return {kMultiThreads, 1, (ipr + kMultiThreads - 1) / kMultiThreads};
    // whole rows keep P ipr of the 256 threads busy; 32-item slices keep
    // ipr / (32 n32) of them busy: the slices when 8 > P n32
    const int P = kMultiThreads / ipr, n32 = (ipr + 31) / 32;
    if (8 > P * n32)
        return {32, kMultiThreads / 32, n32};
    return {ipr, P, 1};
}

// An empty output (out_h or out_w 0) reads and writes nothing, so its
// pointers and pitches are not checked.
__device__ __forceinline__ bool job_valid(const rz_job &j, int C)
{
    const bool dims = j.H >= 1 && j.W >= 1 && j.H <= RZ_MAX_DIM && j.W <= RZ_MAX_DIM && j.out_h >= 0 &&
                      j.out_w >= 0 && j.out_h <= RZ_MAX_DIM && j.out_w <= RZ_MAX_DIM;
    if (!dims || j.out_h == 0 || j.out_w == 0)
        return dims;
    return j.src && j.dst && j.src_pitch >= static_cast<size_t>(j.W) * C &&
           j.dst_pitch >= static_cast<size_t>(j.out_w) * C;
}

template <int C, int LINEAR>
__device__ __forceinline__ long long job_units(const rz_job &j)
{
    if (!job_valid(j, C))
        return 0;
    if (j.out_w == 0 || j.out_h == 0)
        return 0;
    const JobForm f = job_form<C, LINEAR>(j);
    const UnitShape sh = unit_shape(f.ipr);
    const int rows = f.rpl * sh.P;
    return static_cast<long long>((f.rows + rows - 1) / rows) * sh.col_units;
}

// Exact sampling position of output index d on an axis of n_in -> n_out
// samples, as quotient and remainder: bilinear (2d+1) n_in - n_out =
// s 2 n_out + r (x = s + r / (2 n_out), the half-pixel source position),
// nearest d n_in = s n_out + r; 0 <= r < den.  The float quotient is within
// one of the floor and corrected by integer checks.
struct AxisPos {
    int s, r;
};

__device__ __forceinline__ int axis_den(int n_out, bool linear) { return linear ? 2 * n_out : n_out; }

__device__ __forceinline__ AxisPos axis_pos(int n_in, int n_out, int d, bool linear)
{
    const long long num = linear ? (2LL * d + 1) * n_in - n_out : static_cast<long long>(d) * n_in;
    const int den = axis_den(n_out, linear);
    const int s = floor_div_exact(num, den);
    return {s, static_cast<int>(num - static_cast<long long>(s) * den)};
}

// The change of the position over D output indices (D n_in / den in the
// same quotient and remainder form), and one such step: the remainders add,
// carrying one into the quotient when they reach den.
__device__ __forceinline__ AxisPos axis_delta(int n_in, int n_out, int D, bool linear)
{
    const long long num = static_cast<long long>(linear ? 2 * D : D) * n_in;
    const int den = axis_den(n_out, linear);
    const int s = floor_div_exact(num, den);
    return {s, static_cast<int>(num - static_cast<long long>(s) * den)};
}

__device__ __forceinline__ void axis_step(AxisPos &p, AxisPos d, int den)
{
    p.s += d.s;
    p.r += d.r;
    if (p.r >= den) {
        p.r -= den;
        p.s += 1;
    }
}

// Sampling entry {left tap, far-tap 11-bit weight} at a position (the plan's
// table entry, clamp border): weight round-half-up(2048 r / den) =
// floor((4096 r + den) / (2 den)) (below 4097 den < 2^30, a 32-bit float
// quotient within one, corrected); taps outside the image folded onto one
// tap with weight 0.  Nearest: the quotient, kept below n_in.
__device__ __forceinline__ int2 axis_entry(AxisPos p, int n_in, int den, bool linear)
{
    if (!linear)
        return make_int2(min(p.s, n_in - 1), 0);
    if (p.s < 0)
        return make_int2(0, 0);
    if (p.s >= n_in - 1)
        return make_int2(n_in - 1, 0);
    const int a = 4096 * p.r + den, b = 2 * den;
    int w = __float2int_rd(__fdividef(static_cast<float>(a), static_cast<float>(b)));
    if (w * b > a)
        w -= 1;
    else if (w * b + b <= a)
        w += 1;
    return make_int2(p.s, w);
}

// hsum_u8 for three channels from two 8-byte loads (row 8-byte aligned; the
// tap pair's bytes o0 .. o0 + 5 lie in the 16 bytes from o0 & ~7): two load
// instructions instead of three, the L1 requests that bound the generic form
__device__ __forceinline__ void hsum3_w8(const uint8_t *row, int o0, uint32_t aw, int (&h)[3])
{
    const uint2 *w = reinterpret_cast<const uint2 *>(row + (o0 & ~7));
    const uint2 a = w[0], b = w[1];
    const int off = o0 & 7;
    const bool up = off >= 4;
    const uint32_t x0 = up ? a.y : a.x, x1 = up ? b.x : a.y, x2 = up ? b.y : b.x;
    const uint32_t sel = 0x3210u + 0x1111u * static_cast<uint32_t>(off & 3);
    const uint32_t lo4 = __byte_perm(x0, x1, sel), hi4 = __byte_perm(x1, x2, sel);
    const uint32_t p01 = __byte_perm(lo4, hi4, 0x4130), p2 = __byte_perm(lo4, hi4, 0x0052);
    h[0] = static_cast<int>(__dp2a_lo(aw, p01, 0u));
    h[1] = static_cast<int>(__dp2a_hi(aw, p01, 0u));
    h[2] = static_cast<int>(__dp2a_lo(aw, p2, 0u));
}

// Exact 2x downscale form: output group g (down2_px(C) pixels) of rows
// y0, y0 + P, ... (kMultiRows of them, those below out_h).
template <int C>
__device__ __forceinline__ void multi_down2(const rz_job &J, int g, int y0, int P)
{
    constexpr int PX = down2_px(C);
    const int full = J.out_w / PX;
    for (int k8 = 0; k8 < kMultiRows; k8++) {
        const int dy = y0 + k8 * P;
        if (dy >= J.out_h)
            break;
        const uint8_t *top = J.src + static_cast<long long>(2 * dy) * J.src_pitch;
        uint8_t *out = J.dst + static_cast<long long>(dy) * J.dst_pitch;
        if (g < full)
            down2_one<C, 1>(top, top + J.src_pitch, out, g);
        else
            down2_row_tail<C, 1>(top, top + J.src_pitch, out, full * PX, J.out_w);
    }
}

// Exact 2x upscale form: source columns 4 g .. 4 g + 3 of source rows
// r0 .. r0 + kUp2Rows - 1 (those below H), output rows 2 r0 ..; the
// unpacked rows above, at and below the current one kept in registers.
template <int C>
__device__ __forceinline__ void multi_up2(const rz_job &J, int g, int r0)
{
    using L = Up2RowsLayout<C>;
    if (r0 >= J.H)
        return;
    const int s0 = g * L::P, np = min(L::P, J.W - s0);
    const int r1 = min(r0 + kUp2Rows, J.H);
    const bool words_in = ((reinterpret_cast<uintptr_t>(J.src) | static_cast<uintptr_t>(J.src_pitch)) & 3) == 0;
    const bool inner = words_in && s0 >= 1 && (s0 - 1) * C - L::LEAD + 4 * L::NW <= J.W * C;
    auto row_ptr = [&](int r) { return J.src + static_cast<long long>(clampi(r, 0, J.H - 1)) * J.src_pitch; };
    uint8_t *out = J.dst + static_cast<long long>(2 * r0) * J.dst_pitch + static_cast<long long>(2 * s0) * C;
    uint32_t lo[3][6], hi[3][6];
    up2_row_lanes<C, RZ_BORDER_CLAMP>(row_ptr(r0 - 1), s0, J.W, inner, lo[0], hi[0]);
    up2_row_lanes<C, RZ_BORDER_CLAMP>(row_ptr(r0), s0, J.W, inner, lo[1], hi[1]);
    auto step = [&](const int ia, const int im, const int ib, int r) {
        up2_row_lanes<C, RZ_BORDER_CLAMP>(row_ptr(r + 1), s0, J.W, inner, lo[ib], hi[ib]);
        uint32_t mlo[6], mhi[6];
#pragma unroll
        for (int k = 0; k < 6; k++) {
            mlo[k] = 48 * lo[im][k] + 0x00200020u;
            mhi[k] = 48 * hi[im][k] + 0x00200020u;
        }
        up2_emit_row<C>(lo[ia], hi[ia], mlo, mhi, out, np);
        up2_emit_row<C>(lo[ib], hi[ib], mlo, mhi, out + J.dst_pitch, np);
        out += 2 * J.dst_pitch;
    };
    for (int r = r0; r < r1; r += 3) {
        step(0, 1, 2, r);
        if (r + 1 >= r1) break;
        step(1, 2, 0, r + 1);
        if (r + 2 >= r1) break;
        step(2, 0, 1, r + 2);
    }
}

template <int C, int LINEAR>
// (registers capped at 64 for four resident CTAs per SM: a few words spill;
// measured faster than five CTAs at 48 registers, where the 2x forms spill
// in their inner loops)
__global__ void __launch_bounds__(kMultiThreads, 4) k_multi(const rz_job *__restrict__ jobs, int njobs, int *status)
{
    __shared__ long long pre[kMultiMaxJobs + 1];   // units before job j
    __shared__ long long warp_sum[kMultiThreads / 32];
    grid_launch_dependents();
    grid_dependency_wait();
    // scan of the jobs' unit counts: each thread sums a run of jobs, the runs
    // are scanned across the block, then each thread writes its run's prefix
    const int per = (njobs + kMultiThreads - 1) / kMultiThreads;
    const int j0 = threadIdx.x * per;
    long long run = 0;
    bool bad = false;
    for (int k = 0; k < per; k++) {
        const int j = j0 + k;
        if (j < njobs) {
            const rz_job J = jobs[j];
            run += job_units<C, LINEAR>(J);
            bad |= !job_valid(J, C);
        }
    }
    if (bad && status && blockIdx.x == 0)
        atomicExch(status, RZ_ERR_ARG);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += v;
    }
    if (lane == 31)
        warp_sum[warp] = incl;
    __syncthreads();
    long long before = incl - run;
    for (int w = 0; w < warp; w++)
        before += warp_sum[w];
    for (int k = 0; k < per; k++) {
        const int j = j0 + k;
        if (j < njobs) {
            pre[j] = before;
            before += job_units<C, LINEAR>(jobs[j]);
        }
    }
    if (threadIdx.x == kMultiThreads - 1)
        pre[njobs] = before;   // the last thread's runs end the list
    __syncthreads();
    const long long total = pre[njobs];
    for (long long u = blockIdx.x; u < total; u += gridDim.x) {
        // the job: the last j with pre[j] <= u (empty jobs share their prefix)
        int lo = 0, hi = njobs - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (pre[mid] <= u)
                lo = mid;
            else
                hi = mid - 1;
        }
        const rz_job J = jobs[lo];
        const long long local = u - pre[lo];
        const JobForm F = job_form<C, LINEAR>(J);
        const UnitShape sh = unit_shape(F.ipr);
        const int rb = static_cast<int>(local / sh.col_units);
        const int cu = static_cast<int>(local - static_cast<long long>(rb) * sh.col_units);
        const int p = static_cast<int>(threadIdx.x) / sh.qw;   // row lane
        const int q = cu * sh.qw + static_cast<int>(threadIdx.x) - p * sh.qw;
        if (q >= F.ipr || p >= sh.P)
            continue;
        if constexpr (LINEAR) {
            if (F.form == kFormDown2) {
                multi_down2<C>(J, q, rb * kMultiRows * sh.P + p, sh.P);
                continue;
            }
            if constexpr (C != 1) {
                if (F.form == kFormUp2) {
                    multi_up2<C>(J, q, (rb * sh.P + p) * kUp2Rows);
                    continue;
                }
            }
        }
        const int x0 = 4 * q;
        const int npx = min(4, J.out_w - x0);
        // the quad's columns, one position stepped by one column (past the
        // row's end the step runs on: those columns fold onto the last
        // sample and are not stored)
        int xs[4], xw[4];
        {
            const int den = axis_den(J.out_w, LINEAR);
            AxisPos px = axis_pos(J.W, J.out_w, x0, LINEAR);
            const AxisPos d1 = axis_delta(J.W, J.out_w, 1, LINEAR);
#pragma unroll
            for (int k = 0; k < 4; k++) {
                if (k > 0)
                    axis_step(px, d1, den);
                const int2 xe = axis_entry(px, J.W, den, LINEAR);
                xs[k] = xe.x;
                xw[k] = xe.y;
            }
        }
        const int row_bytes = J.W * C;
        const bool words_in = ((reinterpret_cast<uintptr_t>(J.src) | static_cast<uintptr_t>(J.src_pitch)) & 3) == 0;
        const bool words8_in = ((reinterpret_cast<uintptr_t>(J.src) | static_cast<uintptr_t>(J.src_pitch)) & 7) == 0;
        const int ybase = rb * kMultiRows * sh.P + p;
        // the lane's rows ybase, ybase + P, ...: one position stepped by P rows
        const int yden = axis_den(J.out_h, LINEAR);
        AxisPos py = axis_pos(J.H, J.out_h, ybase, LINEAR);
        const AxisPos dP = axis_delta(J.H, J.out_h, sh.P, LINEAR);
        for (int k8 = 0; k8 < kMultiRows; k8++) {
            const int dy = ybase + k8 * sh.P;
            if (dy >= J.out_h)
                break;
            if (k8 > 0)
                axis_step(py, dP, yden);
            const int2 ye = axis_entry(py, J.H, yden, LINEAR);
            const uint8_t *top = J.src + static_cast<long long>(ye.x) * J.src_pitch;
            const uint8_t *bot =
                J.src + static_cast<long long>(LINEAR ? min(ye.x + 1, J.H - 1) : ye.x) * J.src_pitch;
            const int B1 = ye.y, B0 = 2048 - B1;
            int q[4][C];
#pragma unroll
            for (int k = 0; k < 4; k++) {
                const int o0 = xs[k] * C;
                if (!LINEAR) {
#pragma unroll
                    for (int c = 0; c < C; c++)
                        q[k][c] = top[o0 + c];
                    continue;
                }
                int hT[C], hB[C];
                const uint32_t aw = static_cast<uint32_t>(2048 - xw[k]) | (static_cast<uint32_t>(xw[k]) << 16);
                bool done = false;
                if constexpr (C == 3) {
                    if (words8_in && (o0 & ~7) + 16 <= row_bytes) {
                        hsum3_w8(top, o0, aw, hT);
                        hsum3_w8(bot, o0, aw, hB);
                        done = true;
                    }
                }
                if (!done) {
                    if (words_in && o0 + 12 <= row_bytes) {   // far tap inside: xs <= W - 2
                        hsum_u8<C>(top, o0, aw, hT);
                        hsum_u8<C>(bot, o0, aw, hB);
                    } else {
                        const int o1 = min(xs[k] + 1, J.W - 1) * C;
#pragma unroll
                        for (int c = 0; c < C; c++) {
                            hT[c] = (2048 - xw[k]) * top[o0 + c] + xw[k] * top[o1 + c];
                            hB[c] = (2048 - xw[k]) * bot[o0 + c] + xw[k] * bot[o1 + c];
                        }
                    }
                }
#pragma unroll
                for (int c = 0; c < C; c++)
                    q[k][c] = (B0 * hT[c] + B1 * hB[c] + (1 << 21)) >> 22;
            }
            uint8_t *op = J.dst + static_cast<long long>(dy) * J.dst_pitch + static_cast<long long>(x0) * C;
            if (npx == 4 && (reinterpret_cast<uintptr_t>(op) & 3) == 0) {
                uint32_t *o = reinterpret_cast<uint32_t *>(op);
                if constexpr (C == 1) {
                    o[0] = pack4(q[0][0], q[1][0], q[2][0], q[3][0]);
                } else if constexpr (C == 3) {
                    o[0] = pack4(q[0][0], q[0][1], q[0][2], q[1][0]);
                    o[1] = pack4(q[1][1], q[1][2], q[2][0], q[2][1]);
                    o[2] = pack4(q[2][2], q[3][0], q[3][1], q[3][2]);
                } else {
#pragma unroll
                    for (int k = 0; k < 4; k++)
                        o[k] = pack4(q[k][0], q[k][1], q[k][2], q[k][3]);
                }
            } else {
                for (int k = 0; k < npx; k++)
#pragma unroll
                    for (int c = 0; c < C; c++)
                        op[k * C + c] = static_cast<uint8_t>(q[k][c]);
            }
        }
    }
}

}  // namespace

int launch_multi(const rz_job *jobs, int njobs, int C, int mode, int *status, bool pdl, void *stream)
{
    using Fn = void (*)(const rz_job *, int, int *);
    static const Fn k[2][3] = {{k_multi<1, 0>, k_multi<3, 0>, k_multi<4, 0>},
                               {k_multi<1, 1>, k_multi<3, 1>, k_multi<4, 1>}};
    const int ci = (C == 1) ? 0 : (C == 3 ? 1 : 2);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return static_cast<int>(e);
    cudaLaunchConfig_t cfg = {};
    // four rounds of the CTAs that fit at once (each CTA walks an equal share
    // of the units; units differ in cost by form, and the finer share
    // measured faster than one or two rounds), the per-SM count asked of the
    // runtime once per form
    const Fn fn = k[mode == RZ_LINEAR ? 1 : 0][ci];
    static std::atomic<int> resident[2][3];
    int per_sm = resident[mode == RZ_LINEAR ? 1 : 0][ci].load(std::memory_order_relaxed);
    if (per_sm <= 0) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kMultiThreads, 0);
        if (e != cudaSuccess)
            return static_cast<int>(e);
        per_sm = per_sm > 0 ? per_sm : 1;
        resident[mode == RZ_LINEAR ? 1 : 0][ci].store(per_sm, std::memory_order_relaxed);
    }
    cfg.gridDim = dim3(static_cast<unsigned>(sms * 4 * per_sm), 1, 1);
    cfg.blockDim = dim3(kMultiThreads, 1, 1);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, fn, jobs, njobs, status);
    return static_cast<int>(e);
}

}  // namespace rz
