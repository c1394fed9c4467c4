// Many independent uint8 resizes of different geometries in one launch, for
// small frames whose own launches would each cost more than their work (the
// kernel-call overhead of the object-tracking page, §4.2; CUDA interpolation
// page §8.1 on batching launches).
//
// The jobs sit in a device array the caller fills (so a graph can replay the
// launch).  A persistent grid takes the work in units sized to the job: a
// thread forms four consecutive output columns (a quad) on kMultiRows rows,
// so a unit is kMultiRows rows of 256 quads for rows of 256 quads or more,
// else P row lanes side by side, each on kMultiRows rows (P apart), so that
// narrow frames still keep the CTA busy: either P = 256 / quads-per-row whole
// rows, or, where that leaves more threads idle, eight lanes of 32-quad
// slices of the row (a 640-pixel row: five slices, every thread busy, where
// one whole row per unit would idle 96 of the 256).  Every CTA
// scans the jobs' unit counts into shared memory, then walks units
// grid-stride, finding each unit's job by a binary search.  The arithmetic
// is that of the plan-based kernels: sampling
// indices and 11-bit weights are computed on the fly from the exact rational
// position (no tables; the columns' once per unit, each row's once), the taps
// read as 32-bit words where the layout allows (hsum_u8) and as bytes
// otherwise, the sum (B0 (A0 t0 + A1 t1) + B1 (A0 b0 + A1 b1) + 2^21) >> 22
// (CUDA interpolation page §2.2, §6.2), clamp border (§6.1); nearest takes
// floor(d n_in / n_out) (§2.1).
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

// Unit shape of a job: quads per row lane, row lanes side by side, column
// units (thread t takes quad cu qw + t % qw of row lane t / qw).
struct UnitShape {
    int qw, P, col_units;
};

__device__ __forceinline__ UnitShape unit_shape(const rz_job &j)
{
    const int qpr = (j.out_w + 3) / 4;
    if (qpr >= kMultiThreads)
        return {kMultiThreads, 1, (qpr + kMultiThreads - 1) / kMultiThreads};
    // whole rows keep P qpr of the 256 threads busy; 32-quad slices keep
    // qpr / (32 n32) of them busy: the slices when 8 > P n32
    const int P = kMultiThreads / qpr, n32 = (qpr + 31) / 32;
    if (8 > P * n32)
        return {32, kMultiThreads / 32, n32};
    return {qpr, P, 1};
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

__device__ __forceinline__ long long job_units(const rz_job &j, int C)
{
    if (!job_valid(j, C))
        return 0;
    if (j.out_w == 0 || j.out_h == 0)
        return 0;
    const UnitShape sh = unit_shape(j);
    const int rows = kMultiRows * sh.P;
    return static_cast<long long>((j.out_h + rows - 1) / rows) * sh.col_units;
}

// Sampling entry {left tap, far-tap 11-bit weight} of output index d on an
// axis of n_in -> n_out samples (the plan's table entry, clamp border):
// x = ((2d+1) n_in - n_out) / (2 n_out), floor and remainder exact (the
// float quotient is within one of the floor and corrected by integer
// checks), weight round-half-up(2048 r / den) likewise; taps outside the
// image folded onto one tap with weight 0.  Nearest: floor(d n_in / n_out).
__device__ __forceinline__ int2 entry(int n_in, int n_out, int d, bool linear)
{
    if (!linear) {
        const int s = floor_div_exact(static_cast<long long>(d) * n_in, n_out);
        return make_int2(min(s, n_in - 1), 0);
    }
    const long long num = (2LL * d + 1) * n_in - n_out;
    const int den = 2 * n_out;
    const int s = floor_div_exact(num, den);
    if (s < 0)
        return make_int2(0, 0);
    if (s >= n_in - 1)
        return make_int2(n_in - 1, 0);
    const int r = static_cast<int>(num - static_cast<long long>(s) * den);
    const int w = floor_div_exact(4096LL * r + den, 2 * den);
    return make_int2(s, w);
}

template <int C, int LINEAR>
// (registers capped for five resident CTAs per SM: a few words spill, and the
// kernel, latency-bound, still runs faster with the extra warps)
__global__ void __launch_bounds__(kMultiThreads, 5) k_multi(const rz_job *__restrict__ jobs, int njobs, int *status)
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
            run += job_units(J, C);
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
            before += job_units(jobs[j], C);
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
        const UnitShape sh = unit_shape(J);
        const int rb = static_cast<int>(local / sh.col_units);
        const int cu = static_cast<int>(local - static_cast<long long>(rb) * sh.col_units);
        const int p = static_cast<int>(threadIdx.x) / sh.qw;   // row lane
        const int q = cu * sh.qw + static_cast<int>(threadIdx.x) - p * sh.qw;
        const int x0 = 4 * q;
        if (x0 >= J.out_w || p >= sh.P)
            continue;
        const int npx = min(4, J.out_w - x0);
        int xs[4], xw[4];
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const int2 xe = entry(J.W, J.out_w, min(x0 + k, J.out_w - 1), LINEAR);
            xs[k] = xe.x;
            xw[k] = xe.y;
        }
        const int row_bytes = J.W * C;
        const bool words_in = ((reinterpret_cast<uintptr_t>(J.src) | static_cast<uintptr_t>(J.src_pitch)) & 3) == 0;
        const int ybase = rb * kMultiRows * sh.P + p;
        for (int k8 = 0; k8 < kMultiRows; k8++) {
            const int dy = ybase + k8 * sh.P;
            if (dy >= J.out_h)
                break;
            const int2 ye = entry(J.H, J.out_h, dy, LINEAR);
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
                if (words_in && o0 + 12 <= row_bytes) {   // far tap inside: xs <= W - 2
                    const uint32_t aw = static_cast<uint32_t>(2048 - xw[k]) | (static_cast<uint32_t>(xw[k]) << 16);
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
    // two rounds of the CTAs that fit at once (each CTA walks an equal share
    // of the units), the per-SM count asked of the runtime once per form
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
    cfg.gridDim = dim3(static_cast<unsigned>(sms * 2 * per_sm), 1, 1);
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
