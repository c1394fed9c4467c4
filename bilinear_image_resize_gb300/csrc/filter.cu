// K x K filters for sm_103a: the standalone correlation over the valid
// region, and the bilinear resize with a fused odd K x K epilogue.
//
// Standalone (OpenCL convolution page §2): out[y][x] = sum_{r, c < K}
// w[r K + c] in[y + r][x + c], float32, one channel, 1 <= K <= 64.  For the
// page's widths (8 to 64) the work is K^2 multiply-adds per output, far above
// the bytes moved, so the kernel is bound by the FP32 FMA pipes: a CTA
// stages its input tile (TH + K - 1 rows of kVTW + K - 1 columns, zero past
// the image) and the weights (rows zero-padded to a multiple of 8) in shared
// memory, and each thread keeps a 2 x 8 block of outputs in registers: per
// input row and chunk of 8 filter columns it loads a 16-float window (four
// 16-byte loads) and the chunk's weights of the one or two filter rows that
// meet its two output rows (16-byte broadcast loads), and issues up to 128
// FMAs.  The tile is staged by asynchronous copies (all in flight at once),
// for filters wider than 32 in CTAs of 16 warps (32 output rows: half the
// halo re-read) with rows swizzled so that the window loads are free of bank
// conflicts, narrower ones in CTAs of 8 warps.  (Tensor
// cores take no FP32 operands; TF32 would not hold float32 accuracy, so this
// contraction stays on the FMA pipes.)
//
// Fused (CUDA interpolation page §4.2, any odd K <= 7): a CTA computes the
// bilinear values of its output tile and a K / 2 halo into shared memory
// (rows and columns of the halo clamped to the output grid: the replicate
// border on that grid), then correlates them with the weights, which sit in
// the kernel's parameter bank.  The source taps are read directly (through
// L1), so plans under the wrap rule are served too.
#include <cuda_runtime.h>

#include <cstdint>

#include "rz_device.h"
#include "rz_internal.h"

namespace rz {
namespace {

using namespace dev;

// 4-byte asynchronous copy global -> shared (no register staging), the
// destination zero-filled when `valid` is false (the source is then not read,
// but the address given is inside the image).
__device__ __forceinline__ void cp_async_4(float *dst, const float *src, bool valid)
{
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(d), "l"(src), "r"(valid ? 4 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

template <bool WRAP>
__device__ __forceinline__ float bilinear_f32(const uint8_t *img, long long pitch, int C, int c, int2 xe, int2 ye,
                                              int W, int H)
{
    const float u = __int_as_float(xe.y), v = __int_as_float(ye.y);
    const int c0 = xe.x * C + c, c1 = far_tap<WRAP>(xe.x, W) * C + c;
    const float *top = reinterpret_cast<const float *>(img + (long long)ye.x * pitch);
    const float *bot = reinterpret_cast<const float *>(img + (long long)far_tap<WRAP>(ye.x, H) * pitch);
    const float t0 = __ldg(top + c0), t1 = __ldg(top + c1), b0 = __ldg(bot + c0), b1 = __ldg(bot + c1);
    const float h0 = fmaf(u, t1 - t0, t0), h1 = fmaf(u, b1 - b0, b0);
    return fmaf(v, h1 - h0, h0);
}

// Grid: x walks the output tiles of one image, y the images of a batch.
template <int C, int K, bool WRAP>
__global__ void __launch_bounds__(kFilterThreads) k_resize_filter(const KArgs a, const __grid_constant__ CUtensorMap)
{
    constexpr int R = K / 2, SW = kFTW + 2 * R, SH = kFTH + 2 * R;
    constexpr int RPT = kFTH / (kFilterThreads / kFTW);   // output rows per thread: 8
    constexpr int N = SH * SW;                          // resized values of tile and halo
    constexpr int U = C == 1 ? 4 : 2;                   // values per thread with loads in flight together
    __shared__ float S[C][SH][SW];
    __shared__ int2 tx[SW], ty[SH];
    grid_launch_dependents();
    grid_dependency_wait();
    const int tiles_x = (a.OW + kFTW - 1) / kFTW;
    const int tx0 = (blockIdx.x % tiles_x) * kFTW, ty0 = (blockIdx.x / tiles_x) * kFTH;
    const int x = threadIdx.x % kFTW, yb = (threadIdx.x / kFTW) * RPT;
    // the tile's table entries (halo rows and columns clamped to the grid)
    for (int i = threadIdx.x; i < SW + SH; i += kFilterThreads) {
        if (i < SW)
            tx[i] = __ldg(a.xt + clampi(tx0 - R + i, 0, a.OW - 1));
        else
            ty[i - SW] = __ldg(a.yt + clampi(ty0 - R + (i - SW), 0, a.OH - 1));
    }
    __syncthreads();
    for (int b = blockIdx.y; b < a.batch; b += gridDim.y) {
        const uint8_t *img = a.src + (long long)b * a.src_bstride;
        for (int base = 0; base < N; base += U * kFilterThreads) {
            float v[U][C];
#pragma unroll
            for (int q = 0; q < U; q++) {
                const int i = min(base + q * kFilterThreads + static_cast<int>(threadIdx.x), N - 1);
                const int sy = i / SW, sx = i - sy * SW;
#pragma unroll
                for (int c = 0; c < C; c++)
                    v[q][c] = bilinear_f32<WRAP>(img, a.src_pitch, C, c, tx[sx], ty[sy], a.W, a.H);
            }
#pragma unroll
            for (int q = 0; q < U; q++) {
                const int i = base + q * kFilterThreads + static_cast<int>(threadIdx.x);
                if (i < N) {
                    const int sy = i / SW, sx = i - sy * SW;
#pragma unroll
                    for (int c = 0; c < C; c++)
                        S[c][sy][sx] = v[q][c];
                }
            }
        }
        __syncthreads();
        float acc[RPT][C];
#pragma unroll
        for (int i = 0; i < RPT; i++)
#pragma unroll
            for (int c = 0; c < C; c++)
                acc[i][c] = 0.0f;
        // shared row yb + sr meets output rows yb + i with filter row sr - i
#pragma unroll
        for (int sr = 0; sr < RPT + K - 1; sr++) {
            float v[K][C];
#pragma unroll
            for (int k = 0; k < K; k++)
#pragma unroll
                for (int c = 0; c < C; c++)
                    v[k][c] = S[c][yb + sr][x + k];
#pragma unroll
            for (int i = 0; i < RPT; i++) {
                const int fr = sr - i;
                if (fr < 0 || fr >= K)
                    continue;
#pragma unroll
                for (int k = 0; k < K; k++)
#pragma unroll
                    for (int c = 0; c < C; c++)
                        acc[i][c] = fmaf(a.w[fr * K + k], v[k][c], acc[i][c]);
            }
        }
        const int ox = tx0 + x;
        if (ox < a.OW) {
#pragma unroll
            for (int i = 0; i < RPT; i++) {
                const int oy = ty0 + yb + i;
                if (oy < a.OH) {
                    float *op = reinterpret_cast<float *>(a.dst + (long long)b * a.dst_bstride +
                                                          (long long)oy * a.dst_pitch) + (long long)ox * C;
#pragma unroll
                    for (int c = 0; c < C; c++)
                        __stcs(op + c, acc[i][c]);
                }
            }
        }
        __syncthreads();   // the next image overwrites S
    }
}

// Swizzled rows (the 16-warp form): 16-byte group g of a staged input row
// sits at group g ^ ((g >> 3) & 1):
// with lanes reading 16-float windows eight floats apart, every 16-byte load
// of eight lanes then meets eight distinct bank groups, whatever the window's
// offset (without it lanes t and t + 4 collide).
__device__ __forceinline__ int swz(int e)
{
    const int g = e >> 2;
    return ((g ^ ((g >> 3) & 1)) << 2) | (e & 3);
}

// Standalone valid-region correlation; the layout of shared memory is given
// by filter_valid_smem (TH + K - 1 input tile rows of
// filter_valid_row_floats, then K rows of the weights zero-padded to a
// multiple of 8).  Grid: x walks column tiles, y row tiles.
template <int NT, bool SWZ>
__global__ void __launch_bounds__(NT) k_filter_valid(const float *__restrict__ src, long long src_pitch, int H, int W,
                                                     const float *__restrict__ wgt, int K, float *__restrict__ dst,
                                                     long long dst_pitch)
{
    constexpr int TH = valid_tile_rows(NT);
    extern __shared__ __align__(16) float smem[];
    const int KP = (K + 7) & ~7;
    const int SWF = filter_valid_row_floats(K);
    const int TR = TH + K - 1;   // staged input rows
    float *tile = smem;
    float *ws = smem + TR * SWF;
    const int OH = H - K + 1, OW = W - K + 1;
    const int x0 = blockIdx.x * kVTW, y0 = blockIdx.y * TH;
    grid_launch_dependents();
    grid_dependency_wait();
    // weights and input tile (rows y0 .. y0 + TR - 1, columns x0 .. x0 +
    // SWF - 1, zero past the image: those meet only zero weights or outputs
    // that are not stored) by asynchronous copies, all in flight at once;
    // neighbouring tiles read the same halo, so the copies keep L2 caching
    for (int i = threadIdx.x; i < K * KP; i += NT) {
        const int r = i / KP, c = i - r * KP;
        cp_async_4(ws + i, wgt + r * K + min(c, K - 1), c < K);
    }
    for (int r = 0; r < TR; r++) {
        const int gy = y0 + r;
        const float *row = reinterpret_cast<const float *>(reinterpret_cast<const uint8_t *>(src) +
                                                           (long long)min(gy, H - 1) * src_pitch);
        for (int c = threadIdx.x; c < SWF; c += NT) {
            const int gx = x0 + c;
            cp_async_4(tile + r * SWF + (SWZ ? swz(c) : c), row + min(gx, W - 1), gy < H && gx < W);
        }
    }
    cp_async_wait_all();
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float acc0[8], acc1[8];
#pragma unroll
    for (int j = 0; j < 8; j++)
        acc0[j] = acc1[j] = 0.0f;
    // input row rr (from the thread's first output row) meets output row 0
    // with filter row rr and output row 1 with filter row rr - 1
    for (int rr = 0; rr <= K; rr++) {
        const float *in = tile + (2 * warp + rr) * SWF;
        for (int kc = 0; kc < KP; kc += 8) {
            float win[16];
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const int e = 8 * lane + kc + 4 * q;
                const float4 f = *reinterpret_cast<const float4 *>(in + (SWZ ? swz(e) : e));
                win[4 * q] = f.x; win[4 * q + 1] = f.y; win[4 * q + 2] = f.z; win[4 * q + 3] = f.w;
            }
            if (rr < K) {
                const float *w0 = ws + rr * KP + kc;
                const float4 p = *reinterpret_cast<const float4 *>(w0);
                const float4 q = *reinterpret_cast<const float4 *>(w0 + 4);
                const float wv[8] = {p.x, p.y, p.z, p.w, q.x, q.y, q.z, q.w};
#pragma unroll
                for (int k = 0; k < 8; k++)
#pragma unroll
                    for (int j = 0; j < 8; j++)
                        acc0[j] = fmaf(wv[k], win[j + k], acc0[j]);
            }
            if (rr >= 1) {
                const float *w1 = ws + (rr - 1) * KP + kc;
                const float4 p = *reinterpret_cast<const float4 *>(w1);
                const float4 q = *reinterpret_cast<const float4 *>(w1 + 4);
                const float wv[8] = {p.x, p.y, p.z, p.w, q.x, q.y, q.z, q.w};
#pragma unroll
                for (int k = 0; k < 8; k++)
#pragma unroll
                    for (int j = 0; j < 8; j++)
                        acc1[j] = fmaf(wv[k], win[j + k], acc1[j]);
            }
        }
    }
    const int ox = x0 + 8 * lane;
#pragma unroll
    for (int rr = 0; rr < 2; rr++) {
        const int oy = y0 + 2 * warp + rr;
        if (oy >= OH)
            continue;
        float *op = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(dst) + (long long)oy * dst_pitch) + ox;
        const float *acc = rr ? acc1 : acc0;
        if (ox + 8 <= OW && ((reinterpret_cast<uintptr_t>(op) & 15) == 0)) {
            __stcs(reinterpret_cast<float4 *>(op), make_float4(acc[0], acc[1], acc[2], acc[3]));
            __stcs(reinterpret_cast<float4 *>(op) + 1, make_float4(acc[4], acc[5], acc[6], acc[7]));
        } else {
#pragma unroll
            for (int j = 0; j < 8; j++)
                if (ox + j < OW)
                    op[j] = acc[j];
        }
    }
}

}  // namespace

const void *resize_filter_kernel_for(int C, int K, bool wrap)
{
    using Fn = void (*)(const KArgs, const CUtensorMap);
#define RZ_FILTER_ROW(CC)                                                                                          \
    {k_resize_filter<CC, 1, false>, k_resize_filter<CC, 3, false>, k_resize_filter<CC, 5, false>,               \
     k_resize_filter<CC, 7, false>, k_resize_filter<CC, 1, true>, k_resize_filter<CC, 3, true>,                   \
     k_resize_filter<CC, 5, true>, k_resize_filter<CC, 7, true>}
    static const Fn k[3][8] = {RZ_FILTER_ROW(1), RZ_FILTER_ROW(3), RZ_FILTER_ROW(4)};
#undef RZ_FILTER_ROW
    const int ci = (C == 1) ? 0 : (C == 3 ? 1 : (C == 4 ? 2 : -1));
    if (ci < 0 || K < 1 || K > 7 || K % 2 == 0)
        return nullptr;
    return reinterpret_cast<const void *>(k[ci][(wrap ? 4 : 0) + K / 2]);
}

int launch_filter_valid(const float *src, long long src_pitch, int H, int W, const float *w, int K, float *dst,
                        long long dst_pitch, bool pdl, void *stream)
{
    // wide filters: CTAs of 16 warps (32 output rows, half the halo re-read
    // per output) with swizzled rows; narrower ones: 8 warps (16 rows), more
    // CTAs in flight, plain rows (the swizzle's index arithmetic cost them
    // more than the 2-way bank conflicts it removes: measured 94 against
    // 106 us at K = 8, 715 against 745 us at K = 32 on 4096^2)
    const int NT = valid_threads(K);
    const int OH = H - K + 1, OW = W - K + 1;
    const size_t smem = filter_valid_smem(K, NT);
    const void *fn = NT == 512 ? reinterpret_cast<const void *>(k_filter_valid<512, true>)
                               : reinterpret_cast<const void *>(k_filter_valid<256, false>);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess)
        return static_cast<int>(e);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((OW + kVTW - 1) / kVTW, (OH + valid_tile_rows(NT) - 1) / valid_tile_rows(NT), 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {&src, &src_pitch, &H, &W, &w, &K, &dst, &dst_pitch};
    e = cudaLaunchKernelExC(&cfg, fn, args);
    return static_cast<int>(e);
}

}  // namespace rz
