// K x K correlation over the valid region on the fifth-generation tensor
// cores (tcgen05), for the filter widths where it beats the FP32 FMA kernel
// (filter.cu k_filter_valid).
//
// The correlation of the convolution page ("OpenCL image convolution" §2),
//   out[y][x] = sum_{r, c < K} w[r][c] in[y + r][x + c],
// is, for a tile of 128 output rows (y0 + m) by 32 output columns (x0 + n),
// a sum over the filter rows r of one matrix product each:
//   D[m][n] += sum_t A_r[m][t] T_r[t][n],
//   A_r[m][t] = in[y0 + r + m][x0 + t],   T_r[t][n] = w[r][t - n] (0 when t - n is outside [0, K)),
// with t over K_T = 32 ch >= 32 + K - 1 input columns: T_r is the banded
// Toeplitz matrix of filter row r.  A_r is the staged input tile shifted down
// r rows, so one TMA load of the tile serves every r: the shared-memory
// descriptor of A_r starts r rows (r * 128 bytes) into it, which the 128-byte
// swizzle follows because the hardware swizzles absolute shared addresses
// (the tile is 1024-byte aligned, as the TMA load requires).
//
// Precision: each float is split into hi = its top 19 bits (a TF32 value:
// sign, exponent, 10 mantissa bits) and lo = x - hi, and the products are
// formed as hi*hi + hi*lo + lo*hi (three TF32 MMAs, FP32 accumulation in
// tensor memory), the standard three-pass TF32 scheme for float32 accuracy.
//
// One CTA per output tile (512 threads; the staged tile, its lo part, two
// Toeplitz buffers and the filter take 214 KB of shared memory): thread 0
// loads the input tile by TMA and all threads split it; then warps 0..14
// build T_r (hi and lo) for each filter row into one of two buffers and
// signal it on the buffer's `full` mbarrier, while one lane of warp 15
// issues each row's 3 * 4 ch MMAs (M = 128, N = 32, K = 8) as soon as its
// tile is ready and commits them to the buffer's `empty` mbarrier, which
// hands the buffer back to the builders (no CTA-wide barrier in the loop).  The 128 x 32 float32
// accumulator lives in tensor memory (32 columns) and leaves through
// tcgen05.ld (warp w reads lanes 32w .. 32w + 31).  Every wait is bounded
// (1 s; RZ_ERR_TIMEOUT in the optional status word) and tensor memory is
// always released.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "gbresize.h"

namespace rz {
namespace {

constexpr int kTcRows = 128;                   // output rows per tile (MMA M)
constexpr int kTcCols = 32;                    // output columns per tile (MMA N)
constexpr int kTcInRows = 192;                 // staged input rows (kTcRows + K - 1 <= 191)
constexpr int kTcChunkA = kTcInRows * 128;     // bytes of one 32-float column chunk of the input tile
constexpr int kTcMaxChunks = 3;                // K_T = 32 * chunks >= kTcCols + K - 1 (K <= 65)
constexpr int kTcChunkB = kTcCols * 128;       // bytes of one chunk of a Toeplitz tile
constexpr int kOffA = 0;
constexpr int kOffALo = kTcMaxChunks * kTcChunkA;
constexpr int kOffB = 2 * kTcMaxChunks * kTcChunkA;
constexpr int kBufB = 2 * kTcMaxChunks * kTcChunkB;   // hi and lo of one filter row
constexpr int kOffBar = kOffB + 2 * kBufB;
constexpr int kOffW = kOffBar + 64;
constexpr int kTcMaxK = 64;
constexpr int kTcMinK = 16;                   // below, the FP32 bound of a K x K sum is tighter than three TF32 products hold
constexpr int kTcSmem = kOffW + kTcMaxK * kTcMaxK * 4 + 1024;   // + slack for 1024-byte alignment
constexpr int kTcThreads = 512;
constexpr int kTcBuilders = kTcThreads - 32;    // warps 0..14 build Toeplitz tiles; warp 15 lane 0 issues MMAs
constexpr unsigned long long kTcWaitNs = 1000000000ull;

struct TcArgs {
    float *dst;
    long long dst_pitch;   // bytes
    const float *w;        // K * K, device
    int OH, OW, K, chunks, tiles_x;
    int *status;           // device status word or nullptr
};

__device__ __forceinline__ uint32_t sa(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool bar_try(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity), "r"(100000u)
                 : "memory");
    return ok != 0;
}

// Wait for phase `parity`, at most kTcWaitNs; false (and RZ_ERR_TIMEOUT in the
// status word) on time-out.
__device__ bool bar_wait(uint32_t bar, uint32_t parity, int *status)
{
    if (bar_try(bar, parity))
        return true;
    uint64_t t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    while (!bar_try(bar, parity)) {
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 > kTcWaitNs) {
            if (status)
                atomicExch(status, RZ_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle (start address
// >> 4; leading offset 16 B, unused by swizzled K-major layouts; 8-row
// groups 1024 B apart; descriptor version 1; layout 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr)
{
    return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (1ull << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) |
           (1ull << 46) | (2ull << 61);
}

// Instruction descriptor: D float32, A and B TF32, both K-major, N, M.
constexpr uint32_t kTcIdesc = (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(kTcCols >> 3) << 17) |
                              (static_cast<uint32_t>(kTcRows >> 4) << 24);

__device__ __forceinline__ void mma_tf32(uint32_t d, uint64_t a, uint64_t b, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
                 "l"(a), "l"(b), "r"(kTcIdesc), "r"(accumulate)
                 : "memory");
}

// True on every builder thread when v holds on all of them (a barrier among
// the builders with an AND reduction).
__device__ __forceinline__ bool builders_all(bool v)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 1, %2, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r)
                 : "r"(static_cast<uint32_t>(v)), "n"(kTcBuilders)
                 : "memory");
    return r != 0;
}

__device__ __forceinline__ float tf32_hi(float x) { return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }

__global__ void __launch_bounds__(kTcThreads, 1) k_filter_tc(const TcArgs p, const __grid_constant__ CUtensorMap map)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = sa(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;     // 1024-byte aligned base (128-byte swizzle atoms)
    uint8_t *base = smem_raw + (sb - raw);
    // barriers: the input tile; buffer b built (full + 8 b); buffer b's MMAs done (empty + 8 b)
    const uint32_t bar_tma = sb + kOffBar, bar_full = sb + kOffBar + 8, bar_empty = sb + kOffBar + 24;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + kOffBar + 40);
    int *n_commit = reinterpret_cast<int *>(base + kOffBar + 44);
    float *wsm = reinterpret_cast<float *>(base + kOffW);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int x0 = (blockIdx.x % p.tiles_x) * kTcCols, y0 = (blockIdx.x / p.tiles_x) * kTcRows;
    const int K = p.K, CH = p.chunks;
    asm volatile("griddepcontrol.launch_dependents;" :::);

    if (threadIdx.x == 0) {
        bar_init(bar_tma, 1);
        bar_init(bar_full, 1);
        bar_init(bar_full + 8, 1);
        bar_init(bar_empty, 1);
        bar_init(bar_empty + 8, 1);
        *n_commit = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sa(tmem_slot)),
                     "r"(32u)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // this builder thread's 16-byte units of every Toeplitz tile (the same
    // for every filter row): unit (row n, chunk c, unit q) sits at c *
    // kTcChunkB + n * 128 + (q ^ (n & 7)) * 16 (the 128-byte swizzle) and
    // holds filter columns d = 32 c + 4 q - n + e, e < 4
    constexpr int kUnits = (kTcCols * kTcMaxChunks * 8 + kTcBuilders - 1) / kTcBuilders;
    int uoff[kUnits], ud[kUnits];
    const int units = kTcCols * CH * 8;
#pragma unroll
    for (int k = 0; k < kUnits; k++) {
        const int u = threadIdx.x + k * kTcBuilders;
        const int n = u / (CH * 8), rem = u - n * CH * 8, c = rem >> 3, q = rem & 7;
        uoff[k] = (threadIdx.x < kTcBuilders && u < units) ? c * kTcChunkB + n * 128 + ((q ^ (n & 7)) << 4) : -1;
        ud[k] = c * 32 + q * 4 - n;
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    // inputs may be written by the previous kernel in the stream
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar_tma),
                     "r"(static_cast<uint32_t>(CH * kTcChunkA))
                     : "memory");
        for (int c = 0; c < CH; c++)
            asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
                         "[%0], [%1, {%2, %3}], [%4];" ::"r"(sb + kOffA + c * kTcChunkA),
                         "l"(reinterpret_cast<uint64_t>(&map)), "r"(x0 + 32 * c), "r"(y0), "r"(bar_tma)
                         : "memory");
    }
    for (int i = threadIdx.x; i < K * K; i += kTcThreads)
        wsm[i] = __ldg(p.w + i);
    bool ok = bar_wait(bar_tma, 0, p.status);
    // hi / lo split of the staged tile, elementwise (so the swizzled layout stays)
    {
        float4 *a4 = reinterpret_cast<float4 *>(base + kOffA);
        float4 *l4 = reinterpret_cast<float4 *>(base + kOffALo);
        const int n4 = CH * kTcChunkA / 16;
        for (int i = threadIdx.x; i < n4; i += kTcThreads) {
            const float4 v = a4[i];
            const float4 h = make_float4(tf32_hi(v.x), tf32_hi(v.y), tf32_hi(v.z), tf32_hi(v.w));
            a4[i] = h;
            l4[i] = make_float4(v.x - h.x, v.y - h.y, v.z - h.z, v.w - h.w);
        }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic writes -> tensor-core reads
    ok = __syncthreads_and(ok ? 1 : 0) != 0;   // one decision for the whole CTA

    if (threadIdx.x < kTcBuilders) {
        // builders: Toeplitz tile of filter row r into buffer r & 1 once the
        // MMAs of row r - 2 have released it; one arrival per tile
        for (int r = 0; r < K && ok; r++) {
            const int buf = r & 1;
            const bool freed = r < 2 || bar_wait(bar_empty + 8 * buf, ((r >> 1) - 1) & 1, p.status);
            ok = builders_all(freed);   // the same decision in every builder: the named barriers stay matched
            if (!ok)
                break;
            uint8_t *bh = base + kOffB + buf * kBufB, *bl = bh + kTcMaxChunks * kTcChunkB;
            const float *wr = wsm + r * K;
#pragma unroll
            for (int k = 0; k < kUnits; k++) {
                if (uoff[k] < 0)
                    continue;
                float v[4];
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const int d = ud[k] + e;
                    v[e] = (d >= 0 && d < K) ? wr[d] : 0.0f;
                }
                const float4 h = make_float4(tf32_hi(v[0]), tf32_hi(v[1]), tf32_hi(v[2]), tf32_hi(v[3]));
                *reinterpret_cast<float4 *>(bh + uoff[k]) = h;
                *reinterpret_cast<float4 *>(bl + uoff[k]) =
                    make_float4(v[0] - h.x, v[1] - h.y, v[2] - h.z, v[3] - h.w);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            asm volatile("bar.sync 1, %0;" ::"n"(kTcBuilders) : "memory");
            if (threadIdx.x == 0)
                asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar_full + 8 * buf) : "memory");
        }
    } else if (threadIdx.x == kTcBuilders) {
        // the issuer: the row's 3 x 4 CH MMAs as soon as its tile is built;
        // descriptors advance by adding (byte offset >> 4) to the start field
        const uint64_t a_hi = smem_desc(sb + kOffA), a_lo = smem_desc(sb + kOffALo);
        for (int r = 0; r < K && ok; r++) {
            const int buf = r & 1;
            ok = bar_wait(bar_full + 8 * buf, (r >> 1) & 1, p.status);
            if (!ok)
                break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint64_t b_hi = smem_desc(sb + kOffB + buf * kBufB);
            const uint64_t b_lo = b_hi + ((kTcMaxChunks * kTcChunkB) >> 4);
#pragma unroll 4
            for (int s = 0; s < 4 * CH; s++) {
                const uint32_t koff = (s & 3) * 32;                                   // 8 TF32 along K
                const uint64_t da = (static_cast<uint32_t>((s >> 2) * kTcChunkA) + r * 128 + koff) >> 4;
                const uint64_t db = (static_cast<uint32_t>((s >> 2) * kTcChunkB) + koff) >> 4;
                mma_tf32(tmem, a_hi + da, b_hi + db, (r > 0 || s > 0) ? 1u : 0u);
                mma_tf32(tmem, a_hi + da, b_lo + db, 1u);
                mma_tf32(tmem, a_lo + da, b_hi + db, 1u);
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                             bar_empty + 8 * buf)
                         : "memory");
            *n_commit = r + 1;
        }
    }
    __syncthreads();
    // the last commit completes after every MMA issued before it
    const int last = *n_commit - 1;
    bool done = last == K - 1 && bar_wait(bar_empty + 8 * (last & 1), (last >> 1) & 1, p.status);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp < 4) {
        uint32_t v[32];
        const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * warp) << 16);
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
            "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
              "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
              "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]),
              "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]),
              "=r"(v[30]), "=r"(v[31])
            : "r"(taddr)
            : "memory");
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        const int row = y0 + 32 * warp + lane;
        if (row < p.OH && ok && done) {
            float *out = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(p.dst) + row * p.dst_pitch) + x0;
            if (x0 + 32 <= p.OW && (reinterpret_cast<uintptr_t>(out) & 15) == 0) {
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4 *>(out + j) = make_float4(
                        __uint_as_float(v[j]), __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]),
                        __uint_as_float(v[j + 3]));
            } else {
#pragma unroll
                for (int j = 0; j < 32; j++)
                    if (x0 + j < p.OW)
                        out[j] = __uint_as_float(v[j]);
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(32u) : "memory");
}

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encoder()
{
    static std::once_flag once;
    static EncodeFn fn = nullptr;
    std::call_once(once, [] {
        void *q = nullptr;
        cudaDriverEntryPointQueryResult r;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000, cudaEnableDefault, &r) ==
                cudaSuccess &&
            r == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(q);
    });
    return fn;
}

std::mutex g_tc_attr_mu;
int g_tc_attr_dev[64];
bool g_tc_attr_set[64];

}  // namespace

// The tensor-core path applies: 16 <= K <= 64, and the source layout the TMA
// tensor map needs (16-byte aligned base, pitch a multiple of 16 bytes).
bool filter_tc_supported(const float *src, long long src_pitch, int K)
{
    return K >= kTcMinK && K <= kTcMaxK && (reinterpret_cast<uintptr_t>(src) & 15) == 0 && (src_pitch & 15) == 0;
}

// Launch the tensor-core correlation; returns a cudaError_t (0 on success,
// cudaErrorInvalidValue when the tensor map cannot be built).
int launch_filter_tc(const float *src, long long src_pitch, int H, int W, const float *w, int K, float *dst,
                     long long dst_pitch, int *status, bool pdl, void *stream)
{
    const int OH = H - K + 1, OW = W - K + 1;
    if (OH <= 0 || OW <= 0)
        return 0;
    EncodeFn enc = encoder();
    if (!enc)
        return static_cast<int>(cudaErrorNotSupported);
    CUtensorMap map;
    std::memset(&map, 0, sizeof(map));
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(W), static_cast<cuuint64_t>(H)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(src_pitch)};
    const cuuint32_t box[2] = {32, kTcInRows};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(src), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return static_cast<int>(cudaErrorInvalidValue);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return static_cast<int>(e);
    {
        std::lock_guard<std::mutex> lk(g_tc_attr_mu);
        if (dev < 0 || dev >= 64)
            return static_cast<int>(cudaErrorInvalidDevice);
        if (!g_tc_attr_set[dev]) {
            e = cudaFuncSetAttribute(k_filter_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
            if (e != cudaSuccess)
                return static_cast<int>(e);
            g_tc_attr_set[dev] = true;
        }
    }
    TcArgs a;
    a.dst = dst;
    a.dst_pitch = dst_pitch;
    a.w = w;
    a.OH = OH;
    a.OW = OW;
    a.K = K;
    a.chunks = (kTcCols + K - 1 + 31) / 32;
    a.tiles_x = (OW + kTcCols - 1) / kTcCols;
    a.status = status;
    const long long tiles = static_cast<long long>(a.tiles_x) * ((OH + kTcRows - 1) / kTcRows);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles), 1, 1);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = kTcSmem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return static_cast<int>(cudaLaunchKernelEx(&cfg, k_filter_tc, a, map));
}

}  // namespace rz
