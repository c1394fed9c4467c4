// Device helpers shared by the kernels (kernels.cu, stream.cu, direct.cu,
// filter.cu, multi.cu, texture.cu): inline PTX for mbarriers, bulk (TMA) copies,
// programmatic dependent launch and cache policies, and the exact sampling
// index the producers derive without touching the tables.  Nothing here is
// part of the C ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "rz_internal.h"

namespace rz {
namespace dev {

// ------------------------------------------------------------------ bounds-checked build
//
// Built with -DRZ_CHECK_BOUNDS (a separate library, for tests), every global
// load and store of the resize kernels goes through the wrappers below, which
// check the address against the extents the kernel recorded at entry
// (bounds_begin: source, output, table block) and every shared-memory copy
// and read window against the CTA's dynamic shared memory.  An access outside
// them is not made: the thread records RZ_ERR_ARG in the status word (the
// first error recorded stays) and goes on with a zero value, and a refused
// bulk copy still completes its barrier's transaction count, so no wait is
// left hanging.  In the normal build the wrappers are the plain accesses.
struct BoundsRec {
    const uint8_t *src, *dst, *tab;
    long long src_n, dst_n, tab_n;
    int *status;
};

#ifdef RZ_CHECK_BOUNDS
static __shared__ BoundsRec g_bounds;

// Record the kernel's extents (every thread writes the same values).
__device__ __forceinline__ void bounds_begin(const KArgs &a)
{
    g_bounds.src = a.src;
    g_bounds.dst = a.dst;
    g_bounds.tab = a.tab;
    g_bounds.src_n = a.src_extent;
    g_bounds.dst_n = a.dst_extent;
    g_bounds.tab_n = a.tab_bytes;
    g_bounds.status = a.status;
}

static __device__ __noinline__ void bounds_fault()
{
    if (g_bounds.status)
        atomicCAS(g_bounds.status, RZ_OK, RZ_ERR_ARG);
}

__device__ __forceinline__ bool in_span(const void *p, long long n, const uint8_t *base, long long extent)
{
    const uint8_t *c = static_cast<const uint8_t *>(p);
    return base != nullptr && n >= 0 && c >= base && c + n <= base + extent;
}

__device__ __forceinline__ bool read_ok(const void *p, long long n)
{
    return in_span(p, n, g_bounds.src, g_bounds.src_n) || in_span(p, n, g_bounds.tab, g_bounds.tab_n);
}

__device__ __forceinline__ bool write_ok(const void *p, long long n) { return in_span(p, n, g_bounds.dst, g_bounds.dst_n); }

extern __shared__ __align__(16) uint8_t rz_dynamic_smem[];

__device__ __forceinline__ bool smem_ok(const void *p, long long n)
{
    uint32_t dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    return in_span(p, n, rz_dynamic_smem, dyn);
}

// Check a shared-memory window [p, p + n) a thread is about to read or write.
#define RZ_SMEM_CHECK(p, n)                                                   \
    do {                                                                      \
        if (!::rz::dev::smem_ok((p), (n))) ::rz::dev::bounds_fault();        \
    } while (0)
#else
__device__ __forceinline__ void bounds_begin(const KArgs &) {}
#define RZ_SMEM_CHECK(p, n) \
    do {                    \
    } while (0)
#endif

// True when [p, p + n) may be read: the CTA's dynamic shared memory for a
// shared address, the source or the tables otherwise (always in the normal
// build); a false result is recorded in the checked build.
__device__ __forceinline__ bool read_guard(const void *p, long long n)
{
#ifdef RZ_CHECK_BOUNDS
    if (!(__isShared(p) ? smem_ok(p, n) : read_ok(p, n))) {
        bounds_fault();
        return false;
    }
#else
    (void)p;
    (void)n;
#endif
    return true;
}

// True when [p, p + n) lies in the CTA's dynamic shared memory (always in the
// normal build); in the checked build a false result is recorded.  Callers
// make the access only when it returns true.
__device__ __forceinline__ bool smem_guard(const void *p, long long n)
{
#ifdef RZ_CHECK_BOUNDS
    if (!smem_ok(p, n)) {
        bounds_fault();
        return false;
    }
#else
    (void)p;
    (void)n;
#endif
    return true;
}

// A float from shared memory (0 and recorded when outside the CTA's dynamic
// shared memory, in the checked build).
__device__ __forceinline__ float lds_f(const float *p) { return smem_guard(p, 4) ? *p : 0.0f; }

// Global loads and stores of the resize kernels (checked in the checked
// build): ld_nc = ld.global.nc (__ldg), ld_cs / st_cs = streaming (__ldcs /
// __stcs), ld_g / st_g = plain.
template <class T>
__device__ __forceinline__ T ld_nc(const T *p)
{
#ifdef RZ_CHECK_BOUNDS
    if (!read_ok(p, sizeof(T))) {
        bounds_fault();
        return T{};
    }
#endif
    return __ldg(p);
}

template <class T>
__device__ __forceinline__ T ld_cs(const T *p)
{
#ifdef RZ_CHECK_BOUNDS
    if (!read_ok(p, sizeof(T))) {
        bounds_fault();
        return T{};
    }
#endif
    return __ldcs(p);
}

template <class T>
__device__ __forceinline__ T ld_g(const T *p)
{
#ifdef RZ_CHECK_BOUNDS
    if (!read_ok(p, sizeof(T))) {
        bounds_fault();
        return T{};
    }
#endif
    return *p;
}

template <class T>
__device__ __forceinline__ void st_cs(T *p, T v)
{
#ifdef RZ_CHECK_BOUNDS
    if (!write_ok(p, sizeof(T))) {
        bounds_fault();
        return;
    }
#endif
    __stcs(p, v);
}

template <class T>
__device__ __forceinline__ void st_g(T *p, T v)
{
#ifdef RZ_CHECK_BOUNDS
    if (!write_ok(p, sizeof(T))) {
        bounds_fault();
        return;
    }
#endif
    *p = v;
}

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

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Complete `bytes` of the barrier's expected transaction count without a
// copy (the checked build's stand-in for a refused bulk copy).
__device__ __forceinline__ void mbar_complete_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.complete_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Barrier among the consumer warps only (the producer warp never joins it).
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

// Consumer barrier that also returns whether `v` held on any consumer thread.
__device__ __forceinline__ bool consumer_any(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "n"(kConsumers)
        : "memory");
    return r != 0;
}

// One bounded wait attempt: the thread may be suspended in hardware until the
// phase completes or about 0.5 ms pass (suspend-time hint), so waiting warps
// do not spin through issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(500000u)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of the barrier, at most limit_ns (kWaitLimitNs).  Between
// attempts the waiting warp sleeps (32 ns, doubling up to 256 ns) so that it
// leaves the issue slots to the warps computing on the same scheduler.  On
// time-out the status word (if given) records RZ_ERR_TIMEOUT and false is
// returned.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, int *status,
                                                  uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_ns();
    unsigned int nap = 32;
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > limit_ns) {
            if (status)
                atomicExch(status, RZ_ERR_TIMEOUT);
            return false;
        }
        __nanosleep(nap);
        if (nap < 256)
            nap <<= 1;
    }
    return true;
}

// Bulk copy global -> this CTA's shared memory, completing on `bar`, with an
// L2 cache policy (createpolicy) attached.  Both addresses 16-byte aligned,
// bytes a multiple of 16.
__device__ __forceinline__ void bulk_load_hint(void *sdst, const void *gsrc, uint32_t bytes, uint64_t *bar,
                                               uint64_t policy)
{
#ifdef RZ_CHECK_BOUNDS
    if (!read_ok(gsrc, bytes) || !smem_ok(sdst, bytes)) {
        bounds_fault();
        mbar_complete_tx(bar, bytes);
        return;
    }
#endif
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_addr(sdst)),
        "l"(gsrc), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Tensor-map copy of one box {words, rows, 1} at coordinates {word, row,
// image} into shared memory, completing on `bar`.  The map's elements are
// 8-byte words and `word` is even, so the copy starts on a 16-byte boundary;
// parts of the box outside the image are zero-filled, not read.
__device__ __forceinline__ void tensor_load_3d(void *sdst, const CUtensorMap *map, int word, int row, int image,
                                               uint64_t *bar, uint64_t policy, uint32_t box_bytes)
{
#ifdef RZ_CHECK_BOUNDS
    // (the tensor map keeps the global side inside the image: parts of the
    // box outside it are zero-filled)
    if (!smem_ok(sdst, box_bytes)) {
        bounds_fault();
        mbar_complete_tx(bar, box_bytes);
        return;
    }
#else
    (void)box_bytes;
#endif
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(sdst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(word), "r"(row), "r"(image), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Bulk copy global -> this CTA's shared memory with the default L2 policy
// (for the sampling tables, which every tile row reads again).
__device__ __forceinline__ void bulk_load(void *sdst, const void *gsrc, uint32_t bytes, uint64_t *bar)
{
#ifdef RZ_CHECK_BOUNDS
    if (!read_ok(gsrc, bytes) || !smem_ok(sdst, bytes)) {
        bounds_fault();
        mbar_complete_tx(bar, bytes);
        return;
    }
#endif
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(sdst)),
        "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// L2 policy for data read once: evicted first, so that the small sampling
// tables (read by every launch) stay resident.
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Programmatic dependent launch: wait until the grids this launch depends on
// have completed and their memory is visible; allow the next grid in the
// stream to start launching.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// Ask the memory system to start moving [p, p + bytes) from HBM into L2 (a
// bulk prefetch, cp.async.bulk.prefetch.L2).  It is a hint: it reads nothing
// into registers or shared memory and cannot change any result, so a kernel
// may issue it before griddepcontrol.wait, while the grid it depends on is
// still running (L2 is the device's point of coherence, so a line that grid
// writes later is updated there).  The range is shrunk inward to 16-byte
// bounds, so every prefetched byte lies inside [p, p + bytes).
__device__ __forceinline__ void l2_prefetch_span(const uint8_t *p, long long bytes)
{
    const uintptr_t a0 = (reinterpret_cast<uintptr_t>(p) + 15) & ~static_cast<uintptr_t>(15);
    const uintptr_t a1 = (reinterpret_cast<uintptr_t>(p) + static_cast<uintptr_t>(bytes)) & ~static_cast<uintptr_t>(15);
#ifdef RZ_CHECK_BOUNDS
    if (bytes > 0 && a1 > a0 && !read_ok(reinterpret_cast<const void *>(a0), static_cast<long long>(a1 - a0))) {
        bounds_fault();
        return;
    }
#endif
    if (bytes > 0 && a1 > a0)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a0), "r"(static_cast<uint32_t>(a1 - a0))
                     : "memory");
}

// Pre-wait prefetch of the source bytes one CTA of a direct kernel will read.
// The CTA's work items are [g0, g0 + n) of a grid laid out `per_unit` items
// per unit (an output row, or a source row for the 2x upscale), `units`
// units in all (units * per_unit < 2^31); item j of unit u reads bytes
// [j GB + lead, j GB + lead + GB + extra) of the NR source rows row(u, k),
// k < NR (row() < 0: none).  Thread t takes the piece (unit u0 + t / NR,
// row k = t % NR), one bulk prefetch clipped to [0, row_bytes) of that row;
// pieces past the block's threads are skipped (a hint may cover less).
template <int NR, class RowFn>
__device__ __forceinline__ void prefetch_items(const uint8_t *img, long long pitch, long long row_bytes, int per_unit,
                                               int units, int g0, int n, int GB, int lead, int extra, RowFn row)
{
    const int g1 = min(g0 + n, units * per_unit);
    if (g0 >= g1) return;
    const int u = g0 / per_unit + static_cast<int>(threadIdx.x) / NR;
    if (u > (g1 - 1) / per_unit) return;
    const int k = static_cast<int>(threadIdx.x) % NR;
    const int jlo = max(g0 - u * per_unit, 0), jhi = min(g1 - u * per_unit, per_unit);
    const long long b0 = max(static_cast<long long>(jlo) * GB + lead, 0LL);
    const long long b1 = min(static_cast<long long>(jhi) * GB + lead + extra, row_bytes);
    const int r = row(u, k);
    if (r < 0 || b1 <= b0) return;
    l2_prefetch_span(img + static_cast<long long>(r) * pitch + b0, b1 - b0);
}

// Bulk copy shared -> global (bulk-group completion).
__device__ __forceinline__ void bulk_store(void *gdst, const void *ssrc, uint32_t bytes)
{
#ifdef RZ_CHECK_BOUNDS
    if (!write_ok(gdst, bytes) || !smem_ok(ssrc, bytes)) {
        bounds_fault();
        return;
    }
#endif
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_addr(ssrc)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N committed bulk-store groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

// Index k in [-1, n] of an axis of n samples mapped inside by the border
// rule (CUDA interpolation page §6.1): clamp repeats the edge sample, mirror
// reflects about it (-1 -> 1, n -> n - 2), wrap repeats the axis (-1 -> n - 1,
// n -> 0); a one-sample axis reads sample 0.  Indices further out map to a
// sample inside (callers use them for no output).  Under clamp this is
// clampi(k, 0, n - 1).
__device__ __forceinline__ int border_index(int k, int n, int border)
{
    if (k < 0)
        return border == RZ_BORDER_WRAP ? n - 1 : (border == RZ_BORDER_MIRROR ? min(1, n - 1) : 0);
    if (k >= n)
        return border == RZ_BORDER_WRAP ? 0 : (border == RZ_BORDER_MIRROR ? max(n - 2, 0) : n - 1);
    return k;
}

// The far tap of a bilinear pair whose near tap is k (0 <= k < n): k + 1,
// or past the last sample sample 0 under the wrap rule, else the last.
template <bool WRAP>
__device__ __forceinline__ int far_tap(int k, int n)
{
    return k + 1 < n ? k + 1 : (WRAP ? 0 : n - 1);
}

__device__ __forceinline__ int ceil_log2(int v) { return v <= 1 ? 0 : 32 - __clz(v - 1); }

// floor(num / den) for 0 < den <= 2^17 and |num / den| < 2^17 + 1, exactly:
// the fast float quotient (num rounded to float, a division within 2 ulp)
// is off by less than 2^-4 there, so its floor is within one of the true
// floor, and 64-bit integer checks correct it.
__device__ __forceinline__ int floor_div_exact(long long num, int den)
{
    int q = __float2int_rd(__fdividef(static_cast<float>(num), static_cast<float>(den)));
    const long long qd = static_cast<long long>(q) * den;
    if (qd > num)
        q -= 1;
    else if (qd + den <= num)
        q += 1;
    return q;
}

// Source row/column sampled by output index d, exactly as the plan's tables
// hold it: bilinear floor(((2d+1) n_in - n_out) / (2 n_out)) folded into
// [0, n_in - 1], where under the mirror rule an entry at the last sample with
// a far tap of non-zero weight is held as the pair (n_in - 2, n_in - 1);
// nearest floor(d n_in / n_out) kept below n_in.  (Wrap plans never reach
// the kernels that call this.)  The producer needs only these indices (not
// the weights) to stage a tile, so it derives them without touching global
// memory.
template <int LINEAR>
__device__ __forceinline__ int sample_index(int n_in, int n_out, int d, int border)
{
    int s;
    if (LINEAR) {
        const long long num = (2LL * d + 1) * n_in - n_out;
        s = floor_div_exact(num, 2 * n_out);
        if (s >= n_in - 1 && border == RZ_BORDER_MIRROR && n_in > 1 && num != static_cast<long long>(s) * 2 * n_out)
            return n_in - 2;
    } else {
        s = floor_div_exact(static_cast<long long>(d) * n_in, n_out);
    }
    return s < 0 ? 0 : (s > n_in - 1 ? n_in - 1 : s);
}

// Exact horizontal tap sum of one staged uint8 row for one output pixel:
// h[c] = A0 * row[o0 + c] + A1 * row[o0 + C + c] (at most 2048 * 255), with
// aw = A0 | A1 << 16.  The 2C tap bytes are fetched as 32-bit words (up to
// 11 bytes past the taps: the staged rows carry 16 bytes of padding), each
// channel's pair is gathered into one 16-bit lane pair by a byte permute, and
// dp2a forms the sum.  For C = 4, o0 must be a multiple of 4.
template <int C>
__device__ __forceinline__ void hsum_u8(const uint8_t *row, int o0, uint32_t aw, int (&h)[C])
{
    if (!read_guard(row + (C == 4 ? o0 : (o0 & ~3)), C == 3 ? 12 : 8)) {
#pragma unroll
        for (int c = 0; c < C; c++)
            h[c] = 0;
        return;
    }
    if constexpr (C == 4) {
        const uint32_t t0 = *reinterpret_cast<const uint32_t *>(row + o0);
        const uint32_t t1 = *reinterpret_cast<const uint32_t *>(row + o0 + 4);
        const uint32_t p01 = __byte_perm(t0, t1, 0x5140);   // c0 pair, c1 pair
        const uint32_t p23 = __byte_perm(t0, t1, 0x7362);   // c2 pair, c3 pair
        h[0] = static_cast<int>(__dp2a_lo(aw, p01, 0u));
        h[1] = static_cast<int>(__dp2a_hi(aw, p01, 0u));
        h[2] = static_cast<int>(__dp2a_lo(aw, p23, 0u));
        h[3] = static_cast<int>(__dp2a_hi(aw, p23, 0u));
    } else {
        const int base = o0 & ~3;
        const uint32_t sel = 0x3210u + 0x1111u * static_cast<uint32_t>(o0 & 3);
        const uint32_t *w = reinterpret_cast<const uint32_t *>(row + base);
        const uint32_t w0 = w[0], w1 = w[1];
        const uint32_t lo4 = __byte_perm(w0, w1, sel);      // bytes o0 .. o0+3
        if constexpr (C == 1) {
            h[0] = static_cast<int>(__dp2a_lo(aw, lo4, 0u));
        } else {
            const uint32_t hi4 = __byte_perm(w1, w[2], sel);  // bytes o0+4 .. o0+7
            const uint32_t p01 = __byte_perm(lo4, hi4, 0x4130);  // t0c0 t1c0 t0c1 t1c1
            const uint32_t p2 = __byte_perm(lo4, hi4, 0x0052);   // t0c2 t1c2
            h[0] = static_cast<int>(__dp2a_lo(aw, p01, 0u));
            h[1] = static_cast<int>(__dp2a_hi(aw, p01, 0u));
            h[2] = static_cast<int>(__dp2a_lo(aw, p2, 0u));
        }
    }
}

// Pack the low bytes of four ints into one word (first int in byte 0).
__device__ __forceinline__ uint32_t pack4(int a, int b, int c, int d)
{
    return __byte_perm(__byte_perm(static_cast<uint32_t>(a), static_cast<uint32_t>(b), 0x0040),
                       __byte_perm(static_cast<uint32_t>(c), static_cast<uint32_t>(d), 0x0040), 0x5410);
}

// ------------------------------------------------------------------ exact 2x downscale

// Exact 2x downscale of uint8 (W = 2 OW, H = 2 OH).  Every column and row then
// samples x = 2d + 1/2, so A0 = A1 = B0 = B1 = 1024 and the bilinear sum
// reduces to out = (t0 + t1 + b0 + b1 + 2) >> 2: the same value, bit for bit.
// The four taps are summed with dp4a; weights of 64 and a start of 128 put
// 64 (sum + 2) in the accumulator (at most 65408), whose byte 1 is the
// rounded result, so byte permutes pack it.

__device__ __forceinline__ uint32_t pick_byte1(uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    return __byte_perm(__byte_perm(a, b, 0x0051), __byte_perm(c, d, 0x0051), 0x5410);
}

// One group of down2_px(C) output pixels: tw / bw are the group's source
// words of the upper / lower row
// (2 down2_px(C) C / 4 words each), o receives the down2_px(C) C / 4 output
// words.
template <int C>
__device__ __forceinline__ void down2_group(const uint32_t *tw, const uint32_t *bw, uint32_t *o)
{
    if constexpr (C == 1) {
        uint32_t s[8];
#pragma unroll
        for (int k = 0; k < 4; k++) {
            s[2 * k] = __dp4a(tw[k], 0x00004040u, __dp4a(bw[k], 0x00004040u, 128u));
            s[2 * k + 1] = __dp4a(tw[k], 0x40400000u, __dp4a(bw[k], 0x40400000u, 128u));
        }
        o[0] = pick_byte1(s[0], s[1], s[2], s[3]);
        o[1] = pick_byte1(s[4], s[5], s[6], s[7]);
    } else if constexpr (C == 3) {
        // 24 source bytes per row = words w0..w5; output pixel q covers source
        // bytes [6q, 6q + 6): channel c sums bytes 6q+c and 6q+3+c
        uint32_t s[12];
#pragma unroll
        for (int q = 0; q < 4; q += 2) {
            // even pixel: bytes 0..5 of words (k, k+1) with k = 3q/2
            const int k = 3 * q / 2;
            s[3 * q + 0] = __dp4a(tw[k], 0x40000040u, __dp4a(bw[k], 0x40000040u, 128u));
            s[3 * q + 1] = __dp4a(tw[k], 0x00004000u,
                                  __dp4a(tw[k + 1], 0x00000040u,
                                         __dp4a(bw[k], 0x00004000u, __dp4a(bw[k + 1], 0x00000040u, 128u))));
            s[3 * q + 2] = __dp4a(tw[k], 0x00400000u,
                                  __dp4a(tw[k + 1], 0x00004000u,
                                         __dp4a(bw[k], 0x00400000u, __dp4a(bw[k + 1], 0x00004000u, 128u))));
            // odd pixel: bytes 2..7 of words (k+1, k+2)
            s[3 * q + 3] = __dp4a(tw[k + 1], 0x00400000u,
                                  __dp4a(tw[k + 2], 0x00004000u,
                                         __dp4a(bw[k + 1], 0x00400000u, __dp4a(bw[k + 2], 0x00004000u, 128u))));
            s[3 * q + 4] = __dp4a(tw[k + 1], 0x40000000u,
                                  __dp4a(tw[k + 2], 0x00400000u,
                                         __dp4a(bw[k + 1], 0x40000000u, __dp4a(bw[k + 2], 0x00400000u, 128u))));
            s[3 * q + 5] = __dp4a(tw[k + 2], 0x40000040u, __dp4a(bw[k + 2], 0x40000040u, 128u));
        }
        o[0] = pick_byte1(s[0], s[1], s[2], s[3]);
        o[1] = pick_byte1(s[4], s[5], s[6], s[7]);
        o[2] = pick_byte1(s[8], s[9], s[10], s[11]);
    } else {
        // C == 4: per output pixel four words; sum byte lanes in two 16-bit-lane
        // halves (each sum <= 1022 fits)
        const uint32_t w[2][4] = {{tw[0], tw[1], bw[0], bw[1]}, {tw[2], tw[3], bw[2], bw[3]}};
#pragma unroll
        for (int p = 0; p < 2; p++) {
            const uint32_t l = __byte_perm(w[p][0], 0, 0x4240) + __byte_perm(w[p][1], 0, 0x4240) +
                               __byte_perm(w[p][2], 0, 0x4240) + __byte_perm(w[p][3], 0, 0x4240) + 0x00020002u;
            const uint32_t h = __byte_perm(w[p][0], 0, 0x4341) + __byte_perm(w[p][1], 0, 0x4341) +
                               __byte_perm(w[p][2], 0, 0x4341) + __byte_perm(w[p][3], 0, 0x4341) + 0x00020002u;
            o[p] = ((l >> 2) & 0x00ff00ffu) | ((h << 6) & 0xff00ff00u);
        }
    }
}

// Exact 2x nearest: output pixel p is source pixel 2p of row 2 dy (floor(d n_in
// / n_out) = 2d).  One group from the upper row's words: the first pixel of
// each source pair, packed by byte permutes (source byte indices in the
// comments).
template <int C>
__device__ __forceinline__ void down2_nearest_group(const uint32_t *tw, uint32_t *o)
{
    if constexpr (C == 1) {
        o[0] = __byte_perm(tw[0], tw[1], 0x6420);   // 0 2 4 6
        o[1] = __byte_perm(tw[2], tw[3], 0x6420);   // 8 10 12 14
    } else if constexpr (C == 3) {
        o[0] = __byte_perm(tw[0], tw[1], 0x6210);                                  // 0 1 2 6
        o[1] = __byte_perm(__byte_perm(tw[1], tw[2], 0x0043), tw[3], 0x5410);      // 7 8 12 13
        o[2] = __byte_perm(__byte_perm(tw[3], tw[4], 0x0762), tw[5], 0x4210);      // 14 18 19 20
    } else {
        o[0] = tw[0];   // pixel 0
        o[1] = tw[2];   // pixel 2
    }
}

// The row's last pixels of an exact 2x group kernel (fewer than a group),
// byte by byte; kept out of line so that the whole-group path compiles to a
// short straight sequence.
template <int C, int LINEAR>
__device__ __noinline__ void down2_row_tail(const uint8_t *top, const uint8_t *bot, uint8_t *out, int p0, int OW)
{
    for (int p = p0; p < OW; p++)
#pragma unroll
        for (int c = 0; c < C; c++) {
            const int o = 2 * p * C + c;
            if (LINEAR) {
                const int s = ld_g(top + o) + ld_g(top + o + C) + ld_g(bot + o) + ld_g(bot + o + C) + 2;
                st_g(out + p * C + c, static_cast<uint8_t>(s >> 2));
            } else {
                st_g(out + p * C + c, ld_g(top + o));
            }
        }
}

// One group of the exact 2x downscale: the group's source words of its two
// rows (LINEAR = 0: the upper row only), the exact sums, one vector store.
template <int C, int LINEAR>
__device__ __forceinline__ void down2_one(const uint8_t *top, const uint8_t *bot, uint8_t *out, int j)
{
    constexpr int PX = down2_px(C), SB = 2 * PX * C, OB = PX * C;
    uint32_t tw[SB / 4], bw[SB / 4], o[OB / 4];
    if constexpr (C == 3) {
        const uint2 *tp = reinterpret_cast<const uint2 *>(top + SB * j);
        const uint2 *bp = reinterpret_cast<const uint2 *>(bot + SB * j);
#pragma unroll
        for (int k = 0; k < 3; k++) {
            const uint2 t = ld_cs(tp + k);
            tw[2 * k] = t.x; tw[2 * k + 1] = t.y;
            if (LINEAR) {
                const uint2 u = ld_cs(bp + k);
                bw[2 * k] = u.x; bw[2 * k + 1] = u.y;
            }
        }
    } else {
        const uint4 t = ld_cs(reinterpret_cast<const uint4 *>(top + SB * j));
        tw[0] = t.x; tw[1] = t.y; tw[2] = t.z; tw[3] = t.w;
        if (LINEAR) {
            const uint4 u = ld_cs(reinterpret_cast<const uint4 *>(bot + SB * j));
            bw[0] = u.x; bw[1] = u.y; bw[2] = u.z; bw[3] = u.w;
        }
    }
    if (LINEAR)
        down2_group<C>(tw, bw, o);
    else
        down2_nearest_group<C>(tw, o);
    if constexpr (C == 3) {
        uint32_t *op = reinterpret_cast<uint32_t *>(out + OB * j);
        st_cs(op, o[0]);
        st_cs(op + 1, o[1]);
        st_cs(op + 2, o[2]);
    } else {
        st_cs(reinterpret_cast<uint2 *>(out + OB * j), make_uint2(o[0], o[1]));
    }
}

// ------------------------------------------------------------------ byte gathering

// One 32-bit word from four bytes: byte k is byte pos[k] of reg[k], where
// equal id[k] name the same register.  All arguments are compile-time
// constants after unrolling, so the branches fold: a word drawn from one or
// two registers takes one byte permute, from three two, from four three.
__device__ __forceinline__ uint32_t gather_bytes(const uint32_t (&reg)[4], const int (&id)[4],
                                                 const uint32_t (&pos)[4])
{
    int slot[4], first[4], nd = 0;
#pragma unroll
    for (int k = 0; k < 4; k++) {
        slot[k] = -1;
#pragma unroll
        for (int j = 0; j < k; j++)
            if (slot[k] < 0 && id[j] == id[k])
                slot[k] = slot[j];
        if (slot[k] < 0) {
            slot[k] = nd;
            first[nd] = k;
            nd++;
        }
    }
    if (nd <= 2) {
        uint32_t sel = 0;
#pragma unroll
        for (int k = 0; k < 4; k++)
            sel |= (pos[k] + 4u * static_cast<uint32_t>(slot[k])) << (4 * k);
        return __byte_perm(reg[first[0]], nd == 2 ? reg[first[1]] : 0u, sel);
    }
    if (nd == 3) {
        uint32_t s1 = 0, s2 = 0;
#pragma unroll
        for (int k = 0; k < 4; k++) {
            if (slot[k] < 2) {
                s1 |= (pos[k] + 4u * static_cast<uint32_t>(slot[k])) << (4 * k);
                s2 |= static_cast<uint32_t>(k) << (4 * k);
            } else {
                s2 |= (4u + pos[k]) << (4 * k);
            }
        }
        return __byte_perm(__byte_perm(reg[first[0]], reg[first[1]], s1), reg[first[2]], s2);
    }
    const uint32_t lo2 = __byte_perm(reg[0], reg[1], pos[0] | ((4u + pos[1]) << 4));
    const uint32_t hi2 = __byte_perm(reg[2], reg[3], pos[2] | ((4u + pos[3]) << 4));
    return __byte_perm(lo2, hi2, 0x5410);
}

// ------------------------------------------------------------------ exact 2x upscale, pixel lanes, walking rows
//
// The same 9-3-3-1 sum as the column-group exact 2x upscale, for three and
// four channels, laid out so that a horizontal neighbour is a whole register:
// each source pixel is unpacked once into two lane words, lo = {c0, c2} and
// hi = {c1, c3} (16-bit lanes; c3 = 0 for three channels), so the vertical
// sums
//   V = 16 t + 48 m + 32   (t the row above or below, m the middle row)
// and the horizontal ones
//   even output: 3 V[x] + V[x - 1],   odd output: 3 V[x] + V[x + 1]
// are one integer multiply-add per lane word; every lane is 16 S + 128 with S
// the 9-3-3-1 sum (below 2^16), so its high byte is (S + 8) >> 4, the exact
// result (CUDA interpolation page §2.2, §6.2 at weights 1536 and 512).  A
// caller takes four source columns of a run of consecutive source rows (two
// output rows each), keeping the unpacked rows above, at and below the current
// one in registers, so each row is loaded and unpacked once per thread.
template <int C>
struct Up2RowsLayout {
    static constexpr int P = 4;                    // source columns per thread
    static constexpr int LEAD = (4 - C % 4) % 4;   // bytes before column s0 - 1 in its word
    static constexpr int NB = (P + 2) * C;         // bytes of columns s0 - 1 .. s0 + P
    static constexpr int NW = (LEAD + NB + 3) / 4;
    static constexpr int NWO = 2 * P * C / 4;      // output words per output row
};

// Lane word {byte ea, byte eb} of the row's words (eb < 0: {byte ea, 0}),
// each byte in the low half of a 16-bit lane.
template <int NW>
__device__ __forceinline__ uint32_t lane_word(const uint32_t (&w)[NW], int ea, int eb)
{
    const int wa = ea >> 2;
    if (eb < 0)
        return __byte_perm(w[wa], 0u, 0x4440u | static_cast<uint32_t>(ea & 3));
    const int wb = eb >> 2;
    if (wa == wb)
        return __byte_perm(w[wa], 0u, 0x4040u | static_cast<uint32_t>(ea & 3) | (static_cast<uint32_t>(eb & 3) << 8));
    return __byte_perm(w[wa], w[wb], static_cast<uint32_t>(ea & 3) | ((4u + (eb & 3)) << 8)) & 0x00ff00ffu;
}

// Load the words of source columns s0 - 1 .. s0 + P of one row (interior: NW
// aligned words; at the image's left or right edge, or on layouts that are
// not 4-byte aligned: bytes, the columns mapped by the border rule) and
// unpack the P + 2 pixels into lane words.
template <int C, int BORDER>
__device__ __forceinline__ void up2_row_lanes(const uint8_t *row, int s0, int W, bool inner, uint32_t (&lo)[6],
                                              uint32_t (&hi)[6])
{
    using L = Up2RowsLayout<C>;
    uint32_t wd[L::NW];
    if (inner) {
        const uint32_t *w = reinterpret_cast<const uint32_t *>(row + (s0 - 1) * C - L::LEAD);
#pragma unroll
        for (int i = 0; i < L::NW; i++)
            wd[i] = ld_nc(w + i);
    } else {
#pragma unroll
        for (int i = 0; i < L::NW; i++)
            wd[i] = 0;
#pragma unroll
        for (int i = 0; i < L::NB; i++) {
            const int col = BORDER == RZ_BORDER_CLAMP ? clampi(s0 - 1 + i / C, 0, W - 1)
                                                      : border_index(s0 - 1 + i / C, W, BORDER);
            wd[(L::LEAD + i) / 4] |= static_cast<uint32_t>(ld_nc(row + col * C + i % C)) << (8 * ((L::LEAD + i) % 4));
        }
    }
#pragma unroll
    for (int k = 0; k < 6; k++) {
        const int e = L::LEAD + k * C;
        lo[k] = lane_word<L::NW>(wd, e, e + 2);
        hi[k] = lane_word<L::NW>(wd, e + 1, C == 4 ? e + 3 : -1);
    }
}

// Output row 2r (above = row r - 1) or 2r + 1 (above = row r + 1): vertical
// sums with the middle row's 48 m + 32 (mm), horizontal sums, the result
// bytes gathered into words and stored.
template <int C>
__device__ __forceinline__ void up2_emit_row(const uint32_t (&tlo)[6], const uint32_t (&thi)[6],
                                             const uint32_t (&mlo)[6], const uint32_t (&mhi)[6], uint8_t *op, int np)
{
    using L = Up2RowsLayout<C>;
    uint32_t vlo[6], vhi[6];
#pragma unroll
    for (int k = 0; k < 6; k++) {
        vlo[k] = 16 * tlo[k] + mlo[k];
        vhi[k] = 16 * thi[k] + mhi[k];
    }
    // output pixel q: centre column k = q / 2 + 1, even (left neighbour) or
    // odd (right neighbour)
    uint32_t qlo[2 * 4], qhi[2 * 4];
#pragma unroll
    for (int k = 1; k <= 4; k++) {
        qlo[2 * k - 2] = 3 * vlo[k] + vlo[k - 1];
        qhi[2 * k - 2] = 3 * vhi[k] + vhi[k - 1];
        qlo[2 * k - 1] = 3 * vlo[k] + vlo[k + 1];
        qhi[2 * k - 1] = 3 * vhi[k] + vhi[k + 1];
    }
    uint32_t ow[L::NWO];
#pragma unroll
    for (int wo = 0; wo < L::NWO; wo++) {
        uint32_t reg[4];
        int id[4];
        uint32_t pos[4];
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const int ob = 4 * wo + k, q = ob / C, c = ob % C;
            const bool is_hi = (c & 1) != 0;
            reg[k] = is_hi ? qhi[q] : qlo[q];
            id[k] = 2 * q + (is_hi ? 1 : 0);
            pos[k] = c >= 2 ? 3u : 1u;
        }
        ow[wo] = gather_bytes(reg, id, pos);
    }
    const uintptr_t oa = reinterpret_cast<uintptr_t>(op);
    if (np == 4 && L::NWO % 4 == 0 && (oa & 15) == 0) {
#pragma unroll
        for (int i = 0; i < L::NWO; i += 4)
            st_cs(reinterpret_cast<uint4 *>(op) + i / 4, make_uint4(ow[i], ow[i + 1], ow[i + 2], ow[i + 3]));
    } else if (np == 4 && L::NWO % 2 == 0 && (oa & 7) == 0) {
#pragma unroll
        for (int i = 0; i < L::NWO; i += 2)
            st_cs(reinterpret_cast<uint2 *>(op) + i / 2, make_uint2(ow[i], ow[i + 1]));
    } else if (np == 4 && (oa & 3) == 0) {
#pragma unroll
        for (int i = 0; i < L::NWO; i++)
            st_cs(reinterpret_cast<uint32_t *>(op) + i, ow[i]);
    } else {
#pragma unroll
        for (int i = 0; i < 8 * C; i++)
            if (i < 2 * np * C)
                st_g(op + i, static_cast<uint8_t>(ow[i / 4] >> (8 * (i % 4))));
    }
}

// ------------------------------------------------------------------ exact 3:2 downscale

// One group of the exact 3:2 downscale (W = 3 OW / 2, H = 3 OH / 2): output
// pixels 8 j .. 8 j + 7 of one row from source pixels 12 j .. 12 j + 11 of
// its two source rows, ra weighted 3 and rb weighted 1 (each output weights
// its two source columns 3 and 1 the same way), so the exact bilinear sum is
// (sum of b a t + 8) >> 4 with a, b in {1, 3}.  ra, rb and o 4-byte aligned.
template <int C>
__device__ __forceinline__ void down32_group(const uint8_t *ra, const uint8_t *rb, uint8_t *o, int j)
{
    constexpr int PX = 8;          // output pixels
    constexpr int NW = 3 * C;      // source words per row: 12 pixels
    constexpr int NWO = 2 * C;     // output words: 8 pixels
    if constexpr (C >= 3) {
        // vertical sums 3 a + b in 16-bit lanes of even and odd bytes,
        // regrouped into pixel lane words {c0, c2} and {c1, c3 or 0}; a
        // lane word's horizontal 9-3-3-1 sum is then two multiply-adds
        // for two channels: 48 V[x3] + 16 V[x1] + 128 = 16 S + 128 (S at
        // most 16 * 255), whose high byte is (S + 8) >> 4
        const uint32_t *wa = reinterpret_cast<const uint32_t *>(ra + 12 * C * j);
        const uint32_t *wb = reinterpret_cast<const uint32_t *>(rb + 12 * C * j);
        uint32_t ve[NW], vo[NW];
#pragma unroll
        for (int i = 0; i < NW; i++) {
            const uint32_t x = ld_cs(wa + i), y = ld_nc(wb + i);
            ve[i] = 3 * (x & 0x00ff00ffu) + (y & 0x00ff00ffu);
            vo[i] = 3 * __byte_perm(x, 0u, 0x4341u) + __byte_perm(y, 0u, 0x4341u);
        }
        // {lane of source byte e1, lane of e2 (0 for e2 < 0)}
        auto lanes = [&](int e1, int e2) -> uint32_t {
            const uint32_t a = (e1 & 1) ? vo[e1 >> 2] : ve[e1 >> 2];
            const uint32_t s1 = ((e1 >> 1) & 1) ? 0x32u : 0x10u;
            if (e2 < 0)
                return __byte_perm(a, 0u, s1 | 0x4400u);
            const uint32_t b = (e2 & 1) ? vo[e2 >> 2] : ve[e2 >> 2];
            const bool same = (e1 & 1) == (e2 & 1) && (e1 >> 2) == (e2 >> 2);
            const uint32_t s2 = ((e2 >> 1) & 1) ? (same ? 0x32u : 0x76u) : (same ? 0x10u : 0x54u);
            return __byte_perm(a, same ? 0u : b, s1 | (s2 << 8));
        };
        uint32_t ol[PX], oh[PX];
#pragma unroll
        for (int i = 0; i < PX / 2; i++) {
            const int p3 = 3 * i, p1 = 3 * i + 1, p2 = 3 * i + 2;
            const uint32_t ml = 16 * lanes(p1 * C, p1 * C + 2) + 0x00800080u;
            const uint32_t mh = 16 * lanes(p1 * C + 1, C == 4 ? p1 * C + 3 : -1) + 0x00800080u;
            ol[2 * i] = 48 * lanes(p3 * C, p3 * C + 2) + ml;
            oh[2 * i] = 48 * lanes(p3 * C + 1, C == 4 ? p3 * C + 3 : -1) + mh;
            ol[2 * i + 1] = 48 * lanes(p2 * C, p2 * C + 2) + ml;
            oh[2 * i + 1] = 48 * lanes(p2 * C + 1, C == 4 ? p2 * C + 3 : -1) + mh;
        }
        uint32_t *op = reinterpret_cast<uint32_t *>(o + PX * C * j);
#pragma unroll
        for (int wo = 0; wo < NWO; wo++) {
            // output byte q C + c: byte 1 (c = 0, 1) or 3 (c = 2, 3) of
            // ol[q] (c even) or oh[q] (c odd)
            uint32_t reg[4], pos[4];
            int id[4];
#pragma unroll
            for (int k = 0; k < 4; k++) {
                const int ob = 4 * wo + k, q = ob / C, c = ob % C;
                reg[k] = (c & 1) ? oh[q] : ol[q];
                id[k] = 2 * q + (c & 1);
                pos[k] = c >= 2 ? 3u : 1u;
            }
            st_cs(op + wo, gather_bytes(reg, id, pos));
        }
    } else {
        // vertical sums 3 a + b in 16-bit lanes (even and odd bytes)
        uint32_t vl[NW], vh[NW];
        const uint32_t *wa = reinterpret_cast<const uint32_t *>(ra + 12 * C * j);
        const uint32_t *wb = reinterpret_cast<const uint32_t *>(rb + 12 * C * j);
#pragma unroll
        for (int i = 0; i < NW; i++) {
            const uint32_t x = ld_cs(wa + i), y = ld_nc(wb + i);
            vl[i] = 3 * (x & 0x00ff00ffu) + (y & 0x00ff00ffu);
            vh[i] = 3 * ((x >> 8) & 0x00ff00ffu) + ((y >> 8) & 0x00ff00ffu);
        }
        // the 16-bit lane of source byte e of the group (below 2^10)
        auto lane = [&](int e) -> uint32_t {
            const uint32_t wv = (e & 1) ? vh[e >> 2] : vl[e >> 2];
            return ((e >> 1) & 1) ? (wv >> 16) : (wv & 0xffffu);
        };
        uint32_t *op = reinterpret_cast<uint32_t *>(o + PX * C * j);
#pragma unroll
        for (int wo = 0; wo < NWO; wo++) {
            uint32_t q[4];
#pragma unroll
            for (int k = 0; k < 4; k++) {
                const int ob = 4 * wo + k, oc = ob / C, c = ob % C, i = oc >> 1;
                // output 2i: source 3i (3) and 3i + 1 (1); 2i + 1: 3i + 1 (1) and 3i + 2 (3)
                const uint32_t x3 = lane(((oc & 1) ? 3 * i + 2 : 3 * i) * C + c);
                const uint32_t x1 = lane((3 * i + 1) * C + c);
                q[k] = (3 * x3 + x1 + 8) >> 4;
            }
            st_cs(op + wo, q[0] | (q[1] << 8) | (q[2] << 16) | (q[3] << 24));
        }
    }
}

}  // namespace dev
}  // namespace rz
