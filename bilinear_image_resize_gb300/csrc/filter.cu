// Resize + 3x3 filter for float32 HWC images, streamed down column strips.
//
// The fused epilogue filters the RESIZED image: out(y, x) = sum over a, b in
// {-1, 0, 1} of w[a+1][b+1] * R(clamp(y + a), clamp(x + b)), where R is the
// bilinear (or nearest) resize and the clamp replicates R's border (CUDA
// interpolation page, §4.2 fused epilogue; §6.1 replicate border).
//
// Work unit: one strip of TW output columns by TR output rows of one image;
// each of the eight consumer warps takes ceil(TW / 8) columns, at most 62 for
// one channel (two resized columns per lane) and 30 for three or four.  A unit computes R on rows
// dy0 - 1 .. dy1 and columns dx0 - 1 .. dx1 (clamped into the image), and
// samples the source rows those rows list, each once and in increasing order.
//
//   * The producer warp streams a unit's listed source rows through a ring of
//     chunks in shared memory, up to eight rows per chunk, each chunk with its
//     own "full" mbarrier (completed by the copies) and "empty" mbarrier (one
//     arrival per consumer warp).  A chunk of consecutive source rows (the
//     common case) moves as one tensor-map (TMA) box of rows x column span
//     per 2 KB of span; other chunks as one bulk copy per row and block.
//     Large copies keep the per-copy cost of the copy engine low, and almost
//     all of the ring is in flight at any time, so few CTAs keep HBM busy.
//   * Each consumer warp computes one resized row per step at its columns
//     (its outputs and their two neighbours), keeps partial sums of the three
//     output rows that row feeds in registers and takes the neighbours'
//     values by warp shuffle, so each resized value is computed once per unit.  A warp releases a source row
//     as soon as the next resized row no longer samples it, and writes its 30
//     outputs of a row straight from registers to global memory.
//
// Producer and consumers walk the same list: for resized row k with taps
// r0 <= r1 <= r0 + 1 (non-decreasing in k), r0 is new unless it equals the
// last or the one-before-last listed row, and r1 is new unless it equals the
// last.  A warp holds at most two listed rows (two chunks) at a time, so any
// ring of two or more chunks makes progress.
#include <cuda_runtime.h>

#include <cstdint>

#include "rz_device.h"
#include "rz_internal.h"

namespace rz {
namespace {

using namespace dev;

struct UnitGeom {
    int b;          // image within the batch
    int dy0, dy1;   // output rows [dy0, dy1)
    int dx0, dx1;   // output columns [dx0, dx1)
};

__device__ __forceinline__ UnitGeom unit_geom(const KArgs &a, int u)
{
    UnitGeom g;
    const int per_img = a.tiles_x * a.tiles_y;
    g.b = u / per_img;
    const int r = u - g.b * per_img;
    const int ty = r / a.tiles_x;
    const int tx = r - ty * a.tiles_x;
    g.dy0 = ty * a.TR;
    g.dy1 = min(g.dy0 + a.TR, a.OH);
    g.dx0 = tx * a.TW;
    g.dx1 = min(g.dx0 + a.TW, a.OW);
    return g;
}

// The list of distinct source rows, 32 resized rows at a time: lane k takes
// resized row base + k with taps r0 <= r1 (act: the row exists).  Given the
// rows listed before the batch (n) and the second tap of the batch's previous
// row (r1_before, -1 for none), returns the list positions of lane k's taps;
// new0 / new1 tell whether a tap is listed here (at s0 / s1), and `n` and
// `r1_before` move past the batch.
struct ListBatch {
    int s0, s1;
    bool new0, new1;
};

__device__ __forceinline__ ListBatch list_batch(int r0, int r1, bool act, int &n, int &r1_before, int nact)
{
    const int lane = threadIdx.x & 31;
    int prev = __shfl_up_sync(0xffffffffu, r1, 1);
    if (lane == 0)
        prev = r1_before;
    ListBatch b;
    b.new0 = act && r0 > prev;
    b.new1 = act && r1 > max(r0, prev);
    const unsigned m0 = __ballot_sync(0xffffffffu, b.new0), m1 = __ballot_sync(0xffffffffu, b.new1);
    const unsigned lower = (1u << lane) - 1u;
    const int c = n + __popc(m0 & lower) + __popc(m1 & lower);   // rows listed before lane k's row
    b.s0 = b.new0 ? c : c - 1 - (prev - r0);
    b.s1 = b.new1 ? c + (b.new0 ? 1 : 0) : (r1 == r0 ? b.s0 : c - 1);
    n += __popc(m0) + __popc(m1);
    r1_before = __shfl_sync(0xffffffffu, r1, nact - 1);
    return b;
}

// Column span of a unit's source rows: bytes [b_lo, b_lo + nbytes) of a row,
// widened to 16-byte bounds for bulk copies (the row length is then a
// multiple of 16, so the widened span stays inside the row).
__device__ __forceinline__ void unit_span(const KArgs &a, const UnitGeom &g, int C, bool linear, int &b_lo,
                                          int &nbytes)
{
    const int xs0 = a.xt[clampi(g.dx0 - 1, 0, a.OW - 1)].x;
    const int xr = a.xt[clampi(g.dx1, 0, a.OW - 1)].x;
    const int xs1 = linear ? min(xr + 1, a.W - 1) : xr;
    b_lo = xs0 * C * 4;
    int b_hi = (xs1 + 1) * C * 4;
    if (a.tma_in) {
        b_lo &= ~15;
        b_hi = (b_hi + 15) & ~15;
    }
    nbytes = b_hi - b_lo;
}

template <int C, int LINEAR>
__global__ void __launch_bounds__(kThreads, 3) k_filter_stream(const KArgs a, const __grid_constant__ CUtensorMap tmap)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int NCH = a.ring_chunks, G = a.chunk_rows, NB = a.chunk_boxes, BW = a.box_bytes;
    const int LG = __ffs(G) - 1;                 // log2 of the rows per chunk
    const int BB = filter_block_bytes(G, BW);    // bytes per block of a chunk
    const int CB = NB * BB;                      // bytes per chunk
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + NCH;
    int *window = reinterpret_cast<int *>(smem + 16 * NCH);   // producer: listed rows, by position mod 128
    uint8_t *chunks = smem + filter_chunks_off(NCH);
    const int nunits = a.batch * a.tiles_x * a.tiles_y;
    const int GR = gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int c = 0; c < NCH; c++) {
            mbar_init(&full[c], a.tma_in ? 1 : 32);
            mbar_init(&empty[c], kConsumers / 32);
        }
        fence_mbar_init();
    }
    __syncthreads();
    grid_launch_dependents();
    // every thread reads global memory below: wait for the grids this launch
    // depends on
    grid_dependency_wait();

    if (warp == kConsumers / 32) {
        // ---------------- producer warp
        const uint64_t policy = policy_evict_first();
        int slot = 0, use = 0;   // ring chunk of the next chunk, and how often it was filled before
        long long issued = 0;    // chunks issued
        bool ok = true;
        for (int u = blockIdx.x; u < nunits && ok; u += GR) {
            const UnitGeom g = unit_geom(a, u);
            int b_lo, nbytes;
            unit_span(a, g, C, LINEAR, b_lo, nbytes);
            if (nbytes > NB * BW) {
                // the host sizes the blocks from the same spans: unreachable,
                // but shared memory stays in bounds
                if (lane == 0)
                    atomicExch(a.status, RZ_ERR_ARG);
                nbytes = NB * BW;
            }
            const uint8_t *img = a.src + (long long)g.b * a.src_bstride;
            // issue the chunk of list positions [p0, p0 + rows)
            auto issue = [&](int p0, int rows) -> bool {
                if (use > 0) {
                    bool w = true;
                    if (lane == 0)
                        w = mbar_wait_bounded(&empty[slot], (use - 1) & 1, a.status);
                    if (!__shfl_sync(0xffffffffu, w ? 1 : 0, 0))
                        return false;
                }
                uint8_t *cb = chunks + slot * CB;
                const int first = window[p0 & (kFilterListWindow - 1)];
                const int last = window[(p0 + rows - 1) & (kFilterListWindow - 1)];
                const int my_row = window[(p0 + min(lane, rows - 1)) & (kFilterListWindow - 1)];
                if (a.tensor_in && last - first == rows - 1) {
                    // consecutive rows: one box of G rows per block (rows past
                    // the list's end land unused; rows past the image read as 0)
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(NB * G * BW));
                        for (int k = 0; k < NB; k++)
                            tensor_load_3d(cb + k * BB, &tmap, (b_lo + k * BW) / 8, first, g.b, &full[slot], policy);
                    }
                } else if (a.tma_in) {
                    if (lane == 0)
                        mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(rows * nbytes));
                    __syncwarp();
                    if (lane < rows) {
                        const uint8_t *src = img + (long long)my_row * a.src_pitch + b_lo;
                        for (int k = 0; k < NB; k++) {
                            const int bytes = min(BW, nbytes - k * BW);
                            if (bytes > 0)
                                bulk_load_hint(cb + k * BB + lane * BW, src + k * BW, static_cast<uint32_t>(bytes),
                                               &full[slot], policy);
                        }
                    }
                } else {
                    for (int i = 0; i < rows; i++) {
                        const uint8_t *src = img + (long long)window[(p0 + i) & (kFilterListWindow - 1)] * a.src_pitch + b_lo;
                        for (int o = lane; o < nbytes; o += 32) {
                            const int k = o / BW;
                            cb[k * BB + i * BW + (o - k * BW)] = __ldg(src + o);
                        }
                    }
                    mbar_arrive(&full[slot]);   // 32 arrivals: each lane releases its own copies
                }
                ++issued;
                if (++slot == NCH) {
                    slot = 0;
                    ++use;
                }
                return true;
            };
            // walk the list 32 resized rows at a time; lanes record the new
            // rows in the list window, then every complete chunk is issued
            const int ncomp = g.dy1 - g.dy0 + 2;
            int n = 0, r1_before = -1, done = 0;   // rows listed; rows issued in chunks
            for (int base = 0; base < ncomp && ok; base += 32) {
                const int nact = min(32, ncomp - base);
                const bool act = lane < nact;
                const int r0 = a.yt[clampi(g.dy0 - 1 + base + lane, 0, a.OH - 1)].x;
                const int r1 = LINEAR ? min(r0 + 1, a.H - 1) : r0;
                const ListBatch lb = list_batch(r0, r1, act, n, r1_before, nact);
                if (lb.new0)
                    window[lb.s0 & (kFilterListWindow - 1)] = r0;
                if (lb.new1)
                    window[lb.s1 & (kFilterListWindow - 1)] = r1;
                __syncwarp();
                while (ok && n - done >= G) {
                    ok = issue(done, G);
                    done += G;
                }
            }
            if (ok && n > done)
                ok = issue(done, n - done);
        }
        // no copy may still be landing when the CTA exits: wait for the last
        // chunk issued into each ring slot (already complete unless the
        // consumers gave up early)
        if (lane == 0) {
            const long long first = issued > NCH ? issued - NCH : 0;
            for (long long p = first; p < issued; p++)
                mbar_wait_bounded(&full[p % NCH], static_cast<uint32_t>((p / NCH) & 1), nullptr);
        }
        return;
    }

    // ---------------- consumer warps
    // Chunk counters are 32-bit and compared by signed difference: a CTA
    // walks far fewer than 2^31 chunks.
    int wslot = 0, wphase = 0;   // next chunk to wait for: ring slot and phase parity
    int rslot = 0;               // next chunk to release
    unsigned wch = 0, rch = 0, ucb = 0;   // chunks waited for, released; first chunk of the unit
    const float *fchunks = reinterpret_cast<const float *>(chunks);
    constexpr int NCOL = filter_lane_cols(C);   // resized columns per lane: lane + 32 i
    const int CW = (a.TW + kConsumers / 32 - 1) / (kConsumers / 32);   // output columns per warp
    bool ok = true;
    for (int u = blockIdx.x; u < nunits && ok; u += GR) {
        const UnitGeom g = unit_geom(a, u);
        int b_lo, nbytes;
        unit_span(a, g, C, LINEAR, b_lo, nbytes);
        const int nc = g.dx1 - g.dx0;
        // resized column e = lane + 32 i of this warp is dx0 + warp * CW - 1 + e
        // (held at dx1 past the strip: its value only feeds lanes that emit
        // nothing); columns e = 1 .. CW are this warp's outputs
        float uw[NCOL];
        int off0[NCOL][C], off1[NCOL][C];   // float offsets of the taps' channels within a staged row
        bool emit[NCOL];
        const int rel0 = warp * CW - 1 + lane;
#pragma unroll
        for (int i = 0; i < NCOL; i++) {
            const int e = lane + 32 * i, rel = rel0 + 32 * i;
            emit[i] = e >= 1 && e <= CW && rel < nc;
            const int2 xe = a.xt[clampi(g.dx0 + min(rel, nc), 0, a.OW - 1)];
            uw[i] = __int_as_float(xe.y);
            const int x1 = LINEAR ? min(xe.x + 1, a.W - 1) : xe.x;
#pragma unroll
            for (int c = 0; c < C; c++) {
                const int q0 = clampi((xe.x * C + c) * 4 - b_lo, 0, NB * BW - 4);
                const int q1 = clampi((x1 * C + c) * 4 - b_lo, 0, NB * BW - 4);
                off0[i][c] = ((q0 / BW) * BB + q0 % BW) / 4;
                off1[i][c] = ((q1 / BW) * BB + q1 % BW) / 4;
            }
        }
        // the unit's output row at column dx0, advanced one row per step;
        // column i of this lane is rel0 + 32 i pixels on (>= 0 where emitted)
        uint8_t *op = a.dst + (long long)g.b * a.dst_bstride + (long long)g.dy0 * a.dst_pitch +
                      (long long)g.dx0 * C * 4;
        // partial sums of the output rows resized row k contributes to:
        // acc1 for output row k - 1, acc2 for k - 2 (complete after row k);
        // each sums its nine products in the filter's row-major order
        float acc1[NCOL][C], acc2[NCOL][C];
#pragma unroll
        for (int i = 0; i < NCOL; i++)
#pragma unroll
            for (int c = 0; c < C; c++)
                acc1[i][c] = acc2[i][c] = 0.0f;
        const int ncomp = g.dy1 - g.dy0 + 2;
        int n = 0, r1_before = -1;
        // chunks of the previous row's taps (none yet: one below the unit's first)
        unsigned c0_before = ucb - 1, c1_before = ucb - 1;
        int2 ye_next = a.yt[clampi(g.dy0 - 1 + lane, 0, a.OH - 1)];
        for (int base = 0; base < ncomp && ok; base += 32) {
            // the next 32 resized rows: list positions of their taps, the ring
            // chunks and shared-memory rows those land in (16-byte units:
            // shared memory is below 2^20 bytes), and which rows move to a new
            // chunk; the table entries of the batch after are fetched meanwhile
            const int nact = min(32, ncomp - base);
            const int2 ye = ye_next;
            ye_next = a.yt[clampi(g.dy0 - 1 + base + 32 + lane, 0, a.OH - 1)];
            const int r1 = LINEAR ? min(ye.x + 1, a.H - 1) : ye.x;
            const ListBatch lb = list_batch(ye.x, r1, lane < nact, n, r1_before, nact);
            const unsigned bc0 = ucb + (lb.s0 >> LG), bc1 = ucb + (lb.s1 >> LG);
            const unsigned top16 = ((bc0 % NCH) * CB + (lb.s0 & (G - 1)) * BW) >> 4;
            const unsigned bot16 = ((bc1 % NCH) * CB + (lb.s1 & (G - 1)) * BW) >> 4;
            const unsigned bpk = top16 | (bot16 << 16);
            const float bv = __int_as_float(ye.y);
            unsigned prev_c0 = __shfl_up_sync(0xffffffffu, bc0, 1);
            unsigned prev_c1 = __shfl_up_sync(0xffffffffu, bc1, 1);
            if (lane == 0) {
                prev_c0 = c0_before;
                prev_c1 = c1_before;
            }
            // rows whose taps move to a later chunk: the first tap's move
            // releases chunks, the second tap's waits for one
            const unsigned events = __ballot_sync(0xffffffffu, lane < nact && (bc0 != prev_c0 || bc1 != prev_c1));
            c0_before = __shfl_sync(0xffffffffu, bc0, nact - 1);
            c1_before = __shfl_sync(0xffffffffu, bc1, nact - 1);
            for (int j = 0; j < nact; j++) {
                const int k = base + j;
                const unsigned pk = __shfl_sync(0xffffffffu, bpk, j);
                const float v = __shfl_sync(0xffffffffu, bv, j);
                if ((events >> j) & 1u) {
                    const unsigned c0 = __shfl_sync(0xffffffffu, bc0, j);
                    const unsigned c1 = __shfl_sync(0xffffffffu, bc1, j);
                    // release the chunks before this row's first tap (the
                    // previous rows' reads are complete: their values were
                    // shuffled)
                    while (static_cast<int>(c0 - rch) > 0) {
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive(&empty[rslot]);
                        ++rch;
                        if (++rslot == NCH)
                            rslot = 0;
                    }
                    // wait for every chunk up to the second tap's
                    while (static_cast<int>(c1 - wch) >= 0) {
                        if (!mbar_wait_bounded(&full[wslot], static_cast<uint32_t>(wphase), a.status))
                            ok = false;
                        ++wch;
                        if (++wslot == NCH) {
                            wslot = 0;
                            wphase ^= 1;
                        }
                    }
                    if (!__all_sync(0xffffffffu, ok)) {
                        ok = false;
                        break;
                    }
                }
                const float *top = fchunks + (pk & 0xffffu) * 4;
                const float *bot = fchunks + (pk >> 16) * 4;
                const bool store = k >= 2;
#pragma unroll
                for (int c = 0; c < C; c++) {
                    float m[NCOL], l[NCOL], r[NCOL];
#pragma unroll
                    for (int i = 0; i < NCOL; i++) {
                        const float t0 = top[off0[i][c]], t1 = top[off1[i][c]];
                        const float b0 = bot[off0[i][c]], b1 = bot[off1[i][c]];
                        const float hT = fmaf(uw[i], t1 - t0, t0);
                        const float hB = fmaf(uw[i], b1 - b0, b0);
                        m[i] = fmaf(v, hB - hT, hT);
                    }
                    if constexpr (NCOL == 1) {
                        l[0] = __shfl_up_sync(0xffffffffu, m[0], 1);
                        r[0] = __shfl_down_sync(0xffffffffu, m[0], 1);
                    } else {
                        // e = lane and e = lane + 32: the two halves meet
                        // between lane 31's first column and lane 0's second
                        l[0] = __shfl_up_sync(0xffffffffu, m[0], 1);
                        r[0] = __shfl_sync(0xffffffffu, lane == 0 ? m[1] : m[0], (lane + 1) & 31);
                        l[1] = __shfl_sync(0xffffffffu, lane == 31 ? m[0] : m[1], (lane + 31) & 31);
                        r[1] = __shfl_down_sync(0xffffffffu, m[1], 1);
                    }
#pragma unroll
                    for (int i = 0; i < NCOL; i++) {
                        // this row is row a = -1 of output k, a = 0 of k - 1,
                        // a = +1 of k - 2
                        const float a0 = fmaf(a.w[2], r[i], fmaf(a.w[1], m[i], a.w[0] * l[i]));
                        const float a1 = fmaf(a.w[5], r[i], fmaf(a.w[4], m[i], fmaf(a.w[3], l[i], acc1[i][c])));
                        const float a2 = fmaf(a.w[8], r[i], fmaf(a.w[7], m[i], fmaf(a.w[6], l[i], acc2[i][c])));
                        if (store && emit[i])
                            __stcs(reinterpret_cast<float *>(op) + (rel0 + 32 * i) * C + c, a2);
                        acc2[i][c] = a1;
                        acc1[i][c] = a0;
                    }
                }
                if (store)
                    op += a.dst_pitch;
            }
        }
        if (!ok)
            break;
        // the unit's remaining chunks
        ucb += (n + G - 1) >> LG;
        while (static_cast<int>(ucb - rch) > 0) {
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[rslot]);
            ++rch;
            if (++rslot == NCH)
                rslot = 0;
        }
    }
}

}  // namespace

// The fused entry point is bilinear only, so only bilinear kernels exist.
const void *filter_kernel_for(int mode, int C)
{
    using Fn = void (*)(const KArgs, const CUtensorMap);
    static const Fn lin[3] = {k_filter_stream<1, 1>, k_filter_stream<3, 1>, k_filter_stream<4, 1>};
    const int ci = (C == 1) ? 0 : (C == 3 ? 1 : (C == 4 ? 2 : -1));
    if (ci < 0 || mode != RZ_LINEAR)
        return nullptr;
    return reinterpret_cast<const void *>(lin[ci]);
}

}  // namespace rz
