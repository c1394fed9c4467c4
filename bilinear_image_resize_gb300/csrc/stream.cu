// Streaming kernels for sm_103a: each CTA walks column strips of the output
// down a segment of rows, streaming the source rows it needs through a ring
// of chunks in shared memory.  Two consumers share the producer:
//
//   * the K x K filter epilogue (K = 3, 5, 7) on float32 HWC images.  It
//     filters the RESIZED image: out(y, x) = sum over a, b in -K/2 .. K/2 of
//     w[a+K/2][b+K/2] * Z(clamp(y + a), clamp(x + b)), where Z is the
//     bilinear resize and the clamp replicates Z's border (CUDA interpolation
//     page, §4.2 fused epilogue; §6.1 replicate border);
//   * the uint8 bilinear resize in row-separable form.  The exact horizontal
//     sum h = A0 t0 + A1 t1 of a source row is formed once per output column
//     when the row arrives; each output row then needs only the vertical
//     combination (B0 hT + B1 hB + 2^21) >> 22 (CUDA interpolation page §2.2,
//     §6.2).  Both orders give the same exact integer, so this is the same
//     result as the tiled kernel's, with far fewer operations when source
//     rows are shared by several output rows (upscales).
//
// Work unit: one strip of TW output columns by TR output rows of one image.
// A unit computes on rows dy0 - HALO .. dy1 - 1 + HALO (HALO = K / 2 for the
// filter, 0 for the plain resize; clamped into the image) and samples the
// source rows those rows list, each once and in increasing order.
//
//   * The producer warp streams a unit's listed source rows through a ring of
//     chunks, up to eight rows per chunk, each chunk with its own "full"
//     mbarrier (completed by the copies) and "empty" mbarrier (one arrival per
//     consumer warp).  A chunk of consecutive source rows (the common case)
//     moves as one tensor-map (TMA) box of rows x column span per 2 KB of
//     span; other chunks as one bulk copy per row and block.  Large copies
//     keep the per-copy cost of the copy engine low, and almost all of the
//     ring is in flight at any time, so few CTAs keep HBM busy.
//   * Consumer warps walk the same list 32 rows at a time (warp votes), wait
//     for a chunk and release the chunks behind them only on the rows whose
//     taps move to a new chunk, and write their outputs straight from
//     registers to global memory.
//
// Producer and consumers walk the same list: for computed row k with taps
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

// The list of distinct source rows, 32 computed rows at a time: lane k takes
// computed row base + k with taps r0 <= r1 (act: the row exists).  Given the
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

// Column span of a unit's source rows: bytes [b_lo, b_lo + nbytes) of a row
// (elements of ES bytes, computed columns dx0 - HALO .. dx1 - 1 + HALO),
// widened to 16-byte bounds for bulk copies (the row length is then a
// multiple of 16, so the widened span stays inside the row).
template <int ES, int HALO>
__device__ __forceinline__ void unit_span(const KArgs &a, const UnitGeom &g, int C, bool linear, int &b_lo,
                                          int &nbytes)
{
    const int xs0 = a.xt[clampi(g.dx0 - HALO, 0, a.OW - 1)].x;
    const int xr = a.xt[clampi(g.dx1 - 1 + HALO, 0, a.OW - 1)].x;
    const int xs1 = linear ? min(xr + 1, a.W - 1) : xr;
    b_lo = xs0 * C * ES;
    int b_hi = (xs1 + 1) * C * ES;
    if (a.tma_in) {
        b_lo &= ~15;
        b_hi = (b_hi + 15) & ~15;
    }
    nbytes = b_hi - b_lo;
}

// The ring as the kernels see it.
struct Ring {
    int NCH, G, LG, NB, BW, BB, CB;   // chunks, rows per chunk (log2), blocks per row, bytes per block row,
                                      // bytes per block, bytes per chunk
    uint64_t *full, *empty;
    uint8_t *chunks;
};

// ------------------------------------------------------------------ producer

template <int ES, int HALO, int LINEAR>
__device__ void stream_producer(const KArgs &a, const CUtensorMap *tmap, const Ring &rg, int *window, int C)
{
    const int lane = threadIdx.x & 31;
    const int nunits = a.batch * a.tiles_x * a.tiles_y;
    const int NCH = rg.NCH, G = rg.G, NB = rg.NB, BW = rg.BW, BB = rg.BB;
    const uint64_t policy = policy_evict_first();
    int slot = 0, use = 0;   // ring slot of the next chunk, and how often it was filled before
    long long issued = 0;    // chunks issued
    bool ok = true;
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const UnitGeom g = unit_geom(a, u);
        int b_lo, nbytes;
        unit_span<ES, HALO>(a, g, C, LINEAR, b_lo, nbytes);
        if (nbytes > NB * BW) {
            // the host sizes the blocks from the same spans: unreachable, but
            // shared memory stays in bounds
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
                    w = mbar_wait_bounded(&rg.empty[slot], (use - 1) & 1, a.status);
                if (!__shfl_sync(0xffffffffu, w ? 1 : 0, 0))
                    return false;
            }
            uint8_t *cb = rg.chunks + slot * rg.CB;
            const int first = window[p0 & (kStreamListWindow - 1)];
            const int last = window[(p0 + rows - 1) & (kStreamListWindow - 1)];
            const int my_row = window[(p0 + min(lane, rows - 1)) & (kStreamListWindow - 1)];
            if (a.tensor_in && last - first == rows - 1) {
                // consecutive rows: one box of G rows per block (rows past the
                // list's end land unused; rows past the image read as 0)
                if (lane == 0) {
                    mbar_arrive_expect_tx(&rg.full[slot], static_cast<uint32_t>(NB * G * BW));
                    for (int k = 0; k < NB; k++)
                        tensor_load_3d(cb + k * BB, tmap, (b_lo + k * BW) / 8, first, g.b, &rg.full[slot], policy,
                                       static_cast<uint32_t>(G * BW));
                }
            } else if (a.tma_in) {
                if (lane == 0)
                    mbar_arrive_expect_tx(&rg.full[slot], static_cast<uint32_t>(rows * nbytes));
                __syncwarp();
                if (lane < rows) {
                    const uint8_t *src = img + (long long)my_row * a.src_pitch + b_lo;
                    for (int k = 0; k < NB; k++) {
                        const int bytes = min(BW, nbytes - k * BW);
                        if (bytes > 0)
                            bulk_load_hint(cb + k * BB + lane * BW, src + k * BW, static_cast<uint32_t>(bytes),
                                           &rg.full[slot], policy);
                    }
                }
            } else {
                for (int i = 0; i < rows; i++) {
                    const uint8_t *src =
                        img + (long long)window[(p0 + i) & (kStreamListWindow - 1)] * a.src_pitch + b_lo;
                    for (int o = lane; o < nbytes; o += 32) {
                        const int k = o / BW;
                        if (smem_guard(cb + k * BB + i * BW + (o - k * BW), 1))
                            cb[k * BB + i * BW + (o - k * BW)] = ld_nc(src + o);
                    }
                }
                mbar_arrive(&rg.full[slot]);   // 32 arrivals: each lane releases its own copies
            }
            ++issued;
            if (++slot == NCH) {
                slot = 0;
                ++use;
            }
            return true;
        };
        // walk the list 32 computed rows at a time; lanes record the new rows
        // in the list window, then every complete chunk is issued
        const int ncomp = g.dy1 - g.dy0 + 2 * HALO;
        int n = 0, r1_before = -1, done = 0;   // rows listed; rows issued in chunks
        for (int base = 0; base < ncomp && ok; base += 32) {
            const int nact = min(32, ncomp - base);
            const bool act = lane < nact;
            const int r0 = a.yt[clampi(g.dy0 - HALO + base + lane, 0, a.OH - 1)].x;
            const int r1 = LINEAR ? min(r0 + 1, a.H - 1) : r0;
            const ListBatch lb = list_batch(r0, r1, act, n, r1_before, nact);
            if (lb.new0)
                window[lb.s0 & (kStreamListWindow - 1)] = r0;
            if (lb.new1)
                window[lb.s1 & (kStreamListWindow - 1)] = r1;
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
    // chunk issued into each ring slot (already complete unless the consumers
    // gave up early)
    if (lane == 0) {
        const long long first = issued > NCH ? issued - NCH : 0;
        for (long long p = first; p < issued; p++)
            mbar_wait_bounded(&rg.full[p % NCH], static_cast<uint32_t>((p / NCH) & 1), nullptr);
    }
}

// ------------------------------------------------------------------ consumer side of the ring

// A consumer warp's position in the ring.  Chunk counters are 32-bit and
// compared by signed difference: a CTA walks far fewer than 2^31 chunks.
struct Cursor {
    int wslot = 0, wphase = 0;   // next chunk to wait for: ring slot and phase parity
    int rslot = 0;               // next chunk to release
    unsigned wch = 0, rch = 0, ucb = 0;   // chunks waited for, released; first chunk of the unit
};

// Walk the computed rows k = 0 .. ncomp - 1 of unit g (rows dy0 - HALO + k),
// calling row(k, top, bot, wbits, nnew): the shared-memory rows of the taps
// (top == bot when both taps are one row), the row's table weight bits and
// how many source rows the list gained at this row (0, 1 or 2).  Returns
// false if a wait timed out.
template <int HALO, int LINEAR, typename RowFn>
__device__ __forceinline__ bool walk_unit(const KArgs &a, const UnitGeom &g, const Ring &rg, Cursor &cs, RowFn &&row)
{
    const int lane = threadIdx.x & 31;
    const int NCH = rg.NCH, G = rg.G, LG = rg.LG;
    const int ncomp = g.dy1 - g.dy0 + 2 * HALO;
    int n = 0, r1_before = -1;
    // chunks of the previous row's taps (none yet: one below the unit's first)
    unsigned c0_before = cs.ucb - 1, c1_before = cs.ucb - 1;
    int2 ye_next = a.yt[clampi(g.dy0 - HALO + lane, 0, a.OH - 1)];
    bool ok = true;
    for (int base = 0; base < ncomp && ok; base += 32) {
        // the next 32 computed rows: list positions of their taps, the ring
        // chunks and shared-memory rows those land in (16-byte units below
        // 2^14: shared memory is below 232448 bytes), how many rows each adds
        // to the list, and which rows move to a new chunk; the table entries
        // of the batch after are fetched meanwhile
        const int nact = min(32, ncomp - base);
        const int2 ye = ye_next;
        ye_next = a.yt[clampi(g.dy0 - HALO + base + 32 + lane, 0, a.OH - 1)];
        const int r1 = LINEAR ? min(ye.x + 1, a.H - 1) : ye.x;
        const ListBatch lb = list_batch(ye.x, r1, lane < nact, n, r1_before, nact);
        const unsigned bc0 = cs.ucb + (lb.s0 >> LG), bc1 = cs.ucb + (lb.s1 >> LG);
        const unsigned top16 = ((bc0 % NCH) * rg.CB + (lb.s0 & (G - 1)) * rg.BW) >> 4;
        const unsigned bot16 = ((bc1 % NCH) * rg.CB + (lb.s1 & (G - 1)) * rg.BW) >> 4;
        const unsigned nnew = (lb.new0 ? 1u : 0u) + (lb.new1 ? 1u : 0u);
        const unsigned bpk = top16 | (nnew << 14) | (bot16 << 16);
        const int bw = ye.y;
        unsigned prev_c0 = __shfl_up_sync(0xffffffffu, bc0, 1);
        unsigned prev_c1 = __shfl_up_sync(0xffffffffu, bc1, 1);
        if (lane == 0) {
            prev_c0 = c0_before;
            prev_c1 = c1_before;
        }
        // rows whose taps move to a later chunk: the first tap's move releases
        // chunks, the second tap's waits for one
        const unsigned events = __ballot_sync(0xffffffffu, lane < nact && (bc0 != prev_c0 || bc1 != prev_c1));
        c0_before = __shfl_sync(0xffffffffu, bc0, nact - 1);
        c1_before = __shfl_sync(0xffffffffu, bc1, nact - 1);
        for (int j = 0; j < nact; j++) {
            const unsigned pk = __shfl_sync(0xffffffffu, bpk, j);
            const int wbits = __shfl_sync(0xffffffffu, bw, j);
            if ((events >> j) & 1u) {
                const unsigned c0 = __shfl_sync(0xffffffffu, bc0, j);
                const unsigned c1 = __shfl_sync(0xffffffffu, bc1, j);
                // release the chunks before this row's first tap (the previous
                // rows' reads are complete: their values were used)
                while (static_cast<int>(c0 - cs.rch) > 0) {
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&rg.empty[cs.rslot]);
                    ++cs.rch;
                    if (++cs.rslot == NCH)
                        cs.rslot = 0;
                }
                // wait for every chunk up to the second tap's
                while (static_cast<int>(c1 - cs.wch) >= 0) {
                    if (!mbar_wait_bounded(&rg.full[cs.wslot], static_cast<uint32_t>(cs.wphase), a.status))
                        ok = false;
                    ++cs.wch;
                    if (++cs.wslot == NCH) {
                        cs.wslot = 0;
                        cs.wphase ^= 1;
                    }
                }
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
            }
            row(base + j, rg.chunks + (pk & 0x3fffu) * 16, rg.chunks + (pk >> 16) * 16, wbits,
                static_cast<int>((pk >> 14) & 3u));
        }
    }
    if (!ok)
        return false;
    // the unit's remaining chunks
    cs.ucb += (n + G - 1) >> LG;
    while (static_cast<int>(cs.ucb - cs.rch) > 0) {
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&rg.empty[cs.rslot]);
        ++cs.rch;
        if (++cs.rslot == NCH)
            cs.rslot = 0;
    }
    return true;
}

// ------------------------------------------------------------------ consumer: K x K filter (float32)

// K = 2R + 1.  Each warp takes CW output columns; resized column e = lane +
// 32 i of the warp is dx0 + warp * CW - R + e (the true column, clamped to
// the image, up to R past the strip; held there beyond: those values feed
// lanes that emit nothing); columns e = R .. R + CW - 1 are its outputs.  Per
// resized row the lane forms its resized values, takes the neighbours' at
// distances 1 .. R by warp shuffle and adds them into partial sums of the K
// output rows the row feeds (output row k - 2R completes at row k).
template <int C, int LINEAR, int R>
__device__ __forceinline__ bool consume_filter(const KArgs &a, const UnitGeom &g, const Ring &rg, Cursor &cs)
{
    constexpr int K = 2 * R + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int NCOL = filter_lane_cols(C);   // resized columns per lane: lane + 32 i
    const int CW = (a.TW + kConsumers / 32 - 1) / (kConsumers / 32);
    const int NB = rg.NB, BW = rg.BW, BB = rg.BB;
    int b_lo, nbytes;
    unit_span<4, R>(a, g, C, LINEAR, b_lo, nbytes);
    const int nc = g.dx1 - g.dx0;
    float uw[NCOL];
    int off0[NCOL][C], off1[NCOL][C];   // float offsets of the taps' channels within a staged row
    bool emit[NCOL];
    const int rel0 = warp * CW - R + lane;
#pragma unroll
    for (int i = 0; i < NCOL; i++) {
        const int e = lane + 32 * i, rel = rel0 + 32 * i;
        emit[i] = e >= R && e < R + CW && rel < nc;
        const int2 xe = a.xt[clampi(g.dx0 + min(rel, nc + R - 1), 0, a.OW - 1)];
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
    // the unit's output row at column dx0, advanced one row per step; column i
    // of this lane is rel0 + 32 i pixels on (>= 0 where emitted)
    uint8_t *op = a.dst + (long long)g.b * a.dst_bstride + (long long)g.dy0 * a.dst_pitch +
                  (long long)g.dx0 * C * 4;
    // partial sums of the output rows resized row k contributes to: acc[j]
    // for output row k - 1 - j; each sums its K^2 products in the filter's
    // row-major order (none for K = 1: the plain resize, weight 1)
    constexpr int NA = R > 0 ? 2 * R : 1;
    float acc[NA][NCOL][C];
#pragma unroll
    for (int j = 0; j < NA; j++)
#pragma unroll
        for (int i = 0; i < NCOL; i++)
#pragma unroll
            for (int c = 0; c < C; c++)
                acc[j][i][c] = 0.0f;
    return walk_unit<R, LINEAR>(a, g, rg, cs, [&](int k, const uint8_t *top8, const uint8_t *bot8, int wbits, int) {
        const float *top = reinterpret_cast<const float *>(top8);
        const float *bot = reinterpret_cast<const float *>(bot8);
        const float v = __int_as_float(wbits);
        const bool store = k >= 2 * R;
#pragma unroll
        for (int c = 0; c < C; c++) {
            float m[NCOL];
#pragma unroll
            for (int i = 0; i < NCOL; i++) {
                const float t0 = lds_f(top + off0[i][c]), t1 = lds_f(top + off1[i][c]);
                const float b0 = lds_f(bot + off0[i][c]), b1 = lds_f(bot + off1[i][c]);
                const float hT = fmaf(uw[i], t1 - t0, t0);
                const float hB = fmaf(uw[i], b1 - b0, b0);
                m[i] = fmaf(v, hB - hT, hT);
            }
            // nb[d][i]: resized column e + d - R of this lane's column i
            float nb[K][NCOL];
#pragma unroll
            for (int i = 0; i < NCOL; i++)
                nb[R][i] = m[i];
#pragma unroll
            for (int d = 1; d <= R; d++) {
                // column e - d of slot i comes from lane - d, its slot i (slot
                // i - 1 where the lane index wraps); e + d from lane + d, slot
                // i (i + 1 where it wraps): the sender picks
#pragma unroll
                for (int i = 0; i < NCOL; i++) {
                    const float upv = (i > 0 && lane >= 32 - d) ? m[i - 1] : m[i];
                    const float dnv = (i + 1 < NCOL && lane < d) ? m[i + 1] : m[i];
                    nb[R - d][i] = __shfl_sync(0xffffffffu, upv, (lane + 32 - d) & 31);
                    nb[R + d][i] = __shfl_sync(0xffffffffu, dnv, (lane + d) & 31);
                }
            }
#pragma unroll
            for (int i = 0; i < NCOL; i++) {
                // this row is filter row fr of output k - fr (k counted from
                // the unit's first computed row); row 2R completes an output
                float row_sum[K];
#pragma unroll
                for (int fr = 0; fr < K; fr++) {
                    float sacc = fr == 0 ? a.w[fr * K] * nb[0][i] : fmaf(a.w[fr * K], nb[0][i], acc[fr - 1][i][c]);
#pragma unroll
                    for (int b = 1; b < K; b++)
                        sacc = fmaf(a.w[fr * K + b], nb[b][i], sacc);
                    row_sum[fr] = sacc;
                }
                if (store && emit[i])
                    st_cs(reinterpret_cast<float *>(op) + (rel0 + 32 * i) * C + c, row_sum[2 * R]);
#pragma unroll
                for (int j = 0; j < 2 * R; j++)
                    acc[j][i][c] = row_sum[j];
            }
        }
        if (store)
            op += a.dst_pitch;
    });
}

// ------------------------------------------------------------------ consumer: uint8 bilinear, row-separable

// Each warp takes CW output columns, each lane RUN consecutive ones.  The lane
// keeps the exact horizontal sums of the two newest listed source rows at its
// columns in two register buffers (writing a new row over the older one), and
// per output row combines them with the row's weights.
template <int C>
__device__ __forceinline__ bool consume_u8(const KArgs &a, const UnitGeom &g, const Ring &rg, Cursor &cs)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int RUN = stream_u8_run(C);
    const int CW = (a.TW + kConsumers / 32 - 1) / (kConsumers / 32);
    int b_lo, nbytes;
    unit_span<1, 0>(a, g, C, true, b_lo, nbytes);
    const int nc = g.dx1 - g.dx0;
    const int px0 = warp * CW + lane * RUN;   // first output column of this lane, relative to dx0
    const int npx = clampi(min(CW, nc - warp * CW) - lane * RUN, 0, RUN);
    int o0[RUN];        // byte offset of the left tap's first channel in a staged row
    uint32_t aw[RUN];   // {A0, A1} of the column
#pragma unroll
    for (int k = 0; k < RUN; k++) {
        const int2 xe = a.xt[g.dx0 + clampi(px0 + k, 0, nc - 1)];
        o0[k] = clampi(xe.x * C - b_lo, 0, nbytes - C);
        aw[k] = static_cast<uint32_t>(2048 - xe.y) | (static_cast<uint32_t>(xe.y) << 16);
    }
    // outputs leave as 32-bit words when the pixel run starts on a word
    const bool words = npx == RUN &&
                       ((reinterpret_cast<uintptr_t>(a.dst) | static_cast<uintptr_t>(a.dst_pitch) |
                         static_cast<uintptr_t>(a.dst_bstride) | static_cast<uintptr_t>((g.dx0 + px0) * C)) & 3) == 0;
    uint8_t *op = a.dst + (long long)g.b * a.dst_bstride + (long long)g.dy0 * a.dst_pitch +
                  (long long)(g.dx0 + (npx > 0 ? px0 : 0)) * C;
    int h0[RUN][C], h1[RUN][C];   // horizontal sums of the two newest listed rows
#pragma unroll
    for (int k = 0; k < RUN; k++)
#pragma unroll
        for (int c = 0; c < C; c++)
            h0[k][c] = h1[k][c] = 0;
    bool newer1 = false;          // h1 holds the newer row
    return walk_unit<0, 1>(a, g, rg, cs, [&](int, const uint8_t *top, const uint8_t *bot, int wbits, int nnew) {
        // taps: rows (top, bot) are the list's two newest, or the newest twice
        if (nnew == 2) {
#pragma unroll
            for (int k = 0; k < RUN; k++) {
                hsum_u8<C>(top, o0[k], aw[k], h0[k]);
                hsum_u8<C>(bot, o0[k], aw[k], h1[k]);
            }
            newer1 = true;
        } else if (nnew == 1) {
            if (newer1) {
#pragma unroll
                for (int k = 0; k < RUN; k++)
                    hsum_u8<C>(bot, o0[k], aw[k], h0[k]);
            } else {
#pragma unroll
                for (int k = 0; k < RUN; k++)
                    hsum_u8<C>(bot, o0[k], aw[k], h1[k]);
            }
            newer1 = !newer1;
        }
        // weight of the lower tap (the newer row); both taps on one row put
        // all of it there
        const int B1 = top == bot ? 2048 : wbits;
        const int wn = B1, wo = 2048 - B1;   // newer, older
        const int w0 = newer1 ? wo : wn, w1 = newer1 ? wn : wo;
        int q[RUN][C];
#pragma unroll
        for (int k = 0; k < RUN; k++)
#pragma unroll
            for (int c = 0; c < C; c++)
                q[k][c] = (w0 * h0[k][c] + w1 * h1[k][c] + (1 << 21)) >> 22;
        if (words) {
            uint32_t *o = reinterpret_cast<uint32_t *>(op);
            if constexpr (C == 1) {
                st_g(o, pack4(q[0][0], q[1][0], q[2][0], q[3][0]));
            } else if constexpr (C == 3) {
                st_g(o, pack4(q[0][0], q[0][1], q[0][2], q[1][0]));
                st_g(o + 1, pack4(q[1][1], q[1][2], q[2][0], q[2][1]));
                st_g(o + 2, pack4(q[2][2], q[3][0], q[3][1], q[3][2]));
            } else {
#pragma unroll
                for (int k = 0; k < RUN; k++)
                    st_g(o + k, pack4(q[k][0], q[k][1], q[k][2], q[k][3]));
            }
        } else {
#pragma unroll
            for (int k = 0; k < RUN; k++)
                if (k < npx)
#pragma unroll
                    for (int c = 0; c < C; c++)
                        st_g(op + k * C + c, static_cast<uint8_t>(q[k][c]));
        }
        op += a.dst_pitch;
    });
}

// ------------------------------------------------------------------ the kernel

// OP: STREAM_FILTER (float32 + K x K, K = 2R + 1) or STREAM_U8 (uint8
// bilinear).  The uint8 form holds two rows of sums for four pixels per lane.
// CTAs per SM the register budget is set for: 3 for the 3x3 filter, 2 for
// the uint8 form and the 5x5 and one-channel 7x7 filters, 1 for the 7x7
// filter on 3 or 4 channels (whose K - 1 rows of partial sums per channel
// would spill at two).
__host__ __device__ constexpr int stream_min_ctas(int op, int C, int R)
{
    return op == STREAM_U8 ? 2 : (R <= 1 ? 3 : (R == 3 && C > 1 ? 1 : 2));
}

template <int OP, int C, int LINEAR, int R>
__global__ void __launch_bounds__(kThreads, stream_min_ctas(OP, C, R))
    k_stream(const KArgs a, const __grid_constant__ CUtensorMap tmap)
{
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int ES = OP == STREAM_FILTER ? 4 : 1;
    constexpr int HALO = OP == STREAM_FILTER ? R : 0;
    Ring rg;
    rg.NCH = a.ring_chunks;
    rg.G = a.chunk_rows;
    rg.LG = __ffs(rg.G) - 1;
    rg.NB = a.chunk_boxes;
    rg.BW = a.box_bytes;
    rg.BB = stream_block_bytes(rg.G, rg.BW);
    rg.CB = rg.NB * rg.BB;
    rg.full = reinterpret_cast<uint64_t *>(smem);
    rg.empty = rg.full + rg.NCH;
    rg.chunks = smem + stream_chunks_off(rg.NCH);
    int *window = reinterpret_cast<int *>(smem + 16 * rg.NCH);   // producer: listed rows, by position mod 128
    const int nunits = a.batch * a.tiles_x * a.tiles_y;

    if (threadIdx.x == 0) {
        for (int c = 0; c < rg.NCH; c++) {
            mbar_init(&rg.full[c], a.tma_in ? 1 : 32);
            mbar_init(&rg.empty[c], kConsumers / 32);
        }
        fence_mbar_init();
    }
    __syncthreads();
    grid_launch_dependents();
    bounds_begin(a);
    // every thread reads global memory below: wait for the grids this launch
    // depends on
    grid_dependency_wait();

    if (threadIdx.x >= kConsumers) {
        stream_producer<ES, HALO, LINEAR>(a, &tmap, rg, window, C);
        return;
    }
    Cursor cs;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
        const UnitGeom g = unit_geom(a, u);
        bool ok;
        if constexpr (OP == STREAM_FILTER)
            ok = consume_filter<C, LINEAR, R>(a, g, rg, cs);
        else
            ok = consume_u8<C>(a, g, rg, cs);
        if (!ok)
            break;
    }
}

}  // namespace

// Bilinear only: the fused entry point is bilinear by contract, and the
// uint8 streaming form is chosen for bilinear resizes.  R: the filter's
// halo (K = 2R + 1, 0..3; R = 0 with weight 1 is the plain float32 resize);
// ignored for the uint8 form.
const void *stream_kernel_for(int op, int mode, int C, int R)
{
    using Fn = void (*)(const KArgs, const CUtensorMap);
    static const Fn filt[4][3] = {
        {k_stream<STREAM_FILTER, 1, 1, 0>, k_stream<STREAM_FILTER, 3, 1, 0>, k_stream<STREAM_FILTER, 4, 1, 0>},
        {k_stream<STREAM_FILTER, 1, 1, 1>, k_stream<STREAM_FILTER, 3, 1, 1>, k_stream<STREAM_FILTER, 4, 1, 1>},
        {k_stream<STREAM_FILTER, 1, 1, 2>, k_stream<STREAM_FILTER, 3, 1, 2>, k_stream<STREAM_FILTER, 4, 1, 2>},
        {k_stream<STREAM_FILTER, 1, 1, 3>, k_stream<STREAM_FILTER, 3, 1, 3>, k_stream<STREAM_FILTER, 4, 1, 3>}};
    static const Fn u8[3] = {k_stream<STREAM_U8, 1, 1, 0>, k_stream<STREAM_U8, 3, 1, 0>,
                             k_stream<STREAM_U8, 4, 1, 0>};
    const int ci = (C == 1) ? 0 : (C == 3 ? 1 : (C == 4 ? 2 : -1));
    if (ci < 0 || mode != RZ_LINEAR)
        return nullptr;
    if (op == STREAM_FILTER)
        return (R >= 0 && R <= 3) ? reinterpret_cast<const void *>(filt[R][ci]) : nullptr;
    return reinterpret_cast<const void *>(u8[ci]);
}

}  // namespace rz
