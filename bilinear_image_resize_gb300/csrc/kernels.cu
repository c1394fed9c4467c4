// Resize kernels for sm_103a: uint8 and float32 resize and the normalise
// epilogue (the filter epilogues stream strips instead: stream.cu).
//
// Persistent CTAs (as many as fit on the GPU at once) walk the output tiles
// of TR rows x TW columns in a static round-robin.  Each CTA is warp
// specialised:
//   * one producer warp keeps a ring of `stages` tiles of source rows in
//     shared memory.  It plans each tile in a ring of stages + 1 plan
//     entries one tile ahead: the tile's column span and the distinct source
//     rows its output rows sample (two per row for bilinear, one for
//     nearest), derived exactly from the sampling formula with warp votes,
//     without reading memory.  When the consumers release a stage (its
//     "empty" mbarrier) it issues one bulk (TMA) copy per row, or per run of
//     whole consecutive rows, completing on the stage's "full" mbarrier; the
//     normalise family's table entries come along as two more bulk copies.
//     When the source is not 16-byte aligned the warp copies the rows itself;
//   * eight consumer warps compute each tile from shared memory into one of
//     two output buffers (uint8 bilinear as the exact 11-bit fixed-point sum,
//     float32 as two lerps, then the fused epilogue), and one consumer thread
//     writes each output row with one bulk (TMA) store.
// HBM is read once per needed source byte and written once per output byte.
//
// Sampling: CUDA interpolation page (hnwysp.cn/news/129086) §2.1 nearest,
// §2.2 bilinear weights, §6.1 clamp, §6.2 fixed point, §4.2 fused epilogue;
// half-pixel mapping: "From Prototype to Performance: Optimizing OpenCV Resize
// on Volcanic GPUs", "Naive resize with linear sampling".  The per-column and
// per-row tables come from the plan (api.cu), where they are computed exactly.
#include <cuda_runtime.h>

#include <cstdint>

#include "rz_device.h"
#include "rz_internal.h"

namespace rz {
namespace {

using namespace dev;

// ------------------------------------------------------------------ tiles and stages

struct TileGeom {
    int dy0, dy1;       // output rows [dy0, dy1)
    int dx0, dx1;       // output columns [dx0, dx1)
    const uint8_t *src; // this tile's source image
    uint8_t *dst;       // this tile's output image
};

__device__ __forceinline__ TileGeom tile_geom(const KArgs &a, int tile)
{
    TileGeom g;
    const int per_img = a.tiles_x * a.tiles_y;
    const int b = tile / per_img;
    const int r = tile - b * per_img;
    const int ty = r / a.tiles_x;
    const int tx = r - ty * a.tiles_x;
    g.dy0 = ty * a.TR;
    g.dy1 = min(g.dy0 + a.TR, a.OH);
    g.dx0 = tx * a.TW;
    g.dx1 = min(g.dx0 + a.TW, a.OW);
    g.src = a.src + (long long)b * a.src_bstride;
    g.dst = a.dst + (long long)b * a.dst_bstride;
    return g;
}

// Tile plan header, at the start of each plan entry: everything the copies
// and the consumers need beyond the row list and slot map.
struct StageHdr {
    int nrows;   // staged rows (-1: tile rejected)
    int b_lo;    // byte offset, within a source row, of slot byte 0
    int nbytes;  // bytes staged per row
    int tile;    // tile index
    int image;   // image index within the batch
    int xsh;     // staged x (y) table entries start this many entries
    int ysh;     //   before the tile's first column (row): 0 or 1
    int xa, xn;  // x table entries copied: [xa, xa + xn), even bounds
    int ya, yn;  // y table entries copied: [ya, ya + yn), even bounds
    int pad[5];
};
static_assert(sizeof(StageHdr) == 64, "plan header size");

// Producer warp, part 1 (no global memory access): list the source rows of
// `tile` into plan entry `pl`.  Lanes derive the tile's column span and row
// indices in parallel, one computed output row per lane; which rows are new
// and where each lands in the list follow from warp votes (the sampled rows
// never decrease along the output rows); lane 0 records the header.
template <int LINEAR>
__device__ void plan_stage(const KArgs &a, const SmemLayout &L, uint8_t *pl, int tile, int in_es)
{
    const int lane = threadIdx.x & 31;
    StageHdr *h = reinterpret_cast<StageHdr *>(pl);
    int *rows = reinterpret_cast<int *>(pl + L.rows_off);
    int *map = reinterpret_cast<int *>(pl + L.map_off);
    const TileGeom g = tile_geom(a, tile);

    const int nrc = g.dy1 - g.dy0;   // output rows of the tile
    int xv = 0;
    if (lane < 2)
        xv = sample_index<LINEAR>(a.W, a.OW, lane == 0 ? g.dx0 : g.dx1 - 1, a.border);
    int yv = 0;
    if (lane < nrc)
        yv = sample_index<LINEAR>(a.H, a.OH, g.dy0 + lane, a.border);
    const int xs0 = __shfl_sync(0xffffffffu, xv, 0);
    const int xs1r = __shfl_sync(0xffffffffu, xv, 1);
    const int xs1 = LINEAR ? min(xs1r + 1, a.W - 1) : xs1r;
    int b_lo = xs0 * a.C * in_es;
    int b_hi = (xs1 + 1) * a.C * in_es;
    if (a.tma_in) {
        b_lo &= ~15;
        b_hi = (b_hi + 15) & ~15;
    }
    const int nbytes = b_hi - b_lo;

    // Distinct source rows.  Lane k takes output row k (32 rows per pass)
    // with taps r0 <= r1 <= r0 + 1.  Taps never decrease along k, so r0 is
    // already listed exactly when r0 <= r1 of row k - 1, and is then the last
    // or the one-before-last entry listed before row k; r1 is new exactly
    // when it exceeds both.  Counts of new taps on lower lanes (ballots) give
    // each tap its slot.
    int n = 0, r1_before = -1;
    bool overflow = nbytes > a.slot_bytes;
    const unsigned lower = (1u << lane) - 1u;
    for (int base = 0; base < nrc; base += 32) {
        const int k = base + lane;
        const bool act = k < nrc;
        int r0 = 0x7fffffff, r1 = 0x7fffffff;
        if (act) {
            r0 = k < 32 ? yv : sample_index<LINEAR>(a.H, a.OH, g.dy0 + k, a.border);
            r1 = LINEAR ? min(r0 + 1, a.H - 1) : r0;
        }
        int prev_r1 = __shfl_up_sync(0xffffffffu, r1, 1);
        if (lane == 0)
            prev_r1 = r1_before;
        const bool new0 = act && r0 > prev_r1;
        const bool new1 = act && r1 > max(r0, prev_r1);
        const unsigned b0 = __ballot_sync(0xffffffffu, new0), b1 = __ballot_sync(0xffffffffu, new1);
        const int c = n + __popc(b0 & lower) + __popc(b1 & lower);   // entries listed before row k
        const int s0 = new0 ? c : c - 1 - (prev_r1 - r0);
        const int s1 = new1 ? c + (new0 ? 1 : 0) : (r1 == r0 ? s0 : c - 1);
        if (act) {
            if (new0 && s0 < a.max_rows) rows[s0] = r0;
            if (new1 && s1 < a.max_rows) rows[s1] = r1;
            map[2 * k] = s0;
            map[2 * k + 1] = s1;
        }
        n += __popc(b0) + __popc(b1);
        r1_before = __shfl_sync(0xffffffffu, r1, min(31, nrc - 1 - base));
    }
    if (n > a.max_rows)
        overflow = true;
    if (lane == 0) {
        // the host sizes max_rows and slot_bytes from the same indices, so
        // an overflow is unreachable; it guards shared memory
        h->nrows = overflow ? -1 : n;
        h->b_lo = b_lo;
        h->nbytes = nbytes;
        h->tile = tile;
        h->image = tile / (a.tiles_x * a.tiles_y);
        h->xsh = g.dx0 & 1;
        h->ysh = g.dy0 & 1;
        // table entries of the tile's columns and rows, widened to even
        // bounds (16-byte copies)
        h->xa = g.dx0 & ~1;
        h->xn = align_up(g.dx1, 2) - h->xa;
        h->ya = g.dy0 & ~1;
        h->yn = align_up(g.dy1, 2) - h->ya;
    }
    __syncwarp();
}

// Producer warp, part 2: fetch the planned rows.  Bulk path: lane 0 arms
// `full` with the byte count before any copy is issued, and the copies are
// spread over the lanes.  Plain path (unaligned source): the lanes copy the
// bytes and each arrives on `full` (initialised for 32 arrivals).
__device__ void fetch_stage(const KArgs &a, const SmemLayout &L, const uint8_t *pl, uint8_t *st, uint64_t *full,
                            uint64_t policy, bool tables)
{
    const int lane = threadIdx.x & 31;
    const StageHdr *h = reinterpret_cast<const StageHdr *>(pl);
    const int *rows = reinterpret_cast<const int *>(pl + L.rows_off);
    uint8_t *slots = st + L.slots_off;
    const uint8_t *img = a.src + (long long)h->image * a.src_bstride;   // this tile's source image
    const int n = h->nrows, nbytes = h->nbytes, b_lo = h->b_lo;
    if (n < 0 && lane == 0)
        atomicExch(a.status, RZ_ERR_ARG);
    if (tables) {
        // the tile's x entries and y entries, each one bulk copy of a range
        // that starts and ends on an even entry (the plan's tables repeat
        // their end entries past both ends)
        int2 *tx = reinterpret_cast<int2 *>(st + L.tab_off);
        int2 *ty = tx + tab_x_entries(a.TW);
        const int xa = h->xa, xb = h->xa + h->xn;
        const int ya = h->ya, yb = h->ya + h->yn;
        const uint32_t tab_bytes = static_cast<uint32_t>(8 * ((xb - xa) + (yb - ya)));
        if (a.tma_in) {
            const uint32_t bytes = tab_bytes + static_cast<uint32_t>(n > 0 ? n * nbytes : 0);
            if (lane == 0) {
                mbar_arrive_expect_tx(full, bytes);
                bulk_load(tx, a.xt + xa, static_cast<uint32_t>(8 * (xb - xa)), full);
                bulk_load(ty, a.yt + ya, static_cast<uint32_t>(8 * (yb - ya)), full);
            }
            __syncwarp();
            for (int r = lane; r < n; r += 32)
                bulk_load_hint(slots + r * a.slot_bytes, img + (long long)rows[r] * a.src_pitch + b_lo,
                               static_cast<uint32_t>(nbytes), full, policy);
        } else {
            // the tables still move as bulk copies (armed before any lane
            // arrives); the unaligned rows are copied by the lanes, each of
            // which arrives after its own copies
            if (lane == 0) {
                mbar_expect_tx(full, tab_bytes);
                bulk_load(tx, a.xt + xa, static_cast<uint32_t>(8 * (xb - xa)), full);
                bulk_load(ty, a.yt + ya, static_cast<uint32_t>(8 * (yb - ya)), full);
            }
            for (int r = 0; r < n; r++) {
                const uint8_t *src = img + (long long)rows[r] * a.src_pitch + b_lo;
                uint8_t *d = slots + r * a.slot_bytes;
                for (int k = lane; k < nbytes; k += 32)
                    if (smem_guard(d + k, 1))
                        d[k] = ld_nc(src + k);
            }
            __syncwarp();
            mbar_arrive(full);
        }
    } else if (a.tma_in) {
        // a rejected tile completes the phase with no bytes
        if (lane == 0)
            mbar_arrive_expect_tx(full, static_cast<uint32_t>(n > 0 ? n * nbytes : 0));
        __syncwarp();
        if (b_lo == 0 && nbytes == a.src_pitch && nbytes == a.slot_bytes) {
            // whole rows that sit back to back in memory and in the slots:
            // one bulk copy per run of consecutive source rows (a bulk copy
            // has a fixed cost, so fewer, larger copies stream faster)
            if (lane == 0) {
                int r = 0;
                while (r < n) {
                    int e = r + 1;
                    while (e < n && rows[e] == rows[e - 1] + 1)
                        e++;
                    bulk_load_hint(slots + r * a.slot_bytes, img + (long long)rows[r] * a.src_pitch,
                                   static_cast<uint32_t>((e - r) * nbytes), full, policy);
                    r = e;
                }
            }
        } else {
            for (int r = lane; r < n; r += 32)
                bulk_load_hint(slots + r * a.slot_bytes, img + (long long)rows[r] * a.src_pitch + b_lo,
                               static_cast<uint32_t>(nbytes), full, policy);
        }
    } else {
        for (int r = 0; r < n; r++) {
            const uint8_t *src = img + (long long)rows[r] * a.src_pitch + b_lo;
            uint8_t *d = slots + r * a.slot_bytes;
            for (int k = lane; k < nbytes; k += 32)
                if (smem_guard(d + k, 1))
                    d[k] = ld_nc(src + k);
        }
        mbar_arrive(full);   // each lane releases its own copies
    }
}

// One consumer thread: one bulk store per output row of the tile (the
// 16-byte multiple of each row; the ragged tail goes through store_tail).
__device__ void issue_stores(const KArgs &a, const SmemLayout &L, const uint8_t *ob, const TileGeom &g, int planes,
                             int px_bytes)
{
    const int nr = g.dy1 - g.dy0;
    const int row_bytes = (g.dx1 - g.dx0) * px_bytes;
    const int bulk = row_bytes & ~15;
    if (bulk > 0) {
        uint8_t *base = g.dst + (long long)g.dy0 * a.dst_pitch + (long long)g.dx0 * px_bytes;
        for (int c = 0; c < planes; c++)
            for (int i = 0; i < nr; i++)
                bulk_store(base + c * a.dst_plane + i * a.dst_pitch, ob + (c * a.TR + i) * L.out_row_bytes,
                           static_cast<uint32_t>(bulk));
    }
    bulk_commit();
}

// Consumer threads: write the bytes of each output row that the bulk stores
// do not cover (all of them when bulk stores are not allowed).
__device__ void store_tail(const KArgs &a, const SmemLayout &L, const uint8_t *ob, const TileGeom &g, int planes,
                           int px_bytes)
{
    const int nr = g.dy1 - g.dy0;
    const int row_bytes = (g.dx1 - g.dx0) * px_bytes;
    const int bulk = a.tma_out ? (row_bytes & ~15) : 0;
    const int tail = row_bytes - bulk;
    if (tail <= 0)
        return;
    uint8_t *base = g.dst + (long long)g.dy0 * a.dst_pitch + (long long)g.dx0 * px_bytes + bulk;
    const int n = planes * nr * tail;
    for (int k = threadIdx.x; k < n; k += kConsumers) {
        const int row = k / tail, j = k - row * tail;
        const int c = row / nr, i = row - c * nr;
        const uint8_t *sp = ob + (c * a.TR + i) * L.out_row_bytes + bulk + j;
        if (smem_guard(sp, 1))
            st_g(base + c * a.dst_plane + i * a.dst_pitch + j, *sp);
    }
}

// ------------------------------------------------------------------ compute: one tile

struct StageView {
    const uint8_t *slots;
    const int *map;
    const int2 *tx;   // staged x entries (narrow-tile families)
    const int2 *ty;   // staged y entries (narrow-tile families)
    int b_lo, slot_bytes;
};

__device__ __forceinline__ StageView stage_view(const KArgs &a, const SmemLayout &L, const uint8_t *pl,
                                                const uint8_t *st)
{
    StageView v;
    const StageHdr *h = reinterpret_cast<const StageHdr *>(pl);
    v.tx = reinterpret_cast<const int2 *>(st + L.tab_off) + h->xsh;
    v.ty = reinterpret_cast<const int2 *>(st + L.tab_off) + tab_x_entries(a.TW) + h->ysh;
    v.slots = st + L.slots_off;
    v.map = reinterpret_cast<const int *>(pl + L.map_off);
    v.b_lo = h->b_lo;
    v.slot_bytes = a.slot_bytes;
    return v;
}

// uint8 bilinear of one output pixel from two staged rows.  `o0` is the
// byte offset (within the staged rows) of the left tap's first channel; the
// right tap follows C bytes later (at the right image edge the plan gives the
// right tap weight 0, and the bytes read past the row are padding, so the
// product is 0).  Each row's pair of taps is summed exactly by hsum_u8:
//   q = (B0 hT + B1 hB + 2^21) >> 22.
template <int C>
__device__ __forceinline__ void bilinear_u8_px(const uint8_t *top, const uint8_t *bot, int o0, uint32_t aw, int B0,
                                               int B1, int (&q)[C])
{
    int hT[C], hB[C];
    hsum_u8<C>(top, o0, aw, hT);
    hsum_u8<C>(bot, o0, aw, hB);
#pragma unroll
    for (int c = 0; c < C; c++)
        q[c] = (B0 * hT[c] + B1 * hB[c] + (1 << 21)) >> 22;
}

// Generic bilinear / nearest, any ratio.  Each thread takes runs of four
// consecutive output pixels: their column-table entries arrive in two 16-byte
// loads (the tables are 16-byte aligned and carry spare entries past the last
// column), and their outputs leave in 32-bit (uint8) or 128-bit (float)
// shared-memory stores.  uint8 bilinear is
//   out = (B0 (A0 t0 + A1 t1) + B1 (A0 b0 + A1 b1) + 2^21) >> 22
// with A1 = 11-bit weight of the right tap, B1 of the lower row — exact in
// int32 (at most 2048 * 2048 * 255 + 2^21 < 2^31).
template <typename T, int C, int LINEAR>
__device__ void compute_generic(const KArgs &a, const StageView &sv, const TileGeom &g, uint8_t *ob_bytes,
                                int orow_bytes)
{
    constexpr int ES = sizeof(T);
    constexpr int RUN = 4;
    const int nr = g.dy1 - g.dy0, nc = g.dx1 - g.dx0;
    const int nruns = (nc + RUN - 1) / RUN;
    const int lg = min(8, ceil_log2(nruns));
    const int tpr = 1 << lg, rpp = kConsumers >> lg;
    const bool pair_ok = (g.dx0 & 1) == 0;   // 16-byte table loads start on an even column
    for (int rl = threadIdx.x >> lg; rl < nr; rl += rpp) {
        const int2 yw = ld_nc(&a.yt[g.dy0 + rl]);
        const uint8_t *top = sv.slots + sv.map[2 * rl] * sv.slot_bytes;
        const uint8_t *bot = sv.slots + sv.map[2 * rl + 1] * sv.slot_bytes;
        uint8_t *orow = ob_bytes + rl * orow_bytes;
        for (int j = threadIdx.x & (tpr - 1); j < nruns; j += tpr) {
            const int p0 = j * RUN;
            const int npx = min(RUN, nc - p0);
            int2 xw[RUN];
            if (pair_ok) {
                // a row's last run may read up to three entries past the
                // tile's last column (values unused): plan tables keep kTabPad
                // spare entries after their end, and the no-alloc array's
                // column table is followed by its row table
                const int4 v0 = ld_nc(reinterpret_cast<const int4 *>(a.xt + g.dx0 + p0));
                const int4 v1 = ld_nc(reinterpret_cast<const int4 *>(a.xt + g.dx0 + p0 + 2));
                xw[0] = make_int2(v0.x, v0.y);
                xw[1] = make_int2(v0.z, v0.w);
                xw[2] = make_int2(v1.x, v1.y);
                xw[3] = make_int2(v1.z, v1.w);
            } else {
#pragma unroll
                for (int k = 0; k < RUN; k++)
                    xw[k] = p0 + k < nc ? ld_nc(&a.xt[g.dx0 + p0 + k]) : make_int2(0, 0);
            }
            if constexpr (ES == 1) {
                int q[RUN][C];
#pragma unroll
                for (int k = 0; k < RUN; k++) {
                    if (k < npx) {
                        const int o0 = xw[k].x * C - sv.b_lo;
                        if (!LINEAR) {
                            const bool ok = smem_guard(top + o0, C);
#pragma unroll
                            for (int c = 0; c < C; c++)
                                q[k][c] = ok ? top[o0 + c] : 0;
                        } else {
                            const uint32_t aw = static_cast<uint32_t>(2048 - xw[k].y) |
                                                (static_cast<uint32_t>(xw[k].y) << 16);
                            bilinear_u8_px<C>(top, bot, o0, aw, 2048 - yw.y, yw.y, q[k]);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < C; c++)
                            q[k][c] = 0;
                    }
                }
                uint8_t *o = orow + p0 * C;
                if (!smem_guard(o, npx * C))
                    continue;
                if (npx == RUN) {
                    if constexpr (C == 1) {
                        *reinterpret_cast<uint32_t *>(o) = pack4(q[0][0], q[1][0], q[2][0], q[3][0]);
                    } else if constexpr (C == 3) {
                        uint32_t *w = reinterpret_cast<uint32_t *>(o);
                        w[0] = pack4(q[0][0], q[0][1], q[0][2], q[1][0]);
                        w[1] = pack4(q[1][1], q[1][2], q[2][0], q[2][1]);
                        w[2] = pack4(q[2][2], q[3][0], q[3][1], q[3][2]);
                    } else {
                        *reinterpret_cast<uint4 *>(o) = make_uint4(pack4(q[0][0], q[0][1], q[0][2], q[0][3]),
                                                                   pack4(q[1][0], q[1][1], q[1][2], q[1][3]),
                                                                   pack4(q[2][0], q[2][1], q[2][2], q[2][3]),
                                                                   pack4(q[3][0], q[3][1], q[3][2], q[3][3]));
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < RUN; k++)
                        if (k < npx)
#pragma unroll
                            for (int c = 0; c < C; c++)
                                o[k * C + c] = static_cast<uint8_t>(q[k][c]);
                }
            } else {
                const float *ft = reinterpret_cast<const float *>(top);
                const float *fb = reinterpret_cast<const float *>(bot);
                const int lo = sv.b_lo / 4;
                const float v = __int_as_float(yw.y);
                float r[RUN][C];
#pragma unroll
                for (int k = 0; k < RUN; k++) {
                    if (k < npx) {
                        const int o0 = xw[k].x * C - lo;
                        if (!LINEAR) {
                            const bool ok = smem_guard(ft + o0, 4 * C);
#pragma unroll
                            for (int c = 0; c < C; c++)
                                r[k][c] = ok ? ft[o0 + c] : 0.0f;
                        } else {
                            const int o1 = min(xw[k].x + 1, a.W - 1) * C - lo;
                            if (!(smem_guard(ft + o0, 4 * C) && smem_guard(ft + o1, 4 * C) &&
                                  smem_guard(fb + o0, 4 * C) && smem_guard(fb + o1, 4 * C))) {
#pragma unroll
                                for (int c = 0; c < C; c++)
                                    r[k][c] = 0.0f;
                                continue;
                            }
                            const float u = __int_as_float(xw[k].y);
#pragma unroll
                            for (int c = 0; c < C; c++) {
                                const float t0 = ft[o0 + c], t1 = ft[o1 + c];
                                const float b0 = fb[o0 + c], b1 = fb[o1 + c];
                                const float hT = fmaf(u, t1 - t0, t0);
                                const float hB = fmaf(u, b1 - b0, b0);
                                r[k][c] = fmaf(v, hB - hT, hT);
                            }
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < C; c++)
                            r[k][c] = 0.0f;
                    }
                }
                float *o = reinterpret_cast<float *>(orow) + p0 * C;
                if (!smem_guard(o, 4 * npx * C))
                    continue;
                if (npx == RUN) {
                    // RUN * C floats from a 16-byte aligned start: C float4 stores
                    float4 *o4 = reinterpret_cast<float4 *>(o);
#pragma unroll
                    for (int m = 0; m < C; m++) {
                        const int e = 4 * m;
                        o4[m] = make_float4(r[(e + 0) / C][(e + 0) % C], r[(e + 1) / C][(e + 1) % C],
                                            r[(e + 2) / C][(e + 2) % C], r[(e + 3) / C][(e + 3) % C]);
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < RUN; k++)
                        if (k < npx)
#pragma unroll
                            for (int c = 0; c < C; c++)
                                o[k * C + c] = r[k][c];
                }
            }
        }
    }
}

// Exact 2x downscale of uint8 (W = 2 OW, H = 2 OH): see down2_group.  The
// tile's staged span starts at the tile's first source byte, 16-byte aligned
// (the host keeps TW a multiple of 8 columns).
template <int C>
__device__ void compute_down2(const KArgs &a, const StageView &sv, const TileGeom &g, uint8_t *ob, int orow_bytes)
{
    const int nr = g.dy1 - g.dy0, nc = g.dx1 - g.dx0;
    const int ofs0 = 2 * g.dx0 * C - sv.b_lo;    // 0 or a multiple of 16
    constexpr int PX = down2_px(C);              // 8, 4, 2 pixels: 8, 12, 8 output bytes
    constexpr int SW = 2 * PX * C / 4;           // source words per row and group
    const int ngrp = nc / PX;
    const int lg = min(8, ceil_log2(ngrp + 1));
    const int tpr = 1 << lg, rpp = kConsumers >> lg;
    for (int rl = threadIdx.x >> lg; rl < nr; rl += rpp) {
        const uint8_t *top = sv.slots + sv.map[2 * rl] * sv.slot_bytes + ofs0;
        const uint8_t *bot = sv.slots + sv.map[2 * rl + 1] * sv.slot_bytes + ofs0;
        uint8_t *orow = ob + rl * orow_bytes;
        for (int j = threadIdx.x & (tpr - 1); j < ngrp; j += tpr) {
            if (!(smem_guard(top + 4 * SW * j, 4 * SW) && smem_guard(bot + 4 * SW * j, 4 * SW) &&
                  smem_guard(orow + 2 * SW * j, 2 * SW)))
                continue;
            uint32_t tw[SW], bw[SW], o[SW / 2];
            if constexpr (C == 3) {
                const uint2 *tp = reinterpret_cast<const uint2 *>(top + 24 * j);
                const uint2 *bp = reinterpret_cast<const uint2 *>(bot + 24 * j);
#pragma unroll
                for (int k = 0; k < 3; k++) {
                    const uint2 t = tp[k], b = bp[k];
                    tw[2 * k] = t.x; tw[2 * k + 1] = t.y;
                    bw[2 * k] = b.x; bw[2 * k + 1] = b.y;
                }
            } else {
                const uint4 t = *reinterpret_cast<const uint4 *>(top + 16 * j);
                const uint4 b = *reinterpret_cast<const uint4 *>(bot + 16 * j);
                tw[0] = t.x; tw[1] = t.y; tw[2] = t.z; tw[3] = t.w;
                bw[0] = b.x; bw[1] = b.y; bw[2] = b.z; bw[3] = b.w;
            }
            down2_group<C>(tw, bw, o);
            if constexpr (C == 3) {
                uint32_t *op = reinterpret_cast<uint32_t *>(orow + 12 * j);
                op[0] = o[0]; op[1] = o[1]; op[2] = o[2];
            } else {
                *reinterpret_cast<uint2 *>(orow + 8 * j) = make_uint2(o[0], o[1]);
            }
        }
        // columns left over after whole groups
        for (int p = ngrp * PX + (threadIdx.x & (tpr - 1)); p < nc; p += tpr) {
#pragma unroll
            for (int c = 0; c < C; c++) {
                const int o = 2 * p * C + c;
                if (!(smem_guard(top + o, C + 1) && smem_guard(bot + o, C + 1) && smem_guard(orow + p * C + c, 1)))
                    continue;
                const int s = top[o] + top[o + C] + bot[o] + bot[o + C] + 2;
                orow[p * C + c] = static_cast<uint8_t>(s >> 2);
            }
        }
    }
}

// Bilinear + normalise: the uint8 result q of the generic sum, then
// y = q * scale[c] + shift[c] written planar.  Four pixels per thread step.
template <int C>
__device__ void compute_normalize(const KArgs &a, const StageView &sv, const TileGeom &g, uint8_t *ob_bytes,
                                  int orow_bytes)
{
    constexpr int U = 4;
    float *ob = reinterpret_cast<float *>(ob_bytes);
    const int orow_el = orow_bytes / 4;
    const int plane_el = a.TR * orow_el;
    const int nr = g.dy1 - g.dy0, nc = g.dx1 - g.dx0;
    const int lg = min(8, ceil_log2((nc + U - 1) / U));
    const int tpr = 1 << lg, rpp = kConsumers >> lg;
    for (int rl = threadIdx.x >> lg; rl < nr; rl += rpp) {
        const int2 yw = smem_guard(sv.ty + rl, 8) ? sv.ty[rl] : make_int2(0, 0);
        const int B1 = yw.y, B0 = 2048 - B1;
        const uint8_t *top = sv.slots + sv.map[2 * rl] * sv.slot_bytes;
        const uint8_t *bot = sv.slots + sv.map[2 * rl + 1] * sv.slot_bytes;
        for (int c0 = threadIdx.x & (tpr - 1); c0 < nc; c0 += U * tpr) {
            int2 xw[U];
#pragma unroll
            for (int k = 0; k < U; k++) {
                const int cl = c0 + k * tpr;
                xw[k] = cl < nc && smem_guard(sv.tx + cl, 8) ? sv.tx[cl] : make_int2(0, 0);
            }
#pragma unroll
            for (int k = 0; k < U; k++) {
                const int cl = c0 + k * tpr;
                if (cl >= nc)
                    break;
                const uint32_t aw = static_cast<uint32_t>(2048 - xw[k].y) | (static_cast<uint32_t>(xw[k].y) << 16);
                int q[C];
                bilinear_u8_px<C>(top, bot, xw[k].x * C - sv.b_lo, aw, B0, B1, q);
#pragma unroll
                for (int c = 0; c < C; c++)
                    if (smem_guard(ob + c * plane_el + rl * orow_el + cl, 4))
                        ob[c * plane_el + rl * orow_el + cl] = fmaf(static_cast<float>(q[c]), a.scale[c], a.shift[c]);
            }
        }
    }
}

// ------------------------------------------------------------------ the persistent kernel

// OP: 0 plain resize (T, C, LINEAR, VAR), 1 normalise.
template <int OP, typename T, int C, int LINEAR, int VAR>
__global__ void __launch_bounds__(kThreads, 4) k_resize(const KArgs a, const __grid_constant__ CUtensorMap)
{
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int FAM = OP == 1 ? FAM_NORM : (sizeof(T) == 1 ? FAM_U8 : FAM_F32);
    constexpr int IN_ES = fam_in_es(FAM);
    constexpr int PLANES = OP == 1 ? C : 1;
    constexpr int PX_BYTES = OP == 1 ? 4 : C * fam_out_es(FAM);
    const SmemLayout L = smem_layout(FAM, C, a.TR, a.TW, a.max_rows, a.slot_bytes, a.stages);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kMaxStages;
    const int ntiles = a.batch * a.tiles_x * a.tiles_y;
    const int NS = a.stages;
    const int G = gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; s++) {
            mbar_init(&full[s], a.tma_in ? 1 : 32);
            mbar_init(&empty[s], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();
    // the next launch in the stream may begin its set-up now
    grid_launch_dependents();
    bounds_begin(a);

    if (threadIdx.x >= kConsumers) {
        // ---------------- producer warp
        const uint64_t policy = policy_evict_first();
        // plan the first stages before waiting for the grids this launch
        // depends on: planning reads no global memory
        const int NP = NS + 1;
        for (int k = 0; k < NS; k++) {
            const int t = blockIdx.x + k * G;
            if (t < ntiles)
                plan_stage<LINEAR>(a, L, smem + L.plan_off + k * L.plan_bytes, t, IN_ES);
        }
        grid_dependency_wait();
        int it = 0;
        for (int t = blockIdx.x; t < ntiles; t += G, ++it) {
            const int s = it % NS;
            uint8_t *st = smem + L.stage_off + s * L.stage_bytes;
            if (it >= NS) {
                // wait until the consumers have released this stage's previous tile
                bool ok = true;
                if ((threadIdx.x & 31) == 0)
                    ok = mbar_wait_bounded(&empty[s], ((it / NS) - 1) & 1, a.status);
                if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0))
                    break;
            }
            fetch_stage(a, L, smem + L.plan_off + (it % NP) * L.plan_bytes, st, &full[s], policy,
                        fam_tables_in_stage(FAM));
            // plan the next tile while the consumers work.  Tiles it - NS + 1
            // .. it may still be in use; with NS + 1 plan entries the next
            // tile's entry is none of theirs.
            if (it + 1 >= NS && t + G < ntiles)
                plan_stage<LINEAR>(a, L, smem + L.plan_off + ((it + 1) % NP) * L.plan_bytes, t + G, IN_ES);
        }
        return;
    }
    // consumers touch global memory only after the grids this launch depends
    // on are complete
    grid_dependency_wait();

    // ---------------- consumer warps
    int it = 0;
    bool failed = false;
    for (int t = blockIdx.x; t < ntiles; t += G, ++it) {
        const int s = it % NS;
        uint8_t *st = smem + L.stage_off + s * L.stage_bytes;
        const uint8_t *pl = smem + L.plan_off + (it % (NS + 1)) * L.plan_bytes;
        uint8_t *ob = smem + L.out_off + (it & 1) * L.out_bytes;
        // the output buffer is free once the store issued two tiles ago has read it
        if (threadIdx.x == 0 && it >= 2)
            bulk_wait_read<1>();
        // one consumer thread waits for the stage (acquiring the bulk-copied
        // bytes); the other warps wait in the hardware barrier, which issues
        // nothing, and leave it ordered after that thread's acquire.  All
        // consumers leave the loop together if the wait timed out.
        bool ok = true;
        if (threadIdx.x == 0)
            ok = mbar_wait_bounded(&full[s], (it / NS) & 1, a.status);
        if (consumer_any(!ok) || reinterpret_cast<const StageHdr *>(pl)->nrows < 0) {
            failed = true;
            break;
        }
        const TileGeom g = tile_geom(a, t);
        const StageView sv = stage_view(a, L, pl, st);
        if constexpr (OP == 0) {
            if constexpr (VAR == VAR_DOWN2)
                compute_down2<C>(a, sv, g, ob, L.out_row_bytes);
            else
                compute_generic<T, C, LINEAR>(a, sv, g, ob, L.out_row_bytes);
        } else {
            compute_normalize<C>(a, sv, g, ob, L.out_row_bytes);
        }
        fence_proxy_async_smem();
        consumer_sync();
        if (threadIdx.x == 0) {
            mbar_arrive(&empty[s]);          // the stage may be refilled
            if (a.tma_out)
                issue_stores(a, L, ob, g, PLANES, PX_BYTES);
        }
        store_tail(a, L, ob, g, PLANES, PX_BYTES);
    }
    if (threadIdx.x == 0) {
        bulk_wait_read<0>();
        if (failed && a.tma_in) {
            // let bulk loads still in flight land before the CTA leaves
            for (int k = 0; k < NS; k++) {
                const int j = it + k;
                if (blockIdx.x + j * G < ntiles)
                    mbar_wait_bounded(&full[j % NS], (j / NS) & 1, nullptr);
            }
        }
    }
}

// Self-test of the bounded wait: one thread waits on a barrier nothing
// arrives on; the wait must give up after limit_ns and report the time-out.
__global__ void k_wait_selftest(int *status, unsigned long long limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0)
        return;
    mbar_init(&bar, 1);
    fence_mbar_init();
    *status = RZ_OK;
    mbar_wait_bounded(&bar, 0, status, limit_ns);   // writes RZ_ERR_TIMEOUT when it gives up
}

}  // namespace

int launch_wait_selftest(int *status, unsigned long long limit_ns, void *stream)
{
    k_wait_selftest<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, limit_ns);
    return static_cast<int>(cudaGetLastError());
}

const void *kernel_for(int fam, int mode, int variant, int C)
{
    const int ci = (C == 1) ? 0 : (C == 3 ? 1 : (C == 4 ? 2 : -1));
    if (ci < 0)
        return nullptr;
    using Fn = void (*)(const KArgs, const CUtensorMap);
    static const Fn u8[2][3] = {
        {k_resize<0, uint8_t, 1, 0, 0>, k_resize<0, uint8_t, 3, 0, 0>, k_resize<0, uint8_t, 4, 0, 0>},
        {k_resize<0, uint8_t, 1, 1, 0>, k_resize<0, uint8_t, 3, 1, 0>, k_resize<0, uint8_t, 4, 1, 0>}};
    static const Fn u8_down2[3] = {k_resize<0, uint8_t, 1, 1, VAR_DOWN2>, k_resize<0, uint8_t, 3, 1, VAR_DOWN2>,
                                   k_resize<0, uint8_t, 4, 1, VAR_DOWN2>};
    static const Fn f32[2][3] = {
        {k_resize<0, float, 1, 0, 0>, k_resize<0, float, 3, 0, 0>, k_resize<0, float, 4, 0, 0>},
        {k_resize<0, float, 1, 1, 0>, k_resize<0, float, 3, 1, 0>, k_resize<0, float, 4, 1, 0>}};
    static const Fn norm[3] = {k_resize<1, uint8_t, 1, 1, 0>, k_resize<1, uint8_t, 3, 1, 0>,
                               k_resize<1, uint8_t, 4, 1, 0>};
    const int m = mode == RZ_LINEAR ? 1 : 0;
    switch (fam) {
    case FAM_U8:
        if (variant == VAR_DOWN2)
            return m ? reinterpret_cast<const void *>(u8_down2[ci]) : nullptr;
        return reinterpret_cast<const void *>(u8[m][ci]);
    case FAM_F32: return reinterpret_cast<const void *>(f32[m][ci]);
    case FAM_NORM: return m ? reinterpret_cast<const void *>(norm[ci]) : nullptr;
    default: return nullptr;
    }
}

int launch_resize(const void *fn, const KArgs &a, const CUtensorMap &tmap, int grid, size_t smem, bool pdl,
                  void *stream, int threads, int grid_y)
{
    if (grid <= 0 || grid_y <= 0)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), static_cast<unsigned>(grid_y), 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    if (pdl) {
        // overlap this launch's start with the previous kernel's tail; the
        // kernel waits (griddepcontrol.wait) before touching global memory
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return static_cast<int>(cudaLaunchKernelEx(
        &cfg, reinterpret_cast<void (*)(const KArgs, const CUtensorMap)>(const_cast<void *>(fn)), a, tmap));
}

}  // namespace rz
