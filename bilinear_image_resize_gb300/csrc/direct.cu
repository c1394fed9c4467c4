// Direct-load kernels for sm_103a: every thread loads its own source bytes
// and writes its own outputs (the exact 2x uint8 downscale; any ratio with a
// uint8 source, plain or through the normalise epilogue).
//
// For one frame per launch the path is bound by how fast HBM requests get in
// flight after the launch, not by bandwidth: a thread per output group, each
// with two 16- or 24-byte vector loads in flight at once (half a million
// threads for a 4K frame), reaches HBM sooner than a producer warp per CTA
// issuing bulk copies, and there is no stage to plan, no shared memory and
// no barrier.  Each thread forms one group of output pixels (8, 4 or 2
// pixels for 1, 3 or 4 channels) from the two source rows below it with the
// same exact arithmetic as the staged kernel (down2_group: (t0 + t1 + b0 + b1
// + 2) >> 2, CUDA interpolation page §2.2 and §6.2 at A = B = 1024), and
// writes it with one vector store.  Loads and stores bypass L1 and are
// evicted first from L2 (each byte is used once).
//
// Launched as a programmatic dependent launch: the grid may start while the
// previous kernel in the stream finishes, and waits (griddepcontrol.wait)
// before touching memory.
#include <cuda_runtime.h>

#include <cstdint>

#include "rz_device.h"
#include "rz_internal.h"

namespace rz {
namespace {

using namespace dev;

// True for the CTAs that prefetch their source span before the dependency
// wait: the first a.l2_prefetch CTAs in launch order (the host sets it to the
// CTAs resident at once, 0 for none).  Only those can be resident while the
// previous kernel still runs; a CTA of a later wave starts after it has
// finished, when a prefetch just ahead of the CTA's own loads only adds work.
__device__ __forceinline__ bool first_wave_cta(const KArgs &a)
{
    return static_cast<long long>(blockIdx.y) * gridDim.x + blockIdx.x < a.l2_prefetch;
}

// Grid: x covers one image's output groups (kDirectThreads per CTA), y the
// images of a batch, one image per grid row (the host splits batches past
// 65535 images into several launches).  Requirements, checked by the host: W = 2 OW, H = 2 OH; source
// base, pitch and batch stride multiples of the load width (16 bytes for 1
// and 4 channels, 8 for 3); output base, pitch and batch stride multiples of
// the store width (8, 4).  LINEAR = 0 is the exact 2x nearest: every other
// pixel of every other row (only the upper row is read).  First-wave CTAs
// prefetch the source rows they read into L2 before waiting for the previous
// grid (first_wave_cta).
template <int C, int LINEAR>
__global__ void __launch_bounds__(kDirectThreads) k_down2_direct(const KArgs a, const __grid_constant__ CUtensorMap)
{
    constexpr int PX = down2_px(C);       // output pixels per group: 8, 4, 2
    constexpr int SB = 2 * PX * C;        // source bytes per row and group: 16, 24, 16
    grid_launch_dependents();
    bounds_begin(a);
    const int full = a.OW / PX;                // whole groups per row
    const int gpr = full + (a.OW % PX ? 1 : 0);
    if (first_wave_cta(a))
        prefetch_items<LINEAR ? 2 : 1>(a.src + (long long)blockIdx.y * a.src_bstride, a.src_pitch,
                                       (long long)a.W * C, gpr, a.OH, static_cast<int>(blockIdx.x) * kDirectThreads,
                                       kDirectThreads, SB, 0, 0, [](int u, int k) { return 2 * u + k; });
    grid_dependency_wait();
    const int idx = blockIdx.x * kDirectThreads + threadIdx.x;
    if (idx >= a.OH * gpr)
        return;
    const int dy = idx / gpr, j = idx - dy * gpr;
    const uint8_t *top = a.src + (long long)blockIdx.y * a.src_bstride + (long long)(2 * dy) * a.src_pitch;
    uint8_t *out = a.dst + (long long)blockIdx.y * a.dst_bstride + (long long)dy * a.dst_pitch;
    if (j < full)
        down2_one<C, LINEAR>(top, top + a.src_pitch, out, j);
    else
        down2_row_tail<C, LINEAR>(top, top + a.src_pitch, out, full * PX, a.OW);
}

// Any ratio, uint8: bilinear (exact 11-bit fixed point, the tiled kernel's
// arithmetic: hsum_u8 per row, then (B0 hT + B1 hB + 2^21) >> 22) or
// nearest.  A thread takes four consecutive output pixels of one row: their
// four table entries in two 16-byte loads, their taps from the two source
// rows through L1 (neighbouring threads share them), 32-bit words where the
// row layout allows and the taps lie at least 12 bytes before the row's end
// (so no load passes the row), bytes otherwise; the four pixels leave as
// 32-bit words when the output layout allows.  WRAP: the plan's border rule
// is wrap, whose edge entries hold the last sample as the near tap, and the
// far tap past the last sample is sample 0 (far_tap); the clamp and mirror
// rules are in the tables alone.  First-wave CTAs prefetch the source spans
// of their items into L2 before the dependency wait (first_wave_cta).
template <int C, int LINEAR, bool WRAP>
__global__ void __launch_bounds__(kDirectThreads) k_direct(const KArgs a, const __grid_constant__ CUtensorMap)
{
    constexpr int RUN = 4;
    grid_launch_dependents();
    bounds_begin(a);
    const int gpr = (a.OW + RUN - 1) / RUN;
    if (first_wave_cta(a)) {
        // the CTA's source spans into L2 before the dependency wait: one
        // piece per (output row, tap row) of its items, the columns from the
        // plan's tables (written when the plan was made, never by a kernel, so
        // they may be read before the wait)
        const int g0 = blockIdx.x * kDirectThreads, g1 = min(g0 + kDirectThreads, a.OH * gpr);
        const int d0 = g0 / gpr, nr = (g1 - 1) / gpr - d0 + 1;
        const int piece = threadIdx.x;
        if (g0 < g1 && piece < 2 * nr && (LINEAR || (piece & 1) == 0)) {
            const int dy = d0 + (piece >> 1);
            const int jlo = max(g0 - dy * gpr, 0), jhi = min(g1 - dy * gpr, gpr);
            const int y0 = ld_nc(a.yt + dy).x;
            const int r = (piece & 1) ? far_tap<WRAP>(y0, a.H) : y0;
            const int xlo = ld_nc(a.xt + jlo * RUN).x, xhi = ld_nc(a.xt + min(jhi * RUN, a.OW) - 1).x;
            const long long b0 = static_cast<long long>(xlo) * C;
            const long long b1 = min(static_cast<long long>(xhi + 2) * C, static_cast<long long>(a.W) * C);
            if (b1 > b0)
                l2_prefetch_span(a.src + (long long)blockIdx.y * a.src_bstride + (long long)r * a.src_pitch + b0,
                                 b1 - b0);
        }
    }
    grid_dependency_wait();
    const int idx = blockIdx.x * kDirectThreads + threadIdx.x;
    if (idx >= a.OH * gpr)
        return;
    const int dy = idx / gpr, x0 = (idx - dy * gpr) * RUN;
    const int npx = min(RUN, a.OW - x0);
    const int row_bytes = a.W * C;
    // the tables are 16-byte aligned with spare entries past their end, and
    // x0 is a multiple of 4
    const int4 xa = ld_nc(reinterpret_cast<const int4 *>(a.xt + x0));
    const int4 xb = ld_nc(reinterpret_cast<const int4 *>(a.xt + x0 + 2));
    const int xs[RUN] = {xa.x, xa.z, xb.x, xb.z};   // left tap (nearest: the tap)
    const int xw[RUN] = {xa.y, xa.w, xb.y, xb.w};   // right tap's 11-bit weight
    const int2 ye = ld_nc(a.yt + dy);
    const int r0 = ye.x, r1 = LINEAR ? far_tap<WRAP>(ye.x, a.H) : ye.x;
    const int B1 = ye.y, B0 = 2048 - B1;
    const bool words_in = ((reinterpret_cast<uintptr_t>(a.src) | static_cast<uintptr_t>(a.src_pitch) |
                            static_cast<uintptr_t>(a.src_bstride)) & 3) == 0;
    for (int b = blockIdx.y; b < a.batch; b += gridDim.y) {
        const uint8_t *img = a.src + (long long)b * a.src_bstride;
        const uint8_t *top = img + (long long)r0 * a.src_pitch;
        const uint8_t *bot = img + (long long)r1 * a.src_pitch;
        int q[RUN][C];
#pragma unroll
        for (int k = 0; k < RUN; k++) {
            const int o0 = xs[k] * C;
            if (k >= npx) {
#pragma unroll
                for (int c = 0; c < C; c++)
                    q[k][c] = 0;
            } else if (!LINEAR) {
#pragma unroll
                for (int c = 0; c < C; c++)
                    q[k][c] = ld_nc(top + o0 + c);
            } else {
                int hT[C], hB[C];
                // o0 + 12 <= row bytes puts the far tap inside (xs <= W - 2)
                if (words_in && o0 + 12 <= row_bytes) {
                    const uint32_t aw = static_cast<uint32_t>(2048 - xw[k]) | (static_cast<uint32_t>(xw[k]) << 16);
                    hsum_u8<C>(top, o0, aw, hT);
                    hsum_u8<C>(bot, o0, aw, hB);
                } else {
                    const int o1 = far_tap<WRAP>(xs[k], a.W) * C;
#pragma unroll
                    for (int c = 0; c < C; c++) {
                        hT[c] = (2048 - xw[k]) * ld_nc(top + o0 + c) + xw[k] * ld_nc(top + o1 + c);
                        hB[c] = (2048 - xw[k]) * ld_nc(bot + o0 + c) + xw[k] * ld_nc(bot + o1 + c);
                    }
                }
#pragma unroll
                for (int c = 0; c < C; c++)
                    q[k][c] = (B0 * hT[c] + B1 * hB[c] + (1 << 21)) >> 22;
            }
        }
        uint8_t *op = a.dst + (long long)b * a.dst_bstride + (long long)dy * a.dst_pitch + (long long)x0 * C;
        const bool words = npx == RUN && ((reinterpret_cast<uintptr_t>(op)) & 3) == 0;
        if (words) {
            uint32_t *o = reinterpret_cast<uint32_t *>(op);
            if constexpr (C == 1) {
                st_cs(o, pack4(q[0][0], q[1][0], q[2][0], q[3][0]));
            } else if constexpr (C == 3) {
                st_cs(o, pack4(q[0][0], q[0][1], q[0][2], q[1][0]));
                st_cs(o + 1, pack4(q[1][1], q[1][2], q[2][0], q[2][1]));
                st_cs(o + 2, pack4(q[2][2], q[3][0], q[3][1], q[3][2]));
            } else {
#pragma unroll
                for (int k = 0; k < RUN; k++)
                    st_cs(o + k, pack4(q[k][0], q[k][1], q[k][2], q[k][3]));
            }
        } else {
#pragma unroll
            for (int k = 0; k < RUN; k++)
                if (k < npx)
#pragma unroll
                    for (int c = 0; c < C; c++)
                        st_g(op + k * C + c, static_cast<uint8_t>(q[k][c]));
        }
    }
}

// Exact 3:2 bilinear downscale of uint8 (W = 3 OW / 2, H = 3 OH / 2).  Output
// column 2m samples x = 3m + 1/4 (taps 3m, 3m + 1 with weights 3/4, 1/4) and
// 2m + 1 samples 3m + 7/4 (taps 3m + 1, 3m + 2 with 1/4, 3/4), the same for
// rows, so the 11-bit weights are 1536 and 512 and the exact sum (B0 (A0 t0 +
// A1 t1) + B1 (...) + 2^21) >> 22 equals (sum of b a t + 8) >> 4 with a, b in
// {1, 3} (CUDA interpolation page §2.2, §6.2); no tap leaves the image.  A
// thread forms eight output pixels of one row from the two source rows it
// samples over twelve source columns, 12 C bytes per row in 3 C aligned
// words (down32_group: the vertical 3-1 sums lane-wise in 16-bit lanes, then
// for three and four channels regrouped into pixel lane words so that the
// horizontal sums take two channels per multiply-add).  The row's last
// pixels (fewer than eight) take a byte path.  (Written as a loop over the images
// of a batch: without it this kernel compiles to a slower schedule, 4.8
// against 2.9 us for 1080p -> 720p.)  Requirements, checked by the host:
// source base, pitch and batch stride multiples of 4; output ones of 4.
template <int C>
__global__ void __launch_bounds__(kDirectThreads) k_down32_direct(const KArgs a, const __grid_constant__ CUtensorMap)
{
    constexpr int PX = 8;          // output pixels per thread
    constexpr int NW = 3 * C;      // source words per row: 12 pixels
    grid_launch_dependents();
    bounds_begin(a);
    const int full = a.OW / PX;
    const int gpr = full + (a.OW % PX ? 1 : 0);
    if (first_wave_cta(a))
        prefetch_items<2>(a.src + (long long)blockIdx.y * a.src_bstride, a.src_pitch, (long long)a.W * C, gpr, a.OH,
                          static_cast<int>(blockIdx.x) * kDirectThreads, kDirectThreads, 4 * NW, 0, 0,
                          [](int u, int k) { return 3 * (u >> 1) + (k ? 1 : 2 * (u & 1)); });
    grid_dependency_wait();
    const int idx = blockIdx.x * kDirectThreads + threadIdx.x;
    if (idx >= a.OH * gpr)
        return;
    const int oy = idx / gpr, j = idx - oy * gpr;
    // output row 2m + r: the source row weighted 3 is 3m (r = 0) or 3m + 2
    // (r = 1), the one weighted 1 is 3m + 1
    const int m = oy >> 1, r = oy & 1;
    const int ya = 3 * m + 2 * r, yb = 3 * m + 1;
    for (int b = blockIdx.y; b < a.batch; b += gridDim.y) {
        const uint8_t *img = a.src + (long long)b * a.src_bstride;
        const uint8_t *ra = img + (long long)ya * a.src_pitch;
        const uint8_t *rb = img + (long long)yb * a.src_pitch;
        uint8_t *o = a.dst + (long long)b * a.dst_bstride + (long long)oy * a.dst_pitch;
        if (j < full) {
            down32_group<C>(ra, rb, o, j);
        } else {
            // the row's last pixels, fewer than eight: byte by byte
            for (int ox = full * PX; ox < a.OW; ox++) {
                const int i = ox >> 1, s3 = (ox & 1) ? 3 * i + 2 : 3 * i, s1 = 3 * i + 1;
                for (int c = 0; c < C; c++) {
#ifdef RZ_CHECK_BOUNDS
                    const int v = 9 * ld_g(ra + s3 * C + c) + 3 * ld_g(ra + s1 * C + c) + 3 * ld_g(rb + s3 * C + c) +
                                  ld_g(rb + s1 * C + c);
                    st_g(o + ox * C + c, static_cast<uint8_t>((v + 8) >> 4));
#else
                    // (plain accesses here: the wrapper form changes this
                    // kernel's register allocation and slows its main path)
                    const int v = 9 * ra[s3 * C + c] + 3 * ra[s1 * C + c] + 3 * rb[s3 * C + c] + rb[s1 * C + c];
                    o[ox * C + c] = static_cast<uint8_t>((v + 8) >> 4);
#endif
                }
            }
        }
    }
}

// Exact 2x bilinear upscale of uint8 (OW = 2 W, OH = 2 H).  Output column
// X = 2s samples x = s - 1/4 (taps s - 1, s with weights 1/4, 3/4) and
// X = 2s + 1 samples x = s + 1/4 (taps s, s + 1 with 3/4, 1/4); the same for
// rows.  The 11-bit weights are then 512 and 1536, so the exact sum
// (B0 (A0 t0 + A1 t1) + B1 (...) + 2^21) >> 22 equals (V + 8) >> 4 with
// V = sum of b a t over a, b in {1, 3} (CUDA interpolation page §2.2, §6.2).
// A tap outside the source (source column or row -1 or n) reads the sample
// the plan's border rule BORDER names (§6.1: clamp, mirror or wrap;
// border_index); the rule is a template parameter, so the clamp form has no
// test of it.
//
// A thread takes P = 4 source columns s0 .. s0 + 3 of source row r and forms
// output rows 2r and 2r + 1, columns 2 s0 .. 2 s0 + 7, from source rows
// r - 1, r, r + 1 over columns s0 - 1 .. s0 + 4 (clamped).  The bytes of each
// row sit in NW words (32-bit loads for interior groups on a 4-byte-aligned
// layout, assembled from clamped byte loads otherwise), byte e of the group
// at bit 8 (e % 4) of word e / 4.  The arithmetic runs on two bytes at a time
// in 16-bit lanes: word w splits into lo[w] (bytes 4w, 4w + 2) and hi[w]
// (bytes 4w + 1, 4w + 3).  The vertical sums (1 3 and 3 1) are lane-wise and
// scaled by 16, with 32 added, so that the horizontal sum 3 x + x' of two of
// them is 16 V + 128 and its high byte is the result; a byte's horizontal
// neighbour C bytes away lies, for a whole lane pair, in one register of the
// other or the same parity, or across two adjacent ones (one byte permute).
// Every lane stays below 2^16 (at most 16 * 16 * 255 + 128).
template <int C>
struct Up2Layout {
    static constexpr int P = 4;                    // source columns per thread
    static constexpr int NB = (P + 2) * C;         // group bytes: columns s0 - 1 .. s0 + P
    static constexpr int LEAD = (4 - C % 4) % 4;   // bytes before the group in its first word
    static constexpr int NW = (LEAD + NB + 3) / 4;
    static constexpr int NWO = 2 * P * C / 4;      // output words per row: 2, 6, 8
};

// The lane pair {byte e0 + d, byte e0 + 2 + d} of the split words, where the
// pair register (parity a, word w) holds bytes e0 = 4w + a and e0 + 2.
template <int NW>
__device__ __forceinline__ uint32_t lane_pair(const uint32_t (&lo)[NW], const uint32_t (&hi)[NW], int e)
{
    const int ec = max(e, 0);
    const int w = min(ec >> 2, NW - 1), w1 = min(w + 1, NW - 1);
    const uint32_t *src = (ec & 1) ? hi : lo;
    if (((ec >> 1) & 1) == 0)
        return src[w];
    return __byte_perm(src[w], src[w1], 0x5432);   // upper lane of word w, lower lane of w + 1
}

// CTAs per SM that the register budget is set for: six, the most at which
// the one-channel form (the only one launched: three and four channels take
// k_up2_rows) compiles without spills under every border rule.  The kernel is
// issue- and latency-bound, so more resident warps shorten it.
template <int C, int BORDER>
struct Up2Occupancy {
    static constexpr int value = 6;
};

template <int C, int BORDER>
__global__ void __launch_bounds__(kDirectThreads, Up2Occupancy<C, BORDER>::value) k_up2_direct(const KArgs a, const __grid_constant__ CUtensorMap)
{
    using Lay = Up2Layout<C>;
    constexpr int P = Lay::P, NB = Lay::NB, LEAD = Lay::LEAD, NW = Lay::NW, NWO = Lay::NWO;
    grid_launch_dependents();
    bounds_begin(a);
    const int gpr = (a.W + P - 1) / P;
    if (first_wave_cta(a)) {
        // source rows r - 1, r, r + 1 (edge rows of the mirror and wrap rules
        // are left to the loads); the group's words from column s0 - 1
        const int H = a.H;
        prefetch_items<3>(a.src + (long long)blockIdx.y * a.src_bstride, a.src_pitch, (long long)a.W * C, gpr, a.H,
                          static_cast<int>(blockIdx.x) * kDirectThreads, kDirectThreads, P * C, -C - LEAD, 4 * NW - P * C,
                          [H](int u, int k) { return min(max(u - 1 + k, 0), H - 1); });
    }
    grid_dependency_wait();
    const int idx = blockIdx.x * kDirectThreads + threadIdx.x;
    if (idx >= a.H * gpr)
        return;
    const int r = idx / gpr, s0 = (idx - r * gpr) * P;
    const int np = min(P, a.W - s0);
    // (the clamp form spelled as max / min / clampi: this kernel's register
    // allocation, and its speed, follow the exact form of these expressions)
    const int rows[3] = {BORDER == RZ_BORDER_CLAMP ? max(r - 1, 0) : border_index(r - 1, a.H, BORDER), r,
                         BORDER == RZ_BORDER_CLAMP ? min(r + 1, a.H - 1) : border_index(r + 1, a.H, BORDER)};
    const bool words_in = ((reinterpret_cast<uintptr_t>(a.src) | static_cast<uintptr_t>(a.src_pitch) |
                            static_cast<uintptr_t>(a.src_bstride)) & 3) == 0;
    // interior: the words read, [(s0 - 1) C - LEAD, + 4 NW), lie inside the row
    const bool inner = words_in && s0 >= 1 && (s0 - 1) * C - LEAD + 4 * NW <= a.W * C;
    for (int b = blockIdx.y; b < a.batch; b += gridDim.y) {
        const uint8_t *img = a.src + (long long)b * a.src_bstride;
        uint32_t lo[3][NW], hi[3][NW];
#pragma unroll
        for (int k = 0; k < 3; k++) {
            const uint8_t *row = img + (long long)rows[k] * a.src_pitch;
            uint32_t wd[NW];
            if (inner) {
                const uint32_t *w = reinterpret_cast<const uint32_t *>(row + (s0 - 1) * C - LEAD);
#pragma unroll
                for (int i = 0; i < NW; i++)
                    wd[i] = ld_nc(w + i);
            } else {
#pragma unroll
                for (int i = 0; i < NW; i++)
                    wd[i] = 0;
#pragma unroll
                for (int i = 0; i < NB; i++) {
                    const int col = BORDER == RZ_BORDER_CLAMP ? clampi(s0 - 1 + i / C, 0, a.W - 1)
                                                              : border_index(s0 - 1 + i / C, a.W, BORDER);
                    wd[(LEAD + i) / 4] |= static_cast<uint32_t>(ld_nc(row + col * C + i % C)) << (8 * ((LEAD + i) % 4));
                }
            }
#pragma unroll
            for (int i = 0; i < NW; i++) {
                lo[k][i] = wd[i] & 0x00ff00ffu;
                hi[k][i] = __byte_perm(wd[i], 0, 0x4341);   // bytes 1, 3 into the lanes' low bytes
            }
        }
#pragma unroll
        for (int j = 0; j < 2; j++) {
            // vertical sums of output row 2r + j, scaled by 16 and carrying a
            // quarter of the rounding term: 16 (t + 3 m) + 32 with t the
            // source row r - 1 (j = 0) or r + 1 (j = 1), m row r
            uint32_t vl[NW], vh[NW];
#pragma unroll
            for (int i = 0; i < NW; i++) {
                vl[i] = 16 * lo[2 * j][i] + (48 * lo[1][i] + 0x00200020u);
                vh[i] = 16 * hi[2 * j][i] + (48 * hi[1][i] + 0x00200020u);
            }
            // horizontal: for every pair register, the even output (left
            // neighbour 1, itself 3) and the odd output (itself 3, right 1)
            // (only registers holding a byte the outputs use: group bytes
            // LEAD + C .. LEAD + C + P C - 1)
            uint32_t ev[2][NW], od[2][NW];
#pragma unroll
            for (int par = 0; par < 2; par++)
#pragma unroll
                for (int i = 0; i < NW; i++) {
                    const int e0 = 4 * i + par;
                    const bool used = (e0 >= LEAD + C && e0 < LEAD + C + P * C) ||
                                      (e0 + 2 >= LEAD + C && e0 + 2 < LEAD + C + P * C);
                    if (!used) {
                        ev[par][i] = od[par][i] = 0;
                        continue;
                    }
                    // each lane is 16 V + 128 with V the 9-3-3-1 sum, below
                    // 2^16, so its high byte is (V + 8) >> 4: bytes 1 and 3
                    // hold the two results (the only bytes the output
                    // permutes take)
                    const uint32_t m3 = 3 * (par ? vh[i] : vl[i]);
                    const uint32_t l = lane_pair<NW>(vl, vh, e0 - C), rr = lane_pair<NW>(vl, vh, e0 + C);
                    ev[par][i] = l + m3;
                    od[par][i] = m3 + rr;
                }
            // output byte ob: output column oc = ob / C, channel ob % C, from
            // group byte e = LEAD + (oc / 2 + 1) C + ob % C, even or odd
            // output: byte 1 or 3 of its register, picked by byte permutes
            uint32_t ow[NWO];
#pragma unroll
            for (int wo = 0; wo < NWO; wo++) {
                uint32_t reg[4];
                int id[4];
                uint32_t pos[4];
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const int ob = 4 * wo + k, oc = ob / C;
                    const int e = LEAD + (oc / 2 + 1) * C + ob % C;
                    reg[k] = (oc & 1) ? od[e & 1][e >> 2] : ev[e & 1][e >> 2];
                    id[k] = ((oc & 1) * 2 + (e & 1)) * NW + (e >> 2);
                    pos[k] = ((e >> 1) & 1) ? 3u : 1u;
                }
                ow[wo] = gather_bytes(reg, id, pos);
            }
            uint8_t *op = a.dst + (long long)b * a.dst_bstride + (long long)(2 * r + j) * a.dst_pitch +
                          (long long)(2 * s0) * C;
            const uintptr_t oa = reinterpret_cast<uintptr_t>(op);
            if (np == P && NWO % 4 == 0 && (oa & 15) == 0) {
#pragma unroll
                for (int i = 0; i < NWO; i += 4)
                    st_cs(reinterpret_cast<uint4 *>(op) + i / 4, make_uint4(ow[i], ow[i + 1], ow[i + 2], ow[i + 3]));
            } else if (np == P && NWO % 2 == 0 && (oa & 7) == 0) {
#pragma unroll
                for (int i = 0; i < NWO; i += 2)
                    st_cs(reinterpret_cast<uint2 *>(op) + i / 2, make_uint2(ow[i], ow[i + 1]));
            } else if (np == P && (oa & 3) == 0) {
                uint32_t *o = reinterpret_cast<uint32_t *>(op);
#pragma unroll
                for (int i = 0; i < NWO; i++)
                    st_cs(o + i, ow[i]);
            } else {
#pragma unroll
                for (int i = 0; i < 2 * P * C; i++)
                    if (i < 2 * np * C)
                        st_g(op + i, static_cast<uint8_t>(ow[i / 4] >> (8 * (i % 4))));
            }
        }
    }
}

// ------------------------------------------------------------------ exact 2x upscale, pixel lanes, walking rows
//
// (the lane-word helpers up2_row_lanes / up2_emit_row are in rz_device.h,
// shared with the many-geometry launch)
//
// Grid: x covers one image's (row block, column group) items, column groups
// fastest; y the images, one per grid row (the host splits batches past
// 65535).  a.tiles_y = row blocks: block rb takes source rows
// [rb H / nrb, (rb + 1) H / nrb), so the host can size the grid to one wave
// of resident CTAs with rows shared out evenly.  Any layout, any border
// rule.  First-wave CTAs prefetch their source rows into L2 before the
// dependency wait.
template <int C, int BORDER>
__global__ void __launch_bounds__(kDirectThreads) k_up2_rows(const KArgs a, const __grid_constant__ CUtensorMap)
{
    using L = Up2RowsLayout<C>;
    constexpr int P = L::P;
    grid_launch_dependents();
    bounds_begin(a);
    const int gpc = (a.W + P - 1) / P;          // column groups per row block
    const int nrb = a.tiles_y;
    // first row of block rb: rb H / nrb (the host keeps nrb H < 2^32)
    auto block_row = [&](int rb) {
        return static_cast<int>(static_cast<unsigned>(rb) * static_cast<unsigned>(a.H) / static_cast<unsigned>(nrb));
    };
    const uint8_t *img = a.src + (long long)blockIdx.y * a.src_bstride;
    const int g0 = blockIdx.x * kDirectThreads;   // the CTA's first item (gpc * nrb < 2^31)
    if (first_wave_cta(a)) {
        // rows r0 - 1 .. r1 of each row block the CTA touches (at most two:
        // a CTA's 256 items span one boundary when gpc >= 256), over its column
        // span: one piece per row, taken by the threads that issue them
        const int rb0 = g0 / gpc;
        const int per = (a.H + nrb - 1) / nrb + 2;   // rows of the tallest block, with its two neighbours
        const int piece = threadIdx.x;
        if (piece < 2 * per) {
            const int g1 = min(g0 + kDirectThreads, gpc * nrb);
            const int rb = rb0 + (piece >= per ? 1 : 0);
            if (g0 < g1 && rb <= (g1 - 1) / gpc) {
                const int row = min(max(block_row(rb) - 1 + (piece >= per ? piece - per : piece), 0), a.H - 1);
                const int jlo = max(g0 - rb * gpc, 0), jhi = min(g1 - rb * gpc, gpc);
                const long long b0 = max((long long)jlo * P * C - C - L::LEAD, 0LL);
                const long long b1 = min((long long)jhi * P * C + C, (long long)a.W * C);
                if (b1 > b0)
                    l2_prefetch_span(img + (long long)row * a.src_pitch + b0, b1 - b0);
            }
        }
    }
    grid_dependency_wait();
    const int idx = g0 + threadIdx.x;
    if (idx >= gpc * nrb)
        return;
    const int rb = idx / gpc, j = idx - rb * gpc;
    const int s0 = j * P, np = min(P, a.W - s0);
    const int r0 = block_row(rb), r1 = block_row(rb + 1);
    const bool words_in = ((reinterpret_cast<uintptr_t>(a.src) | static_cast<uintptr_t>(a.src_pitch) |
                            static_cast<uintptr_t>(a.src_bstride)) & 3) == 0;
    const bool inner = words_in && s0 >= 1 && (s0 - 1) * C - L::LEAD + 4 * L::NW <= a.W * C;
    auto row_ptr = [&](int r) {
        const int rr = BORDER == RZ_BORDER_CLAMP ? clampi(r, 0, a.H - 1) : border_index(r, a.H, BORDER);
        return img + (long long)rr * a.src_pitch;
    };
    // output rows 2r and 2r + 1 of the current step; the source row below
    // (r + 1) advances by the pitch, mapped by the border rule past the end
    uint8_t *out = a.dst + (long long)blockIdx.y * a.dst_bstride + (long long)(2 * s0) * C +
                   (long long)(2 * r0) * a.dst_pitch;
    const uint8_t *below = img + (long long)(r0 + 1) * a.src_pitch;
    // rows k = 0, 1, 2 of the window rotate through the three buffers
    uint32_t lo[3][6], hi[3][6];
    up2_row_lanes<C, BORDER>(row_ptr(r0 - 1), s0, a.W, inner, lo[0], hi[0]);
    up2_row_lanes<C, BORDER>(row_ptr(r0), s0, a.W, inner, lo[1], hi[1]);
    auto step = [&](const int ia, const int im, const int ib, int r) {
        up2_row_lanes<C, BORDER>(r + 1 < a.H ? below : row_ptr(r + 1), s0, a.W, inner, lo[ib], hi[ib]);
        below += a.src_pitch;
        uint32_t mlo[6], mhi[6];
#pragma unroll
        for (int k = 0; k < 6; k++) {
            mlo[k] = 48 * lo[im][k] + 0x00200020u;
            mhi[k] = 48 * hi[im][k] + 0x00200020u;
        }
        up2_emit_row<C>(lo[ia], hi[ia], mlo, mhi, out, np);
        up2_emit_row<C>(lo[ib], hi[ib], mlo, mhi, out + a.dst_pitch, np);
        out += 2 * a.dst_pitch;
    };
    for (int r = r0; r < r1; r += 3) {
        step(0, 1, 2, r);
        if (r + 1 >= r1) break;
        step(1, 2, 0, r + 1);
        if (r + 2 >= r1) break;
        step(2, 0, 1, r + 2);
    }
}

// Bilinear + normalise, uint8 source, float32 planes out (y = q * scale[c] +
// shift[c] on the exact uint8 result q, CUDA interpolation page §4.2).  A
// warp takes 32 kNormRun consecutive output pixels of one row, lane l the
// pixels l, l + 32, ...: one load instruction then reads the taps of 32
// neighbouring pixels (a short stretch of the source row, few sectors even
// for strong downscales), and each plane store writes 32 consecutive floats.
// Taps, border rules and load rules as in k_direct.
template <int C, bool WRAP>
__global__ void __launch_bounds__(kDirectThreads) k_direct_norm(const KArgs a, const __grid_constant__ CUtensorMap)
{
    constexpr int RUN = kNormRun;
    grid_launch_dependents();
    bounds_begin(a);
    grid_dependency_wait();
    const int wpr = (a.OW + 32 * RUN - 1) / (32 * RUN);   // warps per output row
    const int gw = (blockIdx.x * kDirectThreads + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (gw >= a.OH * wpr)
        return;
    const int dy = gw / wpr, xb = (gw - dy * wpr) * 32 * RUN;
    const int row_bytes = a.W * C;
    int xs[RUN], xw[RUN];
    bool ok[RUN];
#pragma unroll
    for (int k = 0; k < RUN; k++) {
        const int x = xb + lane + 32 * k;
        ok[k] = x < a.OW;
        const int2 e = ld_nc(a.xt + min(x, a.OW - 1));
        xs[k] = e.x;
        xw[k] = e.y;
    }
    const int2 ye = ld_nc(a.yt + dy);
    const int r0 = ye.x, r1 = far_tap<WRAP>(ye.x, a.H);
    const int B1 = ye.y, B0 = 2048 - B1;
    const bool words_in = ((reinterpret_cast<uintptr_t>(a.src) | static_cast<uintptr_t>(a.src_pitch) |
                            static_cast<uintptr_t>(a.src_bstride)) & 3) == 0;
    for (int b = blockIdx.y; b < a.batch; b += gridDim.y) {
        const uint8_t *img = a.src + (long long)b * a.src_bstride;
        const uint8_t *top = img + (long long)r0 * a.src_pitch;
        const uint8_t *bot = img + (long long)r1 * a.src_pitch;
        int q[RUN][C];
#pragma unroll
        for (int k = 0; k < RUN; k++) {
            const int o0 = xs[k] * C;
            int hT[C], hB[C];
            if (words_in && o0 + 12 <= row_bytes) {
                const uint32_t aw = static_cast<uint32_t>(2048 - xw[k]) | (static_cast<uint32_t>(xw[k]) << 16);
                hsum_u8<C>(top, o0, aw, hT);
                hsum_u8<C>(bot, o0, aw, hB);
            } else {
                const int o1 = far_tap<WRAP>(xs[k], a.W) * C;
#pragma unroll
                for (int c = 0; c < C; c++) {
                    hT[c] = (2048 - xw[k]) * ld_nc(top + o0 + c) + xw[k] * ld_nc(top + o1 + c);
                    hB[c] = (2048 - xw[k]) * ld_nc(bot + o0 + c) + xw[k] * ld_nc(bot + o1 + c);
                }
            }
#pragma unroll
            for (int c = 0; c < C; c++)
                q[k][c] = (B0 * hT[c] + B1 * hB[c] + (1 << 21)) >> 22;
        }
#pragma unroll
        for (int c = 0; c < C; c++) {
            float *pl = reinterpret_cast<float *>(a.dst + (long long)b * a.dst_bstride + (long long)c * a.dst_plane +
                                                  (long long)dy * a.dst_pitch) + xb + lane;
#pragma unroll
            for (int k = 0; k < RUN; k++)
                if (ok[k])
                    st_cs(pl + 32 * k, fmaf(static_cast<float>(q[k][c]), a.scale[c], a.shift[c]));
        }
    }
}

// uint8 bilinear, rows walked per thread: a thread takes four consecutive
// output columns of TR consecutive output rows (a.TR) and keeps the exact
// horizontal sums of the two newest source rows it has sampled in registers
// (two buffers, a new row written over the older one).  Output rows sample
// non-decreasing source rows, so each source row's sums are formed once per
// thread however many output rows use it: an upscale by s forms about 1/s
// rows per output row instead of two.  Same arithmetic and load rules as
// k_direct.
template <int C>
__global__ void __launch_bounds__(kDirectThreads) k_direct_rows(const KArgs a, const __grid_constant__ CUtensorMap)
{
    constexpr int RUN = 4;
    grid_launch_dependents();
    bounds_begin(a);
    grid_dependency_wait();
    const int gpr = (a.OW + RUN - 1) / RUN;
    const int segs = (a.OH + a.TR - 1) / a.TR;
    const int idx = blockIdx.x * kDirectThreads + threadIdx.x;
    if (idx >= segs * gpr)
        return;
    const int sg = idx / gpr, x0 = (idx - sg * gpr) * RUN;
    const int dy0 = sg * a.TR, dy1 = min(dy0 + a.TR, a.OH);
    const int npx = min(RUN, a.OW - x0);
    const int row_bytes = a.W * C;
    const int4 xa = ld_nc(reinterpret_cast<const int4 *>(a.xt + x0));
    const int4 xb = ld_nc(reinterpret_cast<const int4 *>(a.xt + x0 + 2));
    const int xs[RUN] = {xa.x, xa.z, xb.x, xb.z};
    const int xw[RUN] = {xa.y, xa.w, xb.y, xb.w};
    uint32_t aw[RUN];
    int o1[RUN];       // right tap's byte offset (clamped at the row end)
    bool wok[RUN];     // word loads stay inside the row
    const bool words_in = ((reinterpret_cast<uintptr_t>(a.src) | static_cast<uintptr_t>(a.src_pitch) |
                            static_cast<uintptr_t>(a.src_bstride)) & 3) == 0;
#pragma unroll
    for (int k = 0; k < RUN; k++) {
        aw[k] = static_cast<uint32_t>(2048 - xw[k]) | (static_cast<uint32_t>(xw[k]) << 16);
        o1[k] = min(xs[k] + 1, a.W - 1) * C;
        wok[k] = words_in && xs[k] * C + 12 <= row_bytes;
    }
    // sums of one source row at this thread's four columns
    auto hrow = [&](const uint8_t *row, int (&h)[RUN][C]) {
#pragma unroll
        for (int k = 0; k < RUN; k++) {
            if (wok[k]) {
                hsum_u8<C>(row, xs[k] * C, aw[k], h[k]);
            } else {
#pragma unroll
                for (int c = 0; c < C; c++)
                    h[k][c] = (2048 - xw[k]) * ld_nc(row + xs[k] * C + c) + xw[k] * ld_nc(row + o1[k] + c);
            }
        }
    };
    for (int b = blockIdx.y; b < a.batch; b += gridDim.y) {
        const uint8_t *img = a.src + (long long)b * a.src_bstride;
        uint8_t *op = a.dst + (long long)b * a.dst_bstride + (long long)dy0 * a.dst_pitch + (long long)x0 * C;
        const bool words = npx == RUN && ((reinterpret_cast<uintptr_t>(op) | static_cast<uintptr_t>(a.dst_pitch)) &
                                          3) == 0;
        int h0[RUN][C], h1[RUN][C];   // the two newest sampled rows' sums
        bool newer1 = false;          // h1 holds the newer row
        int last = -1;                // the newest sampled row
        for (int dy = dy0; dy < dy1; dy++) {
            const int2 ye = ld_nc(a.yt + dy);
            const int r0 = ye.x, r1 = min(ye.x + 1, a.H - 1);
            if (r1 > last) {
                if (r0 > last) {
                    // both taps new: the upper into h0, the lower into h1
                    hrow(img + (long long)r0 * a.src_pitch, h0);
                    hrow(img + (long long)r1 * a.src_pitch, h1);
                    newer1 = true;
                } else if (newer1) {
                    hrow(img + (long long)r1 * a.src_pitch, h0);
                    newer1 = false;
                } else {
                    hrow(img + (long long)r1 * a.src_pitch, h1);
                    newer1 = true;
                }
                last = r1;
            }
            // the taps are (last - 1, last), or last twice at the bottom edge
            const int B1 = r0 == r1 ? 2048 : ye.y;
            const int w0 = newer1 ? 2048 - B1 : B1, w1 = newer1 ? B1 : 2048 - B1;
            int q[RUN][C];
#pragma unroll
            for (int k = 0; k < RUN; k++)
#pragma unroll
                for (int c = 0; c < C; c++)
                    q[k][c] = (w0 * h0[k][c] + w1 * h1[k][c] + (1 << 21)) >> 22;
            if (words) {
                uint32_t *o = reinterpret_cast<uint32_t *>(op);
                if constexpr (C == 1) {
                    st_cs(o, pack4(q[0][0], q[1][0], q[2][0], q[3][0]));
                } else if constexpr (C == 3) {
                    st_cs(o, pack4(q[0][0], q[0][1], q[0][2], q[1][0]));
                    st_cs(o + 1, pack4(q[1][1], q[1][2], q[2][0], q[2][1]));
                    st_cs(o + 2, pack4(q[2][2], q[3][0], q[3][1], q[3][2]));
                } else {
#pragma unroll
                    for (int k = 0; k < RUN; k++)
                        st_cs(o + k, pack4(q[k][0], q[k][1], q[k][2], q[k][3]));
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
        }
    }
}

// Bytes o0 .. o0 + 7 of a row as one 64-bit value (byte o0 lowest), from the
// three aligned 32-bit words that hold them.  The row base is 4-byte aligned
// and o0 + 12 <= the row's bytes, so every word read lies inside the row.
__device__ __forceinline__ uint64_t load_8_bytes(const uint8_t *row, int o0)
{
    const uint32_t *w = reinterpret_cast<const uint32_t *>(row + (o0 & ~3));
    const uint32_t w0 = ld_nc(w), w1 = ld_nc(w + 1), w2 = ld_nc(w + 2);
    const uint32_t sh = 8u * static_cast<uint32_t>(o0 & 3);
    return static_cast<uint64_t>(__funnelshift_r(w1, w2, sh)) << 32 | __funnelshift_r(w0, w1, sh);
}

// BT.601 luma of one pixel, rounded half-up exactly: floor((299 R + 587 G +
// 114 B + 500) / 1000) (the sum is below 2^18).
__device__ __forceinline__ int gray_of(uint32_t r, uint32_t g, uint32_t b)
{
    return static_cast<int>((299u * r + 587u * g + 114u * b + 500u) / 1000u);
}

// The same for a pixel whose channels are bytes 0..2 of px (byte 3 ignored),
// in two byte dot products: the weights split into high and low bytes (299 =
// 256 + 43, 587 = 2 * 256 + 75, 114 = 114), so the sum is 256 dp4a(px, hi) +
// dp4a(px, lo) + 500; floor(s / 1000) is the high word of s * 4294968,
// exact for s < 6.1e6 (4294968 * 1000 - 2^32 = 704).  Weight words for R, G,
// B in bytes 0, 1, 2; for B, G, R the byte order of each word reverses.
constexpr uint32_t kGrayLoRGB = 43u | 75u << 8 | 114u << 16, kGrayHiRGB = 1u | 2u << 8;
constexpr uint32_t kGrayLoBGR = 114u | 75u << 8 | 43u << 16, kGrayHiBGR = 2u << 8 | 1u << 16;
__device__ __forceinline__ int gray_dp4a(uint32_t px, uint32_t lo, uint32_t hi)
{
    const uint32_t s = __dp4a(px, hi, 0u) * 256u + __dp4a(px, lo, 500u);
    return static_cast<int>(__umulhi(s, 4294968u));
}

// Gray of pixel p (0 or 1) of a pair of C-channel pixels packed in v (byte
// 8 p C onwards), with the weight words of the channel order.
template <int C>
__device__ __forceinline__ int gray_in(uint64_t v, int p, uint32_t lo, uint32_t hi)
{
    return gray_dp4a(static_cast<uint32_t>(v >> (8 * p * C)), lo, hi);
}

template <int C>
__device__ __forceinline__ int gray_at(const uint8_t *row, int x, int ir, int ib)
{
    const uint8_t *px = row + x * C;
    return gray_of(ld_nc(px + ir), ld_nc(px + 1), ld_nc(px + ib));
}

// Grayscale conversion fused before the uint8 resize (OpenCV object-tracking
// page §3.1.1: cvtColor to gray, then resize).  Each tap pixel's gray value
// (BT.601, rounded half-up) is formed from its C = 3 or 4 channels (R, G, B
// or B, G, R; a fourth is ignored), then the exact bilinear sum of k_direct
// (or the nearest tap) is taken over the gray values, so the result equals
// resizing the converted image.  A thread takes four consecutive output
// pixels; a tap pair's 2 C bytes come from three aligned words where the
// row allows (as in k_direct), from bytes otherwise; the four gray outputs
// leave as one 32-bit word when aligned.
template <int C, int LINEAR, bool WRAP>
__global__ void __launch_bounds__(kDirectThreads) k_direct_gray(const KArgs a, const __grid_constant__ CUtensorMap)
{
    constexpr int RUN = 4;
    grid_launch_dependents();
    bounds_begin(a);
    grid_dependency_wait();
    const int gpr = (a.OW + RUN - 1) / RUN;
    const int idx = blockIdx.x * kDirectThreads + threadIdx.x;
    if (idx >= a.OH * gpr)
        return;
    const int dy = idx / gpr, x0 = (idx - dy * gpr) * RUN;
    const int npx = min(RUN, a.OW - x0);
    const int row_bytes = a.W * C;
    const int ir = a.bgr ? 2 : 0, ib = a.bgr ? 0 : 2;
    const uint32_t wlo = a.bgr ? kGrayLoBGR : kGrayLoRGB, whi = a.bgr ? kGrayHiBGR : kGrayHiRGB;
    const int4 xa = ld_nc(reinterpret_cast<const int4 *>(a.xt + x0));
    const int4 xb = ld_nc(reinterpret_cast<const int4 *>(a.xt + x0 + 2));
    const int xs[RUN] = {xa.x, xa.z, xb.x, xb.z};
    const int xw[RUN] = {xa.y, xa.w, xb.y, xb.w};
    const int2 ye = ld_nc(a.yt + dy);
    const int r0 = ye.x, r1 = LINEAR ? far_tap<WRAP>(ye.x, a.H) : ye.x;
    const int B1 = ye.y, B0 = 2048 - B1;
    const bool words_in = ((reinterpret_cast<uintptr_t>(a.src) | static_cast<uintptr_t>(a.src_pitch) |
                            static_cast<uintptr_t>(a.src_bstride)) & 3) == 0;
    for (int b = blockIdx.y; b < a.batch; b += gridDim.y) {
        const uint8_t *img = a.src + (long long)b * a.src_bstride;
        const uint8_t *top = img + (long long)r0 * a.src_pitch;
        const uint8_t *bot = img + (long long)r1 * a.src_pitch;
        int q[RUN];
#pragma unroll
        for (int k = 0; k < RUN; k++) {
            if (k >= npx) {
                q[k] = 0;
            } else if (!LINEAR) {
                q[k] = gray_at<C>(top, xs[k], ir, ib);
            } else {
                const int o0 = xs[k] * C;
                int t0, t1, b0, b1;
                if (words_in && o0 + 12 <= row_bytes) {   // far tap inside: xs <= W - 2
                    const uint64_t vt = load_8_bytes(top, o0), vb = load_8_bytes(bot, o0);
                    t0 = gray_in<C>(vt, 0, wlo, whi);
                    t1 = gray_in<C>(vt, 1, wlo, whi);
                    b0 = gray_in<C>(vb, 0, wlo, whi);
                    b1 = gray_in<C>(vb, 1, wlo, whi);
                } else {
                    const int x1 = far_tap<WRAP>(xs[k], a.W);
                    t0 = gray_at<C>(top, xs[k], ir, ib);
                    t1 = gray_at<C>(top, x1, ir, ib);
                    b0 = gray_at<C>(bot, xs[k], ir, ib);
                    b1 = gray_at<C>(bot, x1, ir, ib);
                }
                const int A1 = xw[k], A0 = 2048 - A1;
                q[k] = (B0 * (A0 * t0 + A1 * t1) + B1 * (A0 * b0 + A1 * b1) + (1 << 21)) >> 22;
            }
        }
        uint8_t *op = a.dst + (long long)b * a.dst_bstride + (long long)dy * a.dst_pitch + x0;
        if (npx == RUN && (reinterpret_cast<uintptr_t>(op) & 3) == 0) {
            st_cs(reinterpret_cast<uint32_t *>(op), pack4(q[0], q[1], q[2], q[3]));
        } else {
#pragma unroll
            for (int k = 0; k < RUN; k++)
                if (k < npx)
                    st_g(op + k, static_cast<uint8_t>(q[k]));
        }
    }
}

// Gray of pixel p of a run of NW words of C-channel pixels (byte e of the
// run at bits 8 (e % 4) of word e / 4); p, C and the order compile-time.  A
// three-channel pixel is gathered into one word by a byte permute.
template <int C, bool BGR, int NW>
__device__ __forceinline__ int gray_word_px(const uint32_t (&w)[NW], int p)
{
    const int e = p * C, i = e >> 2, o = e & 3;
    uint32_t px;
    if (C == 4 || o == 0)
        px = w[i];
    else
        px = __byte_perm(w[i], w[min(i + 1, NW - 1)], static_cast<uint32_t>(o | (o + 1) << 4 | (o + 2) << 8));
    return BGR ? gray_dp4a(px, kGrayLoBGR, kGrayHiBGR) : gray_dp4a(px, kGrayLoRGB, kGrayHiRGB);
}

// The row's last pixels of the exact 2x gray kernel (fewer than a group),
// byte by byte; out of line, like down2_row_tail.
template <int C, int LINEAR, bool BGR>
__device__ __noinline__ void gray_down2_row_tail(const uint8_t *top, const uint8_t *bot, uint8_t *out, int p0, int OW)
{
    constexpr int IR = BGR ? 2 : 0, IB = BGR ? 0 : 2;
    for (int p = p0; p < OW; p++) {
        int g = gray_at<C>(top, 2 * p, IR, IB);
        if (LINEAR)
            g = (g + gray_at<C>(top, 2 * p + 1, IR, IB) + gray_at<C>(bot, 2 * p, IR, IB) +
                 gray_at<C>(bot, 2 * p + 1, IR, IB) + 2) >> 2;
        st_g(out + p, static_cast<uint8_t>(g));
    }
}

// Grayscale conversion fused before an exact 2x downscale (W = 2 OW,
// H = 2 OH): bilinear (rounded mean of the 2 x 2 gray values, the exact sum
// at weights 1024) or nearest (the upper-left gray value).  A thread takes
// four output pixels: eight source pixels of each of its two rows in one
// 24- or 32-byte run (three 8-byte or two 16-byte streaming loads), and
// stores the four gray bytes as one word.  One image per grid row (the host
// splits batches past 65535 images).  Requirements, checked by the host:
// source base, pitch and batch stride multiples of 8 bytes (C = 3) or 16
// (C = 4); output ones multiples of 4.
template <int C, int LINEAR, bool BGR>
__global__ void __launch_bounds__(kDirectThreads) k_down2_gray(const KArgs a, const __grid_constant__ CUtensorMap)
{
    constexpr int PX = 4, SB = 2 * PX * C, NW = SB / 4;
    grid_launch_dependents();
    bounds_begin(a);
    const int full = a.OW / PX;
    const int gpr = full + (a.OW % PX ? 1 : 0);
    if (first_wave_cta(a))
        prefetch_items<LINEAR ? 2 : 1>(a.src + (long long)blockIdx.y * a.src_bstride, a.src_pitch,
                                       (long long)a.W * C, gpr, a.OH, static_cast<int>(blockIdx.x) * kDirectThreads,
                                       kDirectThreads, SB, 0, 0, [](int u, int k) { return 2 * u + k; });
    grid_dependency_wait();
    const int idx = blockIdx.x * kDirectThreads + threadIdx.x;
    if (idx >= a.OH * gpr)
        return;
    const int dy = idx / gpr, j = idx - dy * gpr;
    const uint8_t *top = a.src + (long long)blockIdx.y * a.src_bstride + (long long)(2 * dy) * a.src_pitch;
    const uint8_t *bot = top + a.src_pitch;
    uint8_t *out = a.dst + (long long)blockIdx.y * a.dst_bstride + (long long)dy * a.dst_pitch;
    if (j >= full) {
        gray_down2_row_tail<C, LINEAR, BGR>(top, bot, out, full * PX, a.OW);
        return;
    }
    uint32_t tw[NW], bw[NW];
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
        const uint4 *tp = reinterpret_cast<const uint4 *>(top + SB * j);
        const uint4 *bp = reinterpret_cast<const uint4 *>(bot + SB * j);
#pragma unroll
        for (int k = 0; k < 2; k++) {
            const uint4 t = ld_cs(tp + k);
            tw[4 * k] = t.x; tw[4 * k + 1] = t.y; tw[4 * k + 2] = t.z; tw[4 * k + 3] = t.w;
            if (LINEAR) {
                const uint4 u = ld_cs(bp + k);
                bw[4 * k] = u.x; bw[4 * k + 1] = u.y; bw[4 * k + 2] = u.z; bw[4 * k + 3] = u.w;
            }
        }
    }
    int q[PX];
#pragma unroll
    for (int k = 0; k < PX; k++) {
        q[k] = gray_word_px<C, BGR, NW>(tw, 2 * k);
        if (LINEAR)
            q[k] = (q[k] + gray_word_px<C, BGR, NW>(tw, 2 * k + 1) + gray_word_px<C, BGR, NW>(bw, 2 * k) +
                    gray_word_px<C, BGR, NW>(bw, 2 * k + 1) + 2) >> 2;
    }
    st_cs(reinterpret_cast<uint32_t *>(out + PX * j), pack4(q[0], q[1], q[2], q[3]));
}

// float32 bilinear, a thread per output pixel (all C channels): the lerp form
// h = t0 + u (t1 - t0) on both rows, then the same across rows with v, with
// the tables' float weights (CUDA interpolation page §2.2).  Used for plans
// whose border rule is wrap (WRAP: the far tap past the last sample is
// sample 0); clamp and mirror are in the tables alone.
template <int C, bool WRAP>
__global__ void __launch_bounds__(kDirectThreads) k_direct_f32(const KArgs a, const __grid_constant__ CUtensorMap)
{
    grid_launch_dependents();
    bounds_begin(a);
    grid_dependency_wait();
    const long long idx = static_cast<long long>(blockIdx.x) * kDirectThreads + threadIdx.x;
    if (idx >= static_cast<long long>(a.OH) * a.OW)
        return;
    const int dy = static_cast<int>(idx / a.OW), dx = static_cast<int>(idx - static_cast<long long>(dy) * a.OW);
    const int2 xe = ld_nc(a.xt + dx), ye = ld_nc(a.yt + dy);
    const float u = __int_as_float(xe.y), v = __int_as_float(ye.y);
    const int c0 = xe.x * C, c1 = far_tap<WRAP>(xe.x, a.W) * C;
    const int y1 = far_tap<WRAP>(ye.x, a.H);
    for (int b = blockIdx.y; b < a.batch; b += gridDim.y) {
        const uint8_t *img = a.src + (long long)b * a.src_bstride;
        const float *top = reinterpret_cast<const float *>(img + (long long)ye.x * a.src_pitch);
        const float *bot = reinterpret_cast<const float *>(img + (long long)y1 * a.src_pitch);
        float *op = reinterpret_cast<float *>(a.dst + (long long)b * a.dst_bstride + (long long)dy * a.dst_pitch) +
                    static_cast<long long>(dx) * C;
#pragma unroll
        for (int c = 0; c < C; c++) {
            const float t0 = ld_nc(top + c0 + c), t1 = ld_nc(top + c1 + c);
            const float b0 = ld_nc(bot + c0 + c), b1 = ld_nc(bot + c1 + c);
            const float h0 = fmaf(u, t1 - t0, t0), h1 = fmaf(u, b1 - b0, b0);
            st_cs(op + c, fmaf(v, h1 - h0, h0));
        }
    }
}

}  // namespace

const void *direct_gray_kernel_for(int mode, int C, bool wrap)
{
    using Fn = void (*)(const KArgs, const CUtensorMap);
    static const Fn k[2][2][2] = {{{k_direct_gray<3, 0, false>, k_direct_gray<4, 0, false>},
                                   {k_direct_gray<3, 0, false>, k_direct_gray<4, 0, false>}},
                                  {{k_direct_gray<3, 1, false>, k_direct_gray<4, 1, false>},
                                   {k_direct_gray<3, 1, true>, k_direct_gray<4, 1, true>}}};
    if (C != 3 && C != 4)
        return nullptr;
    const int m = mode == RZ_LINEAR ? 1 : 0;
    return reinterpret_cast<const void *>(k[m][wrap ? 1 : 0][C == 4 ? 1 : 0]);
}

const void *direct_down2_gray_kernel_for(int mode, int C, bool bgr)
{
    using Fn = void (*)(const KArgs, const CUtensorMap);
    static const Fn k[2][2][2] = {{{k_down2_gray<3, 0, false>, k_down2_gray<3, 0, true>},
                                   {k_down2_gray<4, 0, false>, k_down2_gray<4, 0, true>}},
                                  {{k_down2_gray<3, 1, false>, k_down2_gray<3, 1, true>},
                                   {k_down2_gray<4, 1, false>, k_down2_gray<4, 1, true>}}};
    if (C != 3 && C != 4)
        return nullptr;
    return reinterpret_cast<const void *>(k[mode == RZ_LINEAR ? 1 : 0][C == 4 ? 1 : 0][bgr ? 1 : 0]);
}

const void *direct_f32_kernel_for(int C, bool wrap)
{
    using Fn = void (*)(const KArgs, const CUtensorMap);
    static const Fn k[2][3] = {{k_direct_f32<1, false>, k_direct_f32<3, false>, k_direct_f32<4, false>},
                               {k_direct_f32<1, true>, k_direct_f32<3, true>, k_direct_f32<4, true>}};
    const int ci = (C == 1) ? 0 : (C == 3 ? 1 : (C == 4 ? 2 : -1));
    return ci < 0 ? nullptr : reinterpret_cast<const void *>(k[wrap ? 1 : 0][ci]);
}

const void *direct_up2_kernel_for(int C, int border)
{
    using Fn = void (*)(const KArgs, const CUtensorMap);
    // one channel only: three and four channels take k_up2_rows
    static const Fn k[3] = {k_up2_direct<1, RZ_BORDER_CLAMP>, k_up2_direct<1, RZ_BORDER_MIRROR>,
                            k_up2_direct<1, RZ_BORDER_WRAP>};
    if (C != 1 || border < 0 || border > 2)
        return nullptr;
    return reinterpret_cast<const void *>(k[border]);
}

const void *direct_up2_rows_kernel_for(int C, int border)
{
    using Fn = void (*)(const KArgs, const CUtensorMap);
    static const Fn k[3][2] = {{k_up2_rows<3, RZ_BORDER_CLAMP>, k_up2_rows<4, RZ_BORDER_CLAMP>},
                               {k_up2_rows<3, RZ_BORDER_MIRROR>, k_up2_rows<4, RZ_BORDER_MIRROR>},
                               {k_up2_rows<3, RZ_BORDER_WRAP>, k_up2_rows<4, RZ_BORDER_WRAP>}};
    const int ci = C == 3 ? 0 : (C == 4 ? 1 : -1);
    if (ci < 0 || border < 0 || border > 2)
        return nullptr;
    return reinterpret_cast<const void *>(k[border][ci]);
}

const void *direct_down32_kernel_for(int C)
{
    using Fn = void (*)(const KArgs, const CUtensorMap);
    static const Fn k[3] = {k_down32_direct<1>, k_down32_direct<3>, k_down32_direct<4>};
    const int ci = (C == 1) ? 0 : (C == 3 ? 1 : (C == 4 ? 2 : -1));
    return ci < 0 ? nullptr : reinterpret_cast<const void *>(k[ci]);
}

const void *direct_rows_kernel_for(int C)
{
    using Fn = void (*)(const KArgs, const CUtensorMap);
    static const Fn k[3] = {k_direct_rows<1>, k_direct_rows<3>, k_direct_rows<4>};
    const int ci = (C == 1) ? 0 : (C == 3 ? 1 : (C == 4 ? 2 : -1));
    return ci < 0 ? nullptr : reinterpret_cast<const void *>(k[ci]);
}

// Any ratio: op DIRECT_U8 (bilinear or nearest) or DIRECT_NORM (bilinear).
// Nearest taps are always inside, so the wrap form exists for bilinear only.
const void *direct_kernel_for(int op, int mode, int C, bool wrap)
{
    using Fn = void (*)(const KArgs, const CUtensorMap);
    static const Fn u8[3][3] = {{k_direct<1, 0, false>, k_direct<3, 0, false>, k_direct<4, 0, false>},
                                {k_direct<1, 1, false>, k_direct<3, 1, false>, k_direct<4, 1, false>},
                                {k_direct<1, 1, true>, k_direct<3, 1, true>, k_direct<4, 1, true>}};
    static const Fn norm[2][3] = {{k_direct_norm<1, false>, k_direct_norm<3, false>, k_direct_norm<4, false>},
                                  {k_direct_norm<1, true>, k_direct_norm<3, true>, k_direct_norm<4, true>}};
    const int ci = (C == 1) ? 0 : (C == 3 ? 1 : (C == 4 ? 2 : -1));
    if (ci < 0)
        return nullptr;
    const int m = mode == RZ_LINEAR ? 1 : 0;
    if (op == DIRECT_NORM)
        return m ? reinterpret_cast<const void *>(norm[wrap ? 1 : 0][ci]) : nullptr;
    return reinterpret_cast<const void *>(u8[m ? (wrap ? 2 : 1) : 0][ci]);
}

const void *direct_down2_kernel_for(int mode, int C)
{
    using Fn = void (*)(const KArgs, const CUtensorMap);
    static const Fn k[2][3] = {{k_down2_direct<1, 0>, k_down2_direct<3, 0>, k_down2_direct<4, 0>},
                               {k_down2_direct<1, 1>, k_down2_direct<3, 1>, k_down2_direct<4, 1>}};
    const int ci = (C == 1) ? 0 : (C == 3 ? 1 : (C == 4 ? 2 : -1));
    return ci < 0 ? nullptr : reinterpret_cast<const void *>(k[mode == RZ_LINEAR ? 1 : 0][ci]);
}

}  // namespace rz
