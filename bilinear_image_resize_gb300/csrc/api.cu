// C ABI of the resize library: plans (exact sampling tables), argument
// validation, tile selection and kernel launch.  See include/gbresize.h for
// the contract of every entry point.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "gbresize.h"
#include "rz_internal.h"

using rz::KArgs;
using rz::SmemLayout;

namespace {

thread_local int g_last_cuda_error = 0;

int cuda_fail(cudaError_t e)
{
    g_last_cuda_error = static_cast<int>(e);
    if (e == cudaErrorMemoryAllocation)
        return RZ_ERR_NOMEM;
    return RZ_ERR_CUDA;
}

int64_t floor_div(int64_t a, int64_t b)  // b > 0
{
    int64_t q = a / b;
    if ((a % b) != 0 && a < 0)
        q -= 1;
    return q;
}

// Bilinear sampling table of one axis.  Output index d samples
// x = (d + 1/2) n_in / n_out - 1/2 = num / den, num = (2d+1) n_in - n_out,
// den = 2 n_out (Volcanic resize page, "Naive resize with linear sampling").
// ofs = floor(x); the far tap's weight is u = r / den with r = num - ofs*den:
// as 11-bit fixed point round-half-up(2048 u) (CUDA interpolation page §6.2),
// as float rounded once from double.  The sampled position lies in
// [-1/2, n_in - 1/2], so only ofs = -1 or ofs = n_in - 1 has a tap outside,
// which the border rule maps (§6.1; the weights stay those of the unmapped
// position):
//  - clamp: both taps read the same edge sample, so the entry is folded to
//    one tap with weight 0 (value unchanged);
//  - mirror: the outside tap reads the inside neighbour of the edge sample,
//    so the taps stay adjacent and the entry becomes that adjacent pair with
//    the weights exchanged (ofs 0 or n_in - 2, weight 2048 - w, u = 1 - u);
//  - wrap: the outside tap reads the opposite edge sample, so the entry keeps
//    its weight with ofs = n_in - 1, and the kernels take sample 0 as the
//    far tap of ofs = n_in - 1.
// A one-sample axis reads its sample under every rule (folded as clamp).
void axis_linear(int n_in, int n_out, int border, int32_t *ofs, int32_t *q11, float *u)
{
    const int64_t den = 2 * static_cast<int64_t>(n_out);
    for (int64_t d = 0; d < n_out; d++) {
        const int64_t num = (2 * d + 1) * n_in - n_out;
        int64_t s = floor_div(num, den);
        const int64_t r = num - s * den;
        int64_t w = floor_div(4096 * r + den, 2 * den);
        float uf = static_cast<float>(static_cast<double>(r) / static_cast<double>(den));
        const bool outside = s < 0 || (s >= n_in - 1 && r != 0);
        const float uflip = static_cast<float>(static_cast<double>(den - r) / static_cast<double>(den));
        if (outside && border == RZ_BORDER_MIRROR && n_in > 1) {
            s = s < 0 ? 0 : n_in - 2;
            w = 2048 - w;
            uf = uflip;
        } else if (outside && border == RZ_BORDER_WRAP) {
            s = n_in - 1;
        } else if (s < 0) {
            s = 0;
            w = 0;
            uf = 0.0f;
        } else if (s >= n_in - 1) {
            s = n_in - 1;
            w = 0;
            uf = 0.0f;
        }
        if (ofs) ofs[d] = static_cast<int32_t>(s);
        if (q11) q11[d] = static_cast<int32_t>(w);
        if (u) u[d] = uf;
    }
}

// Nearest table: floor(d n_in / n_out), OpenCV INTER_NEAREST (CUDA
// interpolation page §2.1 read as the floor rule).
void axis_nearest(int n_in, int n_out, int32_t *ofs)
{
    for (int64_t d = 0; d < n_out; d++) {
        int64_t s = floor_div(d * n_in, n_out);
        if (s > n_in - 1) s = n_in - 1;
        ofs[d] = static_cast<int32_t>(s);
    }
}

struct TileCfg {
    int TR = 0, TW = 0, tiles_x = 0, tiles_y = 0, max_rows = 0, slot_bytes = 0, stages = 0, variant = 0;
    int tensor = 0, box_words = 0, box_rows = 0;   // tensor-map staging (one box per chunk)
    int stream = 0;   // 0: staged-tile kernel; 1: streaming filter; 2: streaming uint8 bilinear
    int ring_chunks = 0, chunk_rows = 0, chunk_boxes = 0, box_bytes = 0;   // streaming kernels
    size_t smem = 0;
    int grid = 0;
};

// cuTensorMapEncodeTiled, fetched from the driver through the runtime (the
// library links no driver library).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn tensor_encoder()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

}  // namespace

struct rz_plan_s {
    int H, W, OH, OW, mode, device;
    int border = RZ_BORDER_CLAMP;   // bilinear taps outside the source (RZ_BORDER_*)
    std::vector<int32_t> xofs, xq, yofs, yq;
    std::vector<float> xu, yu;
    void *dmem = nullptr;
    size_t dmem_bytes = 0;     // tables and status word, one cudaMalloc block
    int2 *d_xq = nullptr, *d_xf = nullptr, *d_yq = nullptr, *d_yf = nullptr;
    int *d_status = nullptr;
    std::mutex mu;
    struct Entry { int fam, C, batch, halo; TileCfg cfg; };
    std::vector<Entry> cache;
    int over_tr[rz::FAM_COUNT] = {}, over_tw[rz::FAM_COUNT] = {};
    int opt_stages = 0;        // 0: automatic
    int opt_generic = 0;       // 1: never use an exact-ratio specialisation
    int opt_ctas_per_sm = 0;   // 0: as many as fit
    int opt_grid_mode = 0;     // 0: persistent CTAs; 1: one CTA per tile
    int opt_pdl = 1;           // programmatic dependent launch
    int opt_ring_rows = 0;     // streaming kernels: source rows in the ring (0: automatic)
    int opt_u8_kernel = 0;     // uint8 bilinear: 0 automatic, 1 staged tiles, 2 streaming, 3 direct
    int opt_filter_kernel = 0; // filter epilogues: 0 automatic, 1 streaming, 2 tile kernel
    int opt_f32_kernel = 0;    // plain float32 bilinear: 0 automatic (streaming), 1 staged tiles
    int opt_l2_prefetch = 1;   // exact-ratio direct kernels: pre-wait L2 prefetch of the source
};

namespace {

bool valid_mode(int m) { return m == RZ_LINEAR || m == RZ_NEAREST; }
bool valid_border(int b) { return b == RZ_BORDER_CLAMP || b == RZ_BORDER_MIRROR || b == RZ_BORDER_WRAP; }

// Upper bound on the bytes of one staged source row of the tile column
// starting at output column dx0: the tap span rounded out to 16 bytes.
int span_bytes(const rz_plan_s &p, int fam, int C, int dx0, int dx1, int halo)
{
    const int es = rz::fam_in_es(fam);
    const int cx0 = std::clamp(dx0 - halo, 0, p.OW - 1);
    const int cx1 = std::clamp(dx1 - 1 + halo, 0, p.OW - 1);
    const int xs0 = p.xofs[cx0];
    const int xs1 = p.mode == RZ_LINEAR ? std::min(p.xofs[cx1] + 1, p.W - 1) : p.xofs[cx1];
    const int lo = (xs0 * C * es) & ~15;
    const int hi = ((xs1 + 1) * C * es + 15) & ~15;
    return hi - lo;
}

// Bytes reserved per staged row: the widest span, plus 16 bytes of padding
// for the uint8 bilinear kernels, whose 32-bit tap reads may run up to 11
// bytes past a span (onto taps of weight 0).  `pad` = false for the exact 2x
// path, which reads only inside each span.
int max_slot_bytes(const rz_plan_s &p, int fam, int C, int TW, bool pad = true, int halo = -1)
{
    if (halo < 0) halo = rz::fam_halo(fam);
    int m = 0;
    for (int dx0 = 0; dx0 < p.OW; dx0 += TW)
        m = std::max(m, span_bytes(p, fam, C, dx0, std::min(dx0 + TW, p.OW), halo));
    return m + (pad ? rz::fam_slot_pad(fam) : 0);
}

// Largest number of distinct source rows a tile of TR output rows stages,
// counted exactly as the kernel lists them.
int max_tile_rows(const rz_plan_s &p, int TR)
{
    const bool lin = p.mode == RZ_LINEAR;
    int m = 0;
    for (int dy0 = 0; dy0 < p.OH; dy0 += TR) {
        const int dy1 = std::min(dy0 + TR, p.OH);
        int n = 0, last = -1;
        for (int dy = dy0; dy < dy1; dy++) {
            const int r0 = p.yofs[dy];
            const int r1 = lin ? std::min(r0 + 1, p.H - 1) : r0;
            if (r0 > last) { n++; last = r0; }
            if (r1 > last) { n++; last = r1; }
        }
        m = std::max(m, n);
    }
    return m;
}

bool eval_tile(const rz_plan_s &p, int fam, int C, int TR, int TW, int stages, TileCfg *out, bool pad = true)
{
    TileCfg t;
    t.TR = std::max(1, std::min(TR, p.OH));
    t.TW = std::max(1, std::min(TW, p.OW));
    t.tiles_x = (p.OW + t.TW - 1) / t.TW;
    t.tiles_y = (p.OH + t.TR - 1) / t.TR;
    t.slot_bytes = max_slot_bytes(p, fam, C, t.TW, pad);
    t.max_rows = max_tile_rows(p, t.TR);
    t.stages = stages;
    const SmemLayout L = rz::smem_layout(fam, C, t.TR, t.TW, t.max_rows, t.slot_bytes, stages);
    t.smem = static_cast<size_t>(L.total);
    *out = t;
    return L.total <= rz::kMaxSmem;
}

constexpr int kSms = 152;                // GB300; the launch itself asks the device
constexpr int kSoftSmem = 48 * 1024;     // keeps several CTAs resident per SM
constexpr int kDefaultStages = 2;

// True when the plan is an exact 2x downscale on both axes: every column and
// row samples x = 2d + 1/2 (weight 1024 on taps 2d and 2d + 1).
bool is_down2(const rz_plan_s &p)
{
    if (p.mode != RZ_LINEAR || p.W != 2 * p.OW || p.H != 2 * p.OH) return false;
    for (int d = 0; d < p.OW; d++)
        if (p.xofs[d] != 2 * d || p.xq[d] != 1024) return false;
    for (int d = 0; d < p.OH; d++)
        if (p.yofs[d] != 2 * d || p.yq[d] != 1024) return false;
    return true;
}

// True when the plan is an exact 3:2 downscale on both axes: output 2m
// samples 3m + 1/4 (weight 512 on taps 3m, 3m + 1) and 2m + 1 samples
// 3m + 7/4 (weight 1536 on taps 3m + 1, 3m + 2).
bool is_down32(const rz_plan_s &p)
{
    if (p.mode != RZ_LINEAR || 2 * p.W != 3 * p.OW || 2 * p.H != 3 * p.OH) return false;
    auto axis_ok = [](const std::vector<int32_t> &ofs, const std::vector<int32_t> &q, int n) {
        for (int d = 0; d < n; d++) {
            const int m = d / 2;
            if (ofs[d] != (d & 1 ? 3 * m + 1 : 3 * m) || q[d] != (d & 1 ? 1536 : 512)) return false;
        }
        return true;
    };
    return axis_ok(p.xofs, p.xq, p.OW) && axis_ok(p.yofs, p.yq, p.OH);
}

// Automatic tile choice for persistent CTAs.  Plain resize and normalise:
// rows as wide as the output (or the widest power-of-two strip whose staged
// row stays within 16 KB), narrowed while there are fewer than about twelve
// tiles per SM (for balance across SMs), then as many output rows per tile as
// keep the staged ring under 48 KB with that many tiles.  (The filter family
// and uint8 upscales stream strips instead: get_stream_tile.)
TileCfg choose_tile(const rz_plan_s &p, int fam, int C, int batch, int stages, bool down2)
{
    const int out_es = rz::fam_out_es(fam);
    const int px_bytes = fam == rz::FAM_NORM ? 4 : C * out_es;
    TileCfg best;
    if (down2) {
        // the exact 2x path computes little per byte, so the kernel is bound
        // by the source stream: two output rows (four consecutive source
        // rows, one contiguous span) per tile and a ring of two tiles measured
        // best for 4K -> 1080p RGB (8.9 us against 10.4 us for one-row tiles)
        TileCfg t;
        if (max_slot_bytes(p, fam, C, p.OW, false) <= 24576 && eval_tile(p, fam, C, 2, p.OW, stages, &t, false) &&
            t.smem <= static_cast<size_t>(rz::kMaxSmem) / 2)
            return t;
    }
    std::vector<int> tws;
    tws.push_back(p.OW);
    for (int w = 4096; w >= 1; w >>= 1)
        if (w < p.OW) tws.push_back(w);
    auto ok_width = [&](int w) {
        if (w >= p.OW) return true;
        if ((w * px_bytes) % 16 != 0) return false;
        return !down2 || (w % 8) == 0;
    };
    const long long want_tiles = 6LL * kSms;
    int TW = 0;
    for (int w : tws) {
        if (!ok_width(w)) continue;
        const int row_out = px_bytes * std::min(w, p.OW);
        if (max_slot_bytes(p, fam, C, w) > 16384 || row_out > 16384) continue;
        if (TW == 0) TW = w;
        const long long tiles = static_cast<long long>(batch) * p.OH * ((p.OW + w - 1) / w);
        TW = w;
        if (tiles >= want_tiles || w <= 64) break;
    }
    if (TW == 0) {
        // no strip of 16 KB: fall back to the narrowest widths that fit
        for (int w = 32; w >= 1; w >>= 1)
            if (ok_width(w) || w == 1) { TW = w; break; }
    }
    TileCfg t1;
    int st = stages;
    while (!eval_tile(p, fam, C, 1, TW, st, &t1)) {
        if (st > 1) { st--; continue; }
        if (TW == 1) return t1;
        TW = std::max(1, TW / 2);
    }
    best = t1;
    for (int TR = 2; TR <= 64; TR *= 2) {
        TileCfg t;
        if (!eval_tile(p, fam, C, TR, TW, st, &t) || t.smem > static_cast<size_t>(kSoftSmem)) break;
        if (static_cast<long long>(batch) * t.tiles_x * t.tiles_y < want_tiles) break;
        best = t;
        if (TR >= p.OH) break;
    }
    return best;
}

std::mutex g_attr_mu;
std::vector<std::pair<int, const void *>> g_attr_done;  // (device, kernel) with the smem opt-in applied

int ensure_smem_attr(int dev, const void *fn)
{
    std::lock_guard<std::mutex> lk(g_attr_mu);
    for (const auto &e : g_attr_done)
        if (e.first == dev && e.second == fn) return 0;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, rz::kMaxSmem);
    if (e != cudaSuccess) return static_cast<int>(e);
    g_attr_done.push_back({dev, fn});
    return 0;
}

}  // namespace

namespace rz {
// the tensor-core correlation (filter_tc.cu)
bool filter_tc_supported(const float *src, long long src_pitch, int K);
int launch_filter_tc(const float *src, long long src_pitch, int H, int W, const float *w, int K, float *dst,
                     long long dst_pitch, int *status, bool pdl, void *stream);
}  // namespace rz

namespace {

// Filter widths from which the automatic choice takes the tensor cores for
// filter2d_valid_f32 (measured on 4096^2: K = 64, 2.53 against 2.95 ms for
// the FP32 kernel; K = 32, 1.00 against 0.72 ms).
constexpr int kFilterTcMinK = 48;

std::mutex g_occ_mu;
struct OccEntry { int dev; const void *fn; int block; int ctas; };
std::vector<OccEntry> g_occ;   // CTAs of a kernel resident at once on a device

// How many CTAs of `fn` (block threads, no dynamic shared memory) the device
// holds at once: the occupancy calculator's CTAs per SM times the SM count,
// computed once per (device, kernel, block size).
int resident_ctas(int dev, const void *fn, int block, int *out)
{
    std::lock_guard<std::mutex> lk(g_occ_mu);
    for (const auto &e : g_occ)
        if (e.dev == dev && e.fn == fn && e.block == block) {
            *out = e.ctas;
            return 0;
        }
    int per_sm = 0, sms = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, block, 0);
    if (e != cudaSuccess) return static_cast<int>(e);
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return static_cast<int>(e);
    *out = std::max(1, per_sm * sms);
    g_occ.push_back({dev, fn, block, *out});
    return 0;
}

constexpr int kStreamCtaSmem = 74 * 1024;   // three streaming CTAs per SM
constexpr int kStreamMinRows = 8;           // shortest automatic unit (the filter's halo adds 2 rows)

// Units, ring and grid of a streaming kernel (stream.cu).  Units are strips
// of up to the kernel's widest strip (filter_strip / stream_u8_strip),
// narrowed to share the columns evenly; the uint8 form needs each strip's
// source span plus 16 bytes of padding (its 32-bit tap reads) in one 2 KB
// block and narrows the strips until it fits.  The automatic unit height
// splits each strip into as many segments as give every resident CTA about
// one unit, so a source row is staged once per strip segment.  The ring holds
// chunks of eight rows (fewer when the option asks for a small ring), as many
// chunks as keep three CTAs per SM (two at least).  Returns
// RZ_ERR_UNSUPPORTED when the uint8 form does not fit (the caller then uses
// the staged-tile kernel).
int get_stream_tile(rz_plan_s *p, int op, int C, int batch, TileCfg *out, const void **fn_out, int halo)
{
    const void *fn = rz::stream_kernel_for(op, p->mode, C, halo);
    if (!fn) return RZ_ERR_UNSUPPORTED;
    const bool u8 = op == rz::STREAM_U8;
    const int fam = u8 ? rz::FAM_U8 : rz::FAM_FILT;
    const int widest = u8 ? rz::stream_u8_strip(C) : rz::filter_strip(C, halo);
    TileCfg t;
    int strips = (p->OW + widest - 1) / widest;
    int span = 0;
    for (;;) {
        t.TW = (p->OW + strips - 1) / strips;
        if (u8 && t.TW < p->OW) t.TW = std::min(p->OW, (t.TW + 31) / 32 * 32);   // word-aligned output runs
        if (p->over_tw[fam] > 0) t.TW = std::min({p->over_tw[fam], widest, p->OW});
        span = max_slot_bytes(*p, fam, C, t.TW, u8, halo);   // a multiple of 16 (+16 of padding for uint8)
        if (!u8 || span <= 2048) break;
        if (p->over_tw[fam] > 0 || t.TW <= 32) return RZ_ERR_UNSUPPORTED;
        strips++;
    }
    t.tiles_x = (p->OW + t.TW - 1) / t.TW;
    const int BW = std::min(span, 2048);   // a box row: at most 256 eight-byte words
    const int NB = (span + BW - 1) / BW;
    int G = rz::kStreamChunkRows, NCH;
    if (p->opt_ring_rows > 0) {
        while (G > 1 && 2 * G > p->opt_ring_rows) G /= 2;
        NCH = p->opt_ring_rows / G;
    } else {
        const int chunk = NB * rz::stream_block_bytes(G, BW);
        NCH = std::max(2, std::min(rz::kStreamRingMax / G, kStreamCtaSmem / (chunk + 16)));
    }
    while (rz::stream_smem(NCH, G, NB, BW) > rz::kMaxSmem) {
        if (NCH > 2) NCH--;
        else if (G > 1) G /= 2;
        else return RZ_ERR_UNSUPPORTED;
    }
    t.ring_chunks = NCH;
    t.chunk_rows = G;
    t.chunk_boxes = NB;
    t.box_bytes = BW;
    t.slot_bytes = span;
    t.tensor = 1;            // used when the source allows bulk copies
    t.box_words = BW / 8;
    t.box_rows = G;
    t.smem = static_cast<size_t>(rz::stream_smem(NCH, G, NB, BW));
    t.stages = 0;
    t.variant = rz::VAR_GENERIC;
    t.stream = u8 ? 2 : 1;
    int e = ensure_smem_attr(p->device, fn);
    if (e != 0) return cuda_fail(static_cast<cudaError_t>(e));
    int per_sm = 0, sms = 0;
    cudaError_t ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, rz::kThreads, t.smem);
    if (ce != cudaSuccess) return cuda_fail(ce);
    ce = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device);
    if (ce != cudaSuccess) return cuda_fail(ce);
    if (per_sm < 1) return RZ_ERR_ARG;
    if (p->opt_ctas_per_sm > 0) per_sm = std::min(per_sm, p->opt_ctas_per_sm);
    const long long cap = static_cast<long long>(per_sm) * sms;
    int TR;
    if (p->over_tr[fam] > 0) {
        TR = p->over_tr[fam];
    } else {
        const long long segs = std::max<long long>(1, cap / (static_cast<long long>(batch) * t.tiles_x));
        TR = static_cast<int>((p->OH + segs - 1) / segs);
        TR = std::max(TR, std::min(p->OH, kStreamMinRows));
    }
    t.TR = std::max(1, std::min(TR, p->OH));
    t.tiles_y = (p->OH + t.TR - 1) / t.TR;
    const long long units = static_cast<long long>(batch) * t.tiles_x * t.tiles_y;
    if (units > 0x7fffffffLL) return RZ_ERR_UNSUPPORTED;
    t.grid = p->opt_grid_mode == 1 ? static_cast<int>(units) : static_cast<int>(std::min(units, cap));
    p->cache.push_back({fam, C, batch, halo, t});
    *out = t;
    *fn_out = fn;
    return RZ_OK;
}

// The uint8 bilinear resize takes the streaming form for vertical upscales
// of at least kStreamMinPixels outputs, where each source row feeds several
// output rows (measured faster there than the direct kernels), or when the
// option asks for it; not for the exact 2x case.
constexpr long long kStreamMinPixels = 1 << 18;   // smaller outputs: the stream's set-up dominates

bool auto_u8_stream(const rz_plan_s &p)
{
    return p.OH > p.H && static_cast<long long>(p.OH) * p.OW >= kStreamMinPixels;
}

bool want_u8_stream(const rz_plan_s &p, bool down2)
{
    if (p.mode != RZ_LINEAR || down2) return false;
    return p.opt_u8_kernel == 2 || (p.opt_u8_kernel == 0 && auto_u8_stream(p));
}

// Tile and grid for this call: the override if one is set, else the cached
// automatic choice.  Returns an RZ_* status.
int get_tile(rz_plan_s *p, int fam, int C, int batch, TileCfg *out, const void **fn_out, int halo)
{
    std::lock_guard<std::mutex> lk(p->mu);
    for (const auto &e : p->cache)
        if (e.fam == fam && e.C == C && e.batch == batch && e.halo == halo) {
            *out = e.cfg;
            *fn_out = e.cfg.stream ? rz::stream_kernel_for(e.cfg.stream == 2 ? rz::STREAM_U8 : rz::STREAM_FILTER,
                                                           p->mode, C, halo)
                                   : rz::kernel_for(fam, p->mode, e.cfg.variant, C);
            return RZ_OK;
        }
    if (fam == rz::FAM_FILT) return get_stream_tile(p, rz::STREAM_FILTER, C, batch, out, fn_out, halo);
    const int stages = p->opt_stages > 0 ? p->opt_stages : kDefaultStages;
    const bool down2 = fam == rz::FAM_U8 && !p->opt_generic && is_down2(*p);
    if (fam == rz::FAM_U8 && want_u8_stream(*p, down2)) {
        const int rc = get_stream_tile(p, rz::STREAM_U8, C, batch, out, fn_out, 0);
        if (rc != RZ_ERR_UNSUPPORTED) return rc;   // else the staged-tile kernel below
    }
    TileCfg t;
    if (p->over_tr[fam] > 0 && p->over_tw[fam] > 0) {
        // an explicit ring depth must fit as asked; an automatic one shrinks
        int st = stages;
        while (!eval_tile(*p, fam, C, p->over_tr[fam], p->over_tw[fam], st, &t)) {
            if (p->opt_stages > 0 || st == 1) return RZ_ERR_ARG;
            st--;
        }
    } else {
        t = choose_tile(*p, fam, C, batch, stages, down2);
    }
    t.variant = rz::VAR_GENERIC;
    if (down2 && (t.tiles_x == 1 || t.TW % 8 == 0)) t.variant = rz::VAR_DOWN2;
    const void *fn = rz::kernel_for(fam, p->mode, t.variant, C);
    if (!fn) return RZ_ERR_UNSUPPORTED;
    int e = ensure_smem_attr(p->device, fn);
    if (e != 0) return cuda_fail(static_cast<cudaError_t>(e));
    int per_sm = 0, sms = 0;
    cudaError_t ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, rz::kThreads, t.smem);
    if (ce != cudaSuccess) return cuda_fail(ce);
    ce = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device);
    if (ce != cudaSuccess) return cuda_fail(ce);
    if (per_sm < 1) return RZ_ERR_ARG;
    if (p->opt_ctas_per_sm > 0) per_sm = std::min(per_sm, p->opt_ctas_per_sm);
    const long long ntiles = static_cast<long long>(batch) * t.tiles_x * t.tiles_y;
    if (ntiles > 0x7fffffffLL) return RZ_ERR_UNSUPPORTED;
    t.grid = p->opt_grid_mode == 1
                 ? static_cast<int>(ntiles)
                 : static_cast<int>(std::min<long long>(ntiles, static_cast<long long>(per_sm) * sms));
    p->cache.push_back({fam, C, batch, halo, t});
    *out = t;
    *fn_out = fn;
    return RZ_OK;
}

bool overlap(const void *a, size_t na, const void *b, size_t nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

size_t image_extent(int rows, size_t pitch, size_t row_bytes)
{
    return rows <= 0 ? 0 : static_cast<size_t>(rows - 1) * pitch + row_bytes;
}

int check_device(const rz_plan_s *p)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    return dev == p->device ? RZ_OK : RZ_ERR_ARG;
}

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; }

// Direct-load kernels (direct.cu) for uint8-source resizes, unless the
// option asks for staged tiles (1) or streaming (2), and except automatic
// bilinear vertical upscales other than exact 2x (streamed).  Exact 2x
// upscales with the 1-3 weights; exact 2x downscales (bilinear tables of the
// 2x pattern, or nearest at W = 2 OW, H = 2 OH) with vector loads where the
// layout allows; vertical bilinear upscales (option 3) with each thread
// walking rows; everything else one thread per four output pixels.  Returns
// true with *rc set when it handled the call.
bool run_direct(rz_plan_s *p, int fam, KArgs &a, int mode, void *stream, bool do_launch, int *rc)
{
    const int opt = p->opt_u8_kernel;
    const int C = a.C, batch = a.batch;
    const bool wrap = p->border == RZ_BORDER_WRAP && mode == RZ_LINEAR;
    // per_image: the kernel takes exactly one image per grid row, so a batch
    // past 65535 images is split into several launches
    auto launch_grid = [&](const void *fn, long long gx, int block, bool per_image = false) {
        *rc = RZ_OK;
        if (!do_launch) return true;
        CUtensorMap none;
        std::memset(&none, 0, sizeof(none));
        KArgs c = a;
        c.l2_prefetch = 0;
        if (a.l2_prefetch) {
            const int e = resident_ctas(p->device, fn, block, &c.l2_prefetch);
            if (e != 0) {
                *rc = cuda_fail(static_cast<cudaError_t>(e));
                return true;
            }
        }
        for (long long b0 = 0; b0 < batch; b0 += 65535) {
            const int nb = static_cast<int>(std::min<long long>(batch - b0, 65535));
            KArgs d = c;
            if (per_image) {
                d.src = c.src + b0 * c.src_bstride;
                d.dst = c.dst + b0 * c.dst_bstride;
                d.batch = nb;
            }
            const int e = rz::launch_resize(fn, d, none, static_cast<int>(gx), 0, p->opt_pdl != 0, stream, block, nb);
            if (e != 0) {
                *rc = cuda_fail(static_cast<cudaError_t>(e));
                return true;
            }
            if (!per_image) break;   // the kernel strides over every image itself
        }
        return true;
    };
    auto launch = [&](const void *fn, long long threads, bool per_image = false) {
        return launch_grid(fn, (threads + rz::kDirectThreads - 1) / rz::kDirectThreads, rz::kDirectThreads,
                           per_image);
    };
    if (fam == rz::FAM_FILT) {
        // K x K epilogue: the streaming kernel for K = 3, 5, 7 (source rows
        // streamed once, neighbours by shuffle); the tile kernel (filter.cu)
        // for K = 1, for wrap plans, or when the option asks
        const int fopt = p->opt_filter_kernel;
        if (a.ksize == 0) return false;   // the plain float32 resize (f32_family)
        if (a.ksize >= 3 && !wrap && fopt != 2) return false;
        if (fopt == 1) {
            *rc = RZ_ERR_UNSUPPORTED;
            return true;
        }
        const void *ffn = rz::resize_filter_kernel_for(C, a.ksize, wrap);
        if (!ffn) {
            *rc = RZ_ERR_UNSUPPORTED;
            return true;
        }
        a.xt = p->d_xf;
        a.yt = p->d_yf;
        const long long tiles = static_cast<long long>((a.OW + rz::kFTW - 1) / rz::kFTW) *
                                ((a.OH + rz::kFTH - 1) / rz::kFTH);
        return launch_grid(ffn, tiles, rz::kFilterThreads);
    }
    if (fam == rz::FAM_GRAY) {
        // gray conversion then uint8 resize: a thread per four output pixels;
        // exact 2x downscales with vector loads where the layout allows
        a.xt = p->d_xq;
        a.yt = p->d_yq;
        const long long groups = static_cast<long long>(a.OH) * ((a.OW + rz::kDirectRun - 1) / rz::kDirectRun);
        if (!p->opt_generic && a.W == 2 * a.OW && a.H == 2 * a.OH && (mode == RZ_NEAREST || is_down2(*p))) {
            const uintptr_t lw = C == 3 ? 8 : 16;
            const uintptr_t sa = reinterpret_cast<uintptr_t>(a.src) | static_cast<uintptr_t>(a.src_pitch) |
                                 static_cast<uintptr_t>(a.src_bstride);
            const uintptr_t da = reinterpret_cast<uintptr_t>(a.dst) | static_cast<uintptr_t>(a.dst_pitch) |
                                 static_cast<uintptr_t>(a.dst_bstride);
            const void *dfn = rz::direct_down2_gray_kernel_for(mode, C, a.bgr != 0);
            if (dfn && sa % lw == 0 && da % 4 == 0) return launch(dfn, groups, true);
        }
        const void *gfn = rz::direct_gray_kernel_for(mode, C, wrap);
        if (!gfn) return false;
        return launch(gfn, groups);
    }
    if (fam == rz::FAM_F32) {
        // float32 plans with the wrap rule: a thread per output pixel
        if (!wrap) return false;
        const void *ffn = rz::direct_f32_kernel_for(C, true);
        if (!ffn) return false;
        a.xt = p->d_xf;
        a.yt = p->d_yf;
        return launch(ffn, static_cast<long long>(a.OH) * a.OW);
    }
    if (!((fam == rz::FAM_U8 && (opt == 0 || opt == 3)) || (fam == rz::FAM_NORM && opt != 1))) return false;
    if (fam == rz::FAM_U8 && mode == RZ_LINEAR && !p->opt_generic && a.OW == 2 * a.W && a.OH == 2 * a.H) {
        // exact 2x upscale: the 1-3 weights, any layout, any border rule;
        // three and four channels with pixel lanes, each thread walking
        // kUp2RowsPerThread source rows (a uint8 tile override's row count
        // replaces it), one channel in 16-bit lanes of byte pairs
        a.xt = p->d_xq;
        a.yt = p->d_yq;
        const void *rfn = rz::direct_up2_rows_kernel_for(C, p->border);
        if (rfn) {
            // row blocks: as many as one wave of resident threads holds per
            // column group (rows shared out evenly), or the uint8 tile
            // override's rows per block
            const long long gpc = (a.W + 3) / 4;
            long long nrb;
            if (p->over_tr[rz::FAM_U8] > 0) {
                nrb = (a.H + p->over_tr[rz::FAM_U8] - 1) / p->over_tr[rz::FAM_U8];
            } else {
                int ctas = 0;
                const int e = resident_ctas(p->device, rfn, rz::kDirectThreads, &ctas);
                if (e != 0) {
                    *rc = cuda_fail(static_cast<cudaError_t>(e));
                    return true;
                }
                nrb = static_cast<long long>(ctas) * rz::kDirectThreads / std::max(1, std::min(batch, 65535)) / gpc;
            }
            // (the kernel forms rb H / nrb in 32 bits: nrb H < 2^32)
            nrb = std::min<long long>(nrb, 0xFFFFFFFFLL / a.H);
            a.tiles_y = static_cast<int>(std::clamp<long long>(nrb, 1, a.H));
            return launch(rfn, gpc * a.tiles_y, true);
        }
        const void *ufn = rz::direct_up2_kernel_for(C, p->border);
        if (ufn) return launch(ufn, static_cast<long long>(a.H) * ((a.W + rz::kUp2Cols - 1) / rz::kUp2Cols));
    }
    if (fam == rz::FAM_U8 && opt == 0 && mode == RZ_LINEAR && auto_u8_stream(*p) && !is_down2(*p) && !wrap)
        return false;
    a.xt = p->d_xq;
    a.yt = p->d_yq;
    const void *fn = nullptr;
    long long groups = 0;
    if (fam == rz::FAM_U8 && !p->opt_generic && a.W == 2 * a.OW && a.H == 2 * a.OH &&
        (mode == RZ_NEAREST || is_down2(*p))) {
        const uintptr_t lw = C == 3 ? 8 : 16, sw = C == 3 ? 4 : 8;
        const uintptr_t sa = reinterpret_cast<uintptr_t>(a.src) | static_cast<uintptr_t>(a.src_pitch) |
                             static_cast<uintptr_t>(a.src_bstride);
        const uintptr_t da = reinterpret_cast<uintptr_t>(a.dst) | static_cast<uintptr_t>(a.dst_pitch) |
                             static_cast<uintptr_t>(a.dst_bstride);
        if (sa % lw == 0 && da % sw == 0) {
            const void *dfn = rz::direct_down2_kernel_for(mode, C);
            const int px = rz::down2_px(C);
            if (dfn) return launch(dfn, static_cast<long long>(a.OH) * ((a.OW + px - 1) / px), true);
        }
    }
    if (!fn && fam == rz::FAM_U8 && !p->opt_generic && is_down32(*p)) {
        // exact 3:2 downscale: eight output pixels of one row per thread
        const uintptr_t sa = reinterpret_cast<uintptr_t>(a.src) | static_cast<uintptr_t>(a.src_pitch) |
                             static_cast<uintptr_t>(a.src_bstride);
        const uintptr_t da = reinterpret_cast<uintptr_t>(a.dst) | static_cast<uintptr_t>(a.dst_pitch) |
                             static_cast<uintptr_t>(a.dst_bstride);
        const void *dfn = rz::direct_down32_kernel_for(C);
        if (dfn && sa % 4 == 0 && da % 4 == 0) return launch(dfn, static_cast<long long>(a.OH) * ((a.OW + 7) / 8));
    }
    const long long gpr = (a.OW + rz::kDirectRun - 1) / rz::kDirectRun;
    if (!fn && fam == rz::FAM_U8 && mode == RZ_LINEAR && a.OH > a.H && opt == 3 && !wrap) {
        // about 2048 threads per SM, each walking R output rows
        fn = rz::direct_rows_kernel_for(C);
        int sms = 0;
        const cudaError_t ce = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device);
        if (ce != cudaSuccess) {
            *rc = cuda_fail(ce);
            return true;
        }
        int R = p->over_tr[fam];
        if (R <= 0) {
            const long long want = static_cast<long long>(sms) * 2048;
            R = static_cast<int>(std::clamp<long long>((gpr * a.OH * batch + want - 1) / want, 2, 32));
        }
        a.TR = std::min(R, a.OH);
        groups = gpr * ((a.OH + a.TR - 1) / a.TR);
    }
    if (!fn && fam == rz::FAM_NORM) {
        // a warp per 32 kNormRun output pixels of a row
        fn = rz::direct_kernel_for(rz::DIRECT_NORM, mode, C, wrap);
        groups = static_cast<long long>(a.OH) * ((a.OW + 32 * rz::kNormRun - 1) / (32 * rz::kNormRun)) * 32;
    }
    if (!fn) {
        fn = rz::direct_kernel_for(rz::DIRECT_U8, mode, C, wrap);
        groups = gpr * a.OH;
    }
    if (!fn) return false;
    return launch(fn, groups);
}

// The kernel family of a plain float32 resize: bilinear clamp and mirror
// plans run the streaming filter kernel with K = 1 and weight 1 (each
// resized value m is stored as 1 * m = m; the source rows stream once, as for
// the fused filters), unless the option or a float32 tile override asks for
// the staged tiles; wrap plans take the direct float32 kernel, nearest the
// staged tiles (and so does a geometry whose source span does not fit a
// streamed strip: run falls back).
int f32_family(const rz_plan_s *p, int mode, KArgs &extra)
{
    if (!p || mode != RZ_LINEAR || p->border == RZ_BORDER_WRAP || p->opt_f32_kernel != 0 ||
        p->over_tr[rz::FAM_F32] > 0 || p->over_tw[rz::FAM_F32] > 0)
        return rz::FAM_F32;
    extra.ksize = 0;
    extra.w[0] = 1.0f;
    return rz::FAM_FILT;
}

// Shared body of every resize entry point.  `planes` > 0 selects the planar
// (NCHW) output of the normalise epilogue.
int run(rz_plan_s *p, int fam, const void *src, size_t src_pitch, size_t src_bstride, void *dst, size_t dst_pitch,
        size_t dst_bstride, int H, int W, int C, int OH, int OW, int mode, int batch, const rz::KArgs &extra,
        void *stream, bool do_launch = true)
{
    if (!p) return RZ_ERR_ARG;
    if (H != p->H || W != p->W || OH != p->OH || OW != p->OW || mode != p->mode) return RZ_ERR_ARG;
    if (C <= 0 || batch < 0) return RZ_ERR_ARG;
    if (C != 1 && C != 3 && C != 4) return RZ_ERR_UNSUPPORTED;
    if (OH == 0 || OW == 0 || batch == 0) return RZ_OK;
    if (!src || !dst) return RZ_ERR_ARG;
    const int in_es = rz::fam_in_es(fam), out_es = rz::fam_out_es(fam);
    const bool nchw = fam == rz::FAM_NORM;
    const int out_c = (nchw || fam == rz::FAM_GRAY) ? 1 : C;   // interleaved channels of an output row
    const size_t in_row = static_cast<size_t>(W) * C * in_es;
    const size_t out_row = static_cast<size_t>(OW) * out_c * out_es;
    if (src_pitch < in_row || dst_pitch < out_row) return RZ_ERR_ARG;
    if (in_es == 4 && ((src_pitch & 3) || (reinterpret_cast<uintptr_t>(src) & 3))) return RZ_ERR_ARG;
    if (out_es == 4 && ((dst_pitch & 3) || (reinterpret_cast<uintptr_t>(dst) & 3))) return RZ_ERR_ARG;
    const size_t src_img = image_extent(H, src_pitch, in_row);
    const size_t dst_img = nchw ? static_cast<size_t>(C) * OH * dst_pitch : image_extent(OH, dst_pitch, out_row);
    if (batch > 1) {
        if (src_bstride < src_img || dst_bstride < dst_img) return RZ_ERR_ARG;
        if (in_es == 4 && (src_bstride & 3)) return RZ_ERR_ARG;
        if (out_es == 4 && (dst_bstride & 3)) return RZ_ERR_ARG;
    }
    const size_t src_all = batch > 1 ? (batch - 1) * src_bstride + src_img : src_img;
    const size_t dst_all = batch > 1 ? (batch - 1) * dst_bstride + dst_img : dst_img;
    if (overlap(src, src_all, dst, dst_all)) return RZ_ERR_ARG;
    int rc = check_device(p);
    if (rc != RZ_OK) return rc;

    KArgs a = extra;
    a.src = static_cast<const uint8_t *>(src);
    a.src_pitch = static_cast<long long>(src_pitch);
    a.src_bstride = batch > 1 ? static_cast<long long>(src_bstride) : 0;
    a.dst = static_cast<uint8_t *>(dst);
    a.dst_pitch = static_cast<long long>(dst_pitch);
    a.dst_bstride = batch > 1 ? static_cast<long long>(dst_bstride) : 0;
    a.dst_plane = nchw ? static_cast<long long>(OH) * static_cast<long long>(dst_pitch) : 0;
    a.H = H; a.W = W; a.OH = OH; a.OW = OW; a.C = C;
    a.batch = batch;
    a.status = p->d_status;
    a.border = p->border;
    a.l2_prefetch = p->opt_l2_prefetch;
    a.src_extent = static_cast<long long>(src_all);
    a.dst_extent = static_cast<long long>(dst_all);
    a.tab = static_cast<const uint8_t *>(p->dmem);
    a.tab_bytes = static_cast<long long>(p->dmem_bytes);
#ifdef RZ_CHECK_BOUNDS
    // test hook of the checked build: declare the last RZ_CHECK_SHRINK bytes
    // of the source and of the output out of range (the buffers themselves
    // are whole, so an access the kernels should have refused still lands in
    // valid memory)
    if (const char *shrink = std::getenv("RZ_CHECK_SHRINK")) {
        const long long n = std::atoll(shrink);
        a.src_extent = std::max(0LL, a.src_extent - n);
        a.dst_extent = std::max(0LL, a.dst_extent - n);
    }
#endif
    if (run_direct(p, fam, a, mode, stream, do_launch, &rc)) return rc;
    // the staged and streaming kernels take source spans from the tables,
    // which under the wrap rule are not monotone at the edges
    if (p->border == RZ_BORDER_WRAP && mode == RZ_LINEAR) return RZ_ERR_UNSUPPORTED;
    if (fam == rz::FAM_GRAY) return RZ_ERR_UNSUPPORTED;

    TileCfg t;
    const void *fn = nullptr;
    rc = get_tile(p, fam, C, batch, &t, &fn, fam == rz::FAM_FILT ? a.ksize / 2 : 0);
    if (rc == RZ_ERR_UNSUPPORTED && fam == rz::FAM_FILT && a.ksize == 0) {
        // a plain float32 resize whose source span does not fit a streamed
        // strip (very wide rows): the staged tiles take it
        fam = rz::FAM_F32;
        rc = get_tile(p, fam, C, batch, &t, &fn, 0);
    }
    if (rc != RZ_OK) return rc;
    a.TR = t.TR; a.TW = t.TW; a.tiles_x = t.tiles_x; a.tiles_y = t.tiles_y;
    a.max_rows = t.max_rows; a.slot_bytes = t.slot_bytes; a.stages = t.stages;
    a.ring_chunks = t.ring_chunks; a.chunk_rows = t.chunk_rows; a.chunk_boxes = t.chunk_boxes;
    a.box_bytes = t.box_bytes;
    a.tma_in = aligned16(src) && (src_pitch % 16 == 0) && (in_row % 16 == 0) &&
               (a.src_bstride % 16 == 0);
    const int strip_bytes = t.TW * out_c * out_es;
    a.tma_out = aligned16(dst) && (dst_pitch % 16 == 0) && (a.dst_bstride % 16 == 0) &&
                (a.dst_plane % 16 == 0) && (t.tiles_x == 1 || strip_bytes % 16 == 0);
    const bool fl = (fam == rz::FAM_F32 || fam == rz::FAM_FILT);
    a.xt = fl ? p->d_xf : p->d_xq;
    a.yt = fl ? p->d_yf : p->d_yq;
    CUtensorMap tmap;
    std::memset(&tmap, 0, sizeof(tmap));
    a.tensor_in = 0;
    if (t.tensor && a.tma_in) {
        // the image as {8-byte words per row, rows, images}: a box row is
        // the tile's whole column span, so it moves as one long transfer
        EncodeTiledFn enc = tensor_encoder();
        const cuuint64_t dims[3] = {in_row / 8, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(batch)};
        const cuuint64_t bstride = batch > 1 ? a.src_bstride : static_cast<long long>(src_pitch) * H;
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(src_pitch), bstride};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(t.box_words), static_cast<cuuint32_t>(t.box_rows), 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (enc && enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<void *>(src), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS) {
            a.tensor_in = 1;
            a.box_words = t.box_words;
            a.box_rows = t.box_rows;
        }
    }
    if (!do_launch) return RZ_OK;
    const int e = rz::launch_resize(fn, a, tmap, t.grid, t.smem, p->opt_pdl != 0, stream);
    if (e != 0) return cuda_fail(static_cast<cudaError_t>(e));
    return RZ_OK;
}

}  // namespace

namespace rz {
void record_cuda_error(int e) { g_last_cuda_error = e; }
}  // namespace rz

extern "C" {

int resize_axis_table(int n_in, int n_out, int mode, int32_t *ofs, int32_t *w_q11, float *u)
{
    return resize_axis_table_border(n_in, n_out, mode, RZ_BORDER_CLAMP, ofs, w_q11, u);
}

int resize_axis_table_border(int n_in, int n_out, int mode, int border, int32_t *ofs, int32_t *w_q11, float *u)
{
    if (n_in < 1 || n_out < 0 || n_in > RZ_MAX_DIM || n_out > RZ_MAX_DIM || !valid_mode(mode) ||
        !valid_border(border))
        return RZ_ERR_ARG;
    if (mode == RZ_LINEAR) {
        axis_linear(n_in, n_out, border, ofs, w_q11, u);
    } else {
        std::vector<int32_t> tmp(static_cast<size_t>(n_out));
        axis_nearest(n_in, n_out, tmp.data());
        if (ofs) std::memcpy(ofs, tmp.data(), tmp.size() * sizeof(int32_t));
    }
    return RZ_OK;
}

int resize_plan_create(rz_plan *out, int in_h, int in_w, int out_h, int out_w, int mode, void *stream)
{
    return resize_plan_create_border(out, in_h, in_w, out_h, out_w, mode, RZ_BORDER_CLAMP, stream);
}

int resize_plan_create_border(rz_plan *out, int in_h, int in_w, int out_h, int out_w, int mode, int border,
                              void *stream)
{
    if (!out) return RZ_ERR_ARG;
    *out = nullptr;
    if (in_h < 1 || in_w < 1 || out_h < 0 || out_w < 0 || in_h > RZ_MAX_DIM || in_w > RZ_MAX_DIM ||
        out_h > RZ_MAX_DIM || out_w > RZ_MAX_DIM || !valid_mode(mode) || !valid_border(border))
        return RZ_ERR_ARG;
    rz_plan_s *p = new (std::nothrow) rz_plan_s();
    if (!p) return RZ_ERR_NOMEM;
    p->H = in_h; p->W = in_w; p->OH = out_h; p->OW = out_w; p->mode = mode; p->border = border;
    try {
        p->xofs.resize(out_w); p->xq.resize(out_w); p->xu.resize(out_w);
        p->yofs.resize(out_h); p->yq.resize(out_h); p->yu.resize(out_h);
    } catch (...) {
        delete p;
        return RZ_ERR_NOMEM;
    }
    if (mode == RZ_LINEAR) {
        axis_linear(in_w, out_w, border, p->xofs.data(), p->xq.data(), p->xu.data());
        axis_linear(in_h, out_h, border, p->yofs.data(), p->yq.data(), p->yu.data());
    } else {
        axis_nearest(in_w, out_w, p->xofs.data());
        axis_nearest(in_h, out_h, p->yofs.data());
    }
    cudaError_t e = cudaGetDevice(&p->device);
    if (e != cudaSuccess) { delete p; return cuda_fail(e); }

    // one device block: x tables (q11 and float weights), y tables, status word
    const size_t nx = static_cast<size_t>(out_w), ny = static_cast<size_t>(out_h);
    // each table is kTabPad entries (a 16-byte multiple) after the start of
    // its block, which starts on a 16-byte boundary; the kTabPad entries
    // before and the kTabPad (or more) after it repeat its first and last
    // entry, so kernels may read entries in 16-byte pairs and copy a tile's
    // clamped range of entries in one piece
    constexpr size_t kPad = rz::kTabPad;
    const size_t xbytes = ((nx + 2 * kPad) * sizeof(int2) + 15) & ~size_t(15);
    const size_t ybytes = ((ny + 2 * kPad) * sizeof(int2) + 15) & ~size_t(15);
    const size_t off_xf = xbytes, off_yq = 2 * xbytes, off_yf = off_yq + ybytes;
    const size_t off_st = off_yf + ybytes;
    const size_t total = off_st + 16;
    std::vector<uint8_t> host(total, 0);
    int2 *hxq = reinterpret_cast<int2 *>(host.data()), *hxf = reinterpret_cast<int2 *>(host.data() + off_xf);
    int2 *hyq = reinterpret_cast<int2 *>(host.data() + off_yq), *hyf = reinterpret_cast<int2 *>(host.data() + off_yf);
    for (size_t k = 0; nx > 0 && k < xbytes / sizeof(int2); k++) {
        const size_t i = std::min(k < kPad ? 0 : k - kPad, nx - 1);
        int32_t ubits;
        std::memcpy(&ubits, &p->xu[i], 4);
        hxq[k] = make_int2(p->xofs[i], p->xq[i]);
        hxf[k] = make_int2(p->xofs[i], ubits);
    }
    for (size_t k = 0; ny > 0 && k < ybytes / sizeof(int2); k++) {
        const size_t i = std::min(k < kPad ? 0 : k - kPad, ny - 1);
        int32_t vbits;
        std::memcpy(&vbits, &p->yu[i], 4);
        hyq[k] = make_int2(p->yofs[i], p->yq[i]);
        hyf[k] = make_int2(p->yofs[i], vbits);
    }
    e = cudaMalloc(&p->dmem, total);
    if (e != cudaSuccess) { p->dmem = nullptr; delete p; return cuda_fail(e); }
    p->dmem_bytes = total;
    uint8_t *d = static_cast<uint8_t *>(p->dmem);
    p->d_xq = reinterpret_cast<int2 *>(d) + kPad;
    p->d_xf = reinterpret_cast<int2 *>(d + off_xf) + kPad;
    p->d_yq = reinterpret_cast<int2 *>(d + off_yq) + kPad;
    p->d_yf = reinterpret_cast<int2 *>(d + off_yf) + kPad;
    p->d_status = reinterpret_cast<int *>(d + off_st);
    // pageable source: the call returns once the bytes are staged, so `host`
    // may be freed on return
    e = cudaMemcpyAsync(p->dmem, host.data(), total, cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) { cudaFree(p->dmem); delete p; return cuda_fail(e); }
    *out = p;
    return RZ_OK;
}

int resize_plan_destroy(rz_plan p)
{
    if (!p) return RZ_OK;
    int rc = RZ_OK;
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != p->device) cudaSetDevice(p->device);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) rc = cuda_fail(e);
    e = cudaFree(p->dmem);
    if (e != cudaSuccess && rc == RZ_OK) rc = cuda_fail(e);
    if (cur >= 0 && cur != p->device) cudaSetDevice(cur);
    delete p;
    return rc;
}

int resize_plan_status(rz_plan p, int *status)
{
    if (!p) return RZ_ERR_ARG;
    int rc = check_device(p);
    if (rc != RZ_OK) return rc;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
    int v = 0;
    e = cudaMemcpy(&v, p->d_status, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaMemset(p->d_status, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e);
    if (status) *status = v;
    return RZ_OK;
}

int resize_plan_set_tile(rz_plan p, int kind, int tile_rows, int tile_cols)
{
    if (!p || kind < 0 || kind >= rz::FAM_COUNT || kind == 2 || kind == rz::FAM_GRAY || tile_rows < 0 ||
        tile_cols < 0)
        return RZ_ERR_ARG;
    if ((tile_rows == 0) != (tile_cols == 0)) return RZ_ERR_ARG;
    std::lock_guard<std::mutex> lk(p->mu);
    p->over_tr[kind] = tile_rows;
    p->over_tw[kind] = tile_cols;
    p->cache.clear();
    return RZ_OK;
}

int resize_plan_set_option(rz_plan p, int option, int value)
{
    if (!p) return RZ_ERR_ARG;
    std::lock_guard<std::mutex> lk(p->mu);
    switch (option) {
    case RZ_OPT_STAGES:
        if (value < 0 || value > rz::kMaxStages) return RZ_ERR_ARG;
        p->opt_stages = value;
        break;
    case RZ_OPT_GENERIC_ONLY:
        if (value != 0 && value != 1) return RZ_ERR_ARG;
        p->opt_generic = value;
        break;
    case RZ_OPT_CTAS_PER_SM:
        if (value < 0 || value > 32) return RZ_ERR_ARG;
        p->opt_ctas_per_sm = value;
        break;
    case RZ_OPT_GRID_MODE:
        if (value != 0 && value != 1) return RZ_ERR_ARG;
        p->opt_grid_mode = value;
        break;
    case RZ_OPT_PDL:
        if (value != 0 && value != 1) return RZ_ERR_ARG;
        p->opt_pdl = value;
        break;
    case RZ_OPT_RING_ROWS:
        if (value != 0 && (value < 2 || value > rz::kStreamRingMax)) return RZ_ERR_ARG;
        p->opt_ring_rows = value;
        break;
    case RZ_OPT_U8_KERNEL:
        if (value < 0 || value > 3) return RZ_ERR_ARG;
        p->opt_u8_kernel = value;
        break;
    case RZ_OPT_FILTER_KERNEL:
        if (value < 0 || value > 2) return RZ_ERR_ARG;
        p->opt_filter_kernel = value;
        break;
    case RZ_OPT_F32_KERNEL:
        if (value < 0 || value > 1) return RZ_ERR_ARG;
        p->opt_f32_kernel = value;
        break;
    case RZ_OPT_L2_PREFETCH:
        if (value != 0 && value != 1) return RZ_ERR_ARG;
        p->opt_l2_prefetch = value;
        break;
    default:
        return RZ_ERR_ARG;
    }
    p->cache.clear();
    return RZ_OK;
}

int resize_u8(rz_plan p, const uint8_t *src, size_t src_pitch, uint8_t *dst, size_t dst_pitch, int H, int W, int C,
              int out_h, int out_w, int mode, void *stream)
{
    KArgs extra = {};
    return run(p, rz::FAM_U8, src, src_pitch, 0, dst, dst_pitch, 0, H, W, C, out_h, out_w, mode, 1, extra, stream);
}

int resize_f32(rz_plan p, const float *src, size_t src_pitch, float *dst, size_t dst_pitch, int H, int W, int C,
               int out_h, int out_w, int mode, void *stream)
{
    KArgs extra = {};
    const int fam = f32_family(p, mode, extra);
    return run(p, fam, src, src_pitch, 0, dst, dst_pitch, 0, H, W, C, out_h, out_w, mode, 1, extra, stream);
}

int resize_wait_selftest(int *dev_status, int limit_us, void *stream)
{
    if (!dev_status || limit_us < 1 || limit_us > 1000000) return RZ_ERR_ARG;
    const int e = rz::launch_wait_selftest(dev_status, 1000ull * static_cast<unsigned long long>(limit_us), stream);
    return e != 0 ? cuda_fail(static_cast<cudaError_t>(e)) : RZ_OK;
}

int resize_u8_batch(rz_plan p, const uint8_t *src, size_t src_pitch, size_t src_batch_stride, uint8_t *dst,
                    size_t dst_pitch, size_t dst_batch_stride, int batch, int H, int W, int C, int out_h, int out_w,
                    int mode, void *stream)
{
    KArgs extra = {};
    return run(p, rz::FAM_U8, src, src_pitch, src_batch_stride, dst, dst_pitch, dst_batch_stride, H, W, C, out_h,
               out_w, mode, batch, extra, stream);
}

int resize_f32_batch(rz_plan p, const float *src, size_t src_pitch, size_t src_batch_stride, float *dst,
                     size_t dst_pitch, size_t dst_batch_stride, int batch, int H, int W, int C, int out_h, int out_w,
                     int mode, void *stream)
{
    KArgs extra = {};
    const int fam = f32_family(p, mode, extra);
    return run(p, fam, src, src_pitch, src_batch_stride, dst, dst_pitch, dst_batch_stride, H, W, C, out_h,
               out_w, mode, batch, extra, stream);
}

int resize_fused(rz_plan p, const void *src, int src_dtype, size_t src_pitch, void *dst, size_t dst_pitch, int H,
                 int W, int C, int out_h, int out_w, int mode, const rz_epilogue *e, void *stream)
{
    if (!e) return RZ_ERR_ARG;
    KArgs extra = {};
    int fam;
    if (e->kind == RZ_EPI_GRAY_RGB || e->kind == RZ_EPI_GRAY_BGR) {
        if (src_dtype != RZ_U8 || !valid_mode(mode) || C < 3) return RZ_ERR_ARG;
        if (C > 4) return RZ_ERR_UNSUPPORTED;
        fam = rz::FAM_GRAY;
        extra.bgr = e->kind == RZ_EPI_GRAY_BGR ? 1 : 0;
        return run(p, fam, src, src_pitch, e->src_batch_stride, dst, dst_pitch, e->dst_batch_stride, H, W, C, out_h,
                   out_w, mode, e->batch, extra, stream);
    }
    if (mode != RZ_LINEAR) return RZ_ERR_ARG;
    if (e->kind == RZ_EPI_NORMALIZE_NCHW) {
        if (src_dtype != RZ_U8) return RZ_ERR_ARG;
        fam = rz::FAM_NORM;
        if (C < 1 || C > 4) return C < 1 ? RZ_ERR_ARG : RZ_ERR_UNSUPPORTED;
        for (int c = 0; c < C; c++) {
            const double sd = e->std[c], mu = e->mean[c];
            if (!(sd != 0.0) || sd != sd || sd - sd != 0.0 || mu != mu || mu - mu != 0.0) return RZ_ERR_ARG;
            extra.scale[c] = static_cast<float>(1.0 / (255.0 * sd));
            extra.shift[c] = static_cast<float>(-mu / sd);
        }
    } else if (e->kind == RZ_EPI_FILTER3X3) {
        if (src_dtype != RZ_F32) return RZ_ERR_ARG;
        fam = rz::FAM_FILT;
        extra.ksize = 3;
        for (int i = 0; i < 9; i++) extra.w[i] = e->w3x3[i];
    } else if (e->kind == RZ_EPI_FILTER) {
        if (src_dtype != RZ_F32 || e->ksize < 1 || e->ksize % 2 == 0) return RZ_ERR_ARG;
        if (e->ksize > 7) return RZ_ERR_UNSUPPORTED;
        fam = rz::FAM_FILT;
        extra.ksize = e->ksize;
        for (int i = 0; i < e->ksize * e->ksize; i++) extra.w[i] = e->wk[i];
    } else {
        return RZ_ERR_ARG;
    }
    return run(p, fam, src, src_pitch, e->src_batch_stride, dst, dst_pitch, e->dst_batch_stride, H, W, C, out_h,
               out_w, mode, e->batch, extra, stream);
}

int resize_u8_multi(const rz_job *dev_jobs, int njobs, int C, int mode, int *dev_status, void *stream)
{
    if (njobs < 0 || njobs > RZ_MULTI_MAX_JOBS || !valid_mode(mode) || C < 1) return RZ_ERR_ARG;
    if (C != 1 && C != 3 && C != 4) return RZ_ERR_UNSUPPORTED;
    if (njobs == 0) return RZ_OK;
    if (!dev_jobs) return RZ_ERR_ARG;
    const int e = rz::launch_multi(dev_jobs, njobs, C, mode, dev_status, true, stream);
    return e != 0 ? cuda_fail(static_cast<cudaError_t>(e)) : RZ_OK;
}

int filter2d_valid_f32(const float *src, size_t src_pitch, int H, int W, const float *weights, int K, float *dst,
                       size_t dst_pitch, void *stream)
{
    return filter2d_valid_f32_ex(src, src_pitch, H, W, weights, K, dst, dst_pitch, RZ_FILTER_AUTO, nullptr, stream);
}

int filter2d_valid_f32_ex(const float *src, size_t src_pitch, int H, int W, const float *weights, int K, float *dst,
                          size_t dst_pitch, int kernel, int *dev_status, void *stream)
{
    if (kernel != RZ_FILTER_AUTO && kernel != RZ_FILTER_FP32 && kernel != RZ_FILTER_TENSOR) return RZ_ERR_ARG;
    if (H < 0 || W < 0 || K < 1 || H > RZ_MAX_DIM || W > RZ_MAX_DIM) return RZ_ERR_ARG;
    if (K > rz::kMaxFilterK) return RZ_ERR_UNSUPPORTED;
    if (H < K || W < K) return RZ_OK;   // empty output
    if (!src || !dst || !weights) return RZ_ERR_ARG;
    const size_t in_row = static_cast<size_t>(W) * 4, out_row = static_cast<size_t>(W - K + 1) * 4;
    if (src_pitch < in_row || dst_pitch < out_row || (src_pitch & 3) || (dst_pitch & 3) ||
        (reinterpret_cast<uintptr_t>(src) & 3) || (reinterpret_cast<uintptr_t>(dst) & 3) ||
        (reinterpret_cast<uintptr_t>(weights) & 3))
        return RZ_ERR_ARG;
    if (overlap(src, image_extent(H, src_pitch, in_row), dst, image_extent(H - K + 1, dst_pitch, out_row)))
        return RZ_ERR_ARG;
    const bool tc_ok = rz::filter_tc_supported(src, static_cast<long long>(src_pitch), K);
    if (kernel == RZ_FILTER_TENSOR && !tc_ok) return RZ_ERR_UNSUPPORTED;
    const bool tc = kernel == RZ_FILTER_TENSOR || (kernel == RZ_FILTER_AUTO && tc_ok && K >= kFilterTcMinK);
    const int e = tc ? rz::launch_filter_tc(src, static_cast<long long>(src_pitch), H, W, weights, K, dst,
                                            static_cast<long long>(dst_pitch), dev_status, true, stream)
                     : rz::launch_filter_valid(src, static_cast<long long>(src_pitch), H, W, weights, K, dst,
                                               static_cast<long long>(dst_pitch), true, stream);
    return e != 0 ? cuda_fail(static_cast<cudaError_t>(e)) : RZ_OK;
}

int resize_u8_host(rz_plan p, const uint8_t *host_src, size_t host_src_pitch, uint8_t *host_dst, size_t host_dst_pitch,
                   uint8_t *dev_src, size_t dev_src_pitch, uint8_t *dev_dst, size_t dev_dst_pitch, int H, int W,
                   int C, int out_h, int out_w, int mode, void *stream)
{
    if (!p || !host_src || !host_dst || !dev_src || !dev_dst) return RZ_ERR_ARG;
    if (C <= 0 || H != p->H || W != p->W || out_h != p->OH || out_w != p->OW) return RZ_ERR_ARG;
    const size_t in_row = static_cast<size_t>(W) * C, out_row = static_cast<size_t>(out_w) * C;
    if (host_src_pitch < in_row || host_dst_pitch < out_row) return RZ_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // validate the device-side call before queuing any copy
    int rc = run(p, rz::FAM_U8, dev_src, dev_src_pitch, 0, dev_dst, dev_dst_pitch, 0, H, W, C, out_h, out_w, mode, 1,
                 KArgs{}, stream, false);
    if (rc != RZ_OK) return rc;
    cudaError_t e = cudaMemcpy2DAsync(dev_src, dev_src_pitch, host_src, host_src_pitch, in_row, H,
                                      cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e);
    rc = resize_u8(p, dev_src, dev_src_pitch, dev_dst, dev_dst_pitch, H, W, C, out_h, out_w, mode, stream);
    if (rc != RZ_OK) return rc;
    if (out_h > 0 && out_w > 0) {
        e = cudaMemcpy2DAsync(host_dst, host_dst_pitch, dev_dst, dev_dst_pitch, out_row, out_h,
                              cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return RZ_OK;
}

const char *resize_strerror(int code)
{
    switch (code) {
    case RZ_OK: return "ok";
    case RZ_ERR_ARG: return "invalid argument";
    case RZ_ERR_UNSUPPORTED: return "unsupported parameter";
    case RZ_ERR_CUDA: return "CUDA runtime error";
    case RZ_ERR_NOMEM: return "out of memory";
    case RZ_ERR_TIMEOUT: return "kernel timed out waiting for a bulk copy";
    default: return "unknown status";
    }
}

int resize_last_cuda_error(void) { return g_last_cuda_error; }

}  // extern "C"
