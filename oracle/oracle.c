/*
 * CPU oracle for image resize — TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, single-threaded C.  Every output value is computed from its own
 * definition, per pixel, with exact integer (int64) or double arithmetic; there
 * are no tables, no tiling, no vectorisation and nothing shared with the CUDA
 * library.  Only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark load this file; the library's own code never does.
 *
 * Sources (page title, then section):
 *  [VOLCANIC]  "From Prototype to Performance: Optimizing OpenCV Resize on
 *              Volcanic GPUs" — "Naive resize with linear sampling" (the
 *              output->input mapping (dst + 0.5) * inv_scale fed to a linear
 *              sampler with unnormalised coordinates, whose texel centres sit at
 *              +0.5, so that the sampled point is (dst + 0.5) * in/out - 0.5),
 *              "Step 2: Make the GPU version correct first" (output size
 *              int(in * SCALE)).
 *  [INTERP]    "CUDA nearest-neighbour and bilinear interpolation, operator
 *              fusion" (hnwysp.cn/news/129086) — §2.1 nearest, §2.2 bilinear
 *              weights (1-u)(1-v), u(1-v), (1-u)v, uv with i = floor(x),
 *              j = floor(y), u = x - i, v = y - j; §6.1 clamp border;
 *              §6.2 fixed-point arithmetic; §4.2 fusing a 3x3 filter after the
 *              interpolation.
 *  [CONV]      "OpenCL image convolution" (coolbeet.weebly.com/final.html) —
 *              §2 "Image Convolution using CPU": correlation without a kernel
 *              flip, filter index r * width + c with r over rows.
 *  [TRACKING]  "Performance Optimization of Object Tracking Algorithms in
 *              OpenCV on GPUs" — §4.2 kernel merging and Table 10: a merged
 *              kernel computes exactly the composition of the kernels it
 *              replaces; §3.1.1 "Execution Flow": frames are converted to
 *              grayscale (cvtColor, the RGB2Gray kernel) before the resize.
 *
 * Readings where the pages leave a step open (each is also listed in the
 * design notes):
 *  - mapping: x = (dx + 1/2) * W_in / W_out - 1/2 with the ratio of the actual
 *    sizes, held as the exact rational ((2dx+1) W_in - W_out) / (2 W_out);
 *  - border ([INTERP] §6.1 names clamp, mirror and wrap): each tap's integer
 *    index is mapped into [0, n-1] by the border rule, the weights stay
 *    those of the unmapped position; mirror reflects about the edge samples
 *    (index -1 reads 1, index n reads n-2), wrap repeats the axis with
 *    period n;
 *  - u8 weights: 11 fractional bits, A1 = round-half-up(2048 u), A0 = 2048-A1,
 *    the same for B on rows; the four products are summed exactly and rounded
 *    half-up once: (sum + 2^21) >> 22 ([INTERP] §6.2 "fixed point");
 *  - nearest: OpenCV INTER_NEAREST, i = floor(dx * W_in / W_out);
 *  - normalise: y = (q / 255 - mean[c]) / std[c] on the rounded u8 resize
 *    result q, written planar (NCHW);
 *  - 3x3 filter: correlation on the resized grid, replicate border on that
 *    grid, weights used as given (no division by 9);
 *  - grayscale ([TRACKING] §3.1.1 gives no weights): the ITU-R BT.601 luma
 *    weights 0.299 R + 0.587 G + 0.114 B, rounded half-up exactly to u8,
 *    converted per source pixel before the resize samples it.
 *
 * Pixel (x, y), channel c of an interleaved image lives at byte offset
 * y * pitch + (x * C + c) * sizeof(element).  Pitches are in bytes.
 */
#include <stdint.h>
#include <stddef.h>

/* floor(a / b) for b > 0 */
static int64_t floor_div(int64_t a, int64_t b)
{
    int64_t q = a / b;
    if ((a % b) != 0 && a < 0)
        q -= 1;
    return q;
}

static int64_t clamp_index(int64_t k, int64_t n)
{
    if (k < 0)
        return 0;
    if (k > n - 1)
        return n - 1;
    return k;
}

/*
 * Border rule of [INTERP] §6.1 for an integer index k on an axis of n samples:
 *   0  clamp:  the nearest sample inside, k -> min(max(k, 0), n - 1);
 *   1  mirror: reflection about the first and last sample centres, so the
 *              extended axis reads 0 1 .. n-1 n-2 .. 1 0 1 .. (period 2n - 2);
 *              a single sample (n = 1) is read everywhere;
 *   2  wrap:   the axis repeats, k -> k mod n.
 */
static int64_t border_index(int64_t k, int64_t n, int border)
{
    if (border == 1) {
        if (n == 1)
            return 0;
        int64_t period = 2 * (n - 1);
        int64_t m = k % period;
        if (m < 0)
            m += period;
        return m <= n - 1 ? m : period - m;
    }
    if (border == 2) {
        int64_t m = k % n;
        return m < 0 ? m + n : m;
    }
    return clamp_index(k, n);
}

int64_t oracle_border_index(int64_t k, int64_t n, int border)
{
    return border_index(k, n, border);
}

/*
 * Sampling position of output index d on an axis of n_in input and n_out
 * output samples:  x = (d + 1/2) * n_in / n_out - 1/2 = num / den  with
 * num = (2d + 1) n_in - n_out,  den = 2 n_out.
 * Returns i = floor(x) and the remainder r = num - i * den, so u = r / den.
 * [VOLCANIC] "Naive resize with linear sampling"; [INTERP] §2.2.
 */
void oracle_linear_coord(int64_t n_in, int64_t n_out, int64_t d,
                         int64_t *i, int64_t *r, int64_t *den)
{
    int64_t num = (2 * d + 1) * n_in - n_out;
    *den = 2 * n_out;
    *i = floor_div(num, *den);
    *r = num - (*i) * (*den);
}

/* round-half-up(2048 * r / den): the 11-bit fixed-point weight of the far tap. */
int64_t oracle_weight_q11(int64_t r, int64_t den)
{
    return floor_div(4096 * r + den, 2 * den);
}

/* Nearest source index: floor(d * n_in / n_out), kept inside the image. */
int64_t oracle_nearest_index(int64_t n_in, int64_t n_out, int64_t d)
{
    return clamp_index(floor_div(d * n_in, n_out), n_in);
}

/*
 * u8 bilinear, [INTERP] §2.2 with a §6.1 border rule and §6.2 fixed point:
 *   dst = ( B0 A0 s(i,j) + B0 A1 s(i+1,j) + B1 A0 s(i,j+1) + B1 A1 s(i+1,j+1)
 *           + 2^21 ) >> 22
 * where s(i, j) is column i, row j (indices mapped by border_index), and A/B
 * are the 11-bit weights of u/v.
 */
void oracle_linear_u8_border_rows(const uint8_t *src, int64_t src_pitch, int H, int W, int C,
                                  uint8_t *dst, int64_t dst_pitch, int OH, int OW, int border,
                                  int dy0, int dy1)
{
    for (int64_t dy = dy0; dy < dy1 && dy < OH; dy++) {
        int64_t j, rv, dv;
        oracle_linear_coord(H, OH, dy, &j, &rv, &dv);
        int64_t B1 = oracle_weight_q11(rv, dv);
        int64_t B0 = 2048 - B1;
        int64_t j0 = border_index(j, H, border), j1 = border_index(j + 1, H, border);
        for (int64_t dx = 0; dx < OW; dx++) {
            int64_t i, ru, du;
            oracle_linear_coord(W, OW, dx, &i, &ru, &du);
            int64_t A1 = oracle_weight_q11(ru, du);
            int64_t A0 = 2048 - A1;
            int64_t i0 = border_index(i, W, border), i1 = border_index(i + 1, W, border);
            for (int64_t c = 0; c < C; c++) {
                int64_t s00 = src[j0 * src_pitch + i0 * C + c];
                int64_t s10 = src[j0 * src_pitch + i1 * C + c];
                int64_t s01 = src[j1 * src_pitch + i0 * C + c];
                int64_t s11 = src[j1 * src_pitch + i1 * C + c];
                int64_t acc = B0 * A0 * s00 + B0 * A1 * s10 + B1 * A0 * s01 + B1 * A1 * s11;
                dst[dy * dst_pitch + dx * C + c] = (uint8_t)((acc + (1 << 21)) >> 22);
            }
        }
    }
}

/* Clamp border, output rows [dy0, dy1): lets a caller time a bounded sample. */
void oracle_linear_u8_rows(const uint8_t *src, int64_t src_pitch, int H, int W, int C,
                           uint8_t *dst, int64_t dst_pitch, int OH, int OW, int dy0, int dy1)
{
    oracle_linear_u8_border_rows(src, src_pitch, H, W, C, dst, dst_pitch, OH, OW, 0, dy0, dy1);
}

/* All output rows, any border rule. */
void oracle_linear_u8(const uint8_t *src, int64_t src_pitch, int H, int W, int C,
                      uint8_t *dst, int64_t dst_pitch, int OH, int OW, int border)
{
    oracle_linear_u8_border_rows(src, src_pitch, H, W, C, dst, dst_pitch, OH, OW, border, 0, OH);
}

/* u8 nearest, [INTERP] §2.1 read as OpenCV INTER_NEAREST (floor). */
void oracle_nearest_u8(const uint8_t *src, int64_t src_pitch, int H, int W, int C,
                       uint8_t *dst, int64_t dst_pitch, int OH, int OW)
{
    for (int64_t dy = 0; dy < OH; dy++) {
        int64_t j = oracle_nearest_index(H, OH, dy);
        for (int64_t dx = 0; dx < OW; dx++) {
            int64_t i = oracle_nearest_index(W, OW, dx);
            for (int64_t c = 0; c < C; c++)
                dst[dy * dst_pitch + dx * C + c] = src[j * src_pitch + i * C + c];
        }
    }
}

static double f32_at(const float *src, int64_t pitch_bytes, int64_t x, int64_t y, int C, int64_t c)
{
    const char *row = (const char *)src + y * pitch_bytes;
    return (double)((const float *)row)[x * C + c];
}

/*
 * f32 bilinear, evaluated in double with the exact u = r / den:
 *   dst = (1-u)(1-v) s(i,j) + u(1-v) s(i+1,j) + (1-u)v s(i,j+1) + uv s(i+1,j+1)
 * [INTERP] §2.2, §6.1 (indices mapped by border_index).  Output is double,
 * dense, dst[(dy * OW + dx) * C + c].
 */
void oracle_linear_f32(const float *src, int64_t src_pitch, int H, int W, int C,
                       double *dst, int OH, int OW, int border)
{
    for (int64_t dy = 0; dy < OH; dy++) {
        int64_t j, rv, dv;
        oracle_linear_coord(H, OH, dy, &j, &rv, &dv);
        double v = (double)rv / (double)dv;
        int64_t j0 = border_index(j, H, border), j1 = border_index(j + 1, H, border);
        for (int64_t dx = 0; dx < OW; dx++) {
            int64_t i, ru, du;
            oracle_linear_coord(W, OW, dx, &i, &ru, &du);
            double u = (double)ru / (double)du;
            int64_t i0 = border_index(i, W, border), i1 = border_index(i + 1, W, border);
            for (int64_t c = 0; c < C; c++) {
                double s00 = f32_at(src, src_pitch, i0, j0, C, c);
                double s10 = f32_at(src, src_pitch, i1, j0, C, c);
                double s01 = f32_at(src, src_pitch, i0, j1, C, c);
                double s11 = f32_at(src, src_pitch, i1, j1, C, c);
                dst[(dy * OW + dx) * C + c] = (1.0 - u) * (1.0 - v) * s00 + u * (1.0 - v) * s10 +
                                              (1.0 - u) * v * s01 + u * v * s11;
            }
        }
    }
}

/* f32 nearest: a pure copy of the selected sample, so the result is float. */
void oracle_nearest_f32(const float *src, int64_t src_pitch, int H, int W, int C,
                        float *dst, int OH, int OW)
{
    for (int64_t dy = 0; dy < OH; dy++) {
        int64_t j = oracle_nearest_index(H, OH, dy);
        for (int64_t dx = 0; dx < OW; dx++) {
            int64_t i = oracle_nearest_index(W, OW, dx);
            for (int64_t c = 0; c < C; c++)
                dst[(dy * OW + dx) * C + c] = (float)f32_at(src, src_pitch, i, j, C, c);
        }
    }
}

/*
 * Per-channel normalisation of an already resized u8 image q (dense HWC,
 * OH x OW x C), written planar:  out[c][y][x] = (q / 255 - mean[c]) / std[c].
 * The fusion of [INTERP] §4.2 is read, with [TRACKING] §4.2, as leaving the
 * result of the unfused pipeline unchanged, so q is the rounded u8 resize.
 */
void oracle_normalize_nchw(const uint8_t *q, int OH, int OW, int C,
                           const double *mean, const double *std, double *out)
{
    for (int64_t c = 0; c < C; c++)
        for (int64_t y = 0; y < OH; y++)
            for (int64_t x = 0; x < OW; x++) {
                double val = (double)q[(y * OW + x) * C + c];
                out[(c * OH + y) * OW + x] = (val / 255.0 - mean[c]) / std[c];
            }
}

/*
 * 3x3 correlation of a single-channel double image r (dense, OH x OW), the
 * filter centred on each pixel, rows and columns outside the image replaced
 * by the nearest edge row/column:
 *   z[y][x] = sum_{a,b in {-1,0,1}} w[(a+1)*3 + (b+1)] * r[clamp(y+a)][clamp(x+b)]
 * [CONV] §2 (no flip, w[row * 3 + col]); [INTERP] §4.2 (3x3 after resize).
 */
void oracle_filter3x3(const double *r, int OH, int OW, const double *w, double *z)
{
    for (int64_t y = 0; y < OH; y++)
        for (int64_t x = 0; x < OW; x++) {
            double sum = 0.0;
            for (int64_t a = -1; a <= 1; a++)
                for (int64_t b = -1; b <= 1; b++) {
                    int64_t yy = clamp_index(y + a, OH);
                    int64_t xx = clamp_index(x + b, OW);
                    sum += w[(a + 1) * 3 + (b + 1)] * r[yy * OW + xx];
                }
            z[y * OW + x] = sum;
        }
}

/*
 * Grayscale of an interleaved u8 image with C >= 3 channels, [TRACKING]
 * §3.1.1 (cvtColor to grayscale before the resize).  With (R, G, B) the
 * channels (0, 1, 2), or (2, 1, 0) when bgr is set, and any fourth channel
 * ignored:  Y = floor((299 R + 587 G + 114 B + 500) / 1000), which is
 * 0.299 R + 0.587 G + 0.114 B rounded half-up, exactly.  dst is H x W u8.
 */
void oracle_gray_u8(const uint8_t *src, int64_t src_pitch, int H, int W, int C, int bgr,
                    uint8_t *dst, int64_t dst_pitch)
{
    int64_t ir = bgr ? 2 : 0, ib = bgr ? 0 : 2;
    for (int64_t y = 0; y < H; y++)
        for (int64_t x = 0; x < W; x++) {
            const uint8_t *px = src + y * src_pitch + x * C;
            int64_t sum = 299 * (int64_t)px[ir] + 587 * (int64_t)px[1] + 114 * (int64_t)px[ib];
            dst[y * dst_pitch + x] = (uint8_t)((sum + 500) / 1000);
        }
}

/*
 * K x K correlation over the valid region, [CONV] §2 (the filter placed with
 * its first row and column on the output position, each covered input
 * multiplied by its weight, the products summed; no flip):
 *   out[y][x] = sum_{r, c in [0, K)} w[r * K + c] * in[y + r][x + c],
 * 0 <= y <= H - K, 0 <= x <= W - K.  Single channel, dense, double.
 */
void oracle_filter_valid(const double *in, int H, int W, const double *w, int K, double *out)
{
    int64_t OH = H - K + 1, OW = W - K + 1;
    for (int64_t y = 0; y < OH; y++)
        for (int64_t x = 0; x < OW; x++) {
            double sum = 0.0;
            for (int64_t r = 0; r < K; r++)
                for (int64_t c = 0; c < K; c++)
                    sum += w[r * K + c] * in[(y + r) * W + (x + c)];
            out[y * OW + x] = sum;
        }
}

/*
 * K x K correlation (K odd) centred on each pixel of a single-channel image
 * r (OH x OW), rows and columns outside replaced by the nearest edge
 * row/column: the 3x3 rule of oracle_filter3x3 for any odd K,
 *   z[y][x] = sum_{a,b in [-K/2, K/2]} w[(a+K/2)*K + (b+K/2)] r[clamp(y+a)][clamp(x+b)].
 */
void oracle_filter_centred(const double *r, int OH, int OW, const double *w, int K, double *z)
{
    int64_t R = K / 2;
    for (int64_t y = 0; y < OH; y++)
        for (int64_t x = 0; x < OW; x++) {
            double sum = 0.0;
            for (int64_t a = -R; a <= R; a++)
                for (int64_t b = -R; b <= R; b++) {
                    int64_t yy = clamp_index(y + a, OH);
                    int64_t xx = clamp_index(x + b, OW);
                    sum += w[(a + R) * K + (b + R)] * r[yy * OW + xx];
                }
            z[y * OW + x] = sum;
        }
}
