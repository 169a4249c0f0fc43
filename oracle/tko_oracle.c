/*
 * Plain CPU oracle for fused SwiGLU + MoE top-k weight + FP8/FP4 activation cast.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only the test-suite, the smoke check
 * and the benchmark's CPU-baseline / reference legs may load this library. The
 * CUDA path never includes, links or calls anything here, and this file shares
 * no code, header, table or constant generator with it.
 *
 * It is deliberately slow: one element at a time, real-valued steps in double,
 * every encoder a brute-force nearest search over the format's whole grid.
 *
 * What it computes, with the passages it follows:
 *
 *  - Input layout: each expanded-token row of x holds 2H bf16 values, the gate
 *    half x_L at columns [0,H) and the up half x_R at [H,2H).
 *    ("TileKernels从入门到精通" / "TileKernels from Beginner to Master",
 *    zhichai.net/topic/177618752, ch.2 "内存的连体双胞胎：布局的艺术"; English
 *    summary, Chapter 2.)
 *  - Clamp guard: a gate value above the clamp limit is replaced by the limit
 *    and counted (same page, ch.2 "守门员 Clamp"). The page shows the gate's
 *    upper clamp only; the up half is clamped symmetrically to [-L, L] and
 *    counted separately (reading stated in the design notes).
 *  - SwiGLU: x_L * sigmoid(x_L), multiplied elementwise by x_R; then multiplied
 *    by the row's MoE top-k weight, before quantization (ch.2 "算子融合的三重境界",
 *    steps 1 and 2; Shazeer, "GLU Variants Improve Transformer").
 *  - Quantization: per-token or per-block absmax, a scale factor, then the FP8
 *    cast (ch.2 step 3). Formats and granularities from "TileLang + TileKernels：
 *    DeepSeek 的 GPU 内核开发新范式" (zhichai.net/topic/177618740), section
 *    "3. Quantization" table: FP8 E4M3 per-token / per-block, FP4 E2M1, UE8M0
 *    power-of-two scales.
 *
 * Precision: the real-valued activation y is evaluated in double and rounded
 * once to fp32. Everything after that (absmax, the fp32 scale, the quotient
 * y / s that decides a code) is taken in IEEE fp32, the precision the configs
 * fix for the scale; the code is then the round-to-nearest-even, saturating
 * image of that fp32 quotient on the format's grid. Build with
 * -ffp-contract=off and without -ffast-math so every operation is the single
 * IEEE operation written.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define TKO_SCALE_FP32 0
#define TKO_SCALE_UE8M0 1
#define TKO_OUT_E4M3 0
#define TKO_OUT_E2M1 1

/* ---------------------------------------------------------------- formats */

/* OCP FP8 E4M3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits,
 * no infinities, S.1111.111 is NaN, largest finite 448. */
double tko_e4m3_decode(uint8_t code)
{
    int sign = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);          /* subnormal: 0.m * 2^(1-7) */
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7); /* normal: 1.m * 2^(e-7) */
    return sign ? -mag : mag;
}

/* OCP FP4 E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; grid
 * {0, 0.5, 1, 1.5, 2, 3, 4, 6}; no NaN or infinity. Takes the low nibble. */
double tko_e2m1_decode(uint8_t nibble)
{
    int sign = (nibble >> 3) & 1;
    int e = (nibble >> 1) & 0x3;
    int m = nibble & 0x1;
    double mag;
    if (e == 0)
        mag = (double)m * 0.5;                      /* subnormal: 0.m * 2^(1-1) */
    else
        mag = ldexp(1.0 + (double)m / 2.0, e - 1);  /* normal: 1.m * 2^(e-1) */
    return sign ? -mag : mag;
}

/* Round-to-nearest-even with saturation onto the non-negative codes
 * [0, max_code] of a format, by exhaustive search: the nearest grid value wins,
 * and of two equally near neighbours the one with the even code (even mantissa
 * bit) wins. Magnitudes at or beyond the largest finite value saturate to it. */
static int nearest_code(double a, int max_code, double (*decode)(uint8_t))
{
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= max_code; ++c) {
        double d = fabs(decode((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return best;
}

uint8_t tko_e4m3_encode(float v)
{
    if (isnan(v))
        return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0)
        return sign | 0x7E;
    return sign | (uint8_t)nearest_code(a, 0x7E, tko_e4m3_decode);
}

uint8_t tko_e2m1_encode(float v)
{
    /* NaN has no E2M1 code; it is outside the contract and maps to +max. */
    if (isnan(v))
        return 0x7;
    uint8_t sign = signbit(v) ? 0x8 : 0x0;
    double a = fabs((double)v);
    if (a >= 6.0)
        return sign | 0x7;
    return sign | (uint8_t)nearest_code(a, 0x7, tko_e2m1_decode);
}

/* UE8M0: unsigned 8-bit exponent, value 2^(byte-127); 255 is NaN.
 * The scale exponent of a group is the smallest integer k with
 * qmax * 2^k >= amax, found by plain search (exact in double), then clamped to
 * the finite byte range [0, 254]. A group with amax == 0 gets 2^0. */
uint8_t tko_ue8m0_byte(float amax, double qmax)
{
    if (!(amax > 0.0f))
        return 127;
    int k = -300;
    while (qmax * ldexp(1.0, k) < (double)amax)
        ++k;
    if (k < -127)
        k = -127;
    if (k > 127)
        k = 127;
    return (uint8_t)(k + 127);
}

float tko_ue8m0_value(uint8_t byte)
{
    return (float)ldexp(1.0, (int)byte - 127);
}

/* fp32 scale: s = amax / qmax in IEEE fp32; a scale that comes out zero
 * (an all-zero group, or amax so small that the quotient underflows) is
 * replaced by 1 so that every code of the group is a signed zero. */
float tko_fp32_scale(float amax, float qmax)
{
    float s = amax / qmax;
    if (s == 0.0f)
        s = 1.0f;
    return s;
}

/* bf16 is the upper half of an IEEE fp32; widening is exact. */
static double bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------ quantization */

/* Quantize one group of n fp32 values y with the given formats. Writes the
 * n codes (one per byte, low nibble for E2M1) to codes and returns the scale
 * in *scale_f32 (fp32 mode) or *scale_byte (UE8M0 mode). */
static void quantize_group(const float *y, int64_t n, int scale_fmt, int out_fmt,
                           uint8_t *codes, float *scale_f32, uint8_t *scale_byte)
{
    double qmax = (out_fmt == TKO_OUT_E4M3) ? 448.0 : 6.0;
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(y[i]);
        if (a > amax)
            amax = a;
    }
    float s;
    if (scale_fmt == TKO_SCALE_FP32) {
        s = tko_fp32_scale(amax, (float)qmax);
        *scale_f32 = s;
    } else {
        uint8_t b = tko_ue8m0_byte(amax, qmax);
        s = tko_ue8m0_value(b);
        *scale_byte = b;
    }
    for (int64_t i = 0; i < n; ++i) {
        float quotient = y[i] / s; /* IEEE fp32 division */
        codes[i] = (out_fmt == TKO_OUT_E4M3) ? tko_e4m3_encode(quotient)
                                             : tko_e2m1_encode(quotient);
    }
}

/* Quantize rows of fp32 values y [rows, hidden] in groups of `group` columns
 * (group == 0: one group per row). Codes: E4M3 one byte per value
 * [rows, hidden]; E2M1 two per byte [rows, hidden/2], value 2k in the low
 * nibble and value 2k+1 in the high nibble. Scales [rows, hidden/group]:
 * float (fp32 mode) or byte (UE8M0 mode). Returns 0, or -1 on bad sizes. */
int tko_quant_rows_f32(const float *y, int64_t rows, int64_t hidden, int64_t group,
                       int scale_fmt, int out_fmt, uint8_t *q, void *scales)
{
    if (group == 0)
        group = hidden;
    if (rows < 0 || hidden <= 0 || group <= 0 || hidden % group != 0)
        return -1;
    if (out_fmt == TKO_OUT_E2M1 && (group % 2) != 0)
        return -1;
    int64_t ngroups = hidden / group;
    uint8_t codes[65536];
    if (group > 65536)
        return -1;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < ngroups; ++j) {
            const float *yg = y + r * hidden + j * group;
            float sf = 0.0f;
            uint8_t sb = 0;
            quantize_group(yg, group, scale_fmt, out_fmt, codes, &sf, &sb);
            if (scale_fmt == TKO_SCALE_FP32)
                ((float *)scales)[r * ngroups + j] = sf;
            else
                ((uint8_t *)scales)[r * ngroups + j] = sb;
            if (out_fmt == TKO_OUT_E4M3) {
                memcpy(q + r * hidden + j * group, codes, (size_t)group);
            } else {
                uint8_t *dst = q + r * (hidden / 2) + j * (group / 2);
                for (int64_t k = 0; k < group / 2; ++k)
                    dst[k] = (uint8_t)((codes[2 * k] & 0xF) | ((codes[2 * k + 1] & 0xF) << 4));
            }
        }
    }
    return 0;
}

/* Per-channel quantization of y [rows, hidden] (the per-channel granularity
 * of FP8 E4M3 in "TileLang + TileKernels：DeepSeek 的 GPU 内核开发新范式",
 * zhichai.net/topic/177618740, section "3. Quantization", format table): one
 * scale per column j, from the absolute maximum of that column over all rows;
 * every value of the column is scaled by it and encoded exactly as a group is
 * above. Here a column is gathered into a buffer and quantized as one group.
 * Codes [rows, hidden] (E4M3) or [rows, hidden/2] (E2M1, column 2k in the low
 * nibble of byte k, as for rows); scales [hidden]: float (fp32 mode) or byte
 * (UE8M0 mode). Returns 0, or -1 on bad sizes or when out of memory. */
int tko_quant_cols_f32(const float *y, int64_t rows, int64_t hidden, int scale_fmt, int out_fmt,
                       uint8_t *q, void *scales)
{
    if (rows < 0 || hidden <= 0)
        return -1;
    if (out_fmt == TKO_OUT_E2M1 && (hidden % 2) != 0)
        return -1;
    if (rows == 0)
        return 0;
    float *col = malloc((size_t)rows * sizeof(float));
    uint8_t *codes = malloc((size_t)rows);
    if (!col || !codes) {
        free(col);
        free(codes);
        return -1;
    }
    for (int64_t j = 0; j < hidden; ++j) {
        for (int64_t r = 0; r < rows; ++r)
            col[r] = y[r * hidden + j];
        float sf = 0.0f;
        uint8_t sb = 0;
        quantize_group(col, rows, scale_fmt, out_fmt, codes, &sf, &sb);
        if (scale_fmt == TKO_SCALE_FP32)
            ((float *)scales)[j] = sf;
        else
            ((uint8_t *)scales)[j] = sb;
        for (int64_t r = 0; r < rows; ++r) {
            if (out_fmt == TKO_OUT_E4M3) {
                q[r * hidden + j] = codes[r];
            } else {
                uint8_t *byte = q + r * (hidden / 2) + j / 2;
                if (j % 2 == 0)
                    *byte = (uint8_t)((*byte & 0xF0) | (codes[r] & 0xF));
                else
                    *byte = (uint8_t)((*byte & 0x0F) | ((codes[r] & 0xF) << 4));
            }
        }
    }
    free(col);
    free(codes);
    return 0;
}

/* ------------------------------------------------------------------ SwiGLU */

/* y[r, i] for one row: clamp (optional), silu(gate) * up * w, evaluated in
 * double and rounded once to fp32. Adds the clamp counts to cnt[0] (gate
 * values above the limit) and cnt[1] (up values outside [-L, L]). */
static void swiglu_row(const uint16_t *xr, int64_t hidden, double w, int use_clamp,
                       float limit, float *y, int64_t *cnt)
{
    double lim = (double)limit;
    for (int64_t i = 0; i < hidden; ++i) {
        double g = bf16_to_double(xr[i]);
        double u = bf16_to_double(xr[hidden + i]);
        if (use_clamp) {
            if (g > lim) {
                g = lim;
                cnt[0] += 1;
            }
            if (u > lim) {
                u = lim;
                cnt[1] += 1;
            } else if (u < -lim) {
                u = -lim;
                cnt[1] += 1;
            }
        }
        double silu = g / (1.0 + exp(-g)); /* g * sigmoid(g) */
        y[i] = (float)(silu * u * w);
    }
}

/* The fused operation, one row at a time.
 *   x        [rows, 2*hidden] bf16 bit patterns, gate half first
 *   w        [rows] fp32 top-k weights, or NULL for weight 1
 *   q, scales as in tko_quant_rows_f32
 *   counts   int64[2], ADDED to (gate clamps, up clamps); may be NULL
 *   y_out    optional [rows, hidden] fp32 copy of the activation
 * Returns 0, or -1 on bad sizes. */
int tko_swiglu_quant(const uint16_t *x, int64_t rows, int64_t hidden, const float *w,
                     int64_t group, int scale_fmt, int out_fmt, int use_clamp,
                     float clamp_limit, uint8_t *q, void *scales, int64_t *counts,
                     float *y_out)
{
    if (group == 0)
        group = hidden;
    if (rows < 0 || hidden <= 0 || group <= 0 || hidden % group != 0 || hidden > 65536)
        return -1;
    float y[65536];
    int64_t cnt[2] = {0, 0};
    int64_t ngroups = hidden / group;
    int64_t q_row = (out_fmt == TKO_OUT_E4M3) ? hidden : hidden / 2;
    size_t s_elem = (scale_fmt == TKO_SCALE_FP32) ? sizeof(float) : 1;
    for (int64_t r = 0; r < rows; ++r) {
        double wr = w ? (double)w[r] : 1.0;
        swiglu_row(x + r * 2 * hidden, hidden, wr, use_clamp, clamp_limit, y, cnt);
        if (y_out)
            memcpy(y_out + r * hidden, y, (size_t)hidden * sizeof(float));
        int rc = tko_quant_rows_f32(y, 1, hidden, group, scale_fmt, out_fmt,
                                    q + r * q_row,
                                    (uint8_t *)scales + (size_t)(r * ngroups) * s_elem);
        if (rc != 0)
            return rc;
    }
    if (counts) {
        counts[0] += cnt[0];
        counts[1] += cnt[1];
    }
    return 0;
}

/* ------------------------------------------------------------ scale layouts */

#define TKO_LAYOUT_ROW 0
#define TKO_LAYOUT_COL 1
#define TKO_LAYOUT_COL_PACKED 2

/* Padded rows per column of a column-major scale layout: 16 bytes worth of
 * scale elements (4 fp32, 16 UE8M0 bytes), or rows rounded up to 4 for the
 * packed words. */
int64_t tko_scale_ld(int layout, int scale_fmt, int64_t rows)
{
    if (layout == TKO_LAYOUT_COL) {
        int64_t per16 = (scale_fmt == TKO_SCALE_FP32) ? 4 : 16;
        return (rows + per16 - 1) / per16 * per16;
    }
    if (layout == TKO_LAYOUT_COL_PACKED)
        return (rows + 3) / 4 * 4;
    return 0;
}

/* Copy row-major scales [rows, groups] into `layout` (the layouts a
 * following FP8 GEMM reads: "TMA-aligned column-major scale factors" and
 * "packed" UE8M0 in the quantization section of "TileLang + TileKernels",
 * zhichai.net/topic/177618740; the exact placement is this library's
 * reading):
 *   column-major: element (t, j) at j * ld + t;
 *   packed (UE8M0): byte k of 32-bit word m * ld + t is the exponent of group
 *   4m + k of row t (little-endian words: byte address 4 (m ld + t) + k).
 * Padding is not written. Returns 0, or -1 for a combination that has no
 * layout. */
int tko_scales_to_layout(const void *row_major, int64_t rows, int64_t groups, int scale_fmt,
                         int layout, void *out)
{
    int64_t ld = tko_scale_ld(layout, scale_fmt, rows);
    for (int64_t t = 0; t < rows; ++t) {
        for (int64_t j = 0; j < groups; ++j) {
            if (scale_fmt == TKO_SCALE_FP32) {
                float v = ((const float *)row_major)[t * groups + j];
                if (layout == TKO_LAYOUT_ROW)
                    ((float *)out)[t * groups + j] = v;
                else if (layout == TKO_LAYOUT_COL)
                    ((float *)out)[j * ld + t] = v;
                else
                    return -1;
            } else {
                uint8_t v = ((const uint8_t *)row_major)[t * groups + j];
                if (layout == TKO_LAYOUT_ROW)
                    ((uint8_t *)out)[t * groups + j] = v;
                else if (layout == TKO_LAYOUT_COL)
                    ((uint8_t *)out)[j * ld + t] = v;
                else if (groups % 4 == 0)
                    ((uint8_t *)out)[4 * ((j / 4) * ld + t) + (j % 4)] = v;
                else
                    return -1;
            }
        }
    }
    return 0;
}

/* SwiGLU backward (not on the pages; the plain derivation of the forward
 * above). With g' = min(g, L), u' = clamp(u, -L, L) when clamping is on,
 * s = sigmoid(g'), silu(g') = g' s and silu'(g') = s (1 + g' (1 - s)):
 *   dgate = dy * w * u' * silu'(g')   where g <= L, else 0
 *   dup   = dy * w * silu(g')         where |u| <= L, else 0
 *   dw    = sum_i dy_i * silu(g'_i) * u'_i
 * all in double; dx [rows, 2*hidden] (gate half first) rounded once to bf16
 * (nearest even), dw [rows] rounded once to fp32 (may be NULL). x and dy are
 * bf16 bit patterns; w may be NULL (weight 1). A clamped element's gradient
 * is +0. Returns 0, or -1 on bad sizes. */
static uint16_t bf16_rne_from_double(double v);

int tko_swiglu_backward(const uint16_t *x, const uint16_t *dy, int64_t rows, int64_t hidden, const float *w,
                        int use_clamp, float clamp_limit, uint16_t *dx, float *dw)
{
    if (rows < 0 || hidden <= 0)
        return -1;
    double lim = (double)clamp_limit;
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t *xr = x + r * 2 * hidden;
        double wr = w ? (double)w[r] : 1.0;
        double acc = 0.0;
        for (int64_t i = 0; i < hidden; ++i) {
            double g = bf16_to_double(xr[i]);
            double u = bf16_to_double(xr[hidden + i]);
            double d = bf16_to_double(dy[r * hidden + i]);
            int pass_g = 1, pass_u = 1;
            if (use_clamp) {
                if (g > lim) {
                    g = lim;
                    pass_g = 0;
                }
                if (u > lim) {
                    u = lim;
                    pass_u = 0;
                } else if (u < -lim) {
                    u = -lim;
                    pass_u = 0;
                }
            }
            double sig = 1.0 / (1.0 + exp(-g));
            double silu = g * sig;
            double dsilu = sig * (1.0 + g * (1.0 - sig));
            dx[r * 2 * hidden + i] = bf16_rne_from_double(pass_g ? d * wr * u * dsilu : 0.0);
            dx[r * 2 * hidden + hidden + i] = bf16_rne_from_double(pass_u ? d * wr * silu : 0.0);
            acc += d * silu * u;
        }
        if (dw)
            dw[r] = (float)acc;
    }
    return 0;
}

/* Codes stored transposed (the fused-transpose output of "TileKernels从入门到
 * 精通", closing section): out[i * ld + t] = q[t * hidden + i] for t < rows,
 * and 0 for rows <= t < ld. q is the row-major E4M3 code matrix [rows, hidden]. */
int tko_codes_transposed(const uint8_t *q, int64_t rows, int64_t hidden, int64_t ld, uint8_t *out)
{
    if (ld < rows)
        return -1;
    for (int64_t i = 0; i < hidden; ++i)
        for (int64_t t = 0; t < ld; ++t)
            out[i * ld + t] = t < rows ? q[t * hidden + i] : 0;
    return 0;
}

/* ------------------------------------------------------ top-k combine (reduce) */

/* RNE of a double to bf16 (the upper half of an fp32), through fp32: a double
 * rounds to fp32 first only if the fp32 rounding cannot create a bf16 tie, so
 * here the bf16 value is found directly: the nearest bf16 by exhaustive
 * comparison of the two bf16 neighbours of v, ties to the even mantissa. NaN
 * and infinities are outside the contract. */
static uint16_t bf16_rne_from_double(double v)
{
    float f = (float)v;                       /* the bf16 neighbours bracket f's */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t lo_bits = u & 0xffff0000u;        /* toward zero in magnitude */
    uint32_t hi_bits = lo_bits + 0x10000u;     /* next bf16 away from zero */
    float lo, hi;
    memcpy(&lo, &lo_bits, sizeof lo);
    memcpy(&hi, &hi_bits, sizeof hi);
    double dlo = fabs(v - (double)lo), dhi = fabs(v - (double)hi);
    uint32_t pick;
    if (dlo < dhi)
        pick = lo_bits;
    else if (dhi < dlo)
        pick = hi_bits;
    else
        pick = ((lo_bits >> 16) & 1) ? hi_bits : lo_bits;
    return (uint16_t)(pick >> 16);
}

/* The weighted top-k combine after the expert GEMMs ("TileKernels从入门到精通",
 * zhichai.net/topic/177618752, ch.3 "结算中心的减法工程" and "动态寻址": routing
 * weights, quantization factors and a global scale applied while gathering the
 * expert rows through token_topk_to_pos, one read and one write):
 *   out[t, i] = gs * sum_{k < K, pos[t,k] >= 0} w[t,k] * deq(y[pos[t,k], i]),
 * with deq(y) = y for bf16 expert rows (y_fp8 == NULL) or, for E4M3 codes,
 * decode(code) * y_scale[row, i / 128]. The sum is taken in double and
 * rounded once to bf16 (round to nearest even).
 *   y_bf16   [R, hidden] bf16 bits, or NULL when y_fp8 is given
 *   y_fp8    [R, hidden] E4M3 codes, y_scale [R, hidden / 128] fp32
 *   pos      [T, K] int32 row indices into y (-1: empty slot)
 *   w        [T, K] fp32
 *   out      [T, hidden] bf16 bits
 * Returns 0, or -1 on a bad argument (a position outside [0, R)). */
int tko_moe_reduce(const uint16_t *y_bf16, const uint8_t *y_fp8, const float *y_scale, int64_t R,
                   int64_t hidden, const int32_t *pos, const float *w, int64_t T, int64_t K, float gs,
                   uint16_t *out)
{
    if (hidden % 128 != 0 && y_fp8)
        return -1;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t i = 0; i < hidden; ++i) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                int32_t r = pos[t * K + k];
                if (r < 0)
                    continue;
                if (r >= R)
                    return -1;
                double v;
                if (y_fp8)
                    v = tko_e4m3_decode(y_fp8[r * hidden + i]) * (double)y_scale[r * (hidden / 128) + i / 128];
                else
                    v = bf16_to_double(y_bf16[r * hidden + i]);
                acc += (double)w[t * K + k] * v;
            }
            out[t * hidden + i] = bf16_rne_from_double((double)gs * acc);
        }
    }
    return 0;
}
