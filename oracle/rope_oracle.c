/*
 * rope_oracle.c -- plain, slow, single-threaded fp64 CPU oracle for rotary
 * position embedding (RoPE).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg use this file.  It shares no code, header, table or
 * constant with the CUDA library and must never be reached from the product
 * path.
 *
 * Sources (web pages; cited by page title and section):
 *   [RKO]  "Rotary Embedding (RoPE) Kernel Optimization" (skillmd.com),
 *          sections "Overview", "Core Technique / Paired Element Layout",
 *          "Common Pitfalls".
 *   [UNS]  "How Unsloth Optimizes RoPE Embedding Computations in Triton
 *          Kernels", sections "Triton Kernel Architecture for RoPE",
 *          "Dynamic Block Sizing and GPU Occupancy", "Support for Custom
 *          Position IDs", "Usage Examples", "Frequently Asked Questions".
 *   [RET]  "rotary-embedding-torch", sections "flash_attn_with_rotary /
 *          Input Tensor Shapes" and "RotaryEmbedding / Key Parameters".
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes of the repository):
 *   - frequency of pair i is theta^(-2i/rotary_dim) (the pages name theta,
 *     default 10000, but do not print the formula);
 *   - interpolate_factor f scales positions as m / f;
 *   - the cos/sin table is half width, [rows, rotary_dim/2];
 *   - position index -1 marks an unrotated token (pass-through);
 *   - outputs are rounded once, from fp64, to the output type (RNE).
 *
 * Parity pins: every function here is checked in tests/test_oracle_pins.py
 * against closed forms, library routines or brute force; none is unpinned.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif

/* Element types understood by the oracle.  ORACLE_F64 exists only so the
 * invariant tests can run the rotation with no rounding of the output. */
enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F16 = 2, ORACLE_F64 = 3 };
/* Pair layouts [RKO, Core Technique / Paired Element Layout]. */
enum { ORACLE_SPLIT_HALF = 0, ORACLE_INTERLEAVED = 1 };
/* Return codes. */
enum { ORACLE_OK = 0, ORACLE_BAD_ARG = 1, ORACLE_POS_OUT_OF_RANGE = 4 };
/* frequency modes (freqs_for) */
enum { ORACLE_FREQ_LANG = 0, ORACLE_FREQ_PIXEL = 1, ORACLE_FREQ_CONSTANT = 2 };

/* ------------------------------------------------------------------------ */
/* Exact decoding of the 16-bit storage types into fp64.                     */
/* ------------------------------------------------------------------------ */

/* bfloat16 is the upper half of an IEEE binary32; widening is exact. */
double oracle_bf16_to_f64(uint16_t bits)
{
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int e = (bits >> 10) & 0x1f;
    int frac = bits & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)frac, -24);                 /* zero / subnormal */
    else if (e == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), e - 25);     /* 1.frac * 2^(e-15) */
    return sign ? -v : v;
}

/* ------------------------------------------------------------------------ */
/* Round-to-nearest-even directly from fp64 (one rounding, no detour via    */
/* fp32).  Generic over a binary format with p significand bits (implicit   */
/* bit included), minimum normal exponent emin and maximum exponent emax.   */
/* Returns the rounded magnitude as an fp64 value (may be +inf).            */
/* ------------------------------------------------------------------------ */
static double rne_magnitude(double a, int p, int emin, int emax)
{
    int E;
    double q, n, v, maxfin;
    if (a == 0.0 || isinf(a))
        return a;
    (void)frexp(a, &E);            /* a = m * 2^E, m in [0.5, 1) */
    E -= 1;                        /* a in [2^E, 2^(E+1)) */
    if (E < emin)
        E = emin;                  /* subnormal range: fixed quantum */
    q = ldexp(1.0, E - (p - 1));   /* spacing of the format in this binade */
    n = nearbyint(a / q);          /* a / q is exact (power-of-two scale); ties to even */
    v = n * q;
    maxfin = ldexp(ldexp(1.0, p) - 1.0, emax - (p - 1));
    if (v > maxfin)
        return INFINITY;
    return v;
}

uint16_t oracle_f64_to_bf16(double y)
{
    /* bfloat16: p = 8, emin = -126, emax = 127; same exponent field as binary32. */
    int neg = signbit(y) ? 1 : 0;
    double v;
    float f;
    uint32_t w;
    if (isnan(y))
        return (uint16_t)(0x7fc0 | (neg << 15));
    v = rne_magnitude(fabs(y), 8, -126, 127);
    f = (float)v;                  /* exact: v is a bfloat16 value (or inf) */
    memcpy(&w, &f, sizeof w);
    return (uint16_t)((w >> 16) | (uint32_t)(neg << 15));
}

uint16_t oracle_f64_to_f16(double y)
{
    /* binary16: p = 11, emin = -14, emax = 15. */
    int neg = signbit(y) ? 1 : 0;
    double v;
    uint16_t out;
    if (isnan(y))
        return (uint16_t)(0x7e00 | (neg << 15));
    v = rne_magnitude(fabs(y), 11, -14, 15);
    if (isinf(v)) {
        out = 0x7c00;
    } else if (v < ldexp(1.0, -14)) {
        out = (uint16_t)ldexp(v, 24);                 /* subnormal: v = frac * 2^-24 */
    } else {
        int E;
        (void)frexp(v, &E);
        E -= 1;                                       /* v in [2^E, 2^(E+1)) */
        out = (uint16_t)(((E + 15) << 10) | ((int)(ldexp(v, 10 - E)) - 1024));
    }
    return (uint16_t)(out | (neg << 15));
}

/* C's double -> float conversion rounds to nearest even under the default
 * rounding mode, which the oracle never changes. */
float oracle_f64_to_f32(double y) { return (float)y; }

/* ------------------------------------------------------------------------ */
/* Frequencies and the cos/sin table.                                        */
/*   [RET, RotaryEmbedding / Key Parameters]: theta is the base of the       */
/*   frequencies (default 10000); interpolate_factor scales positions        */
/*   (default 1.0).  [RKO, Common Pitfalls]: cos/sin are [seq_len, D/2].      */
/* ------------------------------------------------------------------------ */

/* Inverse frequency of pair i: theta^(-2i / rotary_dim). */
double oracle_inv_freq(double theta, int32_t rotary_dim, int32_t i)
{
    return pow(theta, -(2.0 * (double)i) / (double)rotary_dim);
}

/* Rotation angle of pair i at position m, positions scaled by 1/f. */
double oracle_angle(int64_t m, double interpolate_factor, double inv_freq)
{
    return ((double)m / interpolate_factor) * inv_freq;
}

/* fp64 tables cos/sin [max_pos, rotary_dim/2], row m = position m. */
int oracle_tables_f64(double theta, int32_t rotary_dim, int64_t max_pos,
                      double interpolate_factor, double *cos_out, double *sin_out)
{
    int32_t h, i;
    int64_t m;
    if (theta <= 0.0 || interpolate_factor <= 0.0 || rotary_dim < 2 ||
        (rotary_dim & 1) || max_pos < 0 || !cos_out || !sin_out)
        return ORACLE_BAD_ARG;
    h = rotary_dim / 2;
    for (m = 0; m < max_pos; ++m) {
        for (i = 0; i < h; ++i) {
            double a = oracle_angle(m, interpolate_factor,
                                    oracle_inv_freq(theta, rotary_dim, i));
            cos_out[m * h + i] = cos(a);
            sin_out[m * h + i] = sin(a);
        }
    }
    return ORACLE_OK;
}

/* The same table, each entry rounded once to fp32 (the stored precision). */
int oracle_tables_f32(double theta, int32_t rotary_dim, int64_t max_pos,
                      double interpolate_factor, float *cos_out, float *sin_out)
{
    int32_t h, i;
    int64_t m;
    if (theta <= 0.0 || interpolate_factor <= 0.0 || rotary_dim < 2 ||
        (rotary_dim & 1) || max_pos < 0 || !cos_out || !sin_out)
        return ORACLE_BAD_ARG;
    h = rotary_dim / 2;
    for (m = 0; m < max_pos; ++m) {
        for (i = 0; i < h; ++i) {
            double a = oracle_angle(m, interpolate_factor,
                                    oracle_inv_freq(theta, rotary_dim, i));
            cos_out[m * h + i] = oracle_f64_to_f32(cos(a));
            sin_out[m * h + i] = oracle_f64_to_f32(sin(a));
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Frequency modes, row positions and the XPOS scale.                        */
/*   [RET, RotaryEmbedding / Key Parameters] names the modes freqs_for =     */
/*   'lang' | 'pixel' | 'constant' and use_xpos, but prints no formula.      */
/*   The formulas restated here are the published ones:                      */
/*   - lang: theta^(-2i/rotary_dim) (as above);                              */
/*   - pixel: the Fourier features of Jaegle et al., "Perceiver: General     */
/*     Perception with Iterative Attention" (ICML 2021): frequencies spaced  */
/*     linearly from 1 to max_freq/2, times pi, for positions in [-1, 1];    */
/*   - constant: every pair at frequency 1;                                  */
/*   - XPOS: Sun et al., "A Length-Extrapolatable Transformer" (2022): pair  */
/*     i carries zeta_i = (2i/rotary_dim + gamma) / (1 + gamma); the query   */
/*     at position n is scaled by zeta_i^(n/B) and the key by zeta_i^(-n/B), */
/*     so a query-key product depends on the distance only (gamma = 0.4,     */
/*     B = 512 in the paper).  A common centre c (n - c) cancels likewise.   */
/* ------------------------------------------------------------------------ */

/* Frequency of pair i (h = rotary_dim/2 pairs). */
double oracle_freq_ex(int32_t mode, double theta, double max_freq, int32_t rotary_dim, int32_t i)
{
    const int32_t h = rotary_dim / 2;
    if (mode == ORACLE_FREQ_PIXEL) {
        if (h == 1)
            return M_PI;
        return M_PI * (1.0 + (double)i * (max_freq / 2.0 - 1.0) / (double)(h - 1));
    }
    if (mode == ORACLE_FREQ_CONSTANT)
        return 1.0;
    return oracle_inv_freq(theta, rotary_dim, i);
}

/* Position of table row m. */
double oracle_position(int64_t m, double pos_offset, double pos_divisor)
{
    return pos_offset + (double)m / pos_divisor;
}

/* XPOS scale of pair i at position p: zeta_i^(sign * (p - center) / base). */
double oracle_xpos_scale(int32_t rotary_dim, int32_t i, double p, int32_t sign, double base,
                         double gamma, double center)
{
    const double zeta = (2.0 * (double)i / (double)rotary_dim + gamma) / (1.0 + gamma);
    return pow(zeta, (double)sign * (p - center) / base);
}

static int tables_ex_args_ok(int32_t mode, double theta, double max_freq, int32_t rotary_dim,
                             int64_t rows, double pos_offset, double pos_divisor, int32_t xpos_sign,
                             double xpos_base, double xpos_gamma, double xpos_center)
{
    if (mode != ORACLE_FREQ_LANG && mode != ORACLE_FREQ_PIXEL && mode != ORACLE_FREQ_CONSTANT)
        return 0;
    if (rotary_dim < 2 || (rotary_dim & 1) || rows < 0)
        return 0;
    if (mode == ORACLE_FREQ_LANG && !(theta > 0.0 && isfinite(theta)))
        return 0;
    if (mode == ORACLE_FREQ_PIXEL && !(max_freq > 0.0 && isfinite(max_freq)))
        return 0;
    if (!isfinite(pos_offset) || !(pos_divisor > 0.0 && isfinite(pos_divisor)))
        return 0;
    if (xpos_sign < -1 || xpos_sign > 1)
        return 0;
    if (xpos_sign != 0 && !(xpos_base > 0.0 && isfinite(xpos_base) && xpos_gamma > 0.0 &&
                            isfinite(xpos_gamma) && isfinite(xpos_center)))
        return 0;
    return 1;
}

/* fp64 tables [rows, rotary_dim/2]: row m holds, for pair i,
 *   s * cos(p_m * w_i) and s * sin(p_m * w_i),
 * p_m = pos_offset + m / pos_divisor, w_i the mode's frequency, and s the XPOS
 * scale (1 when xpos_sign == 0). */
int oracle_tables_ex_f64(int32_t mode, double theta, double max_freq, int32_t rotary_dim,
                         int64_t rows, double pos_offset, double pos_divisor, int32_t xpos_sign,
                         double xpos_base, double xpos_gamma, double xpos_center, double *cos_out,
                         double *sin_out)
{
    int32_t h, i;
    int64_t m;
    if (!tables_ex_args_ok(mode, theta, max_freq, rotary_dim, rows, pos_offset, pos_divisor,
                           xpos_sign, xpos_base, xpos_gamma, xpos_center) ||
        !cos_out || !sin_out)
        return ORACLE_BAD_ARG;
    h = rotary_dim / 2;
    for (m = 0; m < rows; ++m) {
        const double p = oracle_position(m, pos_offset, pos_divisor);
        for (i = 0; i < h; ++i) {
            const double a = p * oracle_freq_ex(mode, theta, max_freq, rotary_dim, i);
            const double sc = xpos_sign == 0 ? 1.0
                                             : oracle_xpos_scale(rotary_dim, i, p, xpos_sign,
                                                                 xpos_base, xpos_gamma, xpos_center);
            cos_out[m * h + i] = sc * cos(a);
            sin_out[m * h + i] = sc * sin(a);
        }
    }
    return ORACLE_OK;
}

/* The same tables, each entry rounded once to fp32. */
int oracle_tables_ex_f32(int32_t mode, double theta, double max_freq, int32_t rotary_dim,
                         int64_t rows, double pos_offset, double pos_divisor, int32_t xpos_sign,
                         double xpos_base, double xpos_gamma, double xpos_center, float *cos_out,
                         float *sin_out)
{
    int32_t h, i;
    int64_t m;
    if (!tables_ex_args_ok(mode, theta, max_freq, rotary_dim, rows, pos_offset, pos_divisor,
                           xpos_sign, xpos_base, xpos_gamma, xpos_center) ||
        !cos_out || !sin_out)
        return ORACLE_BAD_ARG;
    h = rotary_dim / 2;
    for (m = 0; m < rows; ++m) {
        const double p = oracle_position(m, pos_offset, pos_divisor);
        for (i = 0; i < h; ++i) {
            const double a = p * oracle_freq_ex(mode, theta, max_freq, rotary_dim, i);
            const double sc = xpos_sign == 0 ? 1.0
                                             : oracle_xpos_scale(rotary_dim, i, p, xpos_sign,
                                                                 xpos_base, xpos_gamma, xpos_center);
            cos_out[m * h + i] = oracle_f64_to_f32(sc * cos(a));
            sin_out[m * h + i] = oracle_f64_to_f32(sc * sin(a));
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Rotation of one head row.                                                 */
/*   [RKO, Overview]: (x1, x2) -> (x1 cos - x2 sin, x1 sin + x2 cos).        */
/*   [RKO, Paired Element Layout]: split-half pairs (x[i], x[i + D/2]),      */
/*   interleaved pairs (x[2i], x[2i+1]).                                     */
/*   [RET, RotaryEmbedding / Key Parameters]: only the first rotary_dim      */
/*   features are rotated; the rest of the row passes through.               */
/*   [UNS, Frequently Asked Questions]: the backward pass is the same        */
/*   rotation with the backward flag set, i.e. by the negated angle.         */
/* x and y hold D fp64 values; c_row and s_row hold rotary_dim/2 values.     */
/* ------------------------------------------------------------------------ */
void oracle_rotate_row_f64(const double *x, double *y, int32_t D, int32_t rotary_dim,
                           int32_t layout, const double *c_row, const double *s_row,
                           int32_t backward)
{
    int32_t h = rotary_dim / 2, i, d;
    for (i = 0; i < h; ++i) {
        int32_t i1 = (layout == ORACLE_INTERLEAVED) ? 2 * i : i;
        int32_t i2 = (layout == ORACLE_INTERLEAVED) ? 2 * i + 1 : i + h;
        double c = c_row[i];
        double s = backward ? -s_row[i] : s_row[i];
        double x1 = x[i1], x2 = x[i2];
        y[i1] = x1 * c - x2 * s;
        y[i2] = x1 * s + x2 * c;
    }
    for (d = rotary_dim; d < D; ++d)
        y[d] = x[d];
}

/* ------------------------------------------------------------------------ */
/* Whole-tensor apply.                                                       */
/*   Tensor layout [B,H,S,D] (seq_before_head = 0) as in [UNS, Usage         */
/*   Examples] and [RET, Input Tensor Shapes], or [B,S,H,D]                   */
/*   (seq_before_head = 1) as in [RET, RotaryEmbedding / Key Parameters].    */
/*   Position of token (b, s): pos_idx[s] when pos_idx is given ([UNS,       */
/*   Support for Custom Position IDs]; [RET, Input Tensor Shapes]:           */
/*   rotary_pos_emb_indices (seq_len,)), else s.  -1 = not rotated (the      */
/*   pos_mask of [RET, flash_attn_with_rotary]): the row's bits are copied.  */
/*   cos_tab/sin_tab: fp64 [table_rows, rotary_dim/2].                       */
/*   x_in: elements of type dtype (bits); y_bits: same type, may be NULL;    */
/*   y_f64: fp64 result before the final rounding, may be NULL.              */
/* ------------------------------------------------------------------------ */
static size_t elem_size(int32_t dtype)
{
    switch (dtype) {
    case ORACLE_F32: return 4;
    case ORACLE_BF16: return 2;
    case ORACLE_F16: return 2;
    case ORACLE_F64: return 8;
    default: return 0;
    }
}

static double load_elem(const void *base, int32_t dtype, int64_t k)
{
    switch (dtype) {
    case ORACLE_F32: return (double)((const float *)base)[k];
    case ORACLE_BF16: return oracle_bf16_to_f64(((const uint16_t *)base)[k]);
    case ORACLE_F16: return oracle_f16_to_f64(((const uint16_t *)base)[k]);
    default: return ((const double *)base)[k];
    }
}

static void store_elem(void *base, int32_t dtype, int64_t k, double v)
{
    switch (dtype) {
    case ORACLE_F32: ((float *)base)[k] = oracle_f64_to_f32(v); break;
    case ORACLE_BF16: ((uint16_t *)base)[k] = oracle_f64_to_bf16(v); break;
    case ORACLE_F16: ((uint16_t *)base)[k] = oracle_f64_to_f16(v); break;
    default: ((double *)base)[k] = v; break;
    }
}

int oracle_apply(int32_t dtype, const void *x_in, void *y_bits, double *y_f64,
                 int64_t B, int32_t H, int64_t S, int32_t D, int32_t rotary_dim,
                 int32_t layout, int32_t seq_before_head, int32_t backward,
                 const int32_t *pos_idx, const double *cos_tab, const double *sin_tab,
                 int64_t table_rows)
{
    size_t es = elem_size(dtype);
    int32_t h = rotary_dim / 2, d;
    int64_t b, s, hh;
    double xrow[4096], yrow[4096];
    int status = ORACLE_OK;

    if (!es || !x_in || B < 0 || H < 0 || S < 0 || D <= 0 || D > 4096 ||
        rotary_dim < 2 || (rotary_dim & 1) || rotary_dim > D ||
        (layout != ORACLE_SPLIT_HALF && layout != ORACLE_INTERLEAVED) ||
        !cos_tab || !sin_tab || table_rows < 0)
        return ORACLE_BAD_ARG;
    if (!pos_idx && S > table_rows)
        return ORACLE_BAD_ARG;

    for (b = 0; b < B; ++b) {
        for (hh = 0; hh < H; ++hh) {
            for (s = 0; s < S; ++s) {
                int64_t row = seq_before_head ? ((b * S + s) * H + hh) * D
                                              : ((b * H + hh) * S + s) * D;
                int64_t r = pos_idx ? (int64_t)pos_idx[s] : s;
                int unrotated = (r == -1);
                if (!unrotated && (r < 0 || r >= table_rows)) {
                    status = ORACLE_POS_OUT_OF_RANGE;   /* rejected: row left as is */
                    unrotated = 1;
                }
                if (unrotated) {
                    /* pass-through: no arithmetic, bits copied */
                    if (y_bits)
                        memcpy((char *)y_bits + row * es, (const char *)x_in + row * es,
                               (size_t)D * es);
                    if (y_f64)
                        for (d = 0; d < D; ++d)
                            y_f64[row + d] = load_elem(x_in, dtype, row + d);
                    continue;
                }
                for (d = 0; d < D; ++d)
                    xrow[d] = load_elem(x_in, dtype, row + d);
                oracle_rotate_row_f64(xrow, yrow, D, rotary_dim, layout,
                                      cos_tab + r * h, sin_tab + r * h, backward);
                for (d = 0; d < D; ++d) {
                    if (y_f64)
                        y_f64[row + d] = yrow[d];
                    if (y_bits) {
                        if (d < rotary_dim)
                            store_elem(y_bits, dtype, row + d, yrow[d]);
                        else            /* tail: bits copied, never re-rounded */
                            memcpy((char *)y_bits + (row + d) * es,
                                   (const char *)x_in + (row + d) * es, es);
                    }
                }
            }
        }
    }
    return status;
}
