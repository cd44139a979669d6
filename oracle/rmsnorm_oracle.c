/*
 * rmsnorm_oracle.c -- plain, slow, obviously correct CPU RMSNorm forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark load this code.  It shares no source,
 * header, helper or table with the CUDA library and never calls it.
 *
 * What it computes (page "A hackable Python ML compiler, part 2"
 * (bittide.aicompass.dev, deplodock write-up), the RMSNorm Loop-IR listing and
 * the epilogue of the generated RMSNorm kernel):
 *
 *     for every row r:
 *         ms[r]   = (1/H) * sum_{j<H} x[r,j]^2          (mean of squares)
 *         rstd[r] = 1 / sqrt(ms[r] + eps)              (eps inside the root)
 *         y[r,j]  = (x[r,j] * rstd[r]) * w[j]          (scale, then weight)
 *
 * Everything is carried in IEEE binary64: inputs are widened exactly, the
 * sum runs sequentially over j, the root is the correctly rounded libm
 * sqrt followed by a true division (no approximate reciprocal square root).
 * No SIMD, no -ffast-math, no reordering beyond the definition above.
 *
 * Fused epilogue (page "CuTe DSL JIT argument generation", section 2.3, and
 * the CuTe DSL control-flow page, section 7: a compile-time epilogue_op, e.g.
 * an optional ReLU, applied to each output value before it is stored):
 * oracle_apply_epilogue_f64 maps every binary64 output v to
 *     kind 0: v,   kind 1: alpha * v,   kind 2: ReLU(v) = v if v > 0 or v is
 *     NaN, else +0,
 * and the bf16 result is the single rounding of the epilogue's output.
 *
 * bfloat16 (the pages never mention it; the plain reading used here):
 * inputs are decoded exactly to binary64, the whole computation above runs
 * in binary64, and the result is rounded ONCE to bfloat16 with
 * round-to-nearest, ties-to-even.  The encoder and decoder are written from
 * the bfloat16 definition (1 sign bit, 8 exponent bits with bias 127,
 * 7 fraction bits; the upper half of an IEEE binary32).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1

/* ---- bfloat16 <-> binary64 --------------------------------------------- */

/* Exact decode: value = (-1)^s * 2^(e-127) * (1 + f/128) for 0 < e < 255,
 * (-1)^s * 2^-126 * (f/128) for e == 0, +-inf / NaN for e == 255. */
double oracle_bf16_to_f64(uint16_t b)
{
    int s = (b >> 15) & 1;
    int e = (b >> 7) & 0xFF;
    int f = b & 0x7F;
    double v;
    if (e == 0xFF) {
        v = (f == 0) ? INFINITY : NAN;
    } else if (e == 0) {
        v = ldexp((double)f, -126 - 7);
    } else {
        v = ldexp((double)(128 + f), e - 127 - 7);
    }
    return s ? -v : v;
}

/* Round half to even of a non-negative binary64 n (exact: n - floor(n) is
 * representable because floor(n) shares n's leading bits). */
static double round_half_even(double n)
{
    double fl = floor(n);
    double frac = n - fl;
    if (frac > 0.5) return fl + 1.0;
    if (frac < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* binary64 -> bfloat16, round-to-nearest-even, one rounding.
 * NaN -> canonical quiet NaN 0x7FC0 (sign kept); overflow -> +-inf. */
uint16_t oracle_f64_to_bf16_rne(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v)) return (uint16_t)(sign | 0x7FC0u);
    double a = fabs(v);
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0) return sign;

    int e2;
    frexp(a, &e2);            /* a = m * 2^e2, m in [0.5, 1) */
    int e = e2 - 1;           /* a in [2^e, 2^(e+1)) */
    if (e < -126) e = -126;   /* subnormal range shares the quantum 2^-133 */
    double q_exp = (double)(e - 7);
    double n = ldexp(a, -(int)q_exp);   /* a / 2^(e-7): exact scaling */
    double r = round_half_even(n);      /* 0 <= r <= 256 */

    uint32_t bits;
    if (a < ldexp(1.0, -126)) {
        /* subnormal: the encoding is r itself; r == 128 lands on the
         * smallest normal 0x0080, which is the correct carry */
        bits = (uint32_t)r;
    } else {
        /* normal: biased exponent e+127, fraction r-128; r == 256 carries
         * into the next binade through the addition */
        bits = ((uint32_t)(e + 127) << 7) + ((uint32_t)r - 128u);
    }
    if (bits >= 0x7F80u) bits = 0x7F80u;  /* rounded past the largest finite */
    return (uint16_t)(sign | bits);
}

/* ---- RMSNorm ------------------------------------------------------------ */

static int check_args(const void* x, const void* w, const void* y,
                      int64_t rows, int64_t hidden)
{
    if (rows < 0 || hidden <= 0) return ORACLE_ERR_ARG;
    if (rows > 0 && (x == 0 || w == 0 || y == 0)) return ORACLE_ERR_ARG;
    return ORACLE_OK;
}

/* One row in binary64: the three steps of the definition in order. */
static void rms_row_f64(const double* xr, const double* w, double* yr,
                        int64_t hidden, double eps)
{
    double acc = 0.0;
    for (int64_t j = 0; j < hidden; ++j) acc += xr[j] * xr[j];
    double ms = acc / (double)hidden;
    double rstd = 1.0 / sqrt(ms + eps);
    for (int64_t j = 0; j < hidden; ++j) yr[j] = (xr[j] * rstd) * w[j];
}

/* binary64 in, binary64 out (used by the pins and as the common core). */
int oracle_rmsnorm_f64(const double* x, const double* w, double* y,
                       int64_t rows, int64_t hidden, double eps)
{
    int st = check_args(x, w, y, rows, hidden);
    if (st) return st;
    for (int64_t r = 0; r < rows; ++r)
        rms_row_f64(x + r * hidden, w, y + r * hidden, hidden, eps);
    return ORACLE_OK;
}

/* binary32 in, binary64 out: every input widened exactly before use. */
int oracle_rmsnorm_f32(const float* x, const float* w, double* y,
                       int64_t rows, int64_t hidden, double eps)
{
    int st = check_args(x, w, y, rows, hidden);
    if (st) return st;
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * hidden;
        double* yr = y + r * hidden;
        double acc = 0.0;
        for (int64_t j = 0; j < hidden; ++j) {
            double v = (double)xr[j];
            acc += v * v;
        }
        double ms = acc / (double)hidden;
        double rstd = 1.0 / sqrt(ms + eps);
        for (int64_t j = 0; j < hidden; ++j)
            yr[j] = ((double)xr[j] * rstd) * (double)w[j];
    }
    return ORACLE_OK;
}

/* bfloat16 bits in; binary64 values out (y64, may be NULL) and the single
 * RNE rounding of each to bfloat16 bits (y16, may be NULL; not both). */
int oracle_rmsnorm_bf16(const uint16_t* x, const uint16_t* w, double* y64,
                        uint16_t* y16, int64_t rows, int64_t hidden, double eps)
{
    int st = check_args(x, w, (y64 ? (const void*)y64 : (const void*)y16),
                        rows, hidden);
    if (st) return st;
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* xr = x + r * hidden;
        double acc = 0.0;
        for (int64_t j = 0; j < hidden; ++j) {
            double v = oracle_bf16_to_f64(xr[j]);
            acc += v * v;
        }
        double ms = acc / (double)hidden;
        double rstd = 1.0 / sqrt(ms + eps);
        for (int64_t j = 0; j < hidden; ++j) {
            double v = (oracle_bf16_to_f64(xr[j]) * rstd)
                       * oracle_bf16_to_f64(w[j]);
            if (y64) y64[r * hidden + j] = v;
            if (y16) y16[r * hidden + j] = oracle_f64_to_bf16_rne(v);
        }
    }
    return ORACLE_OK;
}

/* ---- epilogue ----------------------------------------------------------- */

int oracle_apply_epilogue_f64(double* y, int64_t n, int kind, double alpha)
{
    if (n < 0 || (n > 0 && y == 0) || kind < 0 || kind > 2) return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < n; ++i) {
        double v = y[i];
        if (kind == 1) {
            v = alpha * v;
        } else if (kind == 2) {
            v = (v > 0.0 || isnan(v)) ? v : 0.0;
        }
        y[i] = v;
    }
    return ORACLE_OK;
}

/* Round every element once, binary64 -> bfloat16 (round to nearest even). */
int oracle_f64_to_bf16_array(const double* v, uint16_t* out, int64_t n)
{
    if (n < 0 || (n > 0 && (v == 0 || out == 0))) return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f64_to_bf16_rne(v[i]);
    return ORACLE_OK;
}

/* Per-row mean of squares and reciprocal root, exposed so that tests can
 * check the intermediate quantities of the definition one by one. */
int oracle_rmsnorm_stats_f64(const double* x, double* ms, double* rstd,
                             int64_t rows, int64_t hidden, double eps)
{
    if (rows < 0 || hidden <= 0) return ORACLE_ERR_ARG;
    if (rows > 0 && (x == 0 || ms == 0 || rstd == 0)) return ORACLE_ERR_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        double acc = 0.0;
        for (int64_t j = 0; j < hidden; ++j)
            acc += x[r * hidden + j] * x[r * hidden + j];
        ms[r] = acc / (double)hidden;
        rstd[r] = 1.0 / sqrt(ms[r] + eps);
    }
    return ORACLE_OK;
}
