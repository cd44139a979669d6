/*
 * rowsoftmax_oracle.c -- plain, slow, obviously correct CPU row-wise softmax.
 *
 * TEST INFRASTRUCTURE ONLY (same rules as rmsnorm_oracle.c: loaded only by
 * the tests, the smoke check and the benchmark's CPU-baseline legs; shares
 * nothing with the CUDA library).
 *
 * The compiler write-up ("A hackable Python ML compiler, part 2") names
 * softmax-style small reductions among the ops its generated kernels win on
 * but prints no formula for them.  The plain definition is used, in the
 * numerically stable form that subtracts the row maximum first (the same
 * value in exact arithmetic):
 *
 *     for every row r:
 *         m[r]   = max_j x[r,j]
 *         e[r,j] = exp(x[r,j] - m[r])
 *         s[r]   = sum_j e[r,j]
 *         y[r,j] = e[r,j] / s[r]
 *
 * binary64 throughout, libm exp, a sequential sum, a true division.  IEEE
 * semantics decide the special cases: a NaN anywhere makes its row NaN;
 * a row of -inf gives (-inf) - (-inf) = NaN everywhere; a +inf element gives
 * NaN; -inf elements of an otherwise finite row give exactly 0.
 * bf16 inputs are decoded exactly and each output is rounded once (the
 * encoder of rmsnorm_oracle.c).
 */
#include <math.h>
#include <stdint.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1

double oracle_bf16_to_f64(uint16_t b);
uint16_t oracle_f64_to_bf16_rne(double v);

static int check(const void* x, const void* y, int64_t rows, int64_t cols)
{
    if (rows < 0 || cols <= 0) return ORACLE_ERR_ARG;
    if (rows > 0 && (x == 0 || y == 0)) return ORACLE_ERR_ARG;
    return ORACLE_OK;
}

/* One row: max, exponentials, sum, division -- the four steps in order. */
static void softmax_row(const double* x, double* y, int64_t cols)
{
    double m = x[0];
    for (int64_t j = 1; j < cols; ++j)
        if (x[j] > m) m = x[j];
    double s = 0.0;
    for (int64_t j = 0; j < cols; ++j) {
        y[j] = exp(x[j] - m);
        s += y[j];
    }
    for (int64_t j = 0; j < cols; ++j) y[j] = y[j] / s;
}

int oracle_rowsoftmax_f64(const double* x, double* y, int64_t rows, int64_t cols)
{
    int st = check(x, y, rows, cols);
    if (st) return st;
    for (int64_t r = 0; r < rows; ++r) softmax_row(x + r * cols, y + r * cols, cols);
    return ORACLE_OK;
}

/* binary32 in (widened exactly), binary64 out. */
int oracle_rowsoftmax_f32(const float* x, double* y, int64_t rows, int64_t cols)
{
    int st = check(x, y, rows, cols);
    if (st) return st;
    for (int64_t r = 0; r < rows; ++r) {
        double* yr = y + r * cols;
        for (int64_t j = 0; j < cols; ++j) yr[j] = (double)x[r * cols + j];
        softmax_row(yr, yr, cols);
    }
    return ORACLE_OK;
}

/* bfloat16 bits in; binary64 out (y64) and its single RNE rounding (y16). */
int oracle_rowsoftmax_bf16(const uint16_t* x, double* y64, uint16_t* y16,
                           int64_t rows, int64_t cols)
{
    int st = check(x, y64, rows, cols);
    if (st) return st;
    for (int64_t r = 0; r < rows; ++r) {
        double* yr = y64 + r * cols;
        for (int64_t j = 0; j < cols; ++j) yr[j] = oracle_bf16_to_f64(x[r * cols + j]);
        softmax_row(yr, yr, cols);
        if (y16)
            for (int64_t j = 0; j < cols; ++j)
                y16[r * cols + j] = oracle_f64_to_bf16_rne(yr[j]);
    }
    return ORACLE_OK;
}
