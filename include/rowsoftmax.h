/*
 * rowsoftmax.h -- C ABI of librmsnorm's row-wise softmax (same library,
 * same status codes and conventions as rmsnorm.h).
 *
 * For every row r of a row-major matrix x with `cols` columns:
 *
 *     m[r]   = max_j x[r,j]
 *     y[r,j] = exp(x[r,j] - m[r]) / sum_k exp(x[r,k] - m[r])
 *
 * The compiler write-up "A hackable Python ML compiler, part 2" lists such
 * small reductions (softmax inside SDPA) among the ops its generated kernels
 * win on, without printing a formula; this is the plain definition in the
 * stable form.  fp32 arithmetic: exp(x - m) as a base-2 exponential of
 * (x - m) * log2(e) (CUDA's exp2f for fp32 rows, one SFU instruction for bf16
 * rows), the offset m * log2(e) fused into one FMA for rows whose maximum has
 * |m| < 2^21 and subtracted exactly for larger or non-finite maxima; bf16
 * inputs are widened exactly and each output is rounded once.  Every finite
 * input is in the domain.  IEEE semantics for special values: -inf entries
 * give 0; a row of -inf, or any NaN or +inf in a row, gives a NaN row.
 *
 *  - x, y: DEVICE pointers owned by the caller, rows*cols elements, contiguous
 *    row-major; y == x (in place) is allowed, any other overlap is rejected.
 *  - rows >= 0 (0: OK, no launch); 1 <= cols <= 2^31-1.
 *  - Asynchronous on `stream`; allocates nothing but the whole-grid path's
 *    scratch area (RMSNORM_PATH_GRID, as in rmsnorm.h); kernels are launched
 *    as rmsnorm.h's common contract states (set-up may overlap the kernel
 *    ahead, memory is touched only after it completes); argument errors are
 *    found on the host before any launch (RMSNORM_ERR_INVALID_ARG); a failed
 *    CUDA call returns RMSNORM_ERR_CUDA (see rmsnorm_last_cuda_error).
 */
#ifndef ROWSOFTMAX_H_
#define ROWSOFTMAX_H_

#include "rmsnorm.h"

#ifdef __cplusplus
extern "C" {
#endif

/* y = softmax(x) along the last axis, fp32 tensors.  Defined by: page "A
 * hackable Python ML compiler, part 2", the opening benchmark paragraph
 * (softmax-style small reductions among the generated kernels' wins); the page
 * prints no formula, so the definition above is the plain one. */
rmsnorm_status_t rowsoftmax_fwd_f32(const float* x, float* y, int64_t rows, int64_t cols,
                                    rmsnorm_stream_t stream);

/* The same for bfloat16 tensors (raw 16-bit patterns), fp32 arithmetic; same
 * passage (the page is fp32 only: the single output rounding is this library's
 * reading). */
rmsnorm_status_t rowsoftmax_fwd_bf16(const uint16_t* x, uint16_t* y, int64_t rows,
                                     int64_t cols, rmsnorm_stream_t stream);

/*
 * Either dtype with options: opt->path may be RMSNORM_PATH_AUTO,
 * RMSNORM_PATH_ROWREG (row held in registers; rows up to 64 KiB),
 * RMSNORM_PATH_CLUSTER (each row split over opt->cluster = 2..16 CTAs of a
 * thread-block cluster, row maximum and sum combined through distributed
 * shared memory), RMSNORM_PATH_STAGED (rows staged in shared memory by
 * bulk copies that run ahead into the next rows, then held in registers;
 * needs 16-byte aligned x and y and a row of a multiple of 16 bytes, else
 * RMSNORM_ERR_UNSUPPORTED; opt->chunk_bytes (a power of two, or at least the
 * row) and opt->stages size its copies and its ring of shared-memory slots,
 * zero for the defaults; opt->threads = threads per CTA, a multiple of 32 up
 * to 512; opt->cluster = 2..16 splits each row over a thread-block cluster,
 * maximum and sum combined through distributed shared memory) or
 * RMSNORM_PATH_STREAM (rows streamed twice through a shared-memory ring by
 * bulk copies: first read online maximum and sum, second read the outputs,
 * normally from L2; 16-byte aligned rows, else RMSNORM_ERR_UNSUPPORTED;
 * opt->cluster = 2..16 (any size) splits each row over a thread-block
 * cluster; opt->threads = consumer threads (multiple of 32, <= 480, default 448),
 * opt->chunk_bytes = 2 or 4 vectors of 16 bytes per consumer thread,
 * opt->stages = ring slots), RMSNORM_PATH_GRID (every row over the whole
 * grid, see rmsnorm.h; opt->threads = consumer threads, a multiple of 32 up
 * to 448: takes a scratch area of at most 17 KB from the
 * device's memory pool in stream order; chosen automatically for fewer rows
 * than SMs of 16 MB and more totalling 96 MB or more),
 * RMSNORM_PATH_TWOPASS (the wide-row kernel:
 * reads each row three times, the repeats normally from L2; opt->cluster =
 * 2..16 (any size; the other paths take powers of two) splits each row over
 * a thread-block cluster with one (maximum, sum) exchange per row, which the
 * automatic choice does for few rows too wide for every other kernel;
 * unsplit, rows of at most 2^31 - 1025 vectors, else
 * RMSNORM_ERR_UNSUPPORTED); opt->threads,
 * opt->grid, opt->vec_bytes and opt->wait_timeout_ns as for rmsnorm_fwd_ex.
 * opt->fault_inject (failure-detection tests, test build of the library
 * only): 1 = STAGED, STREAM or GRID withholds each CTA's first bulk copy,
 * 2 = a split row (CLUSTER or GRID, or STAGED, STREAM or TWOPASS with
 * cluster > 1) has CTA rank 0 withhold its first (maximum, sum) pair; the
 * bounded waits then expire (see
 * rmsnorm_last_device_status).  The product library, and any path without
 * that site, return RMSNORM_ERR_UNSUPPORTED; values outside 0..2 are
 * RMSNORM_ERR_INVALID_ARG.  chunk_bytes and stages with any other path, and
 * the other option fields, must be zero (else RMSNORM_ERR_INVALID_ARG).
 * `opt` may be NULL.
 */
rmsnorm_status_t rowsoftmax_fwd_ex(int32_t dtype, const void* x, void* y, int64_t rows,
                                   int64_t cols, const rmsnorm_options_t* opt,
                                   rmsnorm_stream_t stream);

/* What rowsoftmax_fwd_ex would launch (no launch); see rmsnorm_plan. */
rmsnorm_status_t rowsoftmax_plan(int32_t dtype, const void* x, const void* y, int64_t rows,
                                 int64_t cols, const rmsnorm_options_t* opt,
                                 rmsnorm_plan_t* plan);

#ifdef __cplusplus
}
#endif

#endif /* ROWSOFTMAX_H_ */
