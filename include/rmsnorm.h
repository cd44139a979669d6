/*
 * rmsnorm.h -- C ABI of librmsnorm, a fused row-wise RMSNorm forward pass for
 * NVIDIA GB300 (sm_103a).
 *
 * The operation (page "A hackable Python ML compiler, part 2", the RMSNorm
 * Loop-IR listing and the epilogue of the generated kernel) is, for every row
 * r of a row-major matrix x with `hidden` columns:
 *
 *     ms[r]   = (1/hidden) * sum_j x[r,j]^2
 *     rstd[r] = rsqrt(ms[r] + eps)
 *     y[r,j]  = (x[r,j] * rstd[r]) * w[j]
 *
 * Arithmetic is fp32 for both entry points (bf16 inputs are widened exactly;
 * the bf16 output is one round-to-nearest-even rounding of the fp32 product).
 *
 * Common contract of the compute entry points
 * -------------------------------------------
 *  - x, w, y are DEVICE pointers owned by the caller.  x and y hold
 *    rows*hidden elements, contiguous and row-major (row pitch == hidden);
 *    w holds hidden elements.  Any alignment of the element type is accepted;
 *    the library picks the widest vector width the pointers and the row pitch
 *    allow.
 *  - y == x (exact in-place) is allowed; any other overlap of x and y is
 *    rejected.  w may not overlap y.
 *  - The call is asynchronous on `stream` (NULL = the legacy default stream)
 *    and allocates no memory, with one exception: the few-very-wide-rows
 *    kernel (RMSNORM_PATH_GRID: forced through rmsnorm_fwd_ex, and chosen
 *    automatically for fewer rows than SMs of 10 to 40 MiB by RMSNorm and of
 *    16 MiB and more, totalling 96 MiB or more, by the row softmax) takes a
 *    scratch area of at most 17 KB from the current device's default memory
 *    pool in stream order and returns it on the same stream.  Argument errors are detected on the host before any
 *    launch and leave the device untouched.
 *  - Each kernel (all but the whole-grid one, a cooperative launch) is launched
 *    so that its CTAs may be placed and set up before the kernel ahead of it on
 *    `stream` has finished; it reads and writes no global memory until that
 *    kernel has completed and its writes are visible (programmatic dependent
 *    launch), so stream order holds as for any launch.
 *  - rows == 0 returns RMSNORM_OK without a launch.
 *  - The library's only device state is one status word per device, written
 *    by a kernel whose bounded wait ran out (see rmsnorm_last_device_status).
 *
 * Thread safety: calls may be made from several host threads; per-device set-up
 * is done once under a lock.
 */
#ifndef RMSNORM_H_
#define RMSNORM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; spelled out so this header needs no CUDA headers. */
typedef struct CUstream_st* rmsnorm_stream_t;

typedef enum {
    RMSNORM_OK = 0,
    RMSNORM_ERR_INVALID_ARG = 1,  /* bad pointer, size, eps or overlap; nothing launched */
    RMSNORM_ERR_UNSUPPORTED = 2,  /* a forced path/option cannot serve these arguments */
    RMSNORM_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    RMSNORM_ERR_TIMEOUT = 4       /* a kernel's bounded wait expired (device status) */
} rmsnorm_status_t;

typedef enum {
    RMSNORM_DTYPE_F32 = 0,
    RMSNORM_DTYPE_BF16 = 1
} rmsnorm_dtype_t;

/* Kernel families.  AUTO lets the dispatcher choose. */
typedef enum {
    RMSNORM_PATH_AUTO = 0,
    RMSNORM_PATH_ROWREG = 1,   /* single pass, the row held in registers; a group of
                                  threads per row, persistent grid-stride over rows   */
    RMSNORM_PATH_STAGED = 2,   /* rows staged in shared memory by 1-D bulk copies
                                  (cp.async.bulk + mbarrier), multi-stage prefetch    */
    RMSNORM_PATH_CLUSTER = 3,  /* split row: a thread-block cluster per row, slices in
                                  registers, partial sums exchanged through DSMEM     */
    RMSNORM_PATH_TWOPASS = 4,  /* generic fallback: read x twice (any width/alignment);
                                  opt->cluster = 2..16 (any size) splits each row over
                                  a thread-block cluster (partial sums through DSMEM),
                                  which the automatic choice does for few rows too
                                  wide for every other family.  Unsplit (cluster 0
                                  or 1): rows of at most 2^31 - 1025 vectors, else
                                  RMSNORM_ERR_UNSUPPORTED */
    RMSNORM_PATH_PAGE = 5,     /* comparison only, never automatic: the compiler write-up's
                                  schedule (one 256-thread CTA per row, whole row staged
                                  in shared memory, 4-byte accesses, 3-level tree); rows
                                  up to the shared-memory limit (about 56K elements) */
    RMSNORM_PATH_RINGREG = 6,  /* wide rows (up to 128 KB, 16-byte aligned x, w, y and
                                  pitch): rows streamed through a shared-memory ring by
                                  bulk copies and held in registers, the weight row in
                                  shared memory; opt->threads = consumer threads,
                                  opt->chunk_bytes = 2 or 4 vectors per consumer thread
                                  (x 16 bytes x threads), opt->stages = ring slots */
    RMSNORM_PATH_STREAM = 7,   /* row softmax only (rowsoftmax_fwd_ex): each row streamed
                                  twice through a shared-memory ring by bulk copies, the
                                  first read from DRAM (online maximum and sum), the second
                                  normally from L2 (outputs); one CTA per SM; opt->cluster =
                                  2..16 splits each row over a thread-block cluster */
    RMSNORM_PATH_GRID = 8      /* few rows of tens of MB (16-byte aligned x, w, y and
                                  pitch): every row over the whole grid in turn (one CTA
                                  per SM, a cooperative launch), streamed twice through
                                  each CTA's shared-memory ring so that the second read of
                                  a row finds it in L2; the CTAs' partial results meet in
                                  a scratch area of at most 17 KB that the call takes from
                                  the device's default memory pool in stream order
                                  (cudaMallocAsync / cudaFreeAsync on `stream`); opt->grid
                                  = CTAs (at most one per SM), opt->threads = consumer
                                  threads (multiple of 32, <= 448), opt->chunk_bytes =
                                  2 or 4 vectors per consumer thread, opt->stages = ring
                                  slots (2..32) */
} rmsnorm_path_t;

/* Options for rmsnorm_fwd_ex / rmsnorm_plan.  Zero-initialise, then set what you
 * need; every zero field means "automatic". */
typedef struct {
    int32_t path;            /* rmsnorm_path_t */
    int32_t cluster;         /* CTAs per row for CLUSTER (2, 4, 8, 16), STAGED (1..16)
                                or TWOPASS (1..16) */
    int32_t threads;         /* threads per row group (multiple of 32, <= 1024, or
                                1, 2, 4, 8, 16 for ROWREG: several rows per warp);
                                STAGED: consumer threads, 128 or 256 */
    int32_t grid;            /* CTAs to launch (rounded to the cluster size) */
    int32_t vec_bytes;       /* 16, 8, 4 or 2 (bf16 only); must suit the alignment */
    int32_t chunk_bytes;     /* STAGED: bytes per bulk copy (multiple of 16); RINGREG: see
                                RMSNORM_PATH_RINGREG */
    int32_t stages;          /* STAGED: chunk slots in the shared-memory ring (>= chunks per
                                row slice, <= 32); RINGREG: ring slots (2..32) */
    int32_t weights;         /* STAGED: 1 = weight slice copied to shared memory once,
                                2 = weights read through L1/L2 every row */
    int32_t fault_inject;    /* failure-detection tests only: 1 = the bulk-copy producer
                                (STAGED, RINGREG) withholds its first copy, 2 = one CTA of a
                                split-row cluster withholds its partial sum.  Honoured
                                only by the test build of the library (compiled with
                                RMSNORM_FAULT_INJECT); the product library returns
                                RMSNORM_ERR_UNSUPPORTED for any non-zero value. */
    int32_t reserved;        /* must be 0 */
    int32_t epilogue;        /* fused epilogue applied to each output before the store
                                (any path but PAGE): 0 none, 1 y*epilogue_alpha,
                                2 ReLU (y if y > 0 or y is NaN, else +0) */
    float epilogue_alpha;    /* scale for epilogue 1 (finite) */
    uint64_t wait_timeout_ns;/* limit of every device-side wait; 0 = 2 seconds */
} rmsnorm_options_t;

/* What a call with these arguments would launch. */
typedef struct {
    int32_t path;            /* rmsnorm_path_t actually chosen */
    int32_t cluster;         /* CTAs per row (1 unless split) */
    int32_t threads_per_row; /* threads cooperating on one row (or one slice) */
    int32_t block_threads;   /* threads per CTA */
    int32_t rows_per_cta;    /* rows one CTA works on at a time */
    int32_t grid;            /* CTAs launched */
    int32_t vec_bytes;       /* bytes per global load/store instruction */
    int32_t vecs_per_thread; /* register-resident vectors per thread and row */
    int32_t smem_bytes;      /* dynamic shared memory per CTA */
    int32_t chunk_bytes;     /* STAGED: bytes per bulk copy */
    int32_t stages;          /* STAGED: chunk slots in the ring */
    int32_t weights_staged;  /* STAGED: 1 if the weight slice is held in shared memory */
    char kernel[48];         /* kernel family name, for profiles */
} rmsnorm_plan_t;

/*
 * rmsnorm_fwd_f32 -- y = RMSNorm(x) * w for fp32 tensors.
 * Defined by: page "A hackable Python ML compiler, part 2", the RMSNorm
 * Loop-IR listing (the reduce axis summing x^2, the free axis scaling by the
 * reciprocal root and then by the weight) and the epilogue of the CUDA kernel
 * it generates (rsqrt of sum * (1/H) + eps).
 * x, y: rows*hidden floats (device); w: hidden floats (device);
 * rows >= 0; 1 <= hidden <= 2^31-1; eps finite and >= 0.
 * Returns RMSNORM_OK once launched; RMSNORM_ERR_INVALID_ARG for NULL pointers,
 * bad sizes, bad eps or partial overlap; RMSNORM_ERR_CUDA if a CUDA call fails
 * (see rmsnorm_last_cuda_error).
 */
rmsnorm_status_t rmsnorm_fwd_f32(const float* x, const float* w, float* y,
                                 int64_t rows, int64_t hidden, float eps,
                                 rmsnorm_stream_t stream);

/*
 * rmsnorm_fwd_bf16 -- the same for bfloat16 tensors, passed as raw 16-bit
 * patterns.  Defined by: the same Loop-IR listing and kernel epilogue as
 * rmsnorm_fwd_f32; the page is fp32 only, so the bf16 rounding below is this
 * library's reading, not a passage.  Accumulation, rstd and the products are fp32; each output is
 * rounded once to bfloat16 (round-to-nearest-even).  Arguments and errors as
 * for rmsnorm_fwd_f32.
 */
rmsnorm_status_t rmsnorm_fwd_bf16(const uint16_t* x, const uint16_t* w, uint16_t* y,
                                  int64_t rows, int64_t hidden, float eps,
                                  rmsnorm_stream_t stream);

/*
 * rmsnorm_fwd_ex -- the operation of rmsnorm_fwd_f32 / rmsnorm_fwd_bf16 (same
 * passages); the options have no counterpart in the page: they choose among
 * this library's kernels.  Either dtype, with explicit options (forced kernel family,
 * cluster size, launch shape, wait limit).  `opt` may be NULL (= automatic).
 * Returns RMSNORM_ERR_UNSUPPORTED when a forced option cannot serve the call
 * (e.g. STAGED on a row pitch that is not a multiple of 16 bytes); nothing is
 * launched in that case.
 */
rmsnorm_status_t rmsnorm_fwd_ex(int32_t dtype, const void* x, const void* w, void* y,
                                int64_t rows, int64_t hidden, float eps,
                                const rmsnorm_options_t* opt, rmsnorm_stream_t stream);

/*
 * rmsnorm_fwd_grid_noalloc -- the page has no counterpart: this is an
 * interface variant, not part of the method.  The same result as
 * rmsnorm_fwd_ex with opt->path = RMSNORM_PATH_GRID (every row split over the
 * whole grid; meant for few rows of tens of MB), but the call allocates
 * nothing: the kernel's exchange area (an arrival counter and the CTAs'
 * partial sums, 16512 bytes at most: grids of up to 1024 CTAs) lives in a
 * fixed device array inside the library instead of coming from the memory
 * pool on every call.  For callers that may not allocate device memory while
 * they run -- an engine or plugin host that owns every byte of device memory
 * and accounts for it, code on a path that must not risk an allocation
 * failing or blocking mid-step, or a process whose device has no usable
 * stream-ordered memory pool.
 *  - x, w, y, rows, hidden, eps and stream as for rmsnorm_fwd_f32 /
 *    rmsnorm_fwd_bf16; dtype is RMSNORM_DTYPE_F32 or RMSNORM_DTYPE_BF16.
 *    x, w, y and the row pitch must be 16-byte aligned, else
 *    RMSNORM_ERR_UNSUPPORTED (nothing launched).
 *  - RMSNORM_ERR_UNSUPPORTED too if the grid this device would launch needs
 *    more exchange space than the array holds (more than 1024 CTAs).
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before capturing any stream into a CUDA graph.
 *  - Each call clears the part of the array it uses (cudaMemsetAsync on
 *    `stream`) and then launches.  Every call on a device shares the one
 *    array, so calls whose kernels can overlap on the GPU (other streams, or
 *    other host threads) race with each other and give undefined results:
 *    serialise them, or use rmsnorm_fwd_ex, whose scratch is per call.
 */
rmsnorm_status_t rmsnorm_fwd_grid_noalloc(int32_t dtype, const void* x, const void* w, void* y,
                                          int64_t rows, int64_t hidden, float eps,
                                          rmsnorm_stream_t stream);

/*
 * rmsnorm_plan -- no passage of the page: a query of this library's launch
 * heuristics.  Fill *plan with what rmsnorm_fwd_ex(dtype, x, w, y, rows,
 * hidden, ., opt, .) would launch on the current device, without launching.
 * Pointers are used only for their alignment (they may be any non-NULL values).
 */
rmsnorm_status_t rmsnorm_plan(int32_t dtype, const void* x, const void* w, const void* y,
                              int64_t rows, int64_t hidden,
                              const rmsnorm_options_t* opt, rmsnorm_plan_t* plan);

/*
 * rmsnorm_last_device_status -- no passage of the page defines it: it reports
 * this library's own failure detection (bounded device waits).  Synchronise `stream`, then read and clear the
 * current device's status word.  RMSNORM_OK if no kernel's bounded wait has
 * expired since the last read; RMSNORM_ERR_TIMEOUT otherwise (outputs of the
 * affected call are undefined); RMSNORM_ERR_CUDA if synchronisation failed.
 */
rmsnorm_status_t rmsnorm_last_device_status(rmsnorm_stream_t stream);

/* Static English text for a status code (never NULL).  No passage: diagnostics. */
const char* rmsnorm_status_string(rmsnorm_status_t status);

/*
 * rmsnorm_last_cuda_error -- (no passage: diagnostics) the cudaError_t of the last CUDA runtime call of
 * this library that failed on the calling host thread (0 if none), and clears
 * it.  If msg != NULL and len > 0, writes "<name>: <description>" there
 * (truncated, NUL-terminated).  The library links the CUDA runtime
 * statically, so this -- not the caller's cudaGetLastError -- is where an
 * RMSNORM_ERR_CUDA is explained.
 */
int32_t rmsnorm_last_cuda_error(char* msg, size_t len);

/* 1 in the test build of the library that honours rmsnorm_options_t.fault_inject
 * (compiled with RMSNORM_FAULT_INJECT), 0 in the product library. */
int32_t rmsnorm_fault_injection_enabled(void);

/* ABI version of this header: major*10000 + minor*100 + patch. */
int32_t rmsnorm_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RMSNORM_H_ */
