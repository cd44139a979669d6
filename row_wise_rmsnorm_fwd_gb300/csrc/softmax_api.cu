// softmax_api.cu -- C ABI of the row-wise softmax (include/rowsoftmax.h):
// validation, kernel choice and launch.  Shares the library's per-device
// state (device.h) and status conventions with the RMSNorm entry points.
#include "rowsoftmax.h"
#include "launch.h"
#include "device.h"

#include <cstdio>
#include <cstring>

namespace rmsnorm {
namespace {

constexpr int kSoftmaxWavesF32 = 8;                     // at most this many resident waves
constexpr int kSoftmaxWavesBf16 = 4;
constexpr int64_t kSoftmaxSplitRowBytes = 32768;        // few rows wider than this: split
constexpr int64_t kSoftmaxSplitMinBytes = 16 << 20;     // or few rows totalling this much
constexpr int64_t kSoftmaxStagedChunk = 65536;          // bytes per bulk copy (default)
constexpr int64_t kSoftmaxStagedMinCols = 8192;         // wider fp32 rows go to the staged kernel
constexpr int64_t kSoftmaxStagedMinColsBf16 = 16384;    // wider bf16 rows go to the staged kernel
constexpr int kSoftmaxMaxStagedCluster = 8;             // portable cluster sizes only
constexpr int64_t kSoftmaxSplitStagedMinRowBytes = 240 << 10;  // narrower: three-pass (sm_make_plan)
constexpr int64_t kSoftmaxUnsplitMaxVecs = 0x7FFFFFFFll - 1024;  // three-pass, one CTA per row
constexpr int64_t kSoftmaxStreamMinRowBytes = 128 << 10;   // streamed: rows of at least this
constexpr int64_t kSoftmaxStreamMaxSlice = 400 << 10;      // streamed: split rows above this
constexpr int kSoftmaxStreamMaxCluster = 8;
constexpr int64_t kSoftmaxGridMinRowBytes = 16ll << 20;  // auto: rows over the whole grid
constexpr int64_t kSoftmaxGridMinBytes = 96ll << 20;     // ... for few-row inputs this large
constexpr int kStreamReadAheadChunks = 2;                  // streamed split: see sm_plan_stream
constexpr int kStreamDefaultConsumers = 448;               // streamed: see sm_plan_stream
constexpr int64_t kStreamReadAheadMaxBytes = 48ll << 20;

struct SmCall {
    int dtype;
    int sz;
    uintptr_t x, y;
    int64_t rows, cols;
    rmsnorm_options_t opt;
    DeviceView dv;
};

struct SmPlan {
    int path = 0;
    int cluster = 1;
    int slice_vecs = 0;
    int group = 0;
    int block = 0;
    int rpc = 1;
    int grid = 0;
    int vb = 0;
    int nv = 0;
    int nvec = 0;
    int smem = 0;          // dynamic shared memory (staged path)
    int chunk = 0;         // staged path: bytes per bulk copy
    int nchunks = 0;       // staged path: copies per row
    int nslots = 0;        // staged path: ring slots
    int resident = 0;      // three-pass split: resident clusters
    int scratch = 0;       // grid split: bytes of cleared scratch (cooperative launch)
    int read_ahead = 0;    // streamed split: next-row chunks read during each exchange
    int schedule = 0;      // grid split: row schedule
    int res_chunks = 0;    // grid split: slice chunks kept in shared memory
    KernelFn fn = nullptr;
    const char* name = "";
};

int sm_round_up(int64_t a, int64_t b) { return static_cast<int>(((a + b - 1) / b) * b); }
int sm_pow2_ceil(int64_t v) { int p = 1; while (p < v) p <<= 1; return p; }

rmsnorm_status_t sm_validate(int32_t dtype, const void* x, const void* y, int64_t rows,
                             int64_t cols, const rmsnorm_options_t* opt, SmCall* c) {
    if (dtype != RMSNORM_DTYPE_F32 && dtype != RMSNORM_DTYPE_BF16) return RMSNORM_ERR_INVALID_ARG;
    if (!x || !y) return RMSNORM_ERR_INVALID_ARG;
    if (rows < 0 || cols <= 0 || cols > 0x7FFFFFFFll) return RMSNORM_ERR_INVALID_ARG;
    const int sz = dtype == RMSNORM_DTYPE_F32 ? 4 : 2;
    if (rows > 0 && rows > (INT64_MAX / sz) / cols) return RMSNORM_ERR_INVALID_ARG;
    const uintptr_t ux = reinterpret_cast<uintptr_t>(x), uy = reinterpret_cast<uintptr_t>(y);
    if (ux % sz || uy % sz) return RMSNORM_ERR_INVALID_ARG;
    const uint64_t n = static_cast<uint64_t>(rows) * static_cast<uint64_t>(cols) * sz;
    if (ux != uy && ux < uy + n && uy < ux + n) return RMSNORM_ERR_INVALID_ARG;
    std::memset(c, 0, sizeof(*c));
    c->dtype = dtype;
    c->sz = sz;
    c->x = ux;
    c->y = uy;
    c->rows = rows;
    c->cols = cols;
    if (opt) {
        c->opt = *opt;
        const rmsnorm_options_t& o = *opt;
        if (o.weights || o.reserved || o.epilogue || o.fault_inject < 0 || o.fault_inject > 2)
            return RMSNORM_ERR_INVALID_ARG;
        // fault injection: test build only, and only where its site exists
        // (1: the ring's first copy; 2: a split row's first pair)
        if (o.fault_inject != 0 &&
            (!RMSNORM_FAULT_INJECT ||
             (o.fault_inject == 1 && o.path != RMSNORM_PATH_STAGED &&
              o.path != RMSNORM_PATH_STREAM && o.path != RMSNORM_PATH_GRID) ||
             (o.fault_inject == 2 && o.path != RMSNORM_PATH_CLUSTER && o.path != RMSNORM_PATH_GRID &&
              !((o.path == RMSNORM_PATH_STAGED || o.path == RMSNORM_PATH_TWOPASS ||
                 o.path == RMSNORM_PATH_STREAM) &&
                o.cluster > 1))))
            return RMSNORM_ERR_UNSUPPORTED;
        if (o.path != RMSNORM_PATH_AUTO && o.path != RMSNORM_PATH_ROWREG &&
            o.path != RMSNORM_PATH_TWOPASS && o.path != RMSNORM_PATH_CLUSTER &&
            o.path != RMSNORM_PATH_STAGED && o.path != RMSNORM_PATH_STREAM &&
            o.path != RMSNORM_PATH_GRID)
            return RMSNORM_ERR_INVALID_ARG;
        // chunk and ring sizes shape the ring kernels only
        if ((o.chunk_bytes || o.stages) && o.path != RMSNORM_PATH_STAGED &&
            o.path != RMSNORM_PATH_STREAM && o.path != RMSNORM_PATH_GRID)
            return RMSNORM_ERR_INVALID_ARG;
        if (o.chunk_bytes < 0 || o.chunk_bytes % 16 != 0 || o.stages < 0)
            return RMSNORM_ERR_INVALID_ARG;
        // cluster sizes: powers of two, or any size up to 16 for TWOPASS and STREAM
        if (o.cluster < 0 || o.cluster > 16 ||
            ((o.cluster & (o.cluster - 1)) != 0 && o.path != RMSNORM_PATH_TWOPASS &&
             o.path != RMSNORM_PATH_STREAM))
            return RMSNORM_ERR_INVALID_ARG;
        if (o.cluster > 1 && o.path != RMSNORM_PATH_CLUSTER && o.path != RMSNORM_PATH_STAGED &&
            o.path != RMSNORM_PATH_TWOPASS && o.path != RMSNORM_PATH_STREAM)
            return RMSNORM_ERR_INVALID_ARG;
        const bool sub_warp = o.threads > 0 && o.threads < 32 && (o.threads & (o.threads - 1)) == 0;
        if (o.threads < 0 || (o.threads % 32 != 0 && !sub_warp) || o.threads > 1024 || o.grid < 0)
            return RMSNORM_ERR_INVALID_ARG;
        if (sub_warp && o.path != RMSNORM_PATH_ROWREG) return RMSNORM_ERR_INVALID_ARG;
    }
    return RMSNORM_OK;
}

rmsnorm_status_t sm_pick_vb(const SmCall& c, int* vb) {
    const uintptr_t a = c.x | c.y;
    const int64_t pitch = c.cols * c.sz;
    int widest = c.sz;
    for (int v = 16; v >= c.sz; v >>= 1)
        if (a % v == 0 && pitch % v == 0) { widest = v; break; }
    const int f = c.opt.vec_bytes;
    if (f == 0) { *vb = widest; return RMSNORM_OK; }
    if (f != 2 && f != 4 && f != 8 && f != 16) return RMSNORM_ERR_INVALID_ARG;
    if (f < c.sz || f > widest) return RMSNORM_ERR_UNSUPPORTED;
    *vb = f;
    return RMSNORM_OK;
}

// Register-resident softmax; cluster > 1 splits every row over a cluster.
rmsnorm_status_t sm_plan_rowreg(const SmCall& c, int cluster, SmPlan* P) {
    int vb;
    rmsnorm_status_t st = sm_pick_vb(c, &vb);
    if (st != RMSNORM_OK) return st;
    const int64_t nvec = c.cols / (vb / c.sz);
    const int64_t per = cluster > 1 ? (nvec + cluster - 1) / cluster : nvec;
    int G, NV;
    if (c.opt.threads > 0) {
        G = c.opt.threads;
        const int64_t need = (per + G - 1) / G;
        if (need > 8) return RMSNORM_ERR_UNSUPPORTED;
        NV = sm_pow2_ceil(need);
    } else if (cluster == 1 && c.dtype == RMSNORM_DTYPE_BF16 && per <= 8 * 256) {
        // bf16 rows of up to 2048 vectors: 8 vectors per thread (2 for rows
        // of at most 16 vectors), pow2(vectors / NV) lanes per row.  bf16
        // softmax is instruction bound, and the per-row work (reductions,
        // shuffles) is best spread over many elements per thread.  Measured
        // (% of the HBM roofline) on 128 MB inputs, rows of 64 / 128 / 256 /
        // 512 / 1024 / 2048 elements: 87 / 87 / 89 / 90 / 90 / 90, against
        // 81 / 85 / 85 / 83 / 83 / 69 with 4 vectors per thread; on 512 MB
        // inputs, rows of 4096 / 8192 / 16384: 80 / 81 / 81 against 78 / 77 /
        // 65 (and 62 staged at 16384).
        NV = per <= 16 ? (per >= 2 ? 2 : 1) : 8;
        G = sm_pow2_ceil((per + NV - 1) / NV);
    } else if (cluster == 1 && per <= 32 * 4) {
        // rows of up to 128 vectors: 4 vectors per thread (fewer for rows of
        // fewer than 4) and pow2(vectors / 4) lanes per row, 32 / G rows per
        // warp (as for the RMSNorm register kernel)
        NV = per >= 4 ? 4 : sm_pow2_ceil(per);
        G = sm_pow2_ceil((per + NV - 1) / NV);
    } else {
        NV = 4;
        int64_t g = sm_round_up((per + NV - 1) / NV, 32);
        if (g > softmax_rowreg_max_block(NV)) {
            NV = 8;
            g = sm_round_up((per + NV - 1) / NV, 32);
        }
        if (g > softmax_rowreg_max_block(NV)) return RMSNORM_ERR_UNSUPPORTED;
        G = static_cast<int>(g);
    }
    if (G > softmax_rowreg_max_block(NV)) return RMSNORM_ERR_UNSUPPORTED;
    KernelFn fn = softmax_rowreg_ptr(c.dtype, vb, NV, cluster > 1);
    if (!fn) return RMSNORM_ERR_UNSUPPORTED;
    const int rpc = cluster == 1 ? (G >= 256 ? 1 : 256 / G) : 1;
    const int block = G * rpc;
    int occ = 0;
    if (cached_occupancy(c.dv.dev, c.dv.smem_optin, fn, block, 0, cluster, &occ) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    if (occ <= 0) return RMSNORM_ERR_UNSUPPORTED;
    int grid;
    if (cluster == 1) {
        // Whole waves of resident CTAs, each with three or more row blocks
        // (as for the RMSNorm register kernel), at most 8 waves for fp32 and 4
        // for bf16.  bf16 rows of four or more vectors per thread instead run
        // two CTAs per SM, each through many rows, and bf16 rows of two
        // vectors per thread eight CTAs per SM.  Measured (% of the HBM
        // roofline): fp32 rows of 512 with 2 / 4 / 8 waves 93 / 96 / 97; bf16
        // rows of 1024 / 2048 / 4096 / 8192 elements at 4 vectors per thread
        // 83 / 71 / 76 / 75 with two CTAs per SM against 83 / 66 / 74 / 74
        // with four waves; bf16 rows of 512 at 8 vectors per thread 90 with
        // two CTAs per SM, 87 with eight.
        const int64_t nblocks = (c.rows + rpc - 1) / rpc;
        const int64_t resident = static_cast<int64_t>(c.dv.sms) * occ;
        const int64_t max_waves = c.dtype == RMSNORM_DTYPE_F32 ? kSoftmaxWavesF32 : kSoftmaxWavesBf16;
        int64_t waves = nblocks / (3 * resident);
        waves = waves < 1 ? 1 : (waves > max_waves ? max_waves : waves);
        int64_t target = resident * waves;
        if (c.dtype == RMSNORM_DTYPE_BF16 && NV >= 4) target = 2 * static_cast<int64_t>(c.dv.sms);
        if (c.dtype == RMSNORM_DTYPE_BF16 && NV <= 2 && G < 32)
            target = 8 * static_cast<int64_t>(c.dv.sms);
        grid = static_cast<int>(c.opt.grid > 0 ? c.opt.grid
                                               : (nblocks < target ? nblocks : target));
    } else {
        const int64_t nclusters = c.opt.grid > 0 ? (c.opt.grid + cluster - 1) / cluster
                                                 : (c.rows < occ ? c.rows : occ);
        grid = static_cast<int>(nclusters * cluster);
    }
    *P = SmPlan{};             // every field this plan does not set keeps its default
    P->path = cluster == 1 ? RMSNORM_PATH_ROWREG : RMSNORM_PATH_CLUSTER;
    P->cluster = cluster;
    P->slice_vecs = static_cast<int>(per);
    P->group = G;
    P->block = block;
    P->rpc = rpc;
    P->grid = grid;
    P->vb = vb;
    P->nv = NV;
    P->nvec = static_cast<int>(nvec);
    P->fn = fn;
    P->name = cluster == 1 ? "softmax_rowreg" : "softmax_cluster_rowreg";
    return RMSNORM_OK;
}

// Three-pass kernel; cluster > 1 splits each row over a thread-block cluster
// (slices of whole 32-vector groups, one (maximum, sum) exchange per row).
rmsnorm_status_t sm_plan_threepass(const SmCall& c, int cluster, SmPlan* P) {
    int vb;
    rmsnorm_status_t st = sm_pick_vb(c, &vb);
    if (st != RMSNORM_OK) return st;
    KernelFn fn = cluster > 1 ? softmax_threepass_cluster_ptr(c.dtype, vb)
                              : softmax_threepass_ptr(c.dtype, vb);
    if (!fn) return RMSNORM_ERR_UNSUPPORTED;
    const int64_t nvec = c.cols / (vb / c.sz);
    // The unsplit kernel's 32-bit vector index must not pass 2^31 - 1 one
    // stride after the row's last vector: such rows are split.
    if (cluster == 1 && nvec > kSoftmaxUnsplitMaxVecs) return RMSNORM_ERR_UNSUPPORTED;
    const int64_t slice = cluster > 1 ? sm_round_up((nvec + cluster - 1) / cluster, 32) : nvec;
    const int maxb = cluster > 1 ? split_block() : softmax_threepass_block();
    const int block = c.opt.threads > 0 ? c.opt.threads
                                        : (slice >= maxb ? maxb : sm_round_up(slice, 32));
    int occ = 0;
    if (cached_occupancy(c.dv.dev, c.dv.smem_optin, fn, block, 0, cluster, &occ) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    if (occ <= 0) return RMSNORM_ERR_UNSUPPORTED;
    int64_t grid;
    if (cluster == 1) {
        const int64_t resident = static_cast<int64_t>(c.dv.sms) * occ;
        grid = c.opt.grid > 0 ? c.opt.grid : (c.rows < resident ? c.rows : resident);
    } else {
        const int64_t nclusters = c.opt.grid > 0 ? (c.opt.grid + cluster - 1) / cluster
                                                 : (c.rows < occ ? c.rows : occ);
        grid = nclusters * cluster;
    }
    *P = SmPlan{};             // every field this plan does not set keeps its default
    P->path = RMSNORM_PATH_TWOPASS;
    P->cluster = cluster;
    P->slice_vecs = static_cast<int>(slice);
    P->group = block;
    P->block = block;
    P->rpc = 1;
    P->grid = static_cast<int>(grid);
    P->vb = vb;
    P->nv = 0;
    P->nvec = static_cast<int>(nvec);
    P->fn = fn;
    P->resident = occ;
    P->name = cluster == 1 ? "softmax_threepass" : "softmax_cluster_threepass";
    return RMSNORM_OK;
}

// The three-pass kernel with each row over a cluster of C CTAs (one CTA per
// row would leave the row's whole traffic to one SM).  C (2..16, any size)
// minimises the row time waves(C) / C, waves(C) = rows / resident clusters
// of C, rounded up; ties go to the smaller cluster.
rmsnorm_status_t sm_plan_threepass_split(const SmCall& c, SmPlan* P) {
    SmPlan best;
    int64_t best_waves = 0;
    for (int cl = 2; cl <= 16; ++cl) {
        SmPlan Q;
        const rmsnorm_status_t st = sm_plan_threepass(c, cl, &Q);
        if (st == RMSNORM_ERR_CUDA) return st;
        if (st != RMSNORM_OK) continue;
        const int64_t waves = (c.rows + Q.resident - 1) / Q.resident;
        if (best_waves == 0 || waves * best.cluster < best_waves * cl) {
            best = Q;
            best_waves = waves;
        }
    }
    if (best_waves == 0) return RMSNORM_ERR_UNSUPPORTED;
    *P = best;
    return RMSNORM_OK;
}

// Rows staged in shared memory, then held in registers: 16-byte vectors only
// (the bulk copies need 16-byte aligned rows of a multiple of 16 bytes).  The
// fewest vectors per thread (fp32 4/8/16, bf16 2/4/8) that cover the row with
// at most 512 threads (or opt->threads threads); chunks of
// 64 KB (or opt->chunk_bytes, a power of two; a row shorter than a chunk is
// one chunk); as many ring slots as the shared memory holds, up to 32 (or
// opt->stages).  Measured on 1 GB inputs: chunks of 8, 16, 32 and 64 KB gave
// 58, 66, 71 and 76% of the HBM roofline on bf16 rows of 32000.
rmsnorm_status_t sm_plan_staged(const SmCall& c, int cluster, SmPlan* P) {
    int vb;
    rmsnorm_status_t st = sm_pick_vb(c, &vb);
    if (st != RMSNORM_OK) return st;
    if (vb != 16) return RMSNORM_ERR_UNSUPPORTED;
    const int64_t row_bytes = c.cols * c.sz;
    const int64_t nvec = row_bytes / 16;
    const int64_t per = (nvec + cluster - 1) / cluster;       // vectors per CTA slice
    if (static_cast<int64_t>(cluster - 1) * per >= nvec) return RMSNORM_ERR_UNSUPPORTED;
    const int64_t slice_bytes = per * 16;
    const int max_nc = softmax_staged_max_threads();
    const int nv_min = c.sz == 4 ? 4 : 2, nv_max = c.sz == 4 ? 16 : 8;
    int nv = nv_min, nc;
    if (c.opt.threads > 0) {
        if (c.opt.threads > max_nc) return RMSNORM_ERR_UNSUPPORTED;
        nc = c.opt.threads;
        while (nv < nv_max && static_cast<int64_t>(nv) * nc < per) nv <<= 1;
        if (static_cast<int64_t>(nv) * nc < per) return RMSNORM_ERR_UNSUPPORTED;
    } else {
        while (nv < nv_max && static_cast<int64_t>(nv) * max_nc < per) nv <<= 1;
        if (static_cast<int64_t>(nv) * max_nc < per) return RMSNORM_ERR_UNSUPPORTED;
        nc = sm_round_up((per + nv - 1) / nv, 32);
    }
    KernelFn fn = softmax_staged_ptr(c.dtype, nv, cluster > 1);
    if (!fn) return RMSNORM_ERR_UNSUPPORTED;
    int64_t chunk = c.opt.chunk_bytes ? c.opt.chunk_bytes : kSoftmaxStagedChunk;
    if (chunk >= slice_bytes) {
        chunk = slice_bytes;                             // one chunk per row (slice)
    } else if ((chunk & (chunk - 1)) != 0) {
        return RMSNORM_ERR_UNSUPPORTED;                  // chunks must be a power of two
    }
    const int64_t nchunks = (slice_bytes + chunk - 1) / chunk;
    const int64_t budget = c.dv.smem_optin - kStagedHeaderHost;
    int64_t slots = c.opt.stages ? c.opt.stages : budget / chunk;
    if (!c.opt.stages && slots > kStagedMaxSlotsHost) slots = kStagedMaxSlotsHost;
    if (slots < nchunks || slots > kStagedMaxSlotsHost || slots * chunk > budget)
        return RMSNORM_ERR_UNSUPPORTED;
    const int block = nc;
    const int smem = static_cast<int>(kStagedHeaderHost + slots * chunk);
    int occ = 0;
    if (cached_occupancy(c.dv.dev, c.dv.smem_optin, fn, block, smem, cluster, &occ) !=
        cudaSuccess)
        return RMSNORM_ERR_CUDA;
    if (occ <= 0) return RMSNORM_ERR_UNSUPPORTED;
    int grid;
    if (cluster == 1) {
        const int64_t resident = static_cast<int64_t>(c.dv.sms) * occ;
        grid = static_cast<int>(c.opt.grid > 0 ? c.opt.grid
                                               : (c.rows < resident ? c.rows : resident));
    } else {
        const int64_t nclusters = c.opt.grid > 0 ? (c.opt.grid + cluster - 1) / cluster
                                                 : (c.rows < occ ? c.rows : occ);
        grid = static_cast<int>(nclusters * cluster);
    }
    *P = SmPlan{};             // every field this plan does not set keeps its default
    P->path = RMSNORM_PATH_STAGED;
    P->cluster = cluster;
    P->slice_vecs = static_cast<int>(per);
    P->group = nc;
    P->block = block;
    P->rpc = 1;
    P->grid = grid;
    P->vb = vb;
    P->nv = nv;
    P->nvec = static_cast<int>(nvec);
    P->smem = smem;
    P->chunk = static_cast<int>(chunk);
    P->nchunks = static_cast<int>(nchunks);
    P->nslots = static_cast<int>(slots);
    P->fn = fn;
    P->name = cluster == 1 ? "softmax_staged" : "softmax_cluster_staged";
    return RMSNORM_OK;
}

// Rows streamed twice through the ring (softmax_stream_kernel): 16-byte
// vectors only; 480 consumer threads (or opt->threads, a multiple of 32 up
// to 480) and a producer warp; chunks of v = 4 vectors per consumer thread
// (opt->chunk_bytes may ask for v = 2: 16 * v * consumer threads bytes);
// as many ring slots as shared memory holds, up to 32 (or opt->stages, at
// least 2); one CTA per SM, at most one per row (or slice).  cluster > 1
// splits each row over a thread-block cluster of that many CTAs.
rmsnorm_status_t sm_plan_stream(const SmCall& c, int cluster, SmPlan* P) {
    int vb;
    rmsnorm_status_t st = sm_pick_vb(c, &vb);
    if (st != RMSNORM_OK) return st;
    if (vb != 16) return RMSNORM_ERR_UNSUPPORTED;
    const int64_t row_bytes = c.cols * c.sz;
    const int64_t nvec = row_bytes / 16;
    const int64_t per = (nvec + cluster - 1) / cluster;       // vectors per CTA slice
    if (static_cast<int64_t>(cluster - 1) * per >= nvec) return RMSNORM_ERR_UNSUPPORTED;
    const int64_t slice_bytes = per * 16;
    const int max_nc = softmax_stream_max_threads() - 32;
    // 14 consumer warps by default: eight 28 KB ring slots rather than seven
    // of 30 KB.  Measured (% of the HBM copy peak, 448 / 480 consumer
    // threads): bf16 prefill logits 89.2 / 88.4, fp32 rows of 48000 95.6 /
    // 93.3 and of 65536 96.3 / 95.9, bf16 rows of 100000 93.3 / 92.2 and of
    // 65536 86.8 / 85.9, fp32 prefill logits over clusters of two 85.6 / 84.6.
    const int nc = c.opt.threads > 0 ? c.opt.threads : kStreamDefaultConsumers;
    if (nc % 32 != 0 || nc > max_nc) return RMSNORM_ERR_UNSUPPORTED;
    int v = 4;
    if (c.opt.chunk_bytes != 0) {
        if (c.opt.chunk_bytes == 2 * 16 * nc) v = 2;
        else if (c.opt.chunk_bytes == 4 * 16 * nc) v = 4;
        else return RMSNORM_ERR_UNSUPPORTED;
    }
    const int64_t chunk = static_cast<int64_t>(16) * v * nc;
    const int64_t nchunks = (slice_bytes + chunk - 1) / chunk;
    if (nchunks > 0x7FFFFFFFll) return RMSNORM_ERR_UNSUPPORTED;
    const int64_t budget = c.dv.smem_optin - kStreamHeaderHost;
    int64_t slots = c.opt.stages ? c.opt.stages : budget / chunk;
    if (!c.opt.stages && slots > kStagedMaxSlotsHost) slots = kStagedMaxSlotsHost;
    if (slots < 2 || slots > kStagedMaxSlotsHost || slots * chunk > budget)
        return RMSNORM_ERR_UNSUPPORTED;
    KernelFn fn = softmax_stream_ptr(c.dtype, v, cluster > 1);
    if (!fn) return RMSNORM_ERR_UNSUPPORTED;
    const int block = nc + 32;
    const int smem = static_cast<int>(kStreamHeaderHost + slots * chunk);
    int occ = 0;
    if (cached_occupancy(c.dv.dev, c.dv.smem_optin, fn, block, smem, cluster, &occ) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    if (occ <= 0) return RMSNORM_ERR_UNSUPPORTED;
    int64_t grid;
    if (cluster == 1) {
        const int64_t resident = static_cast<int64_t>(c.dv.sms) * occ;
        grid = c.opt.grid > 0 ? c.opt.grid : (c.rows < resident ? c.rows : resident);
    } else {
        const int64_t nclusters = c.opt.grid > 0 ? (c.opt.grid + cluster - 1) / cluster
                                                 : (c.rows < occ ? c.rows : occ);
        grid = nclusters * cluster;
    }
    *P = SmPlan{};             // every field this plan does not set keeps its default
    P->path = RMSNORM_PATH_STREAM;
    P->cluster = cluster;
    P->slice_vecs = static_cast<int>(per);
    P->group = nc;
    P->block = block;
    P->rpc = 1;
    P->grid = static_cast<int>(grid);
    P->vb = 16;
    P->nv = v;
    P->nvec = static_cast<int>(nvec);
    P->smem = smem;
    P->chunk = static_cast<int>(chunk);
    P->nchunks = static_cast<int>(nchunks);
    P->nslots = static_cast<int>(slots);
    P->fn = fn;
    P->name = cluster == 1 ? "softmax_stream" : "softmax_cluster_stream";
    // A split row's CTAs read the next row's first two chunks while their
    // (maximum, sum) pairs cross the cluster -- for fp32 rows whose rows in
    // flight (resident clusters x row) stay within 48 MiB.  Measured (% of
    // the HBM copy peak, with / without): fp32 rows of 128256 (39 MB in
    // flight) 85.5 / 84.0 and of 262144 over clusters of 4 (38 MiB) 83.6 /
    // 82.0; fp32 rows of 200000 (61 MB) 80.5 / 84.9 and bf16 rows of 262144
    // (39 MB; the consumers, not DRAM, set the pace) 84.1 / 84.9.
    if (cluster > 1 && c.dtype == RMSNORM_DTYPE_F32 &&
        (grid / cluster) * row_bytes <= kStreamReadAheadMaxBytes)
        P->read_ahead = kStreamReadAheadChunks;
    return RMSNORM_OK;
}

// Automatic choice: few rows of wide rows (or large few-row inputs) are split
// over a cluster (up to 8 CTAs, slices of at least 4 KB), as for RMSNorm;
// fp32 rows of more than 8192 elements and bf16 rows of more than 16384 are
// staged through shared memory (measured on 1 GB inputs, % of the HBM
// roofline: fp32 rows of 16384 / 32000 elements 87 / 97 staged against 78 /
// 86 for the best other kernel, rows of 8192 89 in registers against 75
// staged; bf16 rows of 32000 86 staged against 61 in registers, rows of
// 16384 64 in registers against 60 staged); narrower rows are held in
// registers by the register kernel; what neither takes goes to the
// three-pass kernel.
// The streamed kernel with every row over the whole grid (few rows of tens
// of MB): the CTA shape of sm_plan_stream, one CTA per SM, all resident (a
// cooperative launch; opt->grid of them at most), each owning a contiguous
// slice of every row; the CTAs' (maximum, sum) pairs meet in global scratch.
rmsnorm_status_t sm_plan_stream_grid(const SmCall& c, SmPlan* P) {
    int vb;
    rmsnorm_status_t st = sm_pick_vb(c, &vb);
    if (st != RMSNORM_OK) return st;
    if (vb != 16 || c.opt.cluster > 1) return RMSNORM_ERR_UNSUPPORTED;
    const int64_t row_bytes = c.cols * c.sz;
    const int64_t nvec = row_bytes / 16;
    // one producer warp and one exchange warp beside the consumers
    const int max_nc = softmax_stream_max_threads() - 64;
    const int nc = c.opt.threads > 0 ? c.opt.threads : max_nc;
    if (nc % 32 != 0 || nc > max_nc) return RMSNORM_ERR_UNSUPPORTED;
    int v = 4;
    if (c.opt.chunk_bytes != 0) {
        if (c.opt.chunk_bytes == 2 * 16 * nc) v = 2;
        else if (c.opt.chunk_bytes == 4 * 16 * nc) v = 4;
        else return RMSNORM_ERR_UNSUPPORTED;
    }
    const int64_t chunk = static_cast<int64_t>(16) * v * nc;
    const int64_t budget = c.dv.smem_optin - kStreamHeaderHost;
    int64_t slots = c.opt.stages ? c.opt.stages : budget / chunk;
    if (!c.opt.stages && slots > kStagedMaxSlotsHost) slots = kStagedMaxSlotsHost;
    if (slots < 2 || slots > kStagedMaxSlotsHost || slots * chunk > budget)
        return RMSNORM_ERR_UNSUPPORTED;
    KernelFn fn = softmax_grid_ptr(c.dtype, v);
    if (!fn) return RMSNORM_ERR_UNSUPPORTED;
    const int block = nc + 64;
    const int smem = static_cast<int>(kStreamHeaderHost + slots * chunk);
    int occ = 0;
    if (cached_occupancy(c.dv.dev, c.dv.smem_optin, fn, block, smem, 1, &occ) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    if (occ <= 0) return RMSNORM_ERR_UNSUPPORTED;
    int64_t resident = static_cast<int64_t>(c.dv.sms) * occ;
    if (resident > kGridMaxCtasHost) resident = kGridMaxCtasHost;
    if (c.opt.grid > resident) return RMSNORM_ERR_UNSUPPORTED;
    const int64_t grid = c.opt.grid > 0 ? c.opt.grid : resident;
    // the arrival counter counts grid * rows arrivals in 32 bits
    if (c.rows > 0xFFFFFFFFll / grid) return RMSNORM_ERR_UNSUPPORTED;
    const int64_t per = (nvec + grid - 1) / grid;
    *P = SmPlan{};             // every field this plan does not set keeps its default
    P->path = RMSNORM_PATH_GRID;
    P->cluster = 1;
    P->slice_vecs = static_cast<int>(per);
    P->group = nc;
    P->block = block;
    P->rpc = 1;
    P->grid = static_cast<int>(grid);
    P->vb = 16;
    P->nv = v;
    P->nvec = static_cast<int>(nvec);
    P->smem = smem;
    P->chunk = static_cast<int>(chunk);
    P->nchunks = static_cast<int>((per * 16 + chunk - 1) / chunk);
    // Chunks of the next row read while the CTAs' pairs meet.  Measured on
    // fp32 rows (% of the HBM copy peak; 1 / 2 / 3 / 4 / 8 chunks): rows of
    // 16 MiB, four chunks per slice, 63.4 / 65.4 / 66.4 / 68.5 / 68.4 (the
    // whole next slice); 32 MiB, eight chunks, 77.9 / 78.0 / 76.0 / 73.8 /
    // 68.9; 64 MiB, sixteen chunks, 59.8 / 60.4 / 61.4 / 61.7 / 62.7.
    P->read_ahead = P->nchunks <= 4 ? P->nchunks : P->nchunks <= 12 ? 2 : 4;
    // Row schedule: a row's second read interleaved with the next row's first
    // read, or phased (second read, then the next first read).  Measured
    // (interleaved / phased / phased reversed): fp32 rows of 24 MiB 72 / 67 /
    // 67, 32 MiB 76 / 62 / 63, 40 MiB 69 / 62 / 61, 64 MiB 62 / 65 / 62; bf16
    // rows of 64 MiB 61 / 65 / 61.  Interleaving puts about two rows of
    // traffic between a chunk's two reads, more than L2 keeps for the widest
    // rows.
    P->schedule = P->nchunks > 12 ? 1 : 0;
    // Phased rows keep chunks D .. D + R - 1 of every slice in shared memory
    // between the two reads, R = the slots beyond a ring of four: L2 then
    // holds less of the row.  Measured on rows of 64 MiB (R = 0 / 2 / 4):
    // fp32 65.0 / 71.6 / 72.4%, bf16 67.6 / 72.4 / 71.7%.  Narrower rows stay
    // interleaved: phased with resident chunks, fp32 rows of 24 / 32 / 40 MiB
    // measured 58 / 62 / 64% against 71 / 74 / 70%.
    P->res_chunks = grid_resident_chunks(P->schedule, static_cast<int>(slots), P->nchunks,
                                         P->read_ahead, c.opt.stages != 0);
    P->nslots = static_cast<int>(slots) - P->res_chunks;
    P->scratch = grid_scratch_bytes(static_cast<int>(grid));
    P->fn = fn;
    P->name = "softmax_grid_stream";
    return RMSNORM_OK;
}

// The streamed kernel, automatically: rows of at least 128 KB that the
// register-resident staged kernel cannot hold (fp32 rows of more than 32768
// elements, bf16 rows of 65536 and more), from a quarter of the SM count of
// rows up.  Each row is split over C CTAs, C the smallest power of two that
// keeps slices within 400 KB (the rows in flight on all SMs, whose second
// read must find them in L2, then stay within about 60 MB) and, for fewer
// rows than SMs, gives at least half the SMs a slice.  Measured (1 GB
// inputs, % of the measured HBM copy peak; streamed / previous automatic
// choice): fp32 rows of 36000 / 40000 / 65536 elements 95 / 93 / 93 against
// 85 / 82 / 83, of 100000 and 200000 (C = 2) 86 / 87 against 63 / 53, of
// 128256 (prefill logits, C = 2) 83 against 74, of 262144 (C = 4) 87 against
// 66; bf16 rows of 98304 / 128256 91 / 89 against 75 / 69, of 262144 (C = 2)
// 93 against 59; bf16 rows of 49152 86 for the three-pass kernel against 79
// streamed.  One CTA per row where slices of two would do loses on L2
// (fp32 rows of 128256: 78%), clusters of 3, 5 or 6 leave SMs idle.  Few
// rows: 64 rows of 128256 elements take 14.7 us (bf16) and 20.9 us (fp32)
// streamed over clusters of two against 16.3 and 30.1 us for the register
// split, but 8 fp32 rows 10.4 us against 8.7 us, so fewer than a quarter of
// the SM count of rows stay with the register split.
bool sm_stream_eligible(const SmCall& c) {
    const int64_t row_bytes = c.cols * c.sz;
    if (row_bytes < kSoftmaxStreamMinRowBytes) return false;
    if (c.dtype == RMSNORM_DTYPE_F32 && c.cols <= 32768) return false;
    return 4 * c.rows >= c.dv.sms;
}

rmsnorm_status_t sm_plan_stream_auto(const SmCall& c, SmPlan* P) {
    const int64_t row_bytes = c.cols * c.sz;
    int cl = 1;
    while (cl < kSoftmaxStreamMaxCluster && (row_bytes + cl - 1) / cl > kSoftmaxStreamMaxSlice)
        cl <<= 1;
    while (cl < kSoftmaxStreamMaxCluster && 2 * c.rows * cl < c.dv.sms) cl <<= 1;
    for (; cl >= 1; cl >>= 1) {
        SmPlan Q;
        const rmsnorm_status_t st = sm_plan_stream(c, cl, &Q);
        if (st == RMSNORM_ERR_CUDA) return st;
        if (st == RMSNORM_OK) {
            *P = Q;
            return RMSNORM_OK;
        }
    }
    return RMSNORM_ERR_UNSUPPORTED;
}

rmsnorm_status_t sm_make_plan(const SmCall& c, SmPlan* P) {
    switch (c.opt.path) {
        case RMSNORM_PATH_ROWREG: return sm_plan_rowreg(c, 1, P);
        case RMSNORM_PATH_CLUSTER: return sm_plan_rowreg(c, c.opt.cluster ? c.opt.cluster : 2, P);
        case RMSNORM_PATH_TWOPASS:
            return sm_plan_threepass(c, c.opt.cluster ? c.opt.cluster : 1, P);
        case RMSNORM_PATH_STAGED: return sm_plan_staged(c, c.opt.cluster ? c.opt.cluster : 1, P);
        case RMSNORM_PATH_STREAM: return sm_plan_stream(c, c.opt.cluster ? c.opt.cluster : 1, P);
        case RMSNORM_PATH_GRID: return sm_plan_stream_grid(c, P);
        default: break;
    }
    const int64_t row_bytes = c.cols * c.sz;
    rmsnorm_status_t st;
    // Few rows of tens of MB totalling more than L2 can hold at once: each
    // row over the whole grid in turn, so that its second read finds it in
    // L2.  Measured (% of the HBM copy peak, against the three-pass kernel
    // split over clusters, which reads x three times): eight fp32 rows of
    // 64 MiB 72 against 40 (clusters of 12), sixteen rows of 32 MiB 74-79
    // against 31 (8), thirty-two rows of 16 MiB 69 against 45 (4).  Rows of
    // 8 MiB exchange too often: 50 against 67 for the streamed kernel split
    // over clusters of 8 (fp32 and bf16 alike).
    if (c.rows < c.dv.sms && row_bytes >= kSoftmaxGridMinRowBytes &&
        c.rows * row_bytes >= kSoftmaxGridMinBytes) {
        st = sm_plan_stream_grid(c, P);
        if (st == RMSNORM_OK || st == RMSNORM_ERR_CUDA) return st;
    }
    if (sm_stream_eligible(c)) {
        st = sm_plan_stream_auto(c, P);
        if (st == RMSNORM_OK || st == RMSNORM_ERR_CUDA) return st;
    }
    if (c.rows < c.dv.sms && (row_bytes > kSoftmaxSplitRowBytes ||
                              c.rows * row_bytes >= kSoftmaxSplitMinBytes)) {
        int want = 1;
        while (static_cast<int64_t>(want) * 2 * c.rows <= c.dv.sms && want < 8) want <<= 1;
        while (want > 1 && row_bytes / want < 4096) want >>= 1;
        for (int cl = want; cl > 1 && cl <= 16; cl <<= 1) {
            st = sm_plan_rowreg(c, cl, P);
            if (st == RMSNORM_OK || st == RMSNORM_ERR_CUDA) return st;
        }
    }
    if (c.cols > (c.dtype == RMSNORM_DTYPE_BF16 ? kSoftmaxStagedMinColsBf16 : kSoftmaxStagedMinCols)) {
        st = sm_plan_staged(c, 1, P);
        if (st == RMSNORM_OK || st == RMSNORM_ERR_CUDA) return st;
        // Rows too wide for one CTA's registers: split each over the smallest
        // cluster whose slices fit (up to 8 CTAs), where that beats the
        // three-pass kernel.  Measured on 1 GB inputs (% of the HBM roofline,
        // split / three-pass): the three-pass kernel holds up while 304 rows
        // fit L2 for its re-reads (rows of 128-200 KB: 70-80%) and falls to
        // 48-55% on rows of 400 KB and more; the split runs at 54-84% for fp32
        // rows (65536 elements 84 / 69, 100000 64 / 55, 128256 78 / 51,
        // 262144 67 / 49; 48000 72 / 80), and for bf16 rows only when the
        // slices fill the CTAs' registers (128256 elements, 98% full: 72 /
        // 67; 262144, full: 60 / 51; 100000 and 200000, 76% full: 60 / 70
        // and 49 / 54).
        if (row_bytes >= kSoftmaxSplitStagedMinRowBytes) {
            for (int cl = 2; cl <= kSoftmaxMaxStagedCluster; cl <<= 1) {
                SmPlan Q;          // P stays untouched unless the split is taken
                st = sm_plan_staged(c, cl, &Q);
                if (st == RMSNORM_ERR_CUDA) return st;
                if (st != RMSNORM_OK) continue;
                const int64_t capacity = static_cast<int64_t>(softmax_staged_max_threads()) * 8 * 16;
                if (c.dtype == RMSNORM_DTYPE_F32 ||
                    16 * static_cast<int64_t>(Q.slice_vecs) * 16 >= 15 * capacity) {
                    *P = Q;
                    return RMSNORM_OK;
                }
                break;             // bf16 slices not full enough: three-pass
            }
        }
    }
    st = sm_plan_rowreg(c, 1, P);
    if (st == RMSNORM_OK || st == RMSNORM_ERR_CUDA) return st;
    // Few rows too wide for any of the above: the three-pass kernel, each row
    // over a cluster.
    if (c.rows < c.dv.sms) {
        st = sm_plan_threepass_split(c, P);
        if (st == RMSNORM_OK || st == RMSNORM_ERR_CUDA) return st;
    }
    st = sm_plan_threepass(c, 1, P);
    if (st != RMSNORM_ERR_UNSUPPORTED) return st;
    return sm_plan_threepass_split(c, P);   // rows too wide for one CTA's 32-bit index
}

rmsnorm_status_t sm_run(int32_t dtype, const void* x, void* y, int64_t rows, int64_t cols,
                        const rmsnorm_options_t* opt, cudaStream_t stream) {
    SmCall c;
    rmsnorm_status_t st = sm_validate(dtype, x, y, rows, cols, opt, &c);
    if (st != RMSNORM_OK) return st;
    if (rows == 0) return RMSNORM_OK;
    if (current_device(&c.dv) != cudaSuccess) return RMSNORM_ERR_CUDA;
    SmPlan P;
    st = sm_make_plan(c, &P);
    if (st != RMSNORM_OK) return st;
    Params p;
    std::memset(&p, 0, sizeof(p));
    p.x = x;
    p.y = y;
    p.rows = rows;
    p.hidden = static_cast<int32_t>(cols);
    p.nvec = P.nvec;
    p.group = P.group;
    p.rows_per_cta = P.rpc;
    p.cluster = P.cluster;
    p.slice_vecs = P.slice_vecs;
    p.chunk_bytes = P.chunk;
    p.nchunks = P.nchunks;
    p.nslots = P.nslots;
    p.read_ahead = P.read_ahead;
    p.schedule = P.schedule;
    p.resident = P.res_chunks;
    p.status = c.dv.status;
    p.fault = c.opt.fault_inject;
    p.timeout_ns = c.opt.wait_timeout_ns ? c.opt.wait_timeout_ns : kDefaultTimeoutNs;
    LaunchShape s{P.grid, P.block, P.cluster, P.smem};
    if (ensure_prepared(c.dv.dev, P.fn, c.dv.smem_optin) != cudaSuccess) return RMSNORM_ERR_CUDA;
    if (P.scratch > 0) {
        s.cooperative = true;
        if (launch_with_pool_scratch(P.fn, s, stream, p, static_cast<size_t>(P.scratch)) !=
            cudaSuccess)
            return RMSNORM_ERR_CUDA;
        return RMSNORM_OK;
    }
    if (note(launch_ex(P.fn, s, stream, p)) != cudaSuccess) return RMSNORM_ERR_CUDA;
    return RMSNORM_OK;
}

}  // namespace
}  // namespace rmsnorm

using namespace rmsnorm;

extern "C" {

rmsnorm_status_t rowsoftmax_fwd_f32(const float* x, float* y, int64_t rows, int64_t cols,
                                    rmsnorm_stream_t stream) {
    return sm_run(RMSNORM_DTYPE_F32, x, y, rows, cols, nullptr,
                  reinterpret_cast<cudaStream_t>(stream));
}

rmsnorm_status_t rowsoftmax_fwd_bf16(const uint16_t* x, uint16_t* y, int64_t rows,
                                     int64_t cols, rmsnorm_stream_t stream) {
    return sm_run(RMSNORM_DTYPE_BF16, x, y, rows, cols, nullptr,
                  reinterpret_cast<cudaStream_t>(stream));
}

rmsnorm_status_t rowsoftmax_fwd_ex(int32_t dtype, const void* x, void* y, int64_t rows,
                                   int64_t cols, const rmsnorm_options_t* opt,
                                   rmsnorm_stream_t stream) {
    return sm_run(dtype, x, y, rows, cols, opt, reinterpret_cast<cudaStream_t>(stream));
}

rmsnorm_status_t rowsoftmax_plan(int32_t dtype, const void* x, const void* y, int64_t rows,
                                 int64_t cols, const rmsnorm_options_t* opt,
                                 rmsnorm_plan_t* plan) {
    if (!plan) return RMSNORM_ERR_INVALID_ARG;
    SmCall c;
    rmsnorm_status_t st = sm_validate(dtype, x, y, rows, cols, opt, &c);
    if (st != RMSNORM_OK) return st;
    if (current_device(&c.dv) != cudaSuccess) return RMSNORM_ERR_CUDA;
    if (c.rows == 0) c.rows = 1;
    SmPlan P;
    st = sm_make_plan(c, &P);
    if (st != RMSNORM_OK) return st;
    std::memset(plan, 0, sizeof(*plan));
    plan->path = P.path;
    plan->cluster = P.cluster;
    plan->threads_per_row = P.group;
    plan->block_threads = P.block;
    plan->rows_per_cta = P.rpc;
    plan->grid = P.grid;
    plan->vec_bytes = P.vb;
    plan->vecs_per_thread = P.nv;
    plan->smem_bytes = P.smem;
    plan->chunk_bytes = P.chunk;
    plan->stages = P.nslots;
    std::snprintf(plan->kernel, sizeof(plan->kernel), "%s", P.name);
    return RMSNORM_OK;
}

}  // extern "C"
