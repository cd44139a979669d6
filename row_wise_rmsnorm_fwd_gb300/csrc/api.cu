// api.cu -- the C ABI of librmsnorm: argument validation, per-device set-up,
// kernel-family selection (the launch heuristics) and the launch itself.
//
// Operation: page "A hackable Python ML compiler, part 2", RMSNorm Loop IR:
// y[r,j] = (x[r,j] * rsqrt(mean_j x[r,j]^2 + eps)) * w[j].
#include "rmsnorm.h"
#include "launch.h"
#include "device.h"

#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

namespace rmsnorm {

KernelFn rowreg_kernel_ptr(int dtype, int vb, int nv, bool pf, int epi) {
    using Pick = KernelFn (*)(int, int, bool);
    static const Pick table[2][3] = {
        {rowreg_kernel_f32_e0, rowreg_kernel_f32_e1, rowreg_kernel_f32_e2},
        {rowreg_kernel_bf16_e0, rowreg_kernel_bf16_e1, rowreg_kernel_bf16_e2}};
    if (dtype < 0 || dtype > 1 || epi < 0 || epi > 2) return nullptr;
    return table[dtype][epi](vb, nv, pf);
}
int rowreg_max_block(int nv) { return nv >= 4 ? 512 : 1024; }

namespace {

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;   // 2 s

constexpr int kRowregBlocksPerCta = 3;   // row blocks each CTA of the row kernel works on
constexpr int64_t kStagedChunk = 16384;   // bytes per bulk copy
constexpr int64_t kStagedLookahead = 2;   // ring slots beyond one row slice
constexpr int kStagedConsumerWarps = 8;       // default consumer warps per CTA (fp32)
constexpr int kStagedConsumerWarpsBf16 = 4;   // default consumer warps per CTA (bf16)
constexpr int64_t kRowregMaxRowBytes = 32768;   // auto: register-resident up to here
constexpr int64_t kStagedMaxRowBytes = 65536;   // auto: fp32 staged up to here
constexpr int kAutoMaxCluster = 8;              // auto: portable cluster sizes only
constexpr int64_t kSplitMinBytes = 16 << 20;    // auto: split narrow few-row inputs from here
constexpr int kRingregSlots = 3;                 // ring-to-register kernel: ring slots
constexpr int64_t kGridMinRowBytes = 10ll << 20;     // auto: rows over the whole grid from here
constexpr int kGridReadAheadRmsNorm = 2;             // see plan_grid
constexpr int64_t kGridInterleavedMaxRowBytes = 24ll << 20;   // see plan_grid
constexpr int64_t kGridMaxRowBytes = 40ll << 20;     //   to here
constexpr int64_t kRingregLowMaxRowBytes = 57344;    // auto: ringreg for rows above 32 KB to here
constexpr int64_t kRingregHighMinRowBytes = 114688;  // auto: and above this (to 128 KB)
constexpr int64_t kUnsplitMaxVecs = 0x7FFFFFFFll - 1024;  // two-pass, one CTA per row: up to here

struct Call {
    int dtype;
    int sz;                 // element bytes
    uintptr_t x, w, y;
    int64_t rows;
    int64_t hidden;
    rmsnorm_options_t opt;
    int dev;
    const DeviceView* info;
    DeviceView view;
};

struct Plan {
    int path = 0;
    int cluster = 1;
    int group = 0;
    int block = 0;
    int rpc = 1;
    int grid = 0;
    int vb = 0;
    int nv = 0;
    int smem = 0;
    int chunk = 0;
    int nchunks = 0;
    int nslots = 0;
    int w_staged = 0;
    int nvec = 0;
    int slice_vecs = 0;
    int resident = 0;       // resident CTAs per SM, or resident clusters (split rows)
    int scratch = 0;        // grid-split kernels: bytes of cleared scratch (cooperative launch)
    int read_ahead = 0;     // grid-split kernels: next-row chunks read during an exchange
    int schedule = 0;       // grid-split kernels: row schedule
    int res_chunks = 0;     // grid-split kernels: slice chunks kept in shared memory
    KernelFn fn = nullptr;
    const char* name = "";
};

int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }
int round_up(int64_t a, int64_t b) { return static_cast<int>(((a + b - 1) / b) * b); }
int pow2_ceil(int v) { int p = 1; while (p < v) p <<= 1; return p; }
int pow2_floor(int64_t v) { int p = 1; while (static_cast<int64_t>(p) * 2 <= v) p <<= 1; return p; }

// Widest vector width that the pointers and the row pitch allow.
int widest_vb(const Call& c) {
    const uintptr_t a = c.x | c.w | c.y;
    const int64_t pitch = c.hidden * c.sz;
    for (int vb = 16; vb >= c.sz; vb >>= 1)
        if (a % vb == 0 && pitch % vb == 0) return vb;
    return c.sz;
}

rmsnorm_status_t pick_vb(const Call& c, int* vb) {
    const int widest = widest_vb(c);
    const int f = c.opt.vec_bytes;
    if (f == 0) { *vb = widest; return RMSNORM_OK; }
    if (f != 2 && f != 4 && f != 8 && f != 16) return RMSNORM_ERR_INVALID_ARG;
    if (f < c.sz || f > widest) return RMSNORM_ERR_UNSUPPORTED;
    *vb = f;
    return RMSNORM_OK;
}

// Register-resident kernel; cluster > 1 splits each row over a cluster.
rmsnorm_status_t plan_rowreg(const Call& c, int cluster, Plan* P) {
    int vb;
    rmsnorm_status_t st = pick_vb(c, &vb);
    if (st != RMSNORM_OK) return st;
    const int epv = vb / c.sz;
    const int64_t nvec = c.hidden / epv;
    const int64_t per = cluster > 1 ? (nvec + cluster - 1) / cluster : nvec;
    int G, NV;
    if (c.opt.threads > 0) {
        G = c.opt.threads;
        const bool sub_warp = G < 32 && (G & (G - 1)) == 0;   // 1, 2, 4, 8, 16
        if ((G % 32 != 0 && !sub_warp) || G > 1024) return RMSNORM_ERR_INVALID_ARG;
        if (sub_warp && cluster > 1) return RMSNORM_ERR_UNSUPPORTED;
        const int64_t need = (per + G - 1) / G;
        if (need > 8) return RMSNORM_ERR_UNSUPPORTED;
        NV = pow2_ceil(static_cast<int>(need));
    } else if (cluster == 1 && per <= 32 * 4) {
        // rows of up to 128 vectors: 4 vectors per thread (fewer for rows of
        // fewer than 4) and pow2(vectors / 4) lanes per row, so a warp holds
        // 32 / G rows.  Measured (% of the measured HBM peak), bf16 rows of
        // 64 / 128 / 256 / 512 elements: 98 / 103 / 103 / 103 with 4 vectors
        // per thread, against 75 / 75 / 76 / 93 with one or two vectors per
        // thread of a full warp per row.
        NV = per >= 4 ? 4 : pow2_ceil(static_cast<int>(per));
        G = pow2_ceil(ceil_div(per, NV));
    } else {
        // 4 vectors per thread (64 B at 16-byte vectors) with a register double
        // buffer; rows wider than 512 threads x 4 vectors use 8 per thread.
        NV = 4;
        int64_t g = round_up((per + NV - 1) / NV, 32);
        if (g > rowreg_max_block(NV)) {
            NV = 8;
            g = round_up((per + NV - 1) / NV, 32);
        }
        if (g > rowreg_max_block(NV)) return RMSNORM_ERR_UNSUPPORTED;
        // With 16-byte vectors, 3 vectors per thread when that leaves fewer
        // idle lanes than 4 and 4 leaves more than 1/16 of them idle.
        // Measured (% of the measured HBM peak): bf16 rows of 1536 elements
        // 96.4 with 3 x 64 lanes, none idle, against 94.3 with 4 x 64 lanes,
        // a quarter idle; fp32 rows of 768 101.8 against 101.0.  5, 6 or 7
        // vectors (about 120 registers, half the CTAs per SM) measured no
        // better or worse (bf16 rows of 2560: 91.4 with 5 against 96.0).
        if (vb == 16 && NV == 4 && (g * NV - per) * 16 > per) {
            const int64_t g3 = round_up((per + 2) / 3, 32);
            if (g3 <= rowreg_max_block(3) && g3 * 3 - per < g * NV - per) {
                NV = 3;
                g = g3;
            }
        }
        G = static_cast<int>(g);
    }
    if (G > rowreg_max_block(NV)) return RMSNORM_ERR_UNSUPPORTED;
    KernelFn fn = rowreg_kernel_ptr(c.dtype, vb, NV, cluster > 1, c.opt.epilogue);
    if (!fn) return RMSNORM_ERR_UNSUPPORTED;
    const int rpc = cluster == 1 ? (G >= 256 ? 1 : 256 / G) : 1;
    const int block = G * rpc;
    int occ = 0;
    if (cached_occupancy(c.dev, c.info->smem_optin, fn, block, 0, cluster, &occ) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    if (occ <= 0) return RMSNORM_ERR_UNSUPPORTED;
    int grid;
    if (cluster == 1) {
        // Grid-stride over row blocks with k whole waves of resident CTAs, k =
        // the row blocks per resident CTA slot / 3 (at least 1): every CTA
        // works on about three row blocks, so the next-row prefetch has
        // something to fetch and the weight slice loaded per CTA is reused,
        // while CTAs start and finish all the time, which keeps them out of
        // phase (loads, reductions and stores of different CTAs overlap).
        // Measured on GB300 (% of the measured HBM copy peak): c5a with 16 /
        // 48 / 120 / 143 / 431 waves (27 / 9 / 3.6 / 3.0 / 1 row blocks per
        // CTA) 101.5 / 103.3 / 104.3 / 104.2 / 88.9%; c4 with 16 / 35 / 48 /
        // 96 waves (6.7 / 3.1 / 2.2 / 1.1) 102.3 / 103.4 / 104.1 / 98.3%;
        // c3 (3.4 row blocks per slot) 1 wave 12.8 us against 14.9 us with
        // one CTA per row block.  Fewer row blocks than resident slots: one
        // CTA each.
        const int64_t nblocks = (c.rows + rpc - 1) / rpc;
        const int64_t resident = static_cast<int64_t>(c.info->sms) * occ;
        int64_t waves = nblocks / (kRowregBlocksPerCta * resident);
        if (waves < 1) waves = 1;
        const int64_t target = resident * waves;
        grid = static_cast<int>(c.opt.grid > 0 ? c.opt.grid
                                               : (nblocks < target ? nblocks : target));
    } else {
        const int64_t nclusters = c.opt.grid > 0 ? (c.opt.grid + cluster - 1) / cluster
                                                 : (c.rows < occ ? c.rows : occ);
        grid = static_cast<int>(nclusters * cluster);
    }
    P->path = cluster == 1 ? RMSNORM_PATH_ROWREG : RMSNORM_PATH_CLUSTER;
    P->cluster = cluster;
    P->group = G;
    P->block = block;
    P->rpc = rpc;
    P->grid = grid;
    P->vb = vb;
    P->nv = NV;
    P->smem = 0;
    P->nvec = static_cast<int>(nvec);
    P->slice_vecs = static_cast<int>(per);
    P->fn = fn;
    P->name = cluster == 1 ? "rowreg" : "cluster_rowreg";
    return RMSNORM_OK;
}

// Bulk-copy staged kernel; needs 16-byte aligned pointers and row pitch.
// Geometry (measured on GB300): chunks of 16 KB (32 KB for slices of 64 KB
// and more), a ring of chunks-per-slice + 2 slots, and the weight slice in
// shared memory when it fits next to the ring.  Deeper rings cost occupancy
// and measured slower.
rmsnorm_status_t plan_staged(const Call& c, int cluster, Plan* P) {
    if (c.opt.vec_bytes != 0 && c.opt.vec_bytes != 16) return RMSNORM_ERR_UNSUPPORTED;
    if (widest_vb(c) != 16) return RMSNORM_ERR_UNSUPPORTED;
    const int64_t row_bytes = c.hidden * c.sz;
    const int64_t vecs = row_bytes / 16;
    const int64_t slice_vecs = (vecs + cluster - 1) / cluster;
    const int64_t slice_bytes = slice_vecs * 16;
    const int64_t budget = c.info->smem_optin;
    if (slice_bytes + kStagedHeaderHost > budget) return RMSNORM_ERR_UNSUPPORTED;
    int64_t chunk = c.opt.chunk_bytes;
    if (chunk != 0) {
        if (chunk % 16 != 0 || chunk <= 0) return RMSNORM_ERR_INVALID_ARG;
    } else {
        const int64_t pref = slice_bytes >= 4 * kStagedChunk ? 2 * kStagedChunk : kStagedChunk;
        chunk = slice_bytes < pref ? slice_bytes : pref;
    }
    int64_t nchunks = (slice_bytes + chunk - 1) / chunk;
    if (nchunks > kStagedMaxSlotsHost) {
        if (c.opt.chunk_bytes != 0) return RMSNORM_ERR_UNSUPPORTED;
        chunk = round_up((slice_bytes + kStagedMaxSlotsHost - 1) / kStagedMaxSlotsHost, 16);
        nchunks = (slice_bytes + chunk - 1) / chunk;
    }
    // Ring slots: forced, or chunks per slice + lookahead, within the budget.
    const int wmode = c.opt.weights;
    if (wmode < 0 || wmode > 2 || c.opt.stages < 0) return RMSNORM_ERR_INVALID_ARG;
    auto fits = [&](int64_t slots, int64_t wbytes) {
        return kStagedHeaderHost + wbytes + slots * chunk <= budget;
    };
    int64_t want = c.opt.stages > 0 ? c.opt.stages : nchunks + kStagedLookahead;
    if (want > kStagedMaxSlotsHost) want = kStagedMaxSlotsHost;
    if (want < nchunks) return RMSNORM_ERR_UNSUPPORTED;
    bool wstaged;
    if (wmode == 1) {
        wstaged = true;
    } else if (wmode == 2) {
        wstaged = false;
    } else {
        wstaged = fits(want, slice_bytes);
    }
    const int64_t wres = wstaged ? slice_bytes : 0;
    int64_t slots = want;
    while (slots > nchunks && !fits(slots, wres)) --slots;
    if (!fits(slots, wres)) return RMSNORM_ERR_UNSUPPORTED;
    if (c.opt.stages > 0 && slots != c.opt.stages) return RMSNORM_ERR_UNSUPPORTED;
    const int64_t smem = staged_smem_bytes(chunk, static_cast<int>(slots), wres);
    if (smem <= 0 || smem > budget) return RMSNORM_ERR_UNSUPPORTED;
    // Consumer warps: forced through `threads` (128 or 256), else 8, or 4 for
    // bf16 slices of at most 16 KB (measured: 92.5% vs 78.9% on 16 KB bf16
    // rows, but 38.8% vs 51.1% on 128 KB ones).
    int ncw = (c.dtype == RMSNORM_DTYPE_BF16 && slice_bytes <= kStagedChunk)
                  ? kStagedConsumerWarpsBf16 : kStagedConsumerWarps;
    if (c.opt.threads != 0) {
        if (c.opt.threads != 128 && c.opt.threads != 256) return RMSNORM_ERR_UNSUPPORTED;
        ncw = c.opt.threads / 32;
    }
    const int block = 32 * (ncw + 1);
    KernelFn fn = staged_kernel_ptr(c.dtype, ncw, c.opt.epilogue);
    if (!fn) return RMSNORM_ERR_UNSUPPORTED;
    int occ = 0;
    if (cached_occupancy(c.dev, c.info->smem_optin, fn, block, static_cast<int>(smem), cluster, &occ) !=
        cudaSuccess)
        return RMSNORM_ERR_CUDA;
    if (occ <= 0) return RMSNORM_ERR_UNSUPPORTED;
    int grid;
    if (cluster == 1) {
        const int64_t resident = static_cast<int64_t>(c.info->sms) * occ;
        grid = static_cast<int>(c.opt.grid > 0 ? c.opt.grid
                                               : (c.rows < resident ? c.rows : resident));
    } else {
        const int64_t nclusters = c.opt.grid > 0 ? (c.opt.grid + cluster - 1) / cluster
                                                 : (c.rows < occ ? c.rows : occ);
        grid = static_cast<int>(nclusters * cluster);
    }
    P->path = RMSNORM_PATH_STAGED;
    P->cluster = cluster;
    P->group = 32 * ncw;
    P->block = block;
    P->rpc = 1;
    P->grid = grid;
    P->vb = 16;
    P->nv = 0;
    P->smem = static_cast<int>(smem);
    P->chunk = static_cast<int>(chunk);
    P->nchunks = static_cast<int>(nchunks);
    P->nslots = static_cast<int>(slots);
    P->w_staged = wstaged ? 1 : 0;
    P->nvec = static_cast<int>(vecs);
    P->slice_vecs = static_cast<int>(slice_vecs);
    P->fn = fn;
    P->name = cluster == 1 ? "staged_bulk" : "staged_bulk_cluster";
    return RMSNORM_OK;
}

// Ring-to-register kernel for wide rows: 16-byte vectors only (bulk copies
// of whole 16-byte-aligned rows); the fewest vectors per consumer thread (8
// or 16) that cover the row with at most 512 consumer threads (or
// opt->threads consumer threads); chunks of M = 4 vectors per consumer
// thread (32 KB at 512 threads; opt->chunk_bytes may ask for M = 2) and a
// ring of 3 slots (or opt->stages, at least 2).  Measured on 1.5 GB inputs of
// rows from 36 to 128 KB: deeper rings were slower, down to 70-80% of the
// HBM roofline with 16 or more slots, and M = 4 with 3 slots was the best or
// within 3 points of it wherever this kernel is chosen automatically.
rmsnorm_status_t plan_ringreg(const Call& c, Plan* P) {
    if (c.opt.vec_bytes != 0 && c.opt.vec_bytes != 16) return RMSNORM_ERR_UNSUPPORTED;
    if (widest_vb(c) != 16) return RMSNORM_ERR_UNSUPPORTED;
    if (c.opt.weights != 0 || c.opt.cluster > 1) return RMSNORM_ERR_UNSUPPORTED;
    const int64_t row_bytes = c.hidden * c.sz;
    const int64_t nvec = row_bytes / 16;
    const int max_nt = ringreg_max_consumers();
    int nv = 8, nt;
    if (c.opt.threads > 0) {
        nt = c.opt.threads;
        if (nt % 32 != 0 || nt > max_nt) return RMSNORM_ERR_UNSUPPORTED;
        if (static_cast<int64_t>(nv) * nt < nvec) nv = 16;
        if (static_cast<int64_t>(nv) * nt < nvec) return RMSNORM_ERR_UNSUPPORTED;
    } else {
        if (static_cast<int64_t>(nv) * max_nt < nvec) nv = 16;
        if (static_cast<int64_t>(nv) * max_nt < nvec) return RMSNORM_ERR_UNSUPPORTED;
        nt = round_up((nvec + nv - 1) / nv, 32);
    }
    int m = 4;
    if (c.opt.chunk_bytes != 0) {
        if (c.opt.chunk_bytes == 2 * nt * 16) m = 2;
        else if (c.opt.chunk_bytes == 4 * nt * 16) m = 4;
        else return RMSNORM_ERR_UNSUPPORTED;
    }
    const int64_t chunk = static_cast<int64_t>(m) * nt * 16;
    const int64_t nchunks = (row_bytes + chunk - 1) / chunk;
    const int64_t wres = (row_bytes + 127) / 128 * 128;
    const int64_t budget = c.info->smem_optin - kStagedHeaderHost - wres;
    if (c.opt.stages < 0) return RMSNORM_ERR_INVALID_ARG;
    int64_t slots = c.opt.stages ? c.opt.stages : kRingregSlots;
    if (!c.opt.stages && slots * chunk > budget) slots = budget / chunk;
    if (slots < 2 || slots > kStagedMaxSlotsHost || slots * chunk > budget)
        return RMSNORM_ERR_UNSUPPORTED;
    KernelFn fn = ringreg_kernel_ptr(c.dtype, nv, m, c.opt.epilogue);
    if (!fn) return RMSNORM_ERR_UNSUPPORTED;
    const int block = nt + 32;
    const int64_t smem = kStagedHeaderHost + wres + slots * chunk;
    int occ = 0;
    if (cached_occupancy(c.dev, c.info->smem_optin, fn, block, static_cast<int>(smem), 1, &occ) !=
        cudaSuccess)
        return RMSNORM_ERR_CUDA;
    if (occ <= 0) return RMSNORM_ERR_UNSUPPORTED;
    const int64_t resident = static_cast<int64_t>(c.info->sms) * occ;
    P->path = RMSNORM_PATH_RINGREG;
    P->cluster = 1;
    P->group = nt;
    P->block = block;
    P->rpc = 1;
    P->grid = static_cast<int>(c.opt.grid > 0 ? c.opt.grid
                                              : (c.rows < resident ? c.rows : resident));
    P->vb = 16;
    P->nv = nv;
    P->smem = static_cast<int>(smem);
    P->chunk = static_cast<int>(chunk);
    P->nchunks = static_cast<int>(nchunks);
    P->nslots = static_cast<int>(slots);
    P->w_staged = 1;
    P->nvec = static_cast<int>(nvec);
    P->slice_vecs = static_cast<int>(nvec);
    P->fn = fn;
    P->name = "ringreg";
    return RMSNORM_OK;
}

// Generic fallback: any width and alignment.
// Two-pass kernel; cluster > 1 splits each row over a thread-block cluster
// (slices of whole 32-vector groups, CTA totals combined through DSMEM).
rmsnorm_status_t plan_twopass(const Call& c, int cluster, Plan* P) {
    int vb;
    rmsnorm_status_t st = pick_vb(c, &vb);
    if (st != RMSNORM_OK) return st;
    KernelFn fn = cluster > 1 ? twopass_cluster_kernel_ptr(c.dtype, vb, c.opt.epilogue)
                              : twopass_kernel_ptr(c.dtype, vb, c.opt.epilogue);
    if (!fn) return RMSNORM_ERR_UNSUPPORTED;
    const int64_t nvec = c.hidden / (vb / c.sz);
    const int maxb = cluster > 1 ? split_block() : twopass_block();
    // The unsplit kernel's 32-bit vector index must not pass 2^31 - 1 one
    // stride after the row's last vector: rows of 2^31 - 1024 vectors or
    // more (widths near 2^31 elements with one-element vectors) are split.
    if (cluster == 1 && nvec > kUnsplitMaxVecs) return RMSNORM_ERR_UNSUPPORTED;
    const int64_t slice = cluster > 1 ? round_up(ceil_div(nvec, cluster), 32) : nvec;
    int block = c.opt.threads > 0 ? c.opt.threads : (slice >= maxb ? maxb : round_up(slice, 32));
    if (block % 32 != 0 || block > maxb) return RMSNORM_ERR_INVALID_ARG;
    int occ = 0;
    if (cached_occupancy(c.dev, c.info->smem_optin, fn, block, 0, cluster, &occ) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    if (occ <= 0) return RMSNORM_ERR_UNSUPPORTED;
    int grid;
    if (cluster == 1) {
        const int64_t resident = static_cast<int64_t>(c.info->sms) * occ;
        grid = static_cast<int>(c.opt.grid > 0 ? c.opt.grid
                                               : (c.rows < resident ? c.rows : resident));
    } else {
        const int64_t nclusters = c.opt.grid > 0 ? (c.opt.grid + cluster - 1) / cluster
                                                 : (c.rows < occ ? c.rows : occ);
        grid = static_cast<int>(nclusters * cluster);
    }
    P->resident = occ;
    P->path = RMSNORM_PATH_TWOPASS;
    P->cluster = cluster;
    P->group = block;
    P->block = block;
    P->rpc = 1;
    P->grid = grid;
    P->vb = vb;
    P->nv = 0;
    P->nvec = static_cast<int>(nvec);
    P->slice_vecs = static_cast<int>(slice);
    P->fn = fn;
    P->name = cluster == 1 ? "twopass" : "twopass_cluster";
    return RMSNORM_OK;
}

// Every row over the whole grid (rmsnorm_grid_kernel): 16-byte vectors only;
// the streamed kernels' CTA (480 consumer threads, or opt->threads, and a
// producer warp; chunks of 4 vectors per consumer thread, or 2 through
// opt->chunk_bytes; as many ring slots as shared memory holds, or
// opt->stages, at least 2); one CTA per SM, all resident (a cooperative
// launch), opt->grid of them at most; each owns a contiguous slice of every
// row and of w.
rmsnorm_status_t plan_grid(const Call& c, Plan* P) {
    if (c.opt.vec_bytes != 0 && c.opt.vec_bytes != 16) return RMSNORM_ERR_UNSUPPORTED;
    if (widest_vb(c) != 16) return RMSNORM_ERR_UNSUPPORTED;
    if (c.opt.cluster > 1 || c.opt.weights != 0) return RMSNORM_ERR_UNSUPPORTED;
    const int64_t row_bytes = c.hidden * c.sz;
    const int64_t nvec = row_bytes / 16;
    // one producer warp and one exchange warp beside the consumers
    const int max_nc = softmax_stream_max_threads() - 64;
    const int nc = c.opt.threads > 0 ? c.opt.threads : max_nc;
    if (nc % 32 != 0 || nc > max_nc) return RMSNORM_ERR_UNSUPPORTED;
    // Two vectors a consumer thread per chunk (14 KB chunks, twice the ring
    // slots) for the phased rows above kGridInterleavedMaxRowBytes: fp32 rows
    // of 32 MiB measured 63.8 against 61.3% of the HBM copy peak with four.
    int v = row_bytes > kGridInterleavedMaxRowBytes ? 2 : 4;
    if (c.opt.chunk_bytes != 0) {
        if (c.opt.chunk_bytes == 2 * 16 * nc) v = 2;
        else if (c.opt.chunk_bytes == 4 * 16 * nc) v = 4;
        else return RMSNORM_ERR_UNSUPPORTED;
    }
    const int64_t chunk = static_cast<int64_t>(16) * v * nc;
    const int64_t budget = c.info->smem_optin - kStreamHeaderHost;
    if (c.opt.stages < 0) return RMSNORM_ERR_INVALID_ARG;
    int64_t slots = c.opt.stages ? c.opt.stages : budget / chunk;
    if (!c.opt.stages && slots > kStagedMaxSlotsHost) slots = kStagedMaxSlotsHost;
    if (slots < 2 || slots > kStagedMaxSlotsHost || slots * chunk > budget)
        return RMSNORM_ERR_UNSUPPORTED;
    KernelFn fn = rmsnorm_grid_kernel_ptr(c.dtype, v, c.opt.epilogue);
    if (!fn) return RMSNORM_ERR_UNSUPPORTED;
    const int block = nc + 64;
    const int smem = static_cast<int>(kStreamHeaderHost + slots * chunk);
    int occ = 0;
    if (cached_occupancy(c.dev, c.info->smem_optin, fn, block, smem, 1, &occ) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    if (occ <= 0) return RMSNORM_ERR_UNSUPPORTED;
    int64_t resident = static_cast<int64_t>(c.info->sms) * occ;
    if (resident > kGridMaxCtasHost) resident = kGridMaxCtasHost;
    if (c.opt.grid > resident) return RMSNORM_ERR_UNSUPPORTED;
    const int64_t grid = c.opt.grid > 0 ? c.opt.grid : resident;
    // the arrival counter counts grid * rows arrivals in 32 bits
    if (c.rows > 0xFFFFFFFFll / grid) return RMSNORM_ERR_UNSUPPORTED;
    const int64_t slice = (nvec + grid - 1) / grid;
    const int64_t nchunks = (slice * 16 + chunk - 1) / chunk;
    P->path = RMSNORM_PATH_GRID;
    P->cluster = 1;
    P->group = nc;
    P->block = block;
    P->rpc = 1;
    P->grid = static_cast<int>(grid);
    P->vb = 16;
    P->nv = v;
    P->smem = smem;
    P->chunk = static_cast<int>(chunk);
    P->nchunks = static_cast<int>(nchunks);
    P->nslots = static_cast<int>(slots);
    P->w_staged = 0;
    P->nvec = static_cast<int>(nvec);
    P->slice_vecs = static_cast<int>(slice);
    P->scratch = grid_scratch_bytes(static_cast<int>(grid));
    // Chunks of the next row read while the CTAs' sums meet.  Measured on
    // fp32 rows of 16 MiB (w4m, four chunks per slice; % of the HBM copy
    // peak): 1 / 2 / 3 / 4 / 8 chunks 71.8 / 74.3 / 73.5 / 72.0 / 72.4;
    // rows of 10 and 32 MiB within a point of each other at every depth.
    P->read_ahead = kGridReadAheadRmsNorm;
    // Row schedule.  Measured (% of the HBM copy peak; interleaved / phased
    // / phased with the second read reversed, four vectors a thread per
    // chunk): fp32 rows of 16 MiB 74 / 65 / 65, 24 MiB 65 / 62 / 63, 32 MiB
    // 55 / 61 / 61, 40 MiB 50 / 56 / 57, 64 MiB 51 / 54 / 56; bf16 rows of
    // 32 MiB 54 / 62 / 60, 64 MiB 50 / 52 / 55.  With two vectors (the
    // phased rows' chunks) phased in order measured 64 at 32 MiB and 63 at
    // 40 MiB against 58 reversed, reversed 56 against 53 at 64 MiB.
    // Interleaving keeps DRAM reading and writing at once, but puts about
    // two rows of traffic (the next row's reads and this row's writes)
    // between a chunk's two reads, which L2 holds only for rows of up to
    // about 24 MiB.
    P->schedule = row_bytes <= kGridInterleavedMaxRowBytes ? 0
                  : row_bytes <= kGridMaxRowBytes          ? 1
                                                           : 2;
    // No resident chunks (the phased softmax keeps some in shared memory):
    // every second-read step also brings w's chunk through the ring, which
    // wants its slots (fp32 rows of 32 MiB, R = 0 / 2 / 4: 60.6 / 61.8 /
    // 59.4% of the HBM copy peak).
    P->nslots = static_cast<int>(slots);
    P->fn = fn;
    P->name = "grid_stream";
    return RMSNORM_OK;
}

// The write-up's own schedule (comparison only): one CTA of 256 threads per
// row, the whole row staged in shared memory as fp32.
rmsnorm_status_t plan_page(const Call& c, Plan* P) {
    if (c.opt.cluster > 1 || c.opt.threads != 0 || c.opt.vec_bytes > c.sz ||
        c.opt.epilogue != 0)
        return RMSNORM_ERR_UNSUPPORTED;
    const int64_t smem = c.hidden * 4;
    if (smem + 1024 > c.info->smem_optin) return RMSNORM_ERR_UNSUPPORTED;
    if (c.rows > 0x7FFFFFFFll) return RMSNORM_ERR_UNSUPPORTED;
    KernelFn fn = page_kernel_ptr(c.dtype);
    int occ = 0;
    if (cached_occupancy(c.dev, c.info->smem_optin, fn, page_block(), static_cast<int>(smem), 1, &occ) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    if (occ <= 0) return RMSNORM_ERR_UNSUPPORTED;
    P->path = RMSNORM_PATH_PAGE;
    P->cluster = 1;
    P->group = page_block();
    P->block = page_block();
    P->rpc = 1;
    P->grid = static_cast<int>(c.rows);
    P->vb = c.sz;
    P->nv = 0;
    P->smem = static_cast<int>(smem);
    P->nvec = static_cast<int>(c.hidden);
    P->slice_vecs = static_cast<int>(c.hidden);
    P->fn = fn;
    P->name = "page_schedule";
    return RMSNORM_OK;
}

// The launch heuristics, from measurements on GB300 (profiles/kernel_choices.md):
//  - few rows (fewer than SMs): split each row over a cluster (up to the
//    portable 8 CTAs; 16 measured no faster) so that about one CTA per SM
//    works, keeping slices of at least 4 KB;
//  - rows up to 32 KB: register-resident, one CTA (or warp) per row (93-101% of
//    the measured HBM copy peak);
//  - fp32 rows up to 64 KB: shared-memory staged by bulk copies (96%);
//  - wider rows (and bf16 rows above 32 KB): two-pass, the second read served
//    by L2 (81-95%).
// Each choice falls through to the next family if it cannot serve the call.
// The two-pass kernel with each row over a cluster of C CTAs (one CTA per
// row would leave the row's whole traffic to a single SM).  C (2..16, any
// size) minimises the row time waves(C) / C, waves(C) = rows / resident
// clusters of C, rounded up: resident clusters are limited by the SMs of a
// GPC, so for eight rows of 16-byte vectors (one 1024-thread CTA per SM) 16
// CTAs per row take two waves where 12 take one (measured on eight fp32 rows
// of 64 MiB: 409 us with 16, 303 us with 12, 355 us with 8).  Ties go to the
// smaller cluster.
rmsnorm_status_t plan_twopass_split(const Call& c, Plan* P) {
    Plan best;
    int64_t best_waves = 0;
    for (int cl = 2; cl <= 16; ++cl) {
        Plan Q;
        const rmsnorm_status_t st = plan_twopass(c, cl, &Q);
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

rmsnorm_status_t plan_auto(const Call& c, Plan* P) {
    const int64_t row_bytes = c.hidden * c.sz;
    rmsnorm_status_t st;
    // A cluster launch costs about 2 us more than a plain one (measured: c1,
    // 32 rows of 8 KB, 8.2 us split vs 6.3 us plain), so few-row inputs are
    // split only when a row is too wide for one CTA's registers or the input
    // is large enough for the extra SMs to pay.
    const bool split = c.rows < c.info->sms &&
                       (row_bytes > kRowregMaxRowBytes || c.rows * row_bytes >= kSplitMinBytes);
    if (split) {
        // Rows of 10 to 40 MiB: each over the whole grid in turn, its second
        // read (and w) from L2.  Measured (% of the HBM copy peak, whole grid
        // against the cluster two-pass split, which reads x twice): fp32 rows
        // of 10 MiB 63 / 60, 12 MiB 70 / 60, 16 MiB 55-76 / 43-64 (4 to 150
        // rows), 24 MiB 67 / 56, 32 MiB 64 / 55, 36 MiB 64 / 61, 40 MiB 63 /
        // 60; bf16 rows of 12 / 16 / 32 / 40 MiB 68 / 63-70 / 61 / 61 against
        // 60 / 52-53 / 54 / 59.  Outside that range the cluster split wins:
        // rows of 8 MiB 58 / 60 (bf16 55 / 59), whose exchanges come too
        // often, and of 44 and 64 MiB 57 / 58 and 55 / 57, which L2 does not
        // keep beside w between the two reads.
        if (row_bytes >= kGridMinRowBytes && row_bytes <= kGridMaxRowBytes) {
            st = plan_grid(c, P);
            if (st == RMSNORM_OK || st == RMSNORM_ERR_CUDA) return st;
        }
        int want = pow2_floor(c.info->sms / (c.rows > 0 ? c.rows : 1));
        if (want > kAutoMaxCluster) want = kAutoMaxCluster;
        while (want > 1 && row_bytes / want < 4096) want >>= 1;
        for (int cl = want; cl <= 16; cl <<= 1) {
            st = plan_rowreg(c, cl, P);
            if (st == RMSNORM_OK || st == RMSNORM_ERR_CUDA) return st;
        }
        for (int cl = want; cl <= 16; cl <<= 1) {
            st = plan_staged(c, cl, P);
            if (st == RMSNORM_OK || st == RMSNORM_ERR_CUDA) return st;
        }
        // Rows too wide for any cluster's registers or shared memory.
        st = plan_twopass_split(c, P);
        if (st == RMSNORM_OK || st == RMSNORM_ERR_CUDA) return st;
        return plan_twopass(c, 1, P);
    }
    if (row_bytes <= kRowregMaxRowBytes) {
        st = plan_rowreg(c, 1, P);
        if (st == RMSNORM_OK || st == RMSNORM_ERR_CUDA) return st;
    }
    // Wider rows, by measurement (1.5 GB inputs, % of the measured HBM peak):
    //   above 32 to 56 KB: ring-to-register, 92-99% (two-pass 76-99%,
    //     staged 47-72%);
    //   above 56 KB to 112 KB: the two-pass kernel, 95-100%, except fp32 rows
    //     of 64 KB, where the staged kernel's two 32 KB chunks per row give
    //     97% (two-pass 96%; at 56 KB it gave only 67%);
    //   above 112 KB to 128 KB: ring-to-register, 99% (two-pass 91-92%).
    const bool ringreg = (row_bytes > kRowregMaxRowBytes && row_bytes <= kRingregLowMaxRowBytes) ||
                         row_bytes > kRingregHighMinRowBytes;
    if (ringreg) {
        st = plan_ringreg(c, P);
        if (st == RMSNORM_OK || st == RMSNORM_ERR_CUDA) return st;
    }
    if (row_bytes > kRingregLowMaxRowBytes && row_bytes <= kStagedMaxRowBytes &&
        c.dtype == RMSNORM_DTYPE_F32) {
        st = plan_staged(c, 1, P);
        if (st == RMSNORM_OK || st == RMSNORM_ERR_CUDA) return st;
    }
    st = plan_twopass(c, 1, P);
    if (st != RMSNORM_ERR_UNSUPPORTED) return st;
    return plan_twopass_split(c, P);   // rows too wide for one CTA's 32-bit index
}

rmsnorm_status_t make_plan(const Call& c, Plan* P) {
    const int cl = c.opt.cluster;
    if (c.opt.reserved != 0) return RMSNORM_ERR_INVALID_ARG;
    if (c.opt.fault_inject < 0 || c.opt.fault_inject > 2) return RMSNORM_ERR_INVALID_ARG;
    if (c.opt.epilogue < 0 || c.opt.epilogue > 2) return RMSNORM_ERR_INVALID_ARG;
    if (c.opt.epilogue == 1 && !std::isfinite(c.opt.epilogue_alpha)) return RMSNORM_ERR_INVALID_ARG;
    if (c.opt.fault_inject != 0 && !RMSNORM_FAULT_INJECT) return RMSNORM_ERR_UNSUPPORTED;
    if (cl < 0 || cl > 16) return RMSNORM_ERR_INVALID_ARG;
    switch (c.opt.path) {
        case RMSNORM_PATH_AUTO:
            if (cl != 0 || c.opt.threads != 0 || c.opt.chunk_bytes != 0 || c.opt.stages != 0 ||
                c.opt.weights != 0)
                return RMSNORM_ERR_INVALID_ARG;   // launch-shape options need a forced path
            return plan_auto(c, P);
        case RMSNORM_PATH_ROWREG:
            if (cl > 1) return RMSNORM_ERR_INVALID_ARG;
            return plan_rowreg(c, 1, P);
        case RMSNORM_PATH_CLUSTER:
            if (cl == 1 || (cl & (cl - 1)) != 0) return RMSNORM_ERR_INVALID_ARG;
            return plan_rowreg(c, cl == 0 ? 2 : cl, P);
        case RMSNORM_PATH_STAGED:
            return plan_staged(c, cl == 0 ? 1 : cl, P);
        case RMSNORM_PATH_TWOPASS:
            return plan_twopass(c, cl == 0 ? 1 : cl, P);
        case RMSNORM_PATH_PAGE:
            return plan_page(c, P);
        case RMSNORM_PATH_RINGREG:
            if (cl > 1) return RMSNORM_ERR_INVALID_ARG;
            return plan_ringreg(c, P);
        case RMSNORM_PATH_GRID:
            if (cl > 1) return RMSNORM_ERR_INVALID_ARG;
            return plan_grid(c, P);
        default:
            return RMSNORM_ERR_INVALID_ARG;
    }
}

bool ranges_overlap(uintptr_t a, uintptr_t b, uint64_t na, uint64_t nb) {
    return a < b + nb && b < a + na;
}

// Host-side validation; fills `c` on success.
rmsnorm_status_t validate(int32_t dtype, const void* x, const void* w, const void* y,
                          int64_t rows, int64_t hidden, const rmsnorm_options_t* opt,
                          Call* c) {
    if (dtype != RMSNORM_DTYPE_F32 && dtype != RMSNORM_DTYPE_BF16) return RMSNORM_ERR_INVALID_ARG;
    if (!x || !w || !y) return RMSNORM_ERR_INVALID_ARG;
    if (rows < 0 || hidden <= 0 || hidden > 0x7FFFFFFFll) return RMSNORM_ERR_INVALID_ARG;
    const int sz = dtype == RMSNORM_DTYPE_F32 ? 4 : 2;
    if (rows > 0 && rows > (INT64_MAX / sz) / hidden) return RMSNORM_ERR_INVALID_ARG;
    const uintptr_t ux = reinterpret_cast<uintptr_t>(x);
    const uintptr_t uw = reinterpret_cast<uintptr_t>(w);
    const uintptr_t uy = reinterpret_cast<uintptr_t>(y);
    if (ux % sz || uw % sz || uy % sz) return RMSNORM_ERR_INVALID_ARG;
    const uint64_t nbytes = static_cast<uint64_t>(rows) * static_cast<uint64_t>(hidden) * sz;
    const uint64_t wbytes = static_cast<uint64_t>(hidden) * sz;
    if (ux != uy && ranges_overlap(ux, uy, nbytes, nbytes)) return RMSNORM_ERR_INVALID_ARG;
    if (rows > 0 && ranges_overlap(uw, uy, wbytes, nbytes)) return RMSNORM_ERR_INVALID_ARG;
    std::memset(c, 0, sizeof(*c));
    c->dtype = dtype;
    c->sz = sz;
    c->x = ux;
    c->w = uw;
    c->y = uy;
    c->rows = rows;
    c->hidden = hidden;
    if (opt) c->opt = *opt;
    return RMSNORM_OK;
}

rmsnorm_status_t run(int32_t dtype, const void* x, const void* w, void* y, int64_t rows,
                     int64_t hidden, float eps, const rmsnorm_options_t* opt,
                     cudaStream_t stream) {
    Call c;
    rmsnorm_status_t st = validate(dtype, x, w, y, rows, hidden, opt, &c);
    if (st != RMSNORM_OK) return st;
    if (!std::isfinite(eps) || eps < 0.f) return RMSNORM_ERR_INVALID_ARG;
    if (rows == 0) return RMSNORM_OK;
    if (current_device(&c.view) != cudaSuccess) return RMSNORM_ERR_CUDA;
    c.info = &c.view;
    c.dev = c.view.dev;
    Plan P;
    st = make_plan(c, &P);
    if (st != RMSNORM_OK) return st;

    Params p;
    std::memset(&p, 0, sizeof(p));
    p.x = x;
    p.w = w;
    p.y = y;
    p.rows = rows;
    p.hidden = static_cast<int32_t>(hidden);
    p.nvec = P.nvec;
    p.inv_hidden = 1.0f / static_cast<float>(hidden);
    p.eps = eps;
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
    p.w_staged = P.w_staged;
    p.fault = c.opt.fault_inject;
    p.alpha = c.opt.epilogue == 1 ? c.opt.epilogue_alpha : 1.0f;
    p.status = c.info->status;
    p.timeout_ns = c.opt.wait_timeout_ns ? c.opt.wait_timeout_ns : kDefaultTimeoutNs;

    LaunchShape s{P.grid, P.block, P.cluster, P.smem};
    if (ensure_prepared(c.dev, P.fn, c.info->smem_optin) != cudaSuccess) return RMSNORM_ERR_CUDA;
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

// ------------------------------------------- the allocation-free grid call --
//
// rmsnorm_fwd_grid_noalloc runs the whole-grid kernel (RMSNORM_PATH_GRID) with
// its exchange area in this file-scope device array instead of memory taken
// from the pool per call, for callers that must not allocate.  Every GPU that
// loads the library holds one copy of the array until the process exits.
constexpr size_t kNoAllocScratchBytes = kGridScratchBytesHost;   // 16512 bytes: 1024 CTAs
static __device__ __align__(256) unsigned char g_grid_scratch_noalloc[kNoAllocScratchBytes];

// The array's device address, looked up once per device (with that device
// current) on the first call there.
struct NoAllocDevice {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    void* scratch = nullptr;
};
NoAllocDevice g_noalloc_dev[64];

cudaError_t noalloc_scratch(int dev, void** out) {
    if (dev < 0 || dev >= 64) return note(cudaErrorInvalidDevice);
    NoAllocDevice& d = g_noalloc_dev[dev];
    std::call_once(d.once, [&] {
        d.err = cudaGetSymbolAddress(&d.scratch, g_grid_scratch_noalloc);
    });
    *out = d.scratch;
    return note(d.err);
}

rmsnorm_status_t run_grid_noalloc(int32_t dtype, const void* x, const void* w, void* y,
                                  int64_t rows, int64_t hidden, float eps, cudaStream_t stream) {
    rmsnorm_options_t opt;
    std::memset(&opt, 0, sizeof(opt));
    opt.path = RMSNORM_PATH_GRID;
    Call c;
    rmsnorm_status_t st = validate(dtype, x, w, y, rows, hidden, &opt, &c);
    if (st != RMSNORM_OK) return st;
    if (!std::isfinite(eps) || eps < 0.f) return RMSNORM_ERR_INVALID_ARG;
    if (rows == 0) return RMSNORM_OK;
    if (current_device(&c.view) != cudaSuccess) return RMSNORM_ERR_CUDA;
    c.info = &c.view;
    c.dev = c.view.dev;
    Plan P;
    st = make_plan(c, &P);
    if (st != RMSNORM_OK) return st;
    // the grid this device launches must fit the fixed array
    if (P.scratch <= 0 || static_cast<size_t>(P.scratch) > kNoAllocScratchBytes)
        return RMSNORM_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (noalloc_scratch(c.dev, &scratch) != cudaSuccess) return RMSNORM_ERR_CUDA;

    Params p;
    std::memset(&p, 0, sizeof(p));
    p.x = x;
    p.w = w;
    p.y = y;
    p.rows = rows;
    p.hidden = static_cast<int32_t>(hidden);
    p.nvec = P.nvec;
    p.inv_hidden = 1.0f / static_cast<float>(hidden);
    p.eps = eps;
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
    p.alpha = 1.0f;
    p.status = c.info->status;
    p.timeout_ns = kDefaultTimeoutNs;
    p.scratch = scratch;

    LaunchShape s{P.grid, P.block, P.cluster, P.smem};
    s.cooperative = true;
    if (ensure_prepared(c.dev, P.fn, c.info->smem_optin) != cudaSuccess) return RMSNORM_ERR_CUDA;
    // the previous call's counter and partials are still there: clear them
    if (note(cudaMemsetAsync(scratch, 0, static_cast<size_t>(P.scratch), stream)) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    if (note(launch_ex(P.fn, s, stream, p)) != cudaSuccess) return RMSNORM_ERR_CUDA;
    return RMSNORM_OK;
}

}  // namespace
}  // namespace rmsnorm

using namespace rmsnorm;

extern "C" {

rmsnorm_status_t rmsnorm_fwd_f32(const float* x, const float* w, float* y, int64_t rows,
                                 int64_t hidden, float eps, rmsnorm_stream_t stream) {
    return run(RMSNORM_DTYPE_F32, x, w, y, rows, hidden, eps, nullptr,
               reinterpret_cast<cudaStream_t>(stream));
}

rmsnorm_status_t rmsnorm_fwd_bf16(const uint16_t* x, const uint16_t* w, uint16_t* y,
                                  int64_t rows, int64_t hidden, float eps,
                                  rmsnorm_stream_t stream) {
    return run(RMSNORM_DTYPE_BF16, x, w, y, rows, hidden, eps, nullptr,
               reinterpret_cast<cudaStream_t>(stream));
}

rmsnorm_status_t rmsnorm_fwd_ex(int32_t dtype, const void* x, const void* w, void* y,
                                int64_t rows, int64_t hidden, float eps,
                                const rmsnorm_options_t* opt, rmsnorm_stream_t stream) {
    return run(dtype, x, w, y, rows, hidden, eps, opt, reinterpret_cast<cudaStream_t>(stream));
}

rmsnorm_status_t rmsnorm_plan(int32_t dtype, const void* x, const void* w, const void* y,
                              int64_t rows, int64_t hidden, const rmsnorm_options_t* opt,
                              rmsnorm_plan_t* plan) {
    if (!plan) return RMSNORM_ERR_INVALID_ARG;
    Call c;
    rmsnorm_status_t st = validate(dtype, x, w, y, rows, hidden, opt, &c);
    if (st != RMSNORM_OK) return st;
    if (current_device(&c.view) != cudaSuccess) return RMSNORM_ERR_CUDA;
    c.info = &c.view;
    c.dev = c.view.dev;
    if (c.rows == 0) c.rows = 1;   // describe the launch a one-row call would make
    Plan P;
    st = make_plan(c, &P);
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
    plan->weights_staged = P.w_staged;
    std::snprintf(plan->kernel, sizeof(plan->kernel), "%s", P.name);
    return RMSNORM_OK;
}

rmsnorm_status_t rmsnorm_last_device_status(rmsnorm_stream_t stream) {
    DeviceView view;
    if (current_device(&view) != cudaSuccess) return RMSNORM_ERR_CUDA;
    const DeviceView* info = &view;
    if (note(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream))) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    unsigned word = 0;
    if (note(cudaMemcpy(&word, info->status, sizeof(word), cudaMemcpyDeviceToHost)) !=
        cudaSuccess)
        return RMSNORM_ERR_CUDA;
    if (word != 0) {
        const unsigned zero = 0;
        if (note(cudaMemcpy(info->status, &zero, sizeof(zero), cudaMemcpyHostToDevice)) !=
            cudaSuccess)
            return RMSNORM_ERR_CUDA;
    }
    return word == 0 ? RMSNORM_OK : static_cast<rmsnorm_status_t>(word & 0xFFu);
}

const char* rmsnorm_status_string(rmsnorm_status_t status) {
    switch (status) {
        case RMSNORM_OK: return "ok";
        case RMSNORM_ERR_INVALID_ARG: return "invalid argument";
        case RMSNORM_ERR_UNSUPPORTED: return "unsupported option for these arguments";
        case RMSNORM_ERR_CUDA: return "CUDA runtime error";
        case RMSNORM_ERR_TIMEOUT: return "device wait timed out";
        default: return "unknown status";
    }
}

int32_t rmsnorm_last_cuda_error(char* msg, size_t len) {
    const cudaError_t e = take_last_cuda_error();
    if (msg && len > 0)
        std::snprintf(msg, len, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return static_cast<int32_t>(e);
}

rmsnorm_status_t rmsnorm_fwd_grid_noalloc(int32_t dtype, const void* x, const void* w, void* y,
                                          int64_t rows, int64_t hidden, float eps,
                                          rmsnorm_stream_t stream) {
    return run_grid_noalloc(dtype, x, w, y, rows, hidden, eps,
                            reinterpret_cast<cudaStream_t>(stream));
}

int32_t rmsnorm_abi_version(void) { return 10200; }

// Present in every build; non-zero only in the failure-injection test build.
int32_t rmsnorm_fault_injection_enabled(void) { return RMSNORM_FAULT_INJECT; }

}  // extern "C"
