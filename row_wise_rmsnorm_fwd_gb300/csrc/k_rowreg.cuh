// k_rowreg.cuh -- single-pass, register-resident RMSNorm forward.
//
// One group of G threads (a multiple of 32, or a power of two below 32 for
// rows of fewer than 32 vectors: 32 / G rows per warp) owns one row at a
// time; each thread owns NV vectors of VB bytes at vector indices t, t+G,
// t+2G, ... so every load instruction of a warp covers 32*VB contiguous
// bytes (G < 32: consecutive rows, which are contiguous).  The row is
// read from HBM exactly once (streaming, evict-first), kept in registers, and
// written once.  The weight slice of each thread is loaded once per CTA and
// stays in registers for every row the CTA processes.
//
// Schedule per row (page "A hackable Python ML compiler, part 2": the Loop IR
// and the generated kernel's cooperative reduction, redesigned):
//   1. fp32 sum of squares of the thread's elements,
//   2. butterfly shuffle sum within each warp (within each G-lane group when
//      G < 32),
//   3. one shared-memory slot per warp, ONE barrier, then every thread adds
//      its group's warp totals in a fixed order (the page's kernel used a
//      three-level tree with a barrier per level),
//   4. (split rows only) the CTA totals of the C CTAs of a thread-block
//      cluster are exchanged through distributed shared memory,
//   5. rstd = rsqrt(sum * (1/H) + eps), y = (x * rstd) * w, streaming store.
//
// Rows are scheduled persistently: a CTA (or a cluster, for split rows) walks
// row blocks with a grid-wide stride, and the next row's loads are issued
// before the current row's reduction (register double buffer, PF).
//
// Compile-time choices: PF (register prefetch of the next row), WREG (weights
// held in registers across rows, packed; otherwise re-read from L1 per row),
// LD / ST (cache policies of the x loads and y stores, see common.cuh), EPI
// (fused epilogue applied before the store).
#pragma once
#include "common.cuh"

namespace rmsnorm {

template <int NV>
constexpr int rowreg_max_threads() { return NV >= 4 ? 512 : 1024; }

template <typename T, int VB, int NV, bool PF, bool WREG, int LD, int ST, int EPI>
__global__ void __launch_bounds__(rowreg_max_threads<NV>())
rowreg_kernel(const Params p) {
    constexpr int EPV = VecTraits<T, VB>::kElems;
    __shared__ float red[2][32];
    __shared__ ClusterExchange ex;

    pdl_trigger();
    const int G = p.group;
    const int tid = threadIdx.x;
    const int g = tid / G;             // row group inside the CTA
    const int t = tid - g * G;         // thread inside the group
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int wpg = G >> 5;            // warps per group
    const int gw0 = g * wpg;           // first warp of this group

    const int ncta = p.cluster;
    uint32_t rank = 0;
    int64_t unit = blockIdx.x, nunits = gridDim.x;
    if (ncta > 1) {
        rank = cluster_ctarank();
        unit = cluster_id_x();
        nunits = cluster_count_x();
        cluster_exchange_init(&ex);
    }
    pdl_wait();

    // Vector indices this thread owns inside the row (or the CTA's slice).
    const int vbase = (ncta > 1) ? static_cast<int>(rank) * p.slice_vecs : 0;
    const int vlim = (ncta > 1) ? min(p.nvec, vbase + p.slice_vecs) : p.nvec;
    int vidx[NV];
    bool valid[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        vidx[i] = vbase + i * G + t;
        valid[i] = vidx[i] < vlim;
    }

    const char* xb = static_cast<const char*>(p.x);
    const char* wb = static_cast<const char*>(p.w);
    char* yb = static_cast<char*>(p.y);
    const int64_t row_bytes = static_cast<int64_t>(p.hidden) * sizeof(T);

    Vec<VB> wv[NV];
    if (WREG) {
#pragma unroll
        for (int i = 0; i < NV; ++i)
            if (valid[i]) wv[i] = ld_ro<VB>(wb + static_cast<int64_t>(vidx[i]) * VB);
    }

    const int RPC = p.rows_per_cta;
    const int64_t nblocks = (p.rows + RPC - 1) / RPC;

    Vec<VB> cur[NV], nxt[NV];
    auto load_rows = [&](Vec<VB> (&dst)[NV], int64_t rb) {
        const int64_t row = rb * RPC + g;
        if (row < p.rows) {
            const char* src = xb + row * row_bytes;
#pragma unroll
            for (int i = 0; i < NV; ++i)
                if (valid[i])
                    dst[i] = ld_stream<VB, LD>(src + static_cast<int64_t>(vidx[i]) * VB);
        }
    };

    int64_t rb = unit;
    if (rb < nblocks) load_rows(cur, rb);
    uint32_t it = 0;
    for (; rb < nblocks; rb += nunits, ++it) {
        const int64_t nrb = rb + nunits;
        if (PF && nrb < nblocks) load_rows(nxt, nrb);

        const int64_t row = rb * RPC + g;
        const bool row_ok = row < p.rows;

        // 1. sum of squares (two accumulators for instruction-level parallelism)
        float s0 = 0.f, s1 = 0.f;
        if (row_ok) {
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                if (valid[i]) {
#pragma unroll
                    for (int k = 0; k < EPV; ++k) {
                        const float f = get<T, VB>(cur[i], k);
                        if (k & 1) s1 = fmaf(f, f, s1); else s0 = fmaf(f, f, s0);
                    }
                }
            }
        }
        // 2. warp butterfly (lane groups of G when a warp holds several rows)
        float ss = G >= 32 ? warp_allreduce_sum(s0 + s1) : group_allreduce_sum(s0 + s1, G);
        // 3. cross-warp combine: one barrier, fixed order
        if (wpg > 1 || ncta > 1) {
            const int b = it & 1;
            if (lane == 0) red[b][warp] = ss;
            __syncthreads();
            ss = 0.f;
            for (int k = 0; k < wpg; ++k) ss += red[b][gw0 + k];
        }
        // 4. cluster combine over DSMEM (split rows)
        if (ncta > 1) {
            float total;
            const bool ok = cluster_allreduce(&ex, ss, ncta, rank, it, p, &total, tid);
            ss = total;
            if (__syncthreads_or(!ok)) break;   // uniform: stop, then leave cleanly
        }
        // 5. rstd and the scaled store
        const float rstd = rsqrtf(fmaf(ss, p.inv_hidden, p.eps));
        if (row_ok) {
            char* dst = yb + row * row_bytes;
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                if (valid[i]) {
                    Vec<VB> wi;
                    if (WREG) {
                        wi = wv[i];
                        if constexpr (sizeof(T) == 2 && VB >= 4) {
#pragma unroll
                            for (int k = 0; k < VB / 4; ++k) opaque(wi.u[k]);
                        }
                    } else {
                        wi = ld_ro<VB>(wb + static_cast<int64_t>(vidx[i]) * VB);
                    }
                    float o[EPV];
#pragma unroll
                    for (int k = 0; k < EPV; ++k)
                        o[k] = epilogue<EPI>((get<T, VB>(cur[i], k) * rstd) * get<T, VB>(wi, k),
                                             p.alpha);
                    st_stream<VB, ST>(dst + static_cast<int64_t>(vidx[i]) * VB,
                                      pack<T, VB>(o));
                }
            }
        }
        if (PF) {
#pragma unroll
            for (int i = 0; i < NV; ++i) cur[i] = nxt[i];
        } else if (nrb < nblocks) {
            load_rows(cur, nrb);
        }
    }
    // Keep this CTA's shared memory alive until every peer is done with it.
    if (ncta > 1) cluster_sync_all();
}

}  // namespace rmsnorm
