// k_split.cuh -- two- and three-pass row kernels split over a thread-block
// cluster, for few rows too wide for any register- or shared-memory-resident
// kernel (rows of several MB, up to 2^31 - 1 elements).
//
// One cluster of C CTAs (2..16, any size) per row, persistent over rows; CTA
// r of a cluster owns the contiguous slice [r*S, min((r+1)*S, nvec)) of the
// row's vectors, S = Params.slice_vecs.  Neither kernel holds the row: each
// pass streams the CTA's slice again (the repeats usually from L2).
//
//   RMSNorm:  pass 1 sum of squares -> warp butterfly + one shared-memory slot
//             per warp -> CTA totals exchanged through distributed shared
//             memory (cluster_allreduce, bounded wait) -> pass 2 scale by
//             rsqrt(sum/H + eps) and the weight, store.
//   softmax:  pass 1 slice maximum, pass 2 sum of exp relative to the slice
//             maximum, one exchange of the (maximum, sum) pair gives the
//             row's (cluster_pair_allreduce), pass 3 stores exp(x - M) / S.
//
// Few CTAs carry the whole input, so each thread keeps four loads in flight
// in the reading passes and two in the writing pass.  Consecutive passes run
// in opposite directions over the slice, so each starts on the part the
// previous one read last, which is still in L2.  A thread's vectors are
// vbeg + tid + j*blockDim for j < J; 32-bit indices (below 2^31).  Each
// thread sums in blocks of kSplitBlockIters batches, every block from zero,
// and adds the block's sum to its running total, so no fp32 chain grows with
// the row beyond one block plus the number of blocks.
#pragma once
#include "common.cuh"
#include "k_softmax.cuh"

namespace rmsnorm {

constexpr int kSplitThreads = 1024;
constexpr uint32_t kSplitBlockIters = 32;
constexpr uint32_t kSplitReadBatch = 4;    // loads in flight per thread, reading passes
constexpr uint32_t kSplitWriteBatch = 2;   // vectors per thread per step, writing pass

// This CTA's slice [*vbeg, *vend) of a row of nvec vectors.
__device__ __forceinline__ void split_slice(const Params& p, uint32_t rank, uint32_t* vbeg,
                                           uint32_t* vend) {
    const uint32_t n = static_cast<uint32_t>(p.nvec);
    const uint32_t len = static_cast<uint32_t>(p.slice_vecs);
    const uint64_t b = static_cast<uint64_t>(rank) * len;
    *vbeg = b < n ? static_cast<uint32_t>(b) : n;
    const uint32_t room = n - *vbeg;
    *vend = *vbeg + (len < room ? len : room);
}

template <typename T, int VB, int EPI>
__global__ void __launch_bounds__(kSplitThreads, 1) twopass_cluster_kernel(const Params p) {
    pdl_trigger();
    pdl_wait();
    constexpr int EPV = VecTraits<T, VB>::kElems;
    constexpr uint32_t U = kSplitReadBatch, U2 = kSplitWriteBatch;
    __shared__ float red[2][32];
    __shared__ ClusterExchange ex;
    const uint32_t tid = threadIdx.x;
    const uint32_t nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int nwarps = nthr >> 5;

    const uint32_t rank = cluster_ctarank();
    const int64_t unit = cluster_id_x(), nunits = cluster_count_x();
    cluster_exchange_init(&ex);
    uint32_t vbeg, vend;
    split_slice(p, rank, &vbeg, &vend);

    const char* xb = static_cast<const char*>(p.x);
    const char* wb = static_cast<const char*>(p.w);
    char* yb = static_cast<char*>(p.y);
    const int64_t row_bytes = static_cast<int64_t>(p.hidden) * sizeof(T);
    // this thread's vectors: vbeg + tid + j * nthr, j < J
    const uint32_t span = vend - vbeg;
    const uint32_t J = tid < span ? (span - tid + nthr - 1) / nthr : 0;
    const uint32_t B = kSplitBlockIters * U;          // vectors per summing block

    const int64_t stride = static_cast<int64_t>(nthr) * VB;
    const char* wsrc = wb + static_cast<int64_t>(vbeg + tid) * VB;

    uint32_t it = 0;
    for (int64_t row = unit; row < p.rows; row += nunits, ++it) {
        const int64_t soff = row * row_bytes + static_cast<int64_t>(vbeg + tid) * VB;
        const char* src = xb + soff;
        // pass 1, forward: sum of squares
        float s0 = 0.f, s1 = 0.f;
        for (uint32_t jb = 0; jb < J; jb += B) {
            const uint32_t je = J - jb > B ? jb + B : J;
            float t0 = 0.f, t1 = 0.f;
            for (uint32_t j0 = jb; j0 < je; j0 += U) {
                Vec<VB> xv[U];
#pragma unroll
                for (uint32_t u = 0; u < U; ++u)
                    if (j0 + u < je) xv[u] = ld_plain<VB>(src + (j0 + u) * stride);
#pragma unroll
                for (uint32_t u = 0; u < U; ++u) {
                    if (j0 + u < je) {
#pragma unroll
                        for (int k = 0; k < EPV; ++k) {
                            const float f = get<T, VB>(xv[u], k);
                            if (k & 1) t1 = fmaf(f, f, t1); else t0 = fmaf(f, f, t0);
                        }
                    }
                }
            }
            s0 += t0;
            s1 += t1;
        }
        float ss = warp_allreduce_sum(s0 + s1);
        const int b = it & 1;
        if (lane == 0) red[b][warp] = ss;
        __syncthreads();
        ss = 0.f;
        for (int k = 0; k < nwarps; ++k) ss += red[b][k];
        float total;
        const bool ok = cluster_allreduce(&ex, ss, p.cluster, rank, it, p, &total,
                                          static_cast<int>(tid));
        if (__syncthreads_or(!ok)) break;   // uniform: stop, then leave cleanly
        const float rstd = rsqrtf(fmaf(total, p.inv_hidden, p.eps));

        // pass 2, backward: scale, weight, store
        char* dst = yb + soff;
        for (uint32_t g = (J + U2 - 1) / U2; g-- > 0;) {
            const uint32_t j0 = g * U2;
            Vec<VB> xv[U2], wv[U2];
#pragma unroll
            for (uint32_t u = 0; u < U2; ++u) {
                if (j0 + u < J) {
                    xv[u] = ld_stream<VB>(src + (j0 + u) * stride);
                    wv[u] = ld_ro<VB>(wsrc + (j0 + u) * stride);
                }
            }
#pragma unroll
            for (uint32_t u = 0; u < U2; ++u) {
                if (j0 + u < J) {
                    float o[EPV];
#pragma unroll
                    for (int k = 0; k < EPV; ++k)
                        o[k] = epilogue<EPI>((get<T, VB>(xv[u], k) * rstd) * get<T, VB>(wv[u], k),
                                             p.alpha);
                    st_stream<VB>(dst + (j0 + u) * stride, pack<T, VB>(o));
                }
            }
        }
    }
    // Keep this CTA's shared memory alive until every peer is done with it.
    cluster_sync_all();
}

template <typename T, int VB>
__global__ void __launch_bounds__(kSplitThreads, 1) softmax_threepass_cluster_kernel(const Params p) {
    pdl_trigger();
    pdl_wait();
    // bf16 vectors of two or more elements: the packed-pair passes; fp32 (and
    // one-element) vectors: scalar code.
    constexpr bool kPairs = sizeof(T) == 2 && VecTraits<T, VB>::kElems >= 2;
    constexpr int EPV = VecTraits<T, VB>::kElems;
    constexpr uint32_t U = kSplitReadBatch, U2 = kSplitWriteBatch;
    using RV = RowVec<T, VB>;
    __shared__ float red[2][2][32];
    __shared__ PairExchange ex;
    const uint32_t tid = threadIdx.x;
    const uint32_t nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int nwarps = nthr >> 5;
    const char* xb = static_cast<const char*>(p.x);
    char* yb = static_cast<char*>(p.y);
    const int64_t row_bytes = static_cast<int64_t>(p.hidden) * sizeof(T);

    const uint32_t rank = cluster_ctarank();
    const int64_t unit = cluster_id_x(), nunits = cluster_count_x();
    if (tid == 0) {
        mbar_init(smem_addr(&ex.bar[0]), 1);
        mbar_init(smem_addr(&ex.bar[1]), 1);
        fence_mbarrier_init_cluster();
    }
    __syncthreads();
    cluster_sync_all();        // no peer arrives before the barriers exist
    uint32_t vbeg, vend;
    split_slice(p, rank, &vbeg, &vend);
    // this thread's vectors: vbeg + tid + j * nthr, j < J
    const uint32_t span = vend - vbeg;
    const uint32_t J = tid < span ? (span - tid + nthr - 1) / nthr : 0;
    const uint32_t B = kSplitBlockIters * U;          // vectors per summing block
    const uint32_t nblocks = (J + B - 1) / B;
    const int64_t stride = static_cast<int64_t>(nthr) * VB;

    uint32_t it = 0;
    for (int64_t row = unit; row < p.rows; row += nunits, ++it) {
        const int b = it & 1;
        const int64_t soff = row * row_bytes + static_cast<int64_t>(vbeg + tid) * VB;
        const char* src = xb + soff;
        // pass 1, forward: the slice's maximum
        float m = -INFINITY;
        float mk[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        uint32_t mw[2] = {kBf16x2NegInf, kBf16x2NegInf};
        for (uint32_t j0 = 0; j0 < J; j0 += U) {
            Vec<VB> xv[U];
#pragma unroll
            for (uint32_t u = 0; u < U; ++u)
                if (j0 + u < J) xv[u] = ld_plain<VB>(src + (j0 + u) * stride);
#pragma unroll
            for (uint32_t u = 0; u < U; ++u) {
                if (j0 + u < J) {
                    if constexpr (kPairs) {
                        RV::fold_max(xv[u], mk, mw);
                    } else {
#pragma unroll
                        for (int k = 0; k < EPV; ++k) m = fmaxf(m, get<T, VB>(xv[u], k));
                    }
                }
            }
        }
        if constexpr (kPairs) m = running_max(mk, mw);
        m = warp_allreduce_max(m);
        if (lane == 0) red[0][b][warp] = m;
        __syncthreads();
        m = -INFINITY;
        for (int k = 0; k < nwarps; ++k) m = fmaxf(m, red[0][b][k]);
        // pass 2, backward: exponentials relative to the slice's maximum (a
        // slice of -inf keeps -inf: exp(-inf) = 0)
        // (the fused offset for slices of moderate maximum, else the exact
        // form: row_exp_offset_ok), both as (x - ms)*log2e + cs in one loop
        const bool fast = row_exp_offset_ok(m) || m == -INFINITY;
        const float c = m == -INFINITY ? -INFINITY : row_exp_bias<T>() - m * kLog2e;
        const float ms = fast ? 0.f : m, cs = fast ? c : row_exp_bias<T>();
        float sl = 0.f;
        for (uint32_t q = nblocks; q-- > 0;) {
            const uint32_t jb = q * B;
            const uint32_t je = J - jb > B ? jb + B : J;
            typename RV::Sums sums;
            float s0 = 0.f, s1 = 0.f;
            for (uint32_t j0 = jb; j0 < je; j0 += U) {
                Vec<VB> xv[U];
#pragma unroll
                for (uint32_t u = 0; u < U; ++u)
                    if (j0 + u < je) xv[u] = ld_plain<VB>(src + (j0 + u) * stride);
#pragma unroll
                for (uint32_t u = 0; u < U; ++u) {
                    if (j0 + u < je) {
                        if constexpr (kPairs) {
                            RV e;
                            e.widen(xv[u]);
                            e.exp_shift(ms, cs, sums);
                        } else {
#pragma unroll
                            for (int k = 0; k < EPV; ++k) {
                                const float ev =
                                    row_exp_arg<T>(fmaf(get<T, VB>(xv[u], k) - ms, kLog2e, cs));
                                if (k & 1) s1 += ev; else s0 += ev;
                            }
                        }
                    }
                }
            }
            if constexpr (kPairs) sl += sums.total(); else sl += s0 + s1;
        }
        float s = warp_allreduce_sum(sl);
        if (lane == 0) red[1][b][warp] = s;
        __syncthreads();
        s = 0.f;
        for (int k = 0; k < nwarps; ++k) s += red[1][b][k];
        // one exchange of the (maximum, sum) pair gives the row's; the slice
        // sum and pass 3's offset are both corrected for the rounding of
        // their offsets (slice_offset_correction)
        float M, S;
        const float corr = fast ? slice_offset_correction<T>(m, c) : 1.0f;
        const bool ok = cluster_pair_allreduce(&ex, m, s * corr, p.cluster, rank, it, p, &M, &S,
                                               static_cast<int>(tid));
        if (__syncthreads_or(!ok)) break;   // uniform: stop, then leave cleanly
        const bool fast3 = row_exp_offset_ok(M);
        const float c3 = row_exp_bias<T>() - M * kLog2e;
        const float inv = (fast3 ? slice_offset_correction<T>(M, c3) : 1.0f) / S;
        const float ms3 = fast3 ? 0.f : M, cs3 = fast3 ? c3 : row_exp_bias<T>();

        // pass 3, forward: exp(x - M) / S
        char* dst = yb + soff;
        for (uint32_t j0 = 0; j0 < J; j0 += U2) {
            Vec<VB> xv[U2];
#pragma unroll
            for (uint32_t u = 0; u < U2; ++u)
                if (j0 + u < J) xv[u] = ld_stream<VB>(src + (j0 + u) * stride);
#pragma unroll
            for (uint32_t u = 0; u < U2; ++u) {
                if (j0 + u < J) {
                    RV e;
                    e.widen(xv[u]);
                    st_stream<VB>(dst + (j0 + u) * stride, e.exp_shift_scaled(ms3, cs3, inv));
                }
            }
        }
    }
    // Keep this CTA's shared memory alive until every peer is done with it.
    cluster_sync_all();
}

}  // namespace rmsnorm
