// k_softmax.cuh -- row-wise softmax on the register-resident row skeleton.
//
// y[r,j] = exp(x[r,j] - m[r]) / sum_k exp(x[r,k] - m[r]),  m[r] = max_k x[r,k]
//
// exp(x - m) is evaluated as exp2f(x*log2(e) - m*log2(e)) with one fused
// multiply-add: CUDA's exp2f maps to the SFU's base-2 exponential, several
// times cheaper than expf, which keeps the bf16 variant from becoming
// instruction-bound; the identity exp(t) = 2^(t*log2 e) costs at most
// |m|*log2(e)*2^-24 absolute error in the exponent.
//
// The second small reduction the compiler write-up ("A hackable Python ML
// compiler, part 2") lists among its wins, built from the same parts as the
// RMSNorm row kernel: a group of G threads per row holding the row in
// registers as NV vectors of VB bytes, persistent grid-stride row blocks, and
// the warp butterfly + one-slot-per-warp combine -- used twice (max, then
// sum of exponentials).  fp32 arithmetic; bf16 inputs widened exactly and
// each output rounded once.  IEEE special cases follow the definition: -inf
// entries give 0, a row of -inf or any NaN or +inf gives a NaN row.
//
// softmax_threepass_kernel serves rows too wide for registers: one CTA per
// row reads x three times (max, sum, write); the second and third reads are
// normally served by L2.
#pragma once
#include "common.cuh"

namespace rmsnorm {

constexpr float kLog2e = 1.4426950408889634f;

// exp(v - m) as 2^(v*log2e - m*log2e); ml2e = m * log2e.
__device__ __forceinline__ float exp_shifted(float v, float ml2e) {
    return exp2f(fmaf(v, kLog2e, -ml2e));
}

__device__ __forceinline__ float warp_allreduce_max(float v) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}

template <int NV>
constexpr int softmax_max_threads() { return NV >= 4 ? 512 : 1024; }

// PF: the next row's loads are issued before this row's two reductions
// (register double buffer), doubling the bytes in flight for narrow rows.
// With p.cluster > 1 a thread-block cluster of C CTAs shares each row: every
// CTA holds a slice, and the row maximum and the row sum are each combined
// across the cluster through distributed shared memory (bounded waits).
template <typename T, int VB, int NV, bool PF>
__global__ void __launch_bounds__(softmax_max_threads<NV>())
softmax_rowreg_kernel(const Params p) {
    constexpr int EPV = VecTraits<T, VB>::kElems;
    __shared__ float red[2][2][32];      // [max | sum][double buffer][warp]
    __shared__ ClusterExchange exmax, exsum;

    const int G = p.group;
    const int tid = threadIdx.x;
    const int g = tid / G;
    const int t = tid - g * G;
    const int warp = tid >> 5, lane = tid & 31;
    const int wpg = G >> 5;
    const int gw0 = g * wpg;

    const int ncta = p.cluster;
    uint32_t rank = 0;
    int64_t unit = blockIdx.x, nunits = gridDim.x;
    if (ncta > 1) {
        rank = cluster_ctarank();
        unit = cluster_id_x();
        nunits = cluster_count_x();
        cluster_exchange_init(&exmax, ncta, &exsum);
    }
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
    char* yb = static_cast<char*>(p.y);
    const int64_t row_bytes = static_cast<int64_t>(p.hidden) * sizeof(T);
    const int RPC = p.rows_per_cta;
    const int64_t nblocks = (p.rows + RPC - 1) / RPC;

    Vec<VB> cur[NV], nxt[NV];
    auto load_row = [&](Vec<VB> (&dst)[NV], int64_t rb) {
        const int64_t row = rb * RPC + g;
        if (row < p.rows) {
            const char* src = xb + row * row_bytes;
#pragma unroll
            for (int i = 0; i < NV; ++i)
                if (valid[i]) dst[i] = ld_stream<VB>(src + static_cast<int64_t>(vidx[i]) * VB);
        }
    };

    int64_t rb = unit;
    if (rb < nblocks) load_row(cur, rb);
    uint32_t it = 0;
    for (; rb < nblocks; rb += nunits, ++it) {
        const int64_t nrb = rb + nunits;
        if (PF && nrb < nblocks) load_row(nxt, nrb);
        const int64_t row = rb * RPC + g;
        const bool row_ok = row < p.rows;
        const int b = it & 1;
        float e[NV][EPV];
        float m = -INFINITY;
        if (row_ok) {
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                if (valid[i]) {
#pragma unroll
                    for (int k = 0; k < EPV; ++k) {
                        e[i][k] = get<T, VB>(cur[i], k);
                        m = fmaxf(m, e[i][k]);
                    }
                }
            }
        }
        // row maximum
        m = warp_allreduce_max(m);
        if (wpg > 1) {
            if (lane == 0) red[0][b][warp] = m;
            __syncthreads();
            m = -INFINITY;
            for (int k = 0; k < wpg; ++k) m = fmaxf(m, red[0][b][gw0 + k]);
        }
        if (ncta > 1) {
            float cm;
            const bool ok = cluster_allreduce<true>(&exmax, m, ncta, rank, it, p, &cm, tid);
            m = cm;
            if (__syncthreads_or(!ok)) break;   // uniform: stop, then leave cleanly
        }
        // exponentials and their sum
        const float ml2e = m * kLog2e;
        float s0 = 0.f, s1 = 0.f;
        if (row_ok) {
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                if (valid[i]) {
#pragma unroll
                    for (int k = 0; k < EPV; ++k) {
                        e[i][k] = exp_shifted(e[i][k], ml2e);
                        if (k & 1) s1 += e[i][k]; else s0 += e[i][k];
                    }
                }
            }
        }
        float s = warp_allreduce_sum(s0 + s1);
        if (wpg > 1) {
            if (lane == 0) red[1][b][warp] = s;
            __syncthreads();
            s = 0.f;
            for (int k = 0; k < wpg; ++k) s += red[1][b][gw0 + k];
        }
        if (ncta > 1) {
            float cs;
            const bool ok = cluster_allreduce(&exsum, s, ncta, rank, it, p, &cs, tid);
            s = cs;
            if (__syncthreads_or(!ok)) break;
        }
        const float inv = 1.0f / s;
        if (row_ok) {
            char* dst = yb + row * row_bytes;
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                if (valid[i]) {
                    float o[EPV];
#pragma unroll
                    for (int k = 0; k < EPV; ++k) o[k] = e[i][k] * inv;
                    st_stream<VB>(dst + static_cast<int64_t>(vidx[i]) * VB, pack<T, VB>(o));
                }
            }
        }
        if (PF) {
#pragma unroll
            for (int i = 0; i < NV; ++i) cur[i] = nxt[i];
        } else if (nrb < nblocks) {
            load_row(cur, nrb);
        }
    }
    // Keep this CTA's shared memory alive until every peer is done with it.
    if (ncta > 1) cluster_sync_all();
}

constexpr int kSoftmaxWideThreads = 1024;

template <typename T, int VB>
__global__ void __launch_bounds__(kSoftmaxWideThreads) softmax_threepass_kernel(const Params p) {
    constexpr int EPV = VecTraits<T, VB>::kElems;
    __shared__ float red[2][2][32];
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int nwarps = nthr >> 5;
    const char* xb = static_cast<const char*>(p.x);
    char* yb = static_cast<char*>(p.y);
    const int64_t row_bytes = static_cast<int64_t>(p.hidden) * sizeof(T);

    uint32_t it = 0;
    for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x, ++it) {
        const int b = it & 1;
        const char* src = xb + row * row_bytes;
        float m = -INFINITY;
        for (int v = tid; v < p.nvec; v += nthr) {
            const Vec<VB> xv = ld_plain<VB>(src + static_cast<int64_t>(v) * VB);
#pragma unroll
            for (int k = 0; k < EPV; ++k) m = fmaxf(m, get<T, VB>(xv, k));
        }
        m = warp_allreduce_max(m);
        if (lane == 0) red[0][b][warp] = m;
        __syncthreads();
        m = -INFINITY;
        for (int k = 0; k < nwarps; ++k) m = fmaxf(m, red[0][b][k]);
        const float ml2e = m * kLog2e;

        float s0 = 0.f, s1 = 0.f;
        for (int v = tid; v < p.nvec; v += nthr) {
            const Vec<VB> xv = ld_plain<VB>(src + static_cast<int64_t>(v) * VB);
#pragma unroll
            for (int k = 0; k < EPV; ++k) {
                const float ev = exp_shifted(get<T, VB>(xv, k), ml2e);
                if (k & 1) s1 += ev; else s0 += ev;
            }
        }
        float s = warp_allreduce_sum(s0 + s1);
        if (lane == 0) red[1][b][warp] = s;
        __syncthreads();
        s = 0.f;
        for (int k = 0; k < nwarps; ++k) s += red[1][b][k];
        const float inv = 1.0f / s;

        char* dst = yb + row * row_bytes;
        for (int v = tid; v < p.nvec; v += nthr) {
            const int64_t off = static_cast<int64_t>(v) * VB;
            const Vec<VB> xv = ld_stream<VB>(src + off);
            float o[EPV];
#pragma unroll
            for (int k = 0; k < EPV; ++k) o[k] = exp_shifted(get<T, VB>(xv, k), ml2e) * inv;
            st_stream<VB>(dst + off, pack<T, VB>(o));
        }
    }
}

}  // namespace rmsnorm
