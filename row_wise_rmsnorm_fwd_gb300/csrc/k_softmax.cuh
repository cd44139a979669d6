// k_softmax.cuh -- row-wise softmax on the register-resident row skeleton.
//
// y[r,j] = exp(x[r,j] - m[r]) / sum_k exp(x[r,k] - m[r]),  m[r] = max_k x[r,k]
//
// exp(x - m) is evaluated as 2^(x*log2(e) - m*log2(e)) with one fused
// multiply-add and a base-2 exponential (exp2f for fp32 rows, a single SFU
// instruction for bf16 rows: see row_exp), much cheaper than expf, which
// keeps the kernels from becoming instruction-bound; the identity exp(t) =
// 2^(t*log2 e) costs at most |m|*log2(e)*2^-24 absolute error in the
// exponent, a factor common to the whole row.
//
// The second small reduction the compiler write-up ("A hackable Python ML
// compiler, part 2") lists among its wins, built from the same parts as the
// RMSNorm row kernel: a group of G threads per row (a multiple of 32, or a
// power of two below 32 lanes for rows of fewer than 32 vectors) holding the
// row in registers as NV vectors of VB bytes, persistent grid-stride row blocks, and
// the warp butterfly + one-slot-per-warp combine -- used twice (max, then
// sum of exponentials).  fp32 arithmetic; bf16 inputs widened exactly and
// each output rounded once.  IEEE special cases follow the definition: -inf
// entries give 0, a row of -inf or any NaN or +inf gives a NaN row.
//
// softmax_staged_kernel brings rows in through the bulk-copy slot ring
// (k_ring.cuh) and holds each in registers, so that the next rows are already
// in flight while a row's reductions run; rows too wide for one CTA's
// registers are split over a thread-block cluster of such CTAs.
// softmax_threepass_kernel serves the wide rows where that split loses: one
// CTA per row reads x three times (max, sum, write), the second and third
// reads normally served by L2.
#pragma once
#include <type_traits>

#include "k_ring.cuh"

namespace rmsnorm {

constexpr float kLog2e = 1.4426950408889634f;

// Every kernel evaluates every exponential of a row as
// 2^(v*log2e + c) with a per-row constant c = row_exp_bias<T>() - m*log2e.
//   fp32: exp2f, bias 0: e = exp(v - m) itself.
//   bf16: the PTX instruction ex2.approx.ftz.f32 (one SFU operation,
//     relative error about 2^-22, far below bf16's 2^-9), with bias 8: every
//     exponential is scaled by 2^8, which cancels in e / sum, and keeps each
//     one whose output a bf16 can resolve (e >= 2^-133, since sum >= 1) a
//     normal number, so that flushing subnormal results to zero loses
//     nothing.  Any rounding of c is a common factor of the row and cancels
//     too.  exp2f costs several instructions more per element, and bf16 rows
//     carry twice the elements per byte.
template <typename T>
__device__ __forceinline__ float row_exp_bias() {
    return sizeof(T) == 2 ? 8.0f : 0.0f;
}

// The exponential of an argument a = v*log2e + c already formed.
template <typename T>
__device__ __forceinline__ float row_exp_arg(float a) {
    if constexpr (sizeof(T) == 2) {
        float r;
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
        return r;
    } else {
        return exp2f(a);
    }
}

template <typename T>
__device__ __forceinline__ float row_exp(float v, float c) {
    return row_exp_arg<T>(fmaf(v, kLog2e, c));
}

// Whether a row (or slice) whose maximum is m may form its exponent
// arguments as v*log2e + c with the one rounded offset c = bias - m*log2e.
// That offset's rounding (half an ulp of |m|*log2e) is a factor common to
// the row, so it cancels in e / sum -- but only while it is small: for |m|
// near 1e10 it is hundreds, every exponential of the row underflows and the
// row turns into 0/0; for |m| above FLT_MAX / log2(e) the offset itself
// overflows.  |m| < 2^21 keeps it below 2^-4.  Other rows (and rows whose
// maximum is not finite) take the exact form (v - m)*log2e + bias: for every
// element that can contribute (v within about 130 of m) the difference v - m
// is exact (Sterbenz), so that form has the single rounding of the fused
// one, for one more instruction per element.
constexpr float kRowExpOffsetMax = 2097152.0f;   // 2^21

__device__ __forceinline__ bool row_exp_offset_ok(float m) {
    return fabsf(m) < kRowExpOffsetMax;
}

// One exponential with the row's offset: F = the fused form (c), else the
// exact form relative to the maximum m.
template <typename T, bool F>
__device__ __forceinline__ float row_exp_sel(float v, float c, float m) {
    if constexpr (F) {
        return row_exp_arg<T>(fmaf(v, kLog2e, c));
    } else {
        return row_exp_arg<T>(fmaf(v - m, kLog2e, row_exp_bias<T>()));
    }
}

// A split row's slices each form their exponentials with their own offset
// c = bias - m*log2(e), m the slice's maximum, rounded to fp32.  That rounding
// (up to half an ulp of |m|*log2(e): 7.6e-6 for |m| near 100) is a factor
// common to the slice, not to the row, so unlike a whole row's offset it does
// not cancel in e / sum.  This returns 2^-eps, eps = c - (bias - m*log2(e))
// recovered with one fma; the split kernels multiply the slice sum they
// exchange and the slice's output scale by it.  1 for a slice whose maximum
// is not finite (c = -inf, or a NaN row).
template <typename T>
__device__ __forceinline__ float slice_offset_correction(float m, float c) {
    if (!(fabsf(m) < INFINITY)) return 1.0f;
    return exp2f(-fmaf(m, kLog2e, c - row_exp_bias<T>()));
}

// Packed fp32 pairs: the f32x2 forms of fma, add and mul (sm_100 and later)
// do two lanes in one instruction, each lane rounded exactly as the scalar
// fmaf / + / * would be, so a kernel that pairs its elements computes the
// bitwise same values with about half the arithmetic instructions.
__device__ __forceinline__ uint64_t pack_x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpack_x2(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t fma_x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t add_x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t mul_x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Lane-wise maximum of two packed bf16 pairs (a NaN lane yields the other
// operand's lane, as fmaxf does); exact, so it can run before widening.
__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Four running sums of a row's exponentials (element k of a vector adds into
// lane k & 3, the order of a plain loop over k), as two packed pairs or as
// four scalars; total() adds the lanes as (0 + 1) + (2 + 3).
struct PairSums {
    uint64_t s2[2] = {0ull, 0ull};       // two pairs of +0
    __device__ __forceinline__ float total() const {
        float s0, s1, s2a, s3;
        unpack_x2(s2[0], s0, s1);
        unpack_x2(s2[1], s2a, s3);
        return (s0 + s1) + (s2a + s3);
    }
};

struct ScalarSums {
    float sk[4] = {0.f, 0.f, 0.f, 0.f};
    __device__ __forceinline__ float total() const { return (sk[0] + sk[1]) + (sk[2] + sk[3]); }
};

constexpr uint32_t kBf16x2NegInf = 0xFF80FF80u;

// The row's maximum from the running maxima of the loads below: four fp32
// lanes and two packed bf16 pairs.
__device__ __forceinline__ float running_max(const float (&mk)[4], const uint32_t (&mw)[2]) {
    const float m4 = fmaxf(fmaxf(mk[0], mk[1]), fmaxf(mk[2], mk[3]));
    const float w0 = fmaxf(__uint_as_float(mw[0] << 16), __uint_as_float(mw[0] & 0xFFFF0000u));
    const float w1 = fmaxf(__uint_as_float(mw[1] << 16), __uint_as_float(mw[1] & 0xFFFF0000u));
    return fmaxf(m4, fmaxf(w0, w1));
}

// One vector of a bf16 row held as fp32 pairs, and the three per-row passes
// over it: elements 2j and 2j + 1 form pair j.  The maximum is taken on the
// packed bf16 pairs before widening; the exponent arguments, the sums and
// the scaled outputs use the packed fp32 instructions.  (Measured against
// scalar code, % of the HBM roofline: bf16 rows of 512 88 -> 91, of 32000
// 87 -> 88; fp32 rows, whose exp2f takes scalar operands anyway, gained
// nothing and stay scalar.)
template <typename T, int VB>
struct RowPairs {
    static constexpr int kElems = VecTraits<T, VB>::kElems;
    static constexpr int kPairs = kElems / 2;
    static_assert(sizeof(T) == 2 && kElems % 2 == 0, "bf16 vectors of two or more elements");
    using Sums = PairSums;
    uint64_t e[kPairs];

    static __device__ __forceinline__ void fold_max(const Vec<VB>& v, float (&)[4],
                                                    uint32_t (&mw)[2]) {
#pragma unroll
        for (int j = 0; j < kPairs; ++j) mw[j & 1] = max_bf16x2(mw[j & 1], v.u[j]);
    }
    __device__ __forceinline__ void widen(const Vec<VB>& v) {
#pragma unroll
        for (int j = 0; j < kPairs; ++j)
            e[j] = pack_x2(get<T, VB>(v, 2 * j), get<T, VB>(v, 2 * j + 1));
    }
    __device__ __forceinline__ void load(const Vec<VB>& v, float (&mk)[4], uint32_t (&mw)[2]) {
        fold_max(v, mk, mw);
        widen(v);
    }
    // The exponent arguments of pair j: e*log2e + c (F), or (e - m)*log2e +
    // bias (the exact form, see row_exp_offset_ok).
    template <bool F>
    __device__ __forceinline__ void args(int j, float c, float m, float& a0, float& a1) const {
        const uint64_t l2 = pack_x2(kLog2e, kLog2e);
        if constexpr (F) {
            unpack_x2(fma_x2(e[j], l2, pack_x2(c, c)), a0, a1);
        } else {
            const float b = row_exp_bias<T>();
            unpack_x2(fma_x2(add_x2(e[j], pack_x2(-m, -m)), l2, pack_x2(b, b)), a0, a1);
        }
    }
    // e = 2^((e - ms)*log2e + cs) in place, the sums take the exponentials:
    // one loop for both forms of the argument, (ms, cs) = (0, c) or (m, bias).
    __device__ __forceinline__ void exp_shift(float ms, float cs, Sums& s) {
        const uint64_t l2 = pack_x2(kLog2e, kLog2e), n2 = pack_x2(-ms, -ms), c2 = pack_x2(cs, cs);
#pragma unroll
        for (int j = 0; j < kPairs; ++j) {
            float a0, a1;
            unpack_x2(fma_x2(add_x2(e[j], n2), l2, c2), a0, a1);
            e[j] = pack_x2(row_exp_arg<T>(a0), row_exp_arg<T>(a1));
            s.s2[j & 1] = add_x2(s.s2[j & 1], e[j]);
        }
    }
    __device__ __forceinline__ Vec<VB> exp_shift_scaled(float ms, float cs, float inv) const {
        const uint64_t l2 = pack_x2(kLog2e, kLog2e), n2 = pack_x2(-ms, -ms), c2 = pack_x2(cs, cs);
        const uint64_t inv2 = pack_x2(inv, inv);
        float o[kElems];
#pragma unroll
        for (int j = 0; j < kPairs; ++j) {
            float a0, a1;
            unpack_x2(fma_x2(add_x2(e[j], n2), l2, c2), a0, a1);
            unpack_x2(mul_x2(pack_x2(row_exp_arg<T>(a0), row_exp_arg<T>(a1)), inv2), o[2 * j],
                      o[2 * j + 1]);
        }
        return pack<T, VB>(o);
    }
    // e = 2^(argument) in place; the sums take the exponentials.
    template <bool F = true>
    __device__ __forceinline__ void exp(float c, Sums& s, float m = 0.f) {
#pragma unroll
        for (int j = 0; j < kPairs; ++j) {
            float a0, a1;
            args<F>(j, c, m, a0, a1);
            e[j] = pack_x2(row_exp_arg<T>(a0), row_exp_arg<T>(a1));
            s.s2[j & 1] = add_x2(s.s2[j & 1], e[j]);
        }
    }
    // The outputs e * inv, packed for the store.
    __device__ __forceinline__ Vec<VB> scaled(float inv) const {
        const uint64_t inv2 = pack_x2(inv, inv);
        float o[kElems];
#pragma unroll
        for (int j = 0; j < kPairs; ++j) unpack_x2(mul_x2(e[j], inv2), o[2 * j], o[2 * j + 1]);
        return pack<T, VB>(o);
    }
    // The outputs 2^(argument) * inv of widened inputs, packed for the store.
    template <bool F = true>
    __device__ __forceinline__ Vec<VB> exp_scaled(float c, float inv, float m = 0.f) const {
        const uint64_t inv2 = pack_x2(inv, inv);
        float o[kElems];
#pragma unroll
        for (int j = 0; j < kPairs; ++j) {
            float a0, a1;
            args<F>(j, c, m, a0, a1);
            unpack_x2(mul_x2(pack_x2(row_exp_arg<T>(a0), row_exp_arg<T>(a1)), inv2), o[2 * j],
                      o[2 * j + 1]);
        }
        return pack<T, VB>(o);
    }
};

// The same passes in scalar fp32 arithmetic (fp32 rows, and bf16 vectors of
// one element).
template <typename T, int VB>
struct RowScalars {
    static constexpr int kElems = VecTraits<T, VB>::kElems;
    using Sums = ScalarSums;
    float e[kElems];

    static __device__ __forceinline__ void fold_max(const Vec<VB>& v, float (&mk)[4],
                                                    uint32_t (&)[2]) {
#pragma unroll
        for (int k = 0; k < kElems; ++k) mk[k & 3] = fmaxf(mk[k & 3], get<T, VB>(v, k));
    }
    __device__ __forceinline__ void widen(const Vec<VB>& v) {
#pragma unroll
        for (int k = 0; k < kElems; ++k) e[k] = get<T, VB>(v, k);
    }
    __device__ __forceinline__ void load(const Vec<VB>& v, float (&mk)[4], uint32_t (&)[2]) {
#pragma unroll
        for (int k = 0; k < kElems; ++k) {
            e[k] = get<T, VB>(v, k);
            mk[k & 3] = fmaxf(mk[k & 3], e[k]);
        }
    }
    template <bool F = true>
    __device__ __forceinline__ void exp(float c, Sums& s, float m = 0.f) {
#pragma unroll
        for (int k = 0; k < kElems; ++k) {
            e[k] = row_exp_sel<T, F>(e[k], c, m);
            s.sk[k & 3] += e[k];
        }
    }
    __device__ __forceinline__ Vec<VB> scaled(float inv) const {
        float o[kElems];
#pragma unroll
        for (int k = 0; k < kElems; ++k) o[k] = e[k] * inv;
        return pack<T, VB>(o);
    }
    template <bool F = true>
    __device__ __forceinline__ Vec<VB> exp_scaled(float c, float inv, float m = 0.f) const {
        float o[kElems];
#pragma unroll
        for (int k = 0; k < kElems; ++k) o[k] = row_exp_sel<T, F>(e[k], c, m) * inv;
        return pack<T, VB>(o);
    }
    __device__ __forceinline__ Vec<VB> exp_shift_scaled(float ms, float cs, float inv) const {
        float o[kElems];
#pragma unroll
        for (int k = 0; k < kElems; ++k) o[k] = row_exp_arg<T>(fmaf(e[k] - ms, kLog2e, cs)) * inv;
        return pack<T, VB>(o);
    }
};

template <typename T, int VB>
using RowVec = std::conditional_t<(sizeof(T) == 2 && VecTraits<T, VB>::kElems >= 2),
                                  RowPairs<T, VB>, RowScalars<T, VB>>;

__device__ __forceinline__ float warp_allreduce_max(float v) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}

// The same within aligned groups of g lanes (g a power of two, 1..32).
__device__ __forceinline__ float group_allreduce_max(float v, int g) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1)
        if (m < g) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}

// One exchange per row of a (maximum, sum of exponentials) pair over a
// thread-block cluster: the combine of the online softmax.  Each CTA sends
// its slice's maximum m_r and its sum s_r of exp(x - m_r) to every peer; every
// CTA then forms M = max_r m_r and S = sum_r s_r * exp(m_r - M) in rank order,
// so all CTAs hold the bitwise same pair.  Double-buffered by row parity, a
// bounded wait, as cluster_allreduce (common.cuh); the caller passes a block
// barrier after each call.  A slice of -inf only has m_r = -inf and s_r = 0
// and adds exp(-inf) * 0 = 0; a row of -inf gives M = -inf and a NaN sum, as
// the definition does.
struct PairExchange {
    alignas(8) unsigned long long bar[2];
    float2 slot[2][16];
};

// The exchange in two halves, so that a CTA can keep working between them.
// cluster_pair_send: this CTA's pair (m, s) of row iteration `it` to every
// CTA of the cluster (threads lt < ncta send; lt == 0 arms the barrier).
__device__ __forceinline__ void cluster_pair_send(PairExchange* ex, float m, float s, int ncta,
                                                  uint32_t rank, uint32_t it, const Params& p,
                                                  int lt) {
    const uint32_t b = it & 1u;
    const uint32_t bar = smem_addr(&ex->bar[b]);
    if (lt == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(ncta) * 8u);
    bool send = lt < ncta;
#if RMSNORM_FAULT_INJECT
    if (p.fault == kFaultClusterWithholdPartial && rank == 0 && it == 0) send = false;
#else
    (void)p;
#endif
    if (send) {
        const uint32_t peer = static_cast<uint32_t>(lt);
        st_async_v2_f32(map_to_rank(smem_addr(&ex->slot[b][rank]), peer), m, s,
                        map_to_rank(bar, peer));
    }
}

// cluster_pair_wait: wait (bounded) for every CTA's pair of iteration `it`
// and fold them in rank order (every CTA gets the bitwise same result).
// Returns false if the wait expired (the status word is then set).
__device__ __forceinline__ bool cluster_pair_wait(PairExchange* ex, int ncta, uint32_t it,
                                                  const Params& p, float* M, float* S, int lt) {
    const uint32_t b = it & 1u;
    const bool ok = mbar_wait_bounded<true>(smem_addr(&ex->bar[b]), (it >> 1) & 1u,
                                            p.timeout_ns);
    float mx = -INFINITY, sum = 0.f;
    if (ok) {
        for (int c = 0; c < ncta; ++c) mx = fmaxf(mx, ex->slot[b][c].x);
        for (int c = 0; c < ncta; ++c)
            sum += ex->slot[b][c].y * exp2f((ex->slot[b][c].x - mx) * kLog2e);
    } else if (lt == 0) {
        report_timeout(p.status, kSiteClusterExchange);
    }
    *M = mx;
    *S = sum;
    return ok;
}

__device__ __forceinline__ bool cluster_pair_allreduce(PairExchange* ex, float m, float s,
                                                       int ncta, uint32_t rank, uint32_t it,
                                                       const Params& p, float* M, float* S,
                                                       int lt) {
    cluster_pair_send(ex, m, s, ncta, rank, it, p, lt);
    return cluster_pair_wait(ex, ncta, it, p, M, S, lt);
}

// Fold the pair (mo, so) into (m, s): each sum is of exponentials relative
// to its own maximum; the result is relative to max(m, mo).  A pair whose
// maximum is the result's keeps its sum unscaled, so two empty pairs (-inf,
// 0) give (-inf, 0) rather than 0 * 2^NaN.
__device__ __forceinline__ void pair_fold(float& m, float& s, float mo, float so) {
    const float M = fmaxf(m, mo);
    const float a = m == M ? s : s * exp2f((m - M) * kLog2e);
    const float b = mo == M ? so : so * exp2f((mo - M) * kLog2e);
    m = M;
    s = a + b;
}

template <int NV>
constexpr int softmax_max_threads() { return NV >= 4 ? 512 : 1024; }

// PF: the next row's loads are issued before this row's two reductions
// (register double buffer), doubling the bytes in flight per thread.
// CL: a thread-block cluster of p.cluster CTAs shares each row: every CTA
// holds a slice, computes exponentials and their sum relative to its slice's
// maximum, and one exchange of the (maximum, sum) pair through distributed
// shared memory (bounded wait) gives the row's, with which each CTA rescales
// its slice.  A compile-time switch, so that the plain instances carry none of
// the cluster code (measured: with the cluster branches present but idle, 1 KB
// bf16 rows ran about 8% slower).
template <typename T, int VB, int NV, bool PF, bool CL>
__global__ void __launch_bounds__(softmax_max_threads<NV>())
softmax_rowreg_kernel(const Params p) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[2][2][32];      // [max | sum][double buffer][warp]
    __shared__ PairExchange ex;        // cluster split only

    const int G = p.group;
    const int tid = threadIdx.x;
    const int g = tid / G;
    const int t = tid - g * G;
    const int warp = tid >> 5, lane = tid & 31;
    const int wpg = G >> 5;
    const int gw0 = g * wpg;

    const int ncta = CL ? p.cluster : 1;
    uint32_t rank = 0;
    int64_t unit = blockIdx.x, nunits = gridDim.x;
    if (CL) {
        rank = cluster_ctarank();
        unit = cluster_id_x();
        nunits = cluster_count_x();
        if (tid == 0) {
            mbar_init(smem_addr(&ex.bar[0]), 1);
            mbar_init(smem_addr(&ex.bar[1]), 1);
            fence_mbarrier_init_cluster();
        }
        __syncthreads();
        cluster_sync_all();        // no peer arrives before the barriers exist
    }
    const int vbase = CL ? static_cast<int>(rank) * p.slice_vecs : 0;
    const int vlim = CL ? min(p.nvec, vbase + p.slice_vecs) : p.nvec;
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
        RowVec<T, VB> e[NV];
        float mk[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};   // 4 independent chains
        uint32_t mw[2] = {kBf16x2NegInf, kBf16x2NegInf};
        if (row_ok) {
#pragma unroll
            for (int i = 0; i < NV; ++i)
                if (valid[i]) e[i].load(cur[i], mk, mw);
        }
        float m = running_max(mk, mw);
        // row maximum (within lane groups of G when a warp holds several rows)
        m = G >= 32 ? warp_allreduce_max(m) : group_allreduce_max(m, G);
        if (wpg > 1) {
            if (lane == 0) red[0][b][warp] = m;
            __syncthreads();
            m = -INFINITY;
            for (int k = 0; k < wpg; ++k) m = fmaxf(m, red[0][b][gw0 + k]);
        }
        // exponentials and their sum, relative to this CTA's maximum when a
        // cluster splits the row (a slice of -inf keeps -inf: exp(-inf) = 0)
        const bool fast = row_exp_offset_ok(m) || (CL && m == -INFINITY);
        const float c = (CL && m == -INFINITY) ? -INFINITY : row_exp_bias<T>() - m * kLog2e;
        typename RowVec<T, VB>::Sums sums;
        if (row_ok) {
            if (fast) {
#pragma unroll
                for (int i = 0; i < NV; ++i)
                    if (valid[i]) e[i].exp(c, sums);
            } else {
#pragma unroll
                for (int i = 0; i < NV; ++i)
                    if (valid[i]) e[i].template exp<false>(c, sums, m);
            }
        }
        const float sl = sums.total();
        float s = G >= 32 ? warp_allreduce_sum(sl) : group_allreduce_sum(sl, G);
        if (wpg > 1) {
            if (lane == 0) red[1][b][warp] = s;
            __syncthreads();
            s = 0.f;
            for (int k = 0; k < wpg; ++k) s += red[1][b][gw0 + k];
        }
        float inv = 1.0f / s;
        if (CL) {
            // one exchange of the (maximum, sum) pair gives the row's
            const float corr = fast ? slice_offset_correction<T>(m, c) : 1.0f;
            float M, S;
            const bool ok =
                cluster_pair_allreduce(&ex, m, s * corr, ncta, rank, it, p, &M, &S, tid);
            if (__syncthreads_or(!ok)) break;   // uniform: stop, then leave cleanly
            // rescale this slice to the row's maximum
            inv = exp2f((m - M) * kLog2e) * corr / S;
        }
        if (row_ok) {
            char* dst = yb + row * row_bytes;
#pragma unroll
            for (int i = 0; i < NV; ++i)
                if (valid[i]) st_stream<VB>(dst + static_cast<int64_t>(vidx[i]) * VB, e[i].scaled(inv));
        }
        if (PF) {
#pragma unroll
            for (int i = 0; i < NV; ++i) cur[i] = nxt[i];
        } else if (nrb < nblocks) {
            load_row(cur, nrb);
        }
    }
    // Keep this CTA's shared memory alive until every peer is done with it.
    if (CL) cluster_sync_all();
}

// Rows staged in shared memory, then held in registers.  The CTA's rows
// stream through the slot ring in chunks (chunk n of the stream in slot
// n % S); every thread waits for a row's chunks, copies its NV vectors into
// registers (widened to fp32), and after the block's first reduction barrier
// -- every thread has its copy by then -- thread 0 refills the row's slots
// with chunks n + S.  The following rows' loads are thus in flight through
// the whole computation of a row (maximum, exponentials, sum, outputs from
// registers) without taking registers: the register kernel's prefetch needs a
// second register copy of the row, which does not fit for rows of 16 KB and
// more.  No producer warp: 16 warps of 128 registers fill an SM's register
// file, where a 17th warp would cap every thread at 96.  Thread t owns
// vectors t, t + blockDim.x, ... of its row (or slice); chunk_bytes is a
// power of two unless a slice fits one chunk.
// CL: rows too wide for one CTA's registers are split over a thread-block
// cluster of p.cluster CTAs; CTA rank r streams slice r (p.slice_vecs
// vectors) of each of its cluster's rows, computes the exponentials and
// their sum relative to its slice's maximum, and one exchange of the
// (maximum, sum) pair through distributed shared memory (bounded wait) gives
// every CTA the row's maximum and sum, with which it rescales its slice --
// the online-softmax combine, one cluster round trip per row instead of two
// -- while the ring keeps loading the next rows' slices.
constexpr int kSoftmaxStagedMaxThreads = 512;

template <typename T, int NV, bool CL>
__global__ void __launch_bounds__(kSoftmaxStagedMaxThreads) softmax_staged_kernel(const Params p) {
    pdl_trigger();
    pdl_wait();
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    // header: full[32] | red[max|sum][buffer][16 warps] | the cluster pair exchange
    float* red = reinterpret_cast<float*>(smem + 8 * kStagedMaxSlots);
    PairExchange* ex = reinterpret_cast<PairExchange*>(smem + 8 * kStagedMaxSlots + 256);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int NT = blockDim.x;
    const int NW = NT >> 5;
    const int NCH = p.nchunks;
    const int S = p.nslots;
    const int CB = p.chunk_bytes;
    const int ncta = CL ? p.cluster : 1;
    uint32_t rank = 0;
    int64_t unit = blockIdx.x, nunits = gridDim.x;
    if (CL) {
        rank = cluster_ctarank();
        unit = cluster_id_x();
        nunits = cluster_count_x();
    }
    const int64_t row_bytes = static_cast<int64_t>(p.hidden) * sizeof(T);
    const int64_t slice_nom = CL ? static_cast<int64_t>(p.slice_vecs) * 16 : row_bytes;
    const int64_t sbeg = static_cast<int64_t>(rank) * slice_nom;
    const int64_t send = sbeg + slice_nom < row_bytes ? sbeg + slice_nom : row_bytes;
    const int64_t my_bytes = send > sbeg ? send - sbeg : 0;
    const int my_vecs = static_cast<int>(my_bytes / 16);
    const SlotRing ring{full, nullptr, smem + kStagedHeader, S, NCH, CB, my_bytes};
    const uint64_t policy = policy_evict_first();

    int64_t issued = 0;            // chunks issued so far (thread 0's count)
    RingCursor cur{unit, 0, 0};    // the next chunk to issue (thread 0)
    if (tid == 0) {
        for (int k = 0; k < S; ++k) mbar_init(smem_addr(&full[k]), 1);
        fence_mbarrier_init_cluster();
        while (issued < S && ring_issue_next(p, ring, cur, nunits, row_bytes, sbeg, policy, issued))
            ++issued;
    }
    if (CL) {
        if (tid == 0) {
            mbar_init(smem_addr(&ex->bar[0]), 1);
            mbar_init(smem_addr(&ex->bar[1]), 1);
            fence_mbarrier_init_cluster();
        }
        __syncthreads();
        cluster_sync_all();        // no peer arrives before the barriers exist
    } else {
        __syncthreads();
    }

    const int shift = (CB & (CB - 1)) == 0 ? __ffs(CB) - 1 : 31;
    int kidx[NV], off[NV];
    bool valid[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int v = i * NT + tid;
        valid[i] = v < my_vecs;
        kidx[i] = (v * 16) >> shift;                   // chunk of the slice holding vector v
        off[i] = v * 16 - (kidx[i] << shift);           // its byte offset in that chunk
    }
    char* yb = static_cast<char*>(p.y);
    uint32_t it = 0;
    int64_t base = 0;              // stream index of this row's chunk 0
    int slot0 = 0;                 // its slot, base % S
    uint32_t lap0 = 0;             // its phase parity, (base / S) & 1
    for (int64_t row = unit; row < p.rows; row += nunits, ++it, base += NCH) {
        const int b = it & 1;
        bool ok = true;
        for (int k = 0; k < NCH; ++k) {
            int sl = slot0 + k;
            uint32_t par = lap0;
            if (sl >= S) {
                sl -= S;
                par ^= 1u;
            }
            if (!mbar_wait_bounded<false>(smem_addr(&full[sl]), par, p.timeout_ns)) {
                ok = false;
                break;
            }
        }
        RowVec<T, 16> e[NV];
        float mk[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};   // 4 independent chains
        uint32_t mw[2] = {kBf16x2NegInf, kBf16x2NegInf};
        if (ok) {
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                if (valid[i]) {
                    int slot = slot0 + kidx[i];
                    if (slot >= S) slot -= S;
                    e[i].load(as_vec(*reinterpret_cast<const uint4*>(
                                  ring.slots + static_cast<int64_t>(slot) * CB + off[i])),
                              mk, mw);
                }
            }
        }
        float m = warp_allreduce_max(running_max(mk, mw));
        if (lane == 0) red[b * 16 + warp] = m;
        if (__syncthreads_or(!ok)) {
            if (tid == 0) report_timeout(p.status, kSiteStagedFull);
            break;
        }
        // every thread holds its part of the row: refill the row's slots
        if (tid == 0)
            while (issued < base + NCH + S &&
                   ring_issue_next(p, ring, cur, nunits, row_bytes, sbeg, policy, issued))
                ++issued;
        slot0 += NCH;              // NCH <= S: one wrap at most
        if (slot0 >= S) {
            slot0 -= S;
            lap0 ^= 1u;
        }
        m = -INFINITY;
        for (int k = 0; k < NW; ++k) m = fmaxf(m, red[b * 16 + k]);
        // exponentials relative to this CTA's maximum: the whole row's when
        // the row is not split; a slice of -inf keeps -inf (exp(-inf) = 0)
        const bool fast = row_exp_offset_ok(m) || (CL && m == -INFINITY);
        const float c = (CL && m == -INFINITY) ? -INFINITY : row_exp_bias<T>() - m * kLog2e;
        typename RowVec<T, 16>::Sums sums;
        if (fast) {
#pragma unroll
            for (int i = 0; i < NV; ++i)
                if (valid[i]) e[i].exp(c, sums);
        } else {
#pragma unroll
            for (int i = 0; i < NV; ++i)
                if (valid[i]) e[i].template exp<false>(c, sums, m);
        }
        float sum = warp_allreduce_sum(sums.total());
        if (lane == 0) red[32 + b * 16 + warp] = sum;
        __syncthreads();
        sum = 0.f;
        for (int k = 0; k < NW; ++k) sum += red[32 + b * 16 + k];
        float inv = 1.0f / sum;
        if (CL) {
            const float corr = fast ? slice_offset_correction<T>(m, c) : 1.0f;
            float M, S;
            const bool cok =
                cluster_pair_allreduce(ex, m, sum * corr, ncta, rank, it, p, &M, &S, tid);
            if (__syncthreads_or(!cok)) break;   // uniform: stop, then leave cleanly
            // rescale this slice to the row's maximum
            inv = exp2f((m - M) * kLog2e) * corr / S;
        }
        char* dst = yb + row * row_bytes + sbeg;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            if (valid[i]) st_stream<16>(dst + static_cast<int64_t>(i * NT + tid) * 16, e[i].scaled(inv));
    }
    // After a timeout, copies may still be in flight: wait (bounded) for the
    // last S issued before the CTA leaves.  Normally every one was consumed.
    if (tid == 0)
        for (int64_t n = issued > S ? issued - S : 0; n < issued; ++n)
            ring_wait_full(ring, n, p.timeout_ns);
    // Keep this CTA's shared memory alive until every peer is done with it.
    if (CL) cluster_sync_all();
}

constexpr int kSoftmaxWideThreads = 1024;

template <typename T, int VB>
__global__ void __launch_bounds__(kSoftmaxWideThreads) softmax_threepass_kernel(const Params p) {
    pdl_trigger();
    pdl_wait();
    // bf16 vectors of two or more elements: the packed-pair passes; fp32 (and
    // one-element) vectors: scalar code with one maximum chain and two sums,
    // which keeps the kernel at 32 registers and two 1024-thread CTAs per SM
    // (four chains took the fp32 instance to 44 registers, one CTA per SM).
    constexpr bool kPairs = sizeof(T) == 2 && VecTraits<T, VB>::kElems >= 2;
    constexpr int EPV = VecTraits<T, VB>::kElems;
    using RV = RowVec<T, VB>;
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
        if constexpr (kPairs) {
            float mk[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            uint32_t mw[2] = {kBf16x2NegInf, kBf16x2NegInf};
            for (int v = tid; v < p.nvec; v += nthr)
                RV::fold_max(ld_plain<VB>(src + static_cast<int64_t>(v) * VB), mk, mw);
            m = running_max(mk, mw);
        } else {
            for (int v = tid; v < p.nvec; v += nthr) {
                const Vec<VB> xv = ld_plain<VB>(src + static_cast<int64_t>(v) * VB);
#pragma unroll
                for (int k = 0; k < EPV; ++k) m = fmaxf(m, get<T, VB>(xv, k));
            }
        }
        m = warp_allreduce_max(m);
        if (lane == 0) red[0][b][warp] = m;
        __syncthreads();
        m = -INFINITY;
        for (int k = 0; k < nwarps; ++k) m = fmaxf(m, red[0][b][k]);
        const float c = row_exp_bias<T>() - m * kLog2e;
        const bool fast = row_exp_offset_ok(m);

        // pass 2: the sum of exponentials (F: fused offset, else exact form)
        auto pass2 = [&](auto ftag) -> float {
            constexpr bool F = decltype(ftag)::value;
            if constexpr (kPairs) {
                PairSums sums;
                for (int v = tid; v < p.nvec; v += nthr) {
                    RV e;
                    e.widen(ld_plain<VB>(src + static_cast<int64_t>(v) * VB));
                    e.template exp<F>(c, sums, m);
                }
                return sums.total();
            } else {
                float s0 = 0.f, s1 = 0.f;
                for (int v = tid; v < p.nvec; v += nthr) {
                    const Vec<VB> xv = ld_plain<VB>(src + static_cast<int64_t>(v) * VB);
#pragma unroll
                    for (int k = 0; k < EPV; ++k) {
                        const float ev = row_exp_sel<T, F>(get<T, VB>(xv, k), c, m);
                        if (k & 1) s1 += ev; else s0 += ev;
                    }
                }
                return s0 + s1;
            }
        };
        const float sl = fast ? pass2(std::true_type{}) : pass2(std::false_type{});
        float s = warp_allreduce_sum(sl);
        if (lane == 0) red[1][b][warp] = s;
        __syncthreads();
        s = 0.f;
        for (int k = 0; k < nwarps; ++k) s += red[1][b][k];
        const float inv = 1.0f / s;

        // pass 3: the outputs
        char* dst = yb + row * row_bytes;
        auto pass3 = [&](auto ftag) {
            constexpr bool F = decltype(ftag)::value;
            for (int v = tid; v < p.nvec; v += nthr) {
                const int64_t off = static_cast<int64_t>(v) * VB;
                RV e;
                e.widen(ld_stream<VB>(src + off));
                st_stream<VB>(dst + off, e.template exp_scaled<F>(c, inv, m));
            }
        };
        if (fast) pass3(std::true_type{}); else pass3(std::false_type{});
    }
}

}  // namespace rmsnorm
