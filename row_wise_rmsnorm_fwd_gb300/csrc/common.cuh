// common.cuh -- device helpers shared by the RMSNorm kernels (sm_103a).
//
// Element access, the fp32 reduction primitives, the launch-parameter block,
// and inline-PTX wrappers for mbarriers, 1-D bulk copies and cluster
// (distributed shared memory) operations.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#ifndef RMSNORM_FAULT_INJECT
#define RMSNORM_FAULT_INJECT 0
#endif

namespace rmsnorm {

// Failure-injection modes, compiled only into the test build of the library.
enum : int {
    kFaultNone = 0,
    kFaultStagedWithholdCopy = 1,      // producer arms a barrier, issues no copy
    kFaultClusterWithholdPartial = 2,  // one cluster CTA never sends its partial
};

// Fused epilogues, applied to each fp32 output value before the store
// (compile-time choice; the CuTe DSL pages' Constexpr epilogue_op idea).
enum : int {
    kEpiNone = 0,     // y
    kEpiScale = 1,    // y * alpha
    kEpiRelu = 2,     // y if y > 0 or y is NaN, else +0
};

template <int EPI>
__device__ __forceinline__ float epilogue(float v, float alpha) {
    if constexpr (EPI == kEpiScale) {
        return v * alpha;
    } else if constexpr (EPI == kEpiRelu) {
        return (v > 0.f || v != v) ? v : 0.f;
    } else {
        return v;
    }
}

// Device status word codes (low byte = rmsnorm_status_t, next byte = site).
enum : unsigned {
    kStatusTimeout = 4u,
    kSiteClusterExchange = 1u,
    kSiteStagedFull = 2u,
    kSiteStagedEmpty = 3u,
};

// Everything a kernel needs; passed by value (kernel parameter space).
struct Params {
    const void* x;
    const void* w;
    void* y;
    int64_t rows;
    int32_t hidden;        // elements per row
    int32_t nvec;          // vectors per row (hidden / elems_per_vec)
    float inv_hidden;      // 1/hidden, the page's reciprocal-then-multiply mean
    float eps;
    int32_t group;         // threads per row (or per slice)
    int32_t rows_per_cta;  // row groups in one CTA
    int32_t cluster;       // CTAs per row (1 = no split)
    int32_t slice_vecs;    // vectors per CTA slice when cluster > 1
    int32_t chunk_bytes;   // staged path: bytes per bulk copy
    int32_t nchunks;       // staged path: bulk copies per row slice
    int32_t nslots;        // staged path: chunk slots in the shared-memory ring
    int32_t w_staged;      // staged path: weight slice held in shared memory
    int32_t fault;         // failure-detection test builds only (else always 0)
    float alpha;           // epilogue scale (kEpiScale)
    unsigned* status;      // per-device status word
    uint64_t timeout_ns;   // limit for every bounded wait
    void* scratch;         // grid-split kernels: cleared exchange records (else null)
    int32_t read_ahead;    // streamed split rows: next-row chunks read during an exchange
    int32_t schedule;      // grid-split kernels: row schedule (k_grid.cuh)
    int32_t resident;      // grid-split kernels: slice chunks kept in shared memory
};

// ------------------------------------------------------------ element types --

template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int kBytes = 4;
};
template <> struct Elem<__nv_bfloat16> {
    static constexpr int kBytes = 2;
};

// A vector of VB bytes as raw 32-bit words (or one 16-bit word when VB == 2).
template <int VB> struct Vec {
    static constexpr int kWords = VB / 4;
    uint32_t u[kWords];
};
template <> struct Vec<2> {
    static constexpr int kWords = 0;
    uint16_t h;
};

template <typename T, int VB> struct VecTraits {
    static constexpr int kElems = VB / Elem<T>::kBytes;
};

// Load-policy codes for the streamed input x (read exactly once):
//   0  ld.global.cs                                  (cache-streaming)
//   1  ld.global.nc.L1::no_allocate.L2::256B         (no L1 line, 256-B L2 prefetch)
//   2  ld.global.nc.L1::no_allocate                  (no L1 line)
//   3  ld.global.L1::no_allocate.L2::cache_hint      (L2 evict-first policy)
// Store-policy codes for y (written exactly once):
//   0  st.global.cs    1  st.global    2  st.global.L1::no_allocate
template <int LD>
__device__ __forceinline__ uint4 ld_v4(const void* p) {
    uint4 t;
    if constexpr (LD == 0) {
        t = __ldcs(reinterpret_cast<const uint4*>(p));
    } else if constexpr (LD == 1) {
        asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(t.x), "=r"(t.y), "=r"(t.z), "=r"(t.w) : "l"(p));
    } else if constexpr (LD == 2) {
        asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(t.x), "=r"(t.y), "=r"(t.z), "=r"(t.w) : "l"(p));
    } else {
        uint64_t pol;
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
        asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                     : "=r"(t.x), "=r"(t.y), "=r"(t.z), "=r"(t.w) : "l"(p), "l"(pol));
    }
    return t;
}

template <int ST>
__device__ __forceinline__ void st_v4(void* p, uint4 t) {
    if constexpr (ST == 0) {
        __stcs(reinterpret_cast<uint4*>(p), t);
    } else if constexpr (ST == 1) {
        asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
                     :: "l"(p), "r"(t.x), "r"(t.y), "r"(t.z), "r"(t.w) : "memory");
    } else {
        asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1,%2,%3,%4};"
                     :: "l"(p), "r"(t.x), "r"(t.y), "r"(t.z), "r"(t.w) : "memory");
    }
}

// Streaming global load of one vector (x is read exactly once).
template <int VB, int LD = 0>
__device__ __forceinline__ Vec<VB> ld_stream(const void* p) {
    Vec<VB> v;
    if constexpr (VB == 16) {
        uint4 t = ld_v4<LD>(p);
        v.u[0] = t.x; v.u[1] = t.y; v.u[2] = t.z; v.u[3] = t.w;
    } else if constexpr (VB == 8) {
        uint2 t = __ldcs(reinterpret_cast<const uint2*>(p));
        v.u[0] = t.x; v.u[1] = t.y;
    } else if constexpr (VB == 4) {
        v.u[0] = __ldcs(reinterpret_cast<const unsigned int*>(p));
    } else {
        v.h = __ldcs(reinterpret_cast<const unsigned short*>(p));
    }
    return v;
}

// Plain global load (kept in L2 normally: the two-pass kernel reads it again).
template <int VB>
__device__ __forceinline__ Vec<VB> ld_plain(const void* p) {
    Vec<VB> v;
    if constexpr (VB == 16) {
        uint4 t = *reinterpret_cast<const uint4*>(p);
        v.u[0] = t.x; v.u[1] = t.y; v.u[2] = t.z; v.u[3] = t.w;
    } else if constexpr (VB == 8) {
        uint2 t = *reinterpret_cast<const uint2*>(p);
        v.u[0] = t.x; v.u[1] = t.y;
    } else if constexpr (VB == 4) {
        v.u[0] = *reinterpret_cast<const unsigned int*>(p);
    } else {
        v.h = *reinterpret_cast<const unsigned short*>(p);
    }
    return v;
}

// Read-only cached load (the weight vector: small, re-read by every CTA).
template <int VB>
__device__ __forceinline__ Vec<VB> ld_ro(const void* p) {
    Vec<VB> v;
    if constexpr (VB == 16) {
        uint4 t = __ldg(reinterpret_cast<const uint4*>(p));
        v.u[0] = t.x; v.u[1] = t.y; v.u[2] = t.z; v.u[3] = t.w;
    } else if constexpr (VB == 8) {
        uint2 t = __ldg(reinterpret_cast<const uint2*>(p));
        v.u[0] = t.x; v.u[1] = t.y;
    } else if constexpr (VB == 4) {
        v.u[0] = __ldg(reinterpret_cast<const unsigned int*>(p));
    } else {
        v.h = __ldg(reinterpret_cast<const unsigned short*>(p));
    }
    return v;
}

// Streaming global store of one vector (y is written exactly once).
template <int VB, int ST = 0>
__device__ __forceinline__ void st_stream(void* p, const Vec<VB>& v) {
    if constexpr (VB == 16) {
        st_v4<ST>(p, make_uint4(v.u[0], v.u[1], v.u[2], v.u[3]));
    } else if constexpr (VB == 8) {
        __stcs(reinterpret_cast<uint2*>(p), make_uint2(v.u[0], v.u[1]));
    } else if constexpr (VB == 4) {
        __stcs(reinterpret_cast<unsigned int*>(p), v.u[0]);
    } else {
        __stcs(reinterpret_cast<unsigned short*>(p), v.h);
    }
}

// Keep a value opaque to the optimiser inside a loop (it is then neither
// hoisted nor re-expanded outside): used to keep packed bf16 weights packed.
__device__ __forceinline__ void opaque(uint32_t& r) { asm volatile("" : "+r"(r)); }

// Element k of a vector, widened exactly to fp32.
template <typename T, int VB>
__device__ __forceinline__ float get(const Vec<VB>& v, int k) {
    if constexpr (sizeof(T) == 4) {
        return __uint_as_float(v.u[k]);
    } else if constexpr (VB == 2) {
        return __uint_as_float(static_cast<uint32_t>(v.h) << 16);
    } else {
        uint32_t word = v.u[k >> 1];
        return __uint_as_float((k & 1) ? (word & 0xFFFF0000u) : (word << 16));
    }
}

// Build an output vector from fp32 values: fp32 as is, bf16 with one
// round-to-nearest-even rounding per element.
template <typename T, int VB>
__device__ __forceinline__ Vec<VB> pack(const float (&f)[VecTraits<T, VB>::kElems]) {
    Vec<VB> v;
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int k = 0; k < VB / 4; ++k) v.u[k] = __float_as_uint(f[k]);
    } else if constexpr (VB == 2) {
        v.h = __bfloat16_as_ushort(__float2bfloat16_rn(f[0]));
    } else {
#pragma unroll
        for (int k = 0; k < VB / 4; ++k) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(f[2 * k], f[2 * k + 1]);
            v.u[k] = *reinterpret_cast<uint32_t*>(&h2);
        }
    }
    return v;
}

// ------------------------------------------------------------- reductions --

// Butterfly sum over the 32 lanes; every lane ends with the warp total.
__device__ __forceinline__ float warp_allreduce_sum(float v) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

// The same within aligned groups of g lanes (g a power of two, 1..32): lane
// masks below g never cross a group boundary.
__device__ __forceinline__ float group_allreduce_sum(float v, int g) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1)
        if (m < g) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

// ------------------------------------------------------------ status word --

__device__ __forceinline__ void report_timeout(unsigned* status, unsigned site) {
    if (status) atomicCAS(status, 0u, kStatusTimeout | (site << 8));
}

// ------------------------------------------ programmatic dependent launch --
// Every kernel is launched so that it may start while the kernel before it in
// the stream is still running (launch.h).  pdl_trigger lets the next kernel's
// CTAs be scheduled once every CTA of this one has issued it; pdl_wait blocks
// until the kernels before this one have completed and their memory is
// visible.  Each kernel issues pdl_wait before its first global memory access
// (reads of x and w, which the previous kernel may write, and writes of y,
// which it may read), so only launch latency and set-up overlap.  Both are
// no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------- mbarrier (PTX) --

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 :: "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Wait for phase `parity` of an mbarrier with a wall-clock limit.  Returns
// false (without having observed the phase) once `timeout_ns` has passed.
template <bool kCluster>
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t timeout_ns) {
    auto probe = [&]() {
        return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    };
    if (probe()) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (probe()) return true;
        if (global_timer_ns() - t0 > timeout_ns) return false;
    }
}

// --------------------------------------------------- bulk copy (async proxy) --

// 1-D bulk copy global -> this CTA's shared memory, completing `bytes` of
// transaction count on `bar`.  dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        :: "r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy) : "memory");
}

// The same without a cache policy.
__device__ __forceinline__ void bulk_g2s_plain(uint32_t dst, const void* src, uint32_t bytes,
                                               uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// -------------------------------------------------------------- clusters --

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Shared::cluster address of the same variable in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

// Asynchronous stores into the shared memory of a CTA of this cluster (addr
// and bar are shared::cluster addresses in the same CTA): the stored bytes
// complete transaction count on that CTA's mbarrier `bar`, whose phase
// completion releases them at cluster scope.  One one-way trip, no fence.
__device__ __forceinline__ void st_async_f32(uint32_t addr, float v, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];"
                 :: "r"(addr), "f"(v), "r"(bar) : "memory");
}

__device__ __forceinline__ void st_async_v2_f32(uint32_t addr, float a, float b, uint32_t bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];"
        :: "r"(addr), "f"(a), "f"(b), "r"(bar) : "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void fence_mbarrier_init_cluster() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// ------------------------------------------- cluster-wide row sum exchange --

// Shared-memory state of the DSMEM exchange: two slot sets and two mbarriers,
// used alternately by consecutive rows (a peer can be at most one row ahead).
// Each barrier phase takes one local arrival, which also expects the bytes of
// the C slots; every CTA's st.async completes its share.  A peer's bytes may
// land before the local arrival (the transaction count then dips below zero,
// which the mbarrier allows); the phase completes only once both happened.
struct ClusterExchange {
    alignas(8) unsigned long long bar[2];
    float slot[2][16];
};

// Initialise (thread 0) the exchange, make its barriers visible cluster-wide,
// and sync the cluster so no peer stores before initialisation.
__device__ __forceinline__ void cluster_exchange_init(ClusterExchange* ex) {
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&ex->bar[0]), 1);
        mbar_init(smem_addr(&ex->bar[1]), 1);
        fence_mbarrier_init_cluster();
    }
    __syncthreads();
    cluster_sync_all();
}

// Sum `part` (this CTA's value, identical in all participating threads) over
// the cluster.  Every CTA adds the C slots in rank order, so every CTA gets
// the bitwise same result.
// `it` is this CTA's row iteration count and `lt` the caller's index among
// the participating threads (the first `ncta` of them send).  Returns false
// if the bounded wait expired (the status word is then set).  The caller
// must pass a barrier over the participants after this returns and before
// its next call on the same exchange (the slots are reused two rows on).
__device__ __forceinline__ bool cluster_allreduce(ClusterExchange* ex, float part, int ncta,
                                                  uint32_t rank, uint32_t it,
                                                  const Params& p, float* total, int lt) {
    const uint32_t b = it & 1u;
    const uint32_t bar = smem_addr(&ex->bar[b]);
    if (lt == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(ncta) * 4u);
    bool send = lt < ncta;
#if RMSNORM_FAULT_INJECT
    if (p.fault == kFaultClusterWithholdPartial && rank == 0 && it == 0) send = false;
#endif
    if (send) {
        const uint32_t peer = static_cast<uint32_t>(lt);
        st_async_f32(map_to_rank(smem_addr(&ex->slot[b][rank]), peer), part,
                     map_to_rank(bar, peer));
    }
    const bool ok = mbar_wait_bounded<true>(bar, (it >> 1) & 1u, p.timeout_ns);
    float s = 0.f;
    if (ok) {
        for (int c = 0; c < ncta; ++c) s += ex->slot[b][c];
    } else if (lt == 0) {
        report_timeout(p.status, kSiteClusterExchange);
    }
    *total = s;
    return ok;
}

}  // namespace rmsnorm
