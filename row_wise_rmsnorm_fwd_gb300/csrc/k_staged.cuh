// k_staged.cuh -- RMSNorm forward with the row staged in shared memory by
// 1-D bulk copies (cp.async.bulk, async proxy) and mbarrier completion.
//
// Warp 0 is the producer: one lane issues the copies.  Warps 1..W are the
// consumers.  A CTA owns one row (or, with a cluster, one slice of a row) at a
// time; the slice is split into NCH chunks, each with a "full" mbarrier
// (producer arrive + transaction bytes) and an "empty" mbarrier (one arrive per
// consumer warp).  Per row:
//   - consumers wait full[k] chunk by chunk and accumulate the fp32 sum of
//     squares while later chunks are still in flight;
//   - the sum is combined across consumer warps (one named barrier) and, for
//     a split row, across the cluster through distributed shared memory;
//   - consumers normalise chunk k from shared memory, store y with streaming
//     16-byte stores, and release chunk k on empty[k];
//   - the producer refills chunk k with the NEXT row's chunk k as soon as it is
//     released, so the next row's loads overlap this row's stores.
// This is the multi-stage prefetch loop of the CuTe DSL page (prologue fills
// the stages, the steady state consumes stage i while stage i+S is in flight)
// with the stage ring laid over the row itself.
//
// Proxy rule (TileLang InjectFenceProxy page): shared memory written by the
// async proxy (bulk copy) is read here by the generic proxy only after the
// mbarrier wait, which orders it; consumers never write the staging buffer
// with generic stores, so no fence.proxy.async is needed before the refill.
// Generic reads before an async-proxy overwrite (WAR) are ordered by the
// empty-barrier release/acquire.
//
// Every wait is bounded (wall clock); on expiry the kernel records a status
// code, stops issuing work, waits (bounded) for the copies it has issued and
// leaves through the final cluster barrier that every thread reaches.
#pragma once
#include "common.cuh"

namespace rmsnorm {

constexpr int kStagedConsumers = 8;                          // consumer warps
constexpr int kStagedBlock = 32 * (kStagedConsumers + 1);    // + producer warp
constexpr int kStagedMaxChunks = 32;
constexpr int kStagedHeader = 1024;                          // barriers, scratch

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads.
__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool pred) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred q, r;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred r, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, r;\n\t}"
        : "=r"(out) : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads) : "memory");
    return out != 0;
}

template <typename T>
__global__ void __launch_bounds__(kStagedBlock, 1) staged_kernel(const Params p) {
    constexpr int EPV = 16 / static_cast<int>(sizeof(T));
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kStagedMaxChunks;
    float* red = reinterpret_cast<float*>(smem + 16 * kStagedMaxChunks);        // [2][32]
    ClusterExchange* ex = reinterpret_cast<ClusterExchange*>(
        smem + 16 * kStagedMaxChunks + 256);
    unsigned char* buf = smem + kStagedHeader;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int NCH = p.nchunks;
    const int CB = p.chunk_bytes;
    const int ncta = p.cluster;
    constexpr int NC = 32 * kStagedConsumers;

    uint32_t rank = 0;
    int64_t unit = blockIdx.x, nunits = gridDim.x;
    if (ncta > 1) {
        rank = cluster_ctarank();
        unit = cluster_id_x();
        nunits = cluster_count_x();
    }
    const int64_t row_bytes = static_cast<int64_t>(p.hidden) * sizeof(T);
    const int64_t slice_nom = static_cast<int64_t>(p.slice_vecs) * 16;
    const int64_t sbeg = static_cast<int64_t>(rank) * slice_nom;
    const int64_t send = (sbeg + slice_nom < row_bytes) ? sbeg + slice_nom : row_bytes;
    const int64_t my_bytes = send > sbeg ? send - sbeg : 0;

    if (tid == 0) {
        for (int k = 0; k < NCH; ++k) {
            mbar_init(smem_addr(&full[k]), 1);
            mbar_init(smem_addr(&empty[k]), kStagedConsumers);
        }
        if (ncta > 1) {
            mbar_init(smem_addr(&ex->bar[0]), ncta);
            mbar_init(smem_addr(&ex->bar[1]), ncta);
        }
        fence_mbarrier_init_cluster();
    }
    __syncthreads();
    if (ncta > 1) cluster_sync_all();

    auto chunk_len = [&](int k) -> int {
        const int64_t rem = my_bytes - static_cast<int64_t>(k) * CB;
        return rem <= 0 ? 0 : static_cast<int>(rem < CB ? rem : CB);
    };

    if (warp == 0) {
        // ------------------------------------------------------ producer --
        if (lane == 0) {
            const uint64_t policy = policy_evict_first();
            const char* xb = static_cast<const char*>(p.x);
            int64_t last_it = -1;
            uint32_t it = 0;
            bool abort = false;
            for (int64_t rb = unit; rb < p.rows && !abort; rb += nunits, ++it) {
                const char* src = xb + rb * row_bytes + sbeg;
                for (int k = 0; k < NCH; ++k) {
                    if (it > 0 && !mbar_wait_bounded<false>(smem_addr(&empty[k]),
                                                            (it - 1) & 1u, p.timeout_ns)) {
                        report_timeout(p.status, kSiteStagedEmpty);
                        abort = true;
                        break;
                    }
                    const int len = chunk_len(k);
                    const uint32_t fb = smem_addr(&full[k]);
                    if (len > 0) {
                        mbar_arrive_expect_tx(fb, static_cast<uint32_t>(len));
                        bulk_g2s(smem_addr(buf + static_cast<int64_t>(k) * CB), src + k * CB,
                                 static_cast<uint32_t>(len), fb, policy);
                    } else {
                        mbar_arrive(fb);
                    }
                }
                if (!abort) last_it = it;
            }
            // Copies issued for the last row must have landed before this CTA
            // may leave (normally they have: the consumers waited for them).
            if (last_it >= 0) {
                for (int k = 0; k < NCH; ++k)
                    mbar_wait_bounded<false>(smem_addr(&full[k]),
                                             static_cast<uint32_t>(last_it) & 1u, p.timeout_ns);
            }
        }
        __syncwarp();
    } else {
        // ----------------------------------------------------- consumers --
        const int ct = tid - 32;
        const char* wb = static_cast<const char*>(p.w) + sbeg;
        char* yb = static_cast<char*>(p.y);
        uint32_t it = 0;
        for (int64_t rb = unit; rb < p.rows; rb += nunits, ++it) {
            float s0 = 0.f, s1 = 0.f;
            bool ok = true;
            for (int k = 0; k < NCH; ++k) {
                if (!mbar_wait_bounded<false>(smem_addr(&full[k]), it & 1u, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                const int nv = chunk_len(k) >> 4;
                const uint4* c = reinterpret_cast<const uint4*>(buf + static_cast<int64_t>(k) * CB);
                for (int v = ct; v < nv; v += NC) {
                    const uint4 q = c[v];
                    Vec<16> xv;
                    xv.u[0] = q.x; xv.u[1] = q.y; xv.u[2] = q.z; xv.u[3] = q.w;
#pragma unroll
                    for (int e = 0; e < EPV; ++e) {
                        const float f = get<T, 16>(xv, e);
                        if (e & 1) s1 = fmaf(f, f, s1); else s0 = fmaf(f, f, s0);
                    }
                }
            }
            float ss = warp_allreduce_sum(s0 + s1);
            const int b = it & 1;
            if (lane == 0) red[b * 32 + (warp - 1)] = ss;
            named_bar_sync(1, NC);
            ss = 0.f;
            for (int k = 0; k < kStagedConsumers; ++k) ss += red[b * 32 + k];
            if (ncta > 1 && ok) {
                float total;
                ok = cluster_allreduce(ex, ss, ncta, rank, it, p, &total, ct);
                ss = total;
            }
            if (named_bar_or(1, NC, !ok)) {
                if (ct == 0) report_timeout(p.status, kSiteStagedFull);
                break;
            }
            const float rstd = rsqrtf(fmaf(ss, p.inv_hidden, p.eps));
            char* dst = yb + rb * row_bytes + sbeg;
            for (int k = 0; k < NCH; ++k) {
                const int nv = chunk_len(k) >> 4;
                const uint4* c = reinterpret_cast<const uint4*>(buf + static_cast<int64_t>(k) * CB);
                for (int v = ct; v < nv; v += NC) {
                    const uint4 q = c[v];
                    Vec<16> xv;
                    xv.u[0] = q.x; xv.u[1] = q.y; xv.u[2] = q.z; xv.u[3] = q.w;
                    const int64_t off = static_cast<int64_t>(k) * CB + static_cast<int64_t>(v) * 16;
                    const Vec<16> wv = ld_ro<16>(wb + off);
                    float o[EPV];
#pragma unroll
                    for (int e = 0; e < EPV; ++e)
                        o[e] = (get<T, 16>(xv, e) * rstd) * get<T, 16>(wv, e);
                    st_stream<16>(dst + off, pack<T, 16>(o));
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&empty[k]));
            }
        }
    }
    if (ncta > 1) {
        __syncwarp();
        cluster_sync_all();
    }
}

}  // namespace rmsnorm
