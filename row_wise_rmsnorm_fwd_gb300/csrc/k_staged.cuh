// k_staged.cuh -- RMSNorm forward with rows staged in shared memory by 1-D
// bulk copies (cp.async.bulk, async proxy) completing on mbarriers.
//
// Warp 0 is the producer: one lane issues the copies.  Warps 1..NCW are the
// consumers (NCW = 4 or 8).  A CTA owns one row (or, with a cluster, one slice of a row) at a
// time.  The slice is cut into NCH chunks; the chunks of consecutive rows flow
// through a ring of S >= NCH shared-memory slots, each with a "full" mbarrier
// (producer arrive + transaction bytes) and an "empty" mbarrier (one arrive per
// consumer warp).  Chunk number n of the CTA's stream (row n / NCH, chunk
// n % NCH) lives in slot n % S, on that slot's (n / S)-th use.  Per row:
//   - consumers wait full[] chunk by chunk and accumulate the fp32 sum of
//     squares while later chunks are still in flight;
//   - the sum is combined across consumer warps (one named barrier) and, for a
//     split row, across the cluster through distributed shared memory;
//   - consumers normalise each chunk from shared memory, store y with
//     streaming 16-byte stores, and release the slot on empty[];
//   - the producer refills a released slot with the next chunk of the stream,
//     running up to S - NCH chunks ahead into the following rows.
// This is the multi-stage prefetch loop of the CuTe DSL page (a prologue fills
// the stages; the steady state consumes stage i while stage i+S is in flight).
// When it fits, the CTA's weight slice is copied to shared memory once;
// otherwise weights come through L1/L2, loaded in batches of four vectors.
//
// Proxy rule (TileLang InjectFenceProxy page): shared memory written by the
// async proxy (bulk copy) is read by the generic proxy only after the mbarrier
// wait, which orders it; no generic store ever writes a staging slot, so no
// fence.proxy.async is needed before a refill (generic reads followed by an
// async-proxy overwrite are ordered through the empty-barrier release and the
// producer's acquire).
//
// Every wait is bounded (wall clock); on expiry the kernel records a status
// code, stops issuing work, waits (bounded) for the copies it has issued and
// leaves through the final cluster barrier that every thread reaches.
#pragma once
#include "common.cuh"

namespace rmsnorm {

constexpr int kStagedMaxSlots = 32;
constexpr int kStagedHeader = 1024;                          // barriers, scratch
constexpr int kStagedUnroll = 4;                             // vectors per batch

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

__device__ __forceinline__ Vec<16> as_vec(const uint4& q) {
    Vec<16> v;
    v.u[0] = q.x; v.u[1] = q.y; v.u[2] = q.z; v.u[3] = q.w;
    return v;
}

// NCW consumer warps (plus the producer warp).  Registers are capped at 96 so
// that two 9-warp CTAs fit the register file of every SM sub-partition.
template <typename T, int NCW, int EPI>
__global__ void __maxnreg__(96) staged_kernel(const Params p) {
    constexpr int EPV = 16 / static_cast<int>(sizeof(T));
    constexpr int NC = 32 * NCW;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kStagedMaxSlots;
    uint64_t* wbar = empty + kStagedMaxSlots;
    float* red = reinterpret_cast<float*>(smem + 16 * kStagedMaxSlots + 16);     // [2][32]
    ClusterExchange* ex = reinterpret_cast<ClusterExchange*>(
        smem + 16 * kStagedMaxSlots + 16 + 256);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int NCH = p.nchunks;
    const int S = p.nslots;
    const int CB = p.chunk_bytes;
    const int ncta = p.cluster;

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

    // Weight slice (optional) and the slot ring follow the header.
    unsigned char* wsm = smem + kStagedHeader;
    const int64_t wreserve = p.w_staged ? slice_nom : 0;
    unsigned char* ring = wsm + wreserve;

    if (tid == 0) {
        for (int k = 0; k < S; ++k) {
            mbar_init(smem_addr(&full[k]), 1);
            mbar_init(smem_addr(&empty[k]), NCW);
        }
        mbar_init(smem_addr(wbar), 1);
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
            if (p.w_staged) {
                const uint32_t wb = smem_addr(wbar);
                if (my_bytes > 0) {
                    mbar_arrive_expect_tx(wb, static_cast<uint32_t>(my_bytes));
                    bulk_g2s_plain(smem_addr(wsm), static_cast<const char*>(p.w) + sbeg,
                                   static_cast<uint32_t>(my_bytes), wb);
                } else {
                    mbar_arrive(wb);
                }
            }
            const char* xb = static_cast<const char*>(p.x);
            int64_t seq = 0;       // chunks issued so far
            bool abort = false;
            for (int64_t rb = unit; rb < p.rows && !abort; rb += nunits) {
                const char* src = xb + rb * row_bytes + sbeg;
                for (int k = 0; k < NCH; ++k, ++seq) {
                    const int slot = static_cast<int>(seq % S);
                    const int64_t use = seq / S;
                    if (use > 0 && !mbar_wait_bounded<false>(smem_addr(&empty[slot]),
                                                             static_cast<uint32_t>(use - 1) & 1u,
                                                             p.timeout_ns)) {
                        report_timeout(p.status, kSiteStagedEmpty);
                        abort = true;
                        break;
                    }
                    const int len = chunk_len(k);
                    const uint32_t fb = smem_addr(&full[slot]);
#if RMSNORM_FAULT_INJECT
                    if (p.fault == kFaultStagedWithholdCopy && seq == 0 && len > 0) {
                        // Arm the barrier for bytes that never come: every wait on
                        // this phase must run out, nothing is in flight.
                        mbar_arrive_expect_tx(fb, static_cast<uint32_t>(len));
                        continue;
                    }
#endif
                    if (len > 0) {
                        mbar_arrive_expect_tx(fb, static_cast<uint32_t>(len));
                        bulk_g2s(smem_addr(ring + static_cast<int64_t>(slot) * CB),
                                 src + static_cast<int64_t>(k) * CB,
                                 static_cast<uint32_t>(len), fb, policy);
                    } else {
                        mbar_arrive(fb);
                    }
                }
            }
            // Every copy issued must have landed before this CTA may leave
            // (normally it has: the consumers waited for all of them).
            const int64_t first = seq > S ? seq - S : 0;
            for (int64_t n = first; n < seq; ++n)
                mbar_wait_bounded<false>(smem_addr(&full[n % S]),
                                         static_cast<uint32_t>(n / S) & 1u, p.timeout_ns);
            if (p.w_staged) mbar_wait_bounded<false>(smem_addr(wbar), 0u, p.timeout_ns);
        }
        __syncwarp();
    } else {
        // ----------------------------------------------------- consumers --
        const int ct = tid - 32;
        const char* wg = static_cast<const char*>(p.w) + sbeg;
        char* yb = static_cast<char*>(p.y);
        bool ok = true;
        if (p.w_staged)
            ok = mbar_wait_bounded<false>(smem_addr(wbar), 0u, p.timeout_ns);
        uint32_t it = 0;
        int64_t base = 0;          // stream index of this row's chunk 0
        for (int64_t rb = unit; rb < p.rows; rb += nunits, ++it, base += NCH) {
            float s0 = 0.f, s1 = 0.f;
            for (int k = 0; k < NCH && ok; ++k) {
                const int64_t n = base + k;
                const int slot = static_cast<int>(n % S);
                if (!mbar_wait_bounded<false>(smem_addr(&full[slot]),
                                              static_cast<uint32_t>(n / S) & 1u, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                const int nv = chunk_len(k) >> 4;
                const uint4* c = reinterpret_cast<const uint4*>(ring + static_cast<int64_t>(slot) * CB);
                for (int v0 = ct; v0 < nv; v0 += kStagedUnroll * NC) {
                    uint4 q[kStagedUnroll];
#pragma unroll
                    for (int u = 0; u < kStagedUnroll; ++u)
                        if (v0 + u * NC < nv) q[u] = c[v0 + u * NC];
#pragma unroll
                    for (int u = 0; u < kStagedUnroll; ++u) {
                        if (v0 + u * NC < nv) {
                            const Vec<16> xv = as_vec(q[u]);
#pragma unroll
                            for (int e = 0; e < EPV; ++e) {
                                const float f = get<T, 16>(xv, e);
                                if (e & 1) s1 = fmaf(f, f, s1); else s0 = fmaf(f, f, s0);
                            }
                        }
                    }
                }
            }
            float ss = warp_allreduce_sum(s0 + s1);
            const int b = it & 1;
            if (lane == 0) red[b * 32 + (warp - 1)] = ss;
            named_bar_sync(1, NC);
            ss = 0.f;
            for (int k = 0; k < NCW; ++k) ss += red[b * 32 + k];
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
                const int64_t n = base + k;
                const int slot = static_cast<int>(n % S);
                const int nv = chunk_len(k) >> 4;
                const uint4* c = reinterpret_cast<const uint4*>(ring + static_cast<int64_t>(slot) * CB);
                const int64_t koff = static_cast<int64_t>(k) * CB;
                for (int v0 = ct; v0 < nv; v0 += kStagedUnroll * NC) {
                    uint4 q[kStagedUnroll];
                    Vec<16> wv[kStagedUnroll];
#pragma unroll
                    for (int u = 0; u < kStagedUnroll; ++u) {
                        const int v = v0 + u * NC;
                        if (v < nv) {
                            q[u] = c[v];
                            const int64_t off = koff + static_cast<int64_t>(v) * 16;
                            if (p.w_staged)
                                wv[u] = as_vec(*reinterpret_cast<const uint4*>(wsm + off));
                            else
                                wv[u] = ld_ro<16>(wg + off);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < kStagedUnroll; ++u) {
                        const int v = v0 + u * NC;
                        if (v < nv) {
                            const Vec<16> xv = as_vec(q[u]);
                            float o[EPV];
#pragma unroll
                            for (int e = 0; e < EPV; ++e)
                                o[e] = epilogue<EPI>(
                                    (get<T, 16>(xv, e) * rstd) * get<T, 16>(wv[u], e), p.alpha);
                            st_stream<16>(dst + koff + static_cast<int64_t>(v) * 16,
                                          pack<T, 16>(o));
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&empty[slot]));
            }
        }
    }
    if (ncta > 1) {
        __syncwarp();
        cluster_sync_all();
    }
}

}  // namespace rmsnorm
