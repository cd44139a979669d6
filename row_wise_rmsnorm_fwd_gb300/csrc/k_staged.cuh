// k_staged.cuh -- RMSNorm forward with rows staged in shared memory by 1-D
// bulk copies through the slot ring of k_ring.cuh.
//
// Warp 0 is the producer: one lane issues the copies.  Warps 1..NCW are the
// consumers (NCW = 4 or 8).  A CTA owns one row (or, with a cluster, one
// slice of a row) at a time.  Per row:
//   - consumers wait for the chunks one by one and accumulate the fp32 sum of
//     squares while later chunks are still in flight;
//   - the sum is combined across consumer warps (one named barrier) and, for a
//     split row, across the cluster through distributed shared memory;
//   - consumers normalise each chunk from shared memory, store y with
//     streaming 16-byte stores, and release the slot;
//   - the producer refills released slots with the next chunks of the stream,
//     running ahead into the following rows.
// When it fits, the CTA's weight slice is copied to shared memory once;
// otherwise weights come through L1/L2, loaded in batches of four vectors.
//
// Every wait is bounded (wall clock); on expiry the kernel records a status
// code, stops issuing work, waits (bounded) for the copies it has issued and
// leaves through the final cluster barrier that every thread reaches.
#pragma once
#include "k_ring.cuh"

namespace rmsnorm {

constexpr int kStagedUnroll = 4;                             // vectors per batch

// NCW consumer warps (plus the producer warp).  Registers are capped at 96 so
// that two 9-warp CTAs fit the register file of every SM sub-partition.
template <typename T, int NCW, int EPI>
__global__ void __maxnreg__(96) staged_kernel(const Params p) {
    pdl_trigger();
    pdl_wait();
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

    const SlotRing ring{full, empty, wsm + wreserve, S, NCH, CB, my_bytes};

    if (tid == 0) {
        ring_init(ring, NCW);
        mbar_init(smem_addr(wbar), 1);
        if (ncta > 1) {
            mbar_init(smem_addr(&ex->bar[0]), 1);   // one local arrival per phase
            mbar_init(smem_addr(&ex->bar[1]), 1);
        }
        fence_mbarrier_init_cluster();
    }
    __syncthreads();
    if (ncta > 1) cluster_sync_all();

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
            ring_produce(p, ring, unit, nunits, row_bytes, sbeg, policy, kSiteStagedEmpty);
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
        // Slots and phases come from the 64-bit stream index once per chunk.
        // Tracking them incrementally in 32 bits (as the staged softmax does
        // per vector) measured slower here: 91.8% against 95.8% of the HBM
        // roofline on rows of 64 KB.
        int64_t base = 0;          // stream index of this row's chunk 0
        for (int64_t rb = unit; rb < p.rows; rb += nunits, ++it, base += NCH) {
            float s0 = 0.f, s1 = 0.f;
            for (int k = 0; k < NCH && ok; ++k) {
                const int64_t n = base + k;
                const int slot = static_cast<int>(n % S);
                if (!ring_wait_full(ring, n, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                const int nv = ring.chunk_len(k) >> 4;
                const uint4* c = ring.slot_vecs(slot);
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
                const int nv = ring.chunk_len(k) >> 4;
                const uint4* c = ring.slot_vecs(slot);
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
