// k_stream.cuh -- row softmax for many rows too wide for one CTA's registers
// (prefill logits of a large vocabulary: rows of 128256 elements), every row
// streamed twice through the bulk-copy slot ring of k_ring.cuh.
//
// One CTA per SM (or a cluster of CTAs per row, each a slice), one row at a
// time: warp 0's lane 0 produces (the row's chunks, then the same chunks
// again; for a split row, with the next row's first p.read_ahead chunks
// between the two, so that DRAM keeps reading while the cluster combines the
// row's pairs), the other warps consume.
//   pass A: each consumer thread keeps an online pair (m_t, s_t): the
//     maximum of the elements it has seen and the sum of their exponentials
//     relative to it; a chunk that raises m_t first rescales s_t.  At the
//     row's end the pairs are folded over the warp (butterfly) and over the
//     warps (one slot per warp, one named barrier, a fixed-order fold in
//     every thread), which is the online-softmax combine, and give the row's
//     maximum M and sum S.
//   pass B: the same chunks again, the outputs exp(x - M) / S stored from
//     registers.
// The first read comes from DRAM with an L2 keep policy, the second from L2
// (the rows in flight on all SMs, 152 x 513 KB for fp32 prefill logits,
// fit in L2), so DRAM moves x once and y once.  Unlike the register-resident
// and cluster-split kernels no thread holds a row: the ring can take all of
// shared memory, which keeps a row's worth of copies in flight per SM.
//
// Exponent arguments: pass A uses the exact form (x - m_t)*log2e + bias (the
// maximum changes as the row goes by, so a rounded offset would differ from
// thread to thread); pass B uses the fused form with the row's offset where
// row_exp_offset_ok allows it, with the offset's rounding taken out of 1/S
// (slice_offset_correction), else the exact form.  A thread that has seen
// only -inf entries keeps (-inf, 0) and adds nothing; a row of -inf, or with
// a NaN or +inf, ends with a NaN sum and a NaN row, as the definition gives.
#pragma once
#include "k_exchange.cuh"


namespace rmsnorm {

// 15 consumer warps + the producer: four warps per SM sub-partition, up to 128
// registers a thread (a 17th warp would cap them at 96 and spill).
constexpr int kStreamMaxThreads = 512;


__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// This thread's vectors of one chunk, raw (bf16: half the registers of the
// widened pairs): src = its first vector in the slot, vstride = bytes to its
// next one.  kFull: all V vectors are there (no bounds checks), else only
// those below nv (q0 = this thread's first vector index, nc = vectors per
// step).
template <int V, bool kFull>
__device__ __forceinline__ void stream_load(Vec<16> (&raw)[V], const unsigned char* src,
                                            int64_t vstride, int q0, int nc, int nv) {
#pragma unroll
    for (int i = 0; i < V; ++i)
        if (kFull || q0 + i * nc < nv)
            raw[i] = as_vec(*reinterpret_cast<const uint4*>(src + i * vstride));
}

// Pass A on one chunk: fold its maximum into the running pair (m, s), then
// add its exponentials relative to the new maximum.
template <typename T, int V, bool kFull>
__device__ __forceinline__ float2 stream_fold(const Vec<16> (&raw)[V], int q0, int nc, int nv,
                                              float2 ms) {
    using RV = RowVec<T, 16>;
    float mk[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    uint32_t mw[2] = {kBf16x2NegInf, kBf16x2NegInf};
#pragma unroll
    for (int i = 0; i < V; ++i)
        if (kFull || q0 + i * nc < nv) RV::fold_max(raw[i], mk, mw);
    float mt = ms.x, st = ms.y;
    const float mn = fmaxf(mt, running_max(mk, mw));
    if (mn > mt) {
        st *= exp2f((mt - mn) * kLog2e);       // 0 while mt was -inf
        mt = mn;
    }
    const float mu = mt == -INFINITY ? 0.f : mt;   // -inf entries give 0, not NaN
    typename RV::Sums sums;
#pragma unroll
    for (int i = 0; i < V; ++i) {
        if (kFull || q0 + i * nc < nv) {
            RV e;
            e.widen(raw[i]);
            e.template exp<false>(0.f, sums, mu);
        }
    }
    return make_float2(mt, st + sums.total());
}

// Shared-memory header of the streamed kernels: full[32] | empty[32] |
// red[2][32] pairs | the cluster pair exchange (split rows), or the grid
// kernels' warp slots (k_grid.cuh).
constexpr int kStreamHeader = 2048;

// Splits of a row over several CTAs (the whole-grid split is softmax_grid's,
// k_grid.cuh).
enum : int {
    kSplitNone = 0,      // one CTA per row
    kSplitCluster = 1,   // a thread-block cluster per row, pairs through DSMEM
};

// V: 16-byte vectors per consumer thread per chunk (chunk_bytes = 16 * V *
// consumer threads).  SPLIT = kSplitCluster: each row over a thread-block
// cluster of p.cluster CTAs, CTA rank r streaming slice r (p.slice_vecs
// vectors) of its cluster's rows; the CTAs' (maximum, sum) pairs cross the
// cluster once per row through distributed shared memory
// (cluster_pair_allreduce, bounded wait).  Splitting halves (for two CTAs)
// the bytes of rows in flight, which the second read needs to find in L2.
template <typename T, int V, int SPLIT>
__global__ void __launch_bounds__(kStreamMaxThreads, 1) softmax_stream_kernel(const Params p) {
    pdl_trigger();
    pdl_wait();
    constexpr bool CL = SPLIT == kSplitCluster;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kStagedMaxSlots;
    float2* red = reinterpret_cast<float2*>(smem + 16 * kStagedMaxSlots);
    PairExchange* ex = reinterpret_cast<PairExchange*>(smem + 16 * kStagedMaxSlots + 512);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int NCW = static_cast<int>(blockDim.x >> 5) - 1;   // consumer warps
    const int NC = NCW * 32;
    const int NCH = p.nchunks, S = p.nslots, CB = p.chunk_bytes;
    const int64_t row_bytes = static_cast<int64_t>(p.hidden) * sizeof(T);
    const int ncta = CL ? p.cluster : 1;
    uint32_t rank = 0;
    int64_t unit = blockIdx.x, nunits = gridDim.x;
    if (CL) {
        rank = cluster_ctarank();
        unit = cluster_id_x();
        nunits = cluster_count_x();
    }
    const int64_t slice_nom = SPLIT != kSplitNone ? static_cast<int64_t>(p.slice_vecs) * 16
                                                  : row_bytes;
    const int64_t sbeg = static_cast<int64_t>(rank) * slice_nom;
    const int64_t send = sbeg + slice_nom < row_bytes ? sbeg + slice_nom : row_bytes;
    const int64_t my_bytes = send > sbeg ? send - sbeg : 0;
    const SlotRing ring{full, empty, smem + kStreamHeader, S, NCH, CB, my_bytes};

    if (tid == 0) {
        ring_init(ring, NCW);
        if (CL) {
            mbar_init(smem_addr(&ex->bar[0]), 1);
            mbar_init(smem_addr(&ex->bar[1]), 1);
        }
        fence_mbarrier_init_cluster();
    }
    __syncthreads();
    if (CL) cluster_sync_all();        // no peer sends before the barriers exist
    // chunks of the next row read while the cluster combines this row (the
    // planner's choice: measured on fp32 prefill logits, clusters of 2, %
    // of the HBM copy peak, 0 / 1 / 2 / 3 / 4 / 6 chunks 83.6 / 85.0 / 84.9 /
    // 84.6 / 81.2 / 76.6; unsplit rows combine within the CTA and read
    // nothing ahead -- 2 chunks measured 1-2 points lower there)
    const int D = !CL ? 0 : NCH < p.read_ahead ? NCH : p.read_ahead;

    if (warp == 0) {
        // ---------------------------------------------------------- producer --
        if (lane == 0) {
            // first read evict_last (measured against evict_normal: prefill
            // logits bf16 88.6 / 84.7%, fp32 C=2 83.1 / 81.6% of the HBM copy
            // peak), second read evict_first.  Order: row r's first read
            // (less the chunks read ahead), the next row's first D chunks
            // (read while the consumers combine row r), row r's second read.
            const uint64_t keep = policy_evict_last(), done = policy_evict_first();
            if (D == 0) {
                ring_produce(p, ring, unit, nunits, row_bytes, sbeg, keep, kSiteStagedEmpty, 2,
                             done);
            } else {
                const char* xb = static_cast<const char*>(p.x) + sbeg;
                RingCursorSeq c;
                auto push = [&](int64_t row, int k0, int k1, uint64_t pol) {
                    for (int k = k0; k < k1; ++k)
                        ring_push(p, ring, c,
                                  xb + row * row_bytes + static_cast<int64_t>(k) * CB,
                                  ring.chunk_len(k), pol, kSiteStagedEmpty);
                };
                if (unit < p.rows) push(unit, 0, D, keep);
                for (int64_t row = unit; row < p.rows && !c.abort; row += nunits) {
                    push(row, D, NCH, keep);
                    if (row + nunits < p.rows) push(row + nunits, 0, D, keep);
                    push(row, 0, NCH, done);
                }
                ring_drain(p, ring, c);
            }
        }
        __syncwarp();
    } else {
        // -------------------------------------------------------- consumers --
        const int ct = tid - 32;
        const int cw = warp - 1;
        char* yb = static_cast<char*>(p.y);
        int slot = 0;            // the next chunk's slot
        uint32_t lap = 0;        // its phase parity
        bool ok = true;          // warp-uniform; false once a bounded wait expired
        // Wait (bounded) for the next chunk; every lane of the warp agrees.
        auto acquire = [&]() {
            ok = __all_sync(0xffffffffu, ok && mbar_wait_bounded<false>(smem_addr(&full[slot]),
                                                                        lap, p.timeout_ns));
            return ok;
        };
        // The warp has copied its vectors of the chunk: hand the slot back.
        auto release = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&empty[slot]));
            if (++slot == S) {
                slot = 0;
                lap ^= 1u;
            }
        };
        // This thread's first vector in the current slot; vector i of a chunk
        // is i * NC vectors further on.
        auto slot_base = [&]() {
            return ring.slots + static_cast<int64_t>(slot) * CB + static_cast<int64_t>(ct) * 16;
        };
        const int64_t vstride = static_cast<int64_t>(NC) * 16;
        const int full_nv = V * NC;            // vectors of a full chunk

        // pass B: exp(x - M) / S from the same chunks again
        auto pass_b = [&](int64_t row, float M, float Ssum) {
            const bool fast = row_exp_offset_ok(M);
            const float c = row_exp_bias<T>() - M * kLog2e;
            const float Mu = M == -INFINITY ? 0.f : M;
            const float inv = (fast ? slice_offset_correction<T>(M, c) : 1.0f) / Ssum;
            char* dst = yb + row * row_bytes + sbeg + static_cast<int64_t>(ct) * 16;
            auto pass_b_chunk = [&](auto ftag, auto full_tag, int k, int nv) {
                constexpr bool F = decltype(ftag)::value;
                constexpr bool kFull = decltype(full_tag)::value;
                Vec<16> raw[V];
                stream_load<V, kFull>(raw, slot_base(), vstride, ct, NC, nv);
                release();
                char* cdst = dst + static_cast<int64_t>(k) * CB;
#pragma unroll
                for (int i = 0; i < V; ++i) {
                    if (kFull || ct + i * NC < nv) {
                        RowVec<T, 16> e;
                        e.widen(raw[i]);
                        st_stream<16>(cdst + i * vstride, e.template exp_scaled<F>(c, inv, Mu));
                    }
                }
            };
            if (fast) {
#pragma unroll 1
                for (int k = 0; k < NCH && acquire(); ++k) {
                    const int nv = ring.chunk_len(k) >> 4;
                    if (nv == full_nv) pass_b_chunk(std::true_type{}, std::true_type{}, k, nv);
                    else pass_b_chunk(std::true_type{}, std::false_type{}, k, nv);
                }
            } else {               // rows of large or non-finite maximum: rare
#pragma unroll 1
                for (int k = 0; k < NCH && acquire(); ++k)
                    pass_b_chunk(std::false_type{}, std::false_type{}, k, ring.chunk_len(k) >> 4);
            }
        };
        // pass A on chunk k (acquired): fold it into the online (maximum, sum)
        // pair (m, s) of this thread's elements; the pairs are summed in blocks
        // of kSumBlockChunks chunks, each folded from an empty pair, into
        // (mt, st) (no fp32 chain grows with the row)
        auto first_read = [&](int k, float2& ms) {
            const int nv = ring.chunk_len(k) >> 4;
            Vec<16> raw[V];
            if (nv == full_nv) {
                stream_load<V, true>(raw, slot_base(), vstride, ct, NC, nv);
                release();
                ms = stream_fold<T, V, true>(raw, ct, NC, nv, ms);
            } else {
                stream_load<V, false>(raw, slot_base(), vstride, ct, NC, nv);
                release();
                ms = stream_fold<T, V, false>(raw, ct, NC, nv, ms);
            }
        };
        // The CTA's pair of a row: warp butterfly, one slot per warp, a
        // fixed-order fold in every thread.  False (uniform) once a wait ran
        // out.
        auto cta_pair = [&](float mt, float st, uint32_t it, float& M, float& Ssum) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float mo = __shfl_xor_sync(0xffffffffu, mt, o);
                const float so = __shfl_xor_sync(0xffffffffu, st, o);
                pair_fold(mt, st, mo, so);
            }
            const int b = it & 1;
            if (lane == 0) red[b * 32 + cw] = make_float2(mt, st);
            if (named_bar_or(1, NC, !ok)) {
                if (ct == 0) report_timeout(p.status, kSiteStagedFull);
                return false;
            }
            M = -INFINITY;
            Ssum = 0.f;
            for (int w = 0; w < NCW; ++w)
                pair_fold(M, Ssum, red[b * 32 + w].x, red[b * 32 + w].y);
            return true;
        };

        if (D == 0) {
            uint32_t it = 0;
            for (int64_t row = unit; row < p.rows; row += nunits, ++it) {
                float mt = -INFINITY, st = 0.f;
                float2 ms = make_float2(-INFINITY, 0.f);
#pragma unroll 1
                for (int k = 0; k < NCH && acquire(); ++k) {
                    first_read(k, ms);
                    if ((k + 1) % kSumBlockChunks == 0) {
                        pair_fold(mt, st, ms.x, ms.y);
                        ms = make_float2(-INFINITY, 0.f);
                    }
                }
                pair_fold(mt, st, ms.x, ms.y);
                float M, Ssum;
                if (!cta_pair(mt, st, it, M, Ssum)) break;
                if (CL) {
                    // the row's pair from the cluster's CTA pairs (one exchange)
                    float Mr, Sr;
                    const bool cok =
                        cluster_pair_allreduce(ex, M, Ssum, ncta, rank, it, p, &Mr, &Sr, ct);
                    if (named_bar_or(1, NC, !cok)) break;   // uniform: stop, leave cleanly
                    M = Mr;
                    Ssum = Sr;
                }
                pass_b(row, M, Ssum);
            }
        } else {
            // The next row's first D chunks are read while the cluster
            // combines this row's pairs; a row's pass A then starts at D.
            float2 ms = make_float2(-INFINITY, 0.f);
            int n = 0;             // chunks folded into ms / the current block
            float mt = -INFINITY, st = 0.f;
            auto block = [&]() {
                if (++n % kSumBlockChunks == 0) {
                    pair_fold(mt, st, ms.x, ms.y);
                    ms = make_float2(-INFINITY, 0.f);
                }
            };
            if (unit < p.rows)
                for (int k = 0; k < D && acquire(); ++k) {
                    first_read(k, ms);
                    block();
                }
            uint32_t it = 0;
            for (int64_t row = unit; row < p.rows; row += nunits, ++it) {
#pragma unroll 1
                for (int k = D; k < NCH && acquire(); ++k) {
                    first_read(k, ms);
                    block();
                }
                pair_fold(mt, st, ms.x, ms.y);
                float M, Ssum;
                if (!cta_pair(mt, st, it, M, Ssum)) break;
                // the row's pair from the cluster's CTA pairs (one exchange)
                cluster_pair_send(ex, M, Ssum, ncta, rank, it, p, ct);
                mt = -INFINITY;
                st = 0.f;
                ms = make_float2(-INFINITY, 0.f);
                n = 0;
                if (row + nunits < p.rows)
                    for (int k = 0; k < D && acquire(); ++k) {
                        first_read(k, ms);
                        block();
                    }
                float Mr, Sr;
                const bool cok = cluster_pair_wait(ex, ncta, it, p, &Mr, &Sr, ct) && ok;
                if (named_bar_or(1, NC, !cok)) break;   // uniform: stop, leave cleanly
                pass_b(row, Mr, Sr);
            }
        }
    }
    // Keep this CTA's shared memory alive until every peer is done with it.
    if (CL) cluster_sync_all();
}

}  // namespace rmsnorm
