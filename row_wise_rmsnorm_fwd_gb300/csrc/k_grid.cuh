// k_grid.cuh -- RMSNorm and row softmax for few rows, each too wide for any
// one cluster to keep on chip (rows of tens of MB): every row is split over
// the whole grid, one CTA per SM, each CTA owning one contiguous slice of
// every row (and of w), and the CTAs' partial results meet in a small global
// scratch area (grid_exchange, k_exchange.cuh).
//
// One row in flight needs less L2 than the several rows a cluster-per-row
// split keeps in flight, so the whole grid reads the row's slices from DRAM
// (first read, L2 evict_last) and the second read finds them in L2 as far as
// L2 keeps them.
// Rows are pipelined: CTA g streams, through its bulk-copy ring, its slice of
// row 0 (first read), then for every row r, chunk by chunk, row r's chunk
// again (second read: the outputs, with row r's result) followed by a chunk
// of row r + 1 (its first read).  DRAM thus sees the writes of one row and
// the reads of the next interleaved (as a streaming kernel's), not a read
// phase, a stall and a write phase; and L2 holds about one row, since row
// r's lines are read for the last time (evict_first) as fast as row r + 1's
// arrive.  The grid fold of row r + 1 runs beside the streaming: the
// consumer warps hand their partials to the CTA's exchange warp (shared
// memory, an mbarrier) and read the first p.read_ahead chunks of row r + 2
// while that warp posts the CTA's partial, waits for the other CTAs and folds
// theirs; the consumers then take the row's result from it (shared memory,
// a second mbarrier), and the second pass of row r + 1 interleaves with row
// r + 2's remaining chunks.
//
// That interleaving puts about two rows of traffic (the next row's reads,
// this row's writes) between a chunk's two reads, more than L2 keeps for the
// widest rows; for those the planner takes a phased schedule (p.schedule):
// row r's whole second read, then row r + 1's first read (after the chunks
// read ahead), with the second read in chunk order or reversed.  Phased, a
// CTA may also keep chunks D .. D + R - 1 of its slice (p.resident, after the
// D chunks read ahead) in shared memory beside the ring from the first read
// to the second, so that L2 holds less of the row; the second read takes
// them first, which frees their slots before the next row's first read
// refills them.
//
//   RMSNorm:  first read: sum of squares; the grid adds the CTA sums;
//             second read: (x * rstd) * w (w's chunk follows x's in the ring,
//             L2 evict_last: every row reads all of w).
//   softmax:  first read: online (maximum, sum) pair per thread; the grid
//             folds the CTA pairs; second read: exp(x - M) / S.
//
// One producer warp (lane 0: ring_push in the order above), 14 consumer
// warps and the exchange warp, whose polls, partial loads and release fence
// (which waits for the SM's output stores in flight) run off the consumers'
// path.  Every wait is bounded (the status word records an expiry and the
// kernel leaves cleanly).
//
// Measured (fp32 softmax, 1 GB in and out): the second read finds the row in
// L2 for rows of 16 MiB (DRAM reads 1.00 x the input), half of it for rows
// of 32 MiB (1.36 x) and a sixth of it for rows of 64 MiB (1.87 x): L2 keeps
// far less than its capacity of a row streamed beside its outputs.
#pragma once
#include "k_stream.cuh"

namespace rmsnorm {

enum : int { kGridOpRmsNorm = 0, kGridOpSoftmax = 1 };
// Row schedules (p.schedule): the second read of row r interleaved chunk by
// chunk with the first read of row r + 1; or phased -- row r's second read,
// then row r + 1's first read -- with the second read in chunk order or
// reversed.
enum : int { kGridInterleaved = 0, kGridPhased = 1, kGridPhasedReversed = 2 };
// Resident slots (phased schedule): at most kGridMaxResident chunks of a
// slice kept in shared memory between a row's two reads; their barriers sit
// in the header from kGridResBarOffset.
constexpr int kGridMaxResident = 16;
constexpr int kGridResBarOffset = 1088;


// Per-thread statistic of a first read: RMSNorm a running sum of squares,
// softmax a running (maximum, sum) pair; both summed in blocks of chunks each
// started from zero (no fp32 chain grows with the row).
template <int OP>
struct GridStat {
    float m = -INFINITY, s = 0.f;                 // running total
    float bm = -INFINITY, b0 = 0.f, b1 = 0.f;     // the current block
    int chunks = 0;
    __device__ __forceinline__ void close_block() {
        if constexpr (OP == kGridOpSoftmax) {
            pair_fold(m, s, bm, b0);
            bm = -INFINITY;
            b0 = 0.f;
        } else {
            s += b0 + b1;
            b0 = b1 = 0.f;
        }
    }
    __device__ __forceinline__ void end_chunk() {
        if (++chunks == kSumBlockChunks) {
            close_block();
            chunks = 0;
        }
    }
};

template <int OP, typename T, int V, int EPI>
__global__ void __launch_bounds__(kStreamMaxThreads, 1) grid_kernel(const Params p) {
    pdl_trigger();
    pdl_wait();
    constexpr int EPV = VecTraits<T, 16>::kElems;
    constexpr bool kSm = OP == kGridOpSoftmax;
    extern __shared__ __align__(128) unsigned char smem[];
    // header: full[32] | empty[32] | red[2][32] pairs | xbar[4] | xres[2] pairs |
    // (at kGridResBarOffset) rfull[16] | rempty[16]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kStagedMaxSlots;
    float2* red = reinterpret_cast<float2*>(smem + 16 * kStagedMaxSlots);
    // xbar[b]: the consumer warps' partials of exchanges b, b + 2, ... are in
    // red[b]; xbar[2 + b]: the exchange's result is in xres[b]
    uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + 16 * kStagedMaxSlots + 512);
    float2* xres = reinterpret_cast<float2*>(smem + 16 * kStagedMaxSlots + 512 + 32);
    // resident slot i holds chunk D + i of the current row from its first
    // read to its second (rfull: landed; rempty: read by every consumer warp)
    uint64_t* rfull = reinterpret_cast<uint64_t*>(smem + kGridResBarOffset);
    uint64_t* rempty = rfull + kGridMaxResident;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int NCW = static_cast<int>(blockDim.x >> 5) - 2;   // consumer warps 1 .. NCW
    const int NC = NCW * 32;
    const int NCH = p.nchunks, S = p.nslots, CB = p.chunk_bytes;
    const int G = gridDim.x, g = blockIdx.x;
    const int64_t row_bytes = static_cast<int64_t>(p.hidden) * sizeof(T);
    const int64_t slice_nom = static_cast<int64_t>(p.slice_vecs) * 16;
    const int64_t sbeg = static_cast<int64_t>(g) * slice_nom;
    const int64_t send = sbeg + slice_nom < row_bytes ? sbeg + slice_nom : row_bytes;
    const int64_t my_bytes = send > sbeg ? send - sbeg : 0;
    const SlotRing ring{full, empty, smem + kStreamHeader, S, NCH, CB, my_bytes};
    unsigned char* const rslots = smem + kStreamHeader + static_cast<int64_t>(S) * CB;
    const int64_t rows = p.rows;

    // first reads of a row before the rest (all of row 0's; the read-ahead of
    // the later rows, p.read_ahead chunks: the planner's choice)
    const int D = NCH < p.read_ahead ? NCH : p.read_ahead;
    const int sched = p.schedule;
    // chunks D .. D + R - 1 of every row stay in shared memory between the
    // two reads (phased schedule only; the planner keeps D + R <= NCH)
    const int R = sched == kGridPhased ? p.resident : 0;
    auto is_res = [&](int k) { return k >= D && k < D + R; };
    // the chunk of second-read step kk: resident chunks first, then the others
    // in order (reversed for kGridPhasedReversed)
    auto b_chunk = [&](int kk) {
        if (sched == kGridPhasedReversed) return NCH - 1 - kk;
        if (kk < R) return D + kk;
        const int j = kk - R;
        return j < D ? j : j + R;
    };

    if (tid == 0) {
        ring_init(ring, NCW);
        mbar_init(smem_addr(&xbar[0]), NCW);
        mbar_init(smem_addr(&xbar[1]), NCW);
        mbar_init(smem_addr(&xbar[2]), 1);
        mbar_init(smem_addr(&xbar[3]), 1);
        for (int i = 0; i < R; ++i) {
            mbar_init(smem_addr(&rfull[i]), 1);
            mbar_init(smem_addr(&rempty[i]), NCW);
        }
        fence_mbarrier_init_cluster();
    }
    __syncthreads();

    if (warp == 0) {
        // ---------------------------------------------------------- producer --
        if (lane == 0) {
            const uint64_t keep = policy_evict_last(), wpol = policy_evict_last();
            const uint64_t done = policy_evict_first();
            const char* xb = static_cast<const char*>(p.x) + sbeg;
            const char* wsrc = static_cast<const char*>(p.w) + sbeg;
            RingCursorSeq c;
            int64_t res_last[kGridMaxResident];   // last row each resident slot was loaded for
            for (int i = 0; i < kGridMaxResident; ++i) res_last[i] = -1;
            auto first = [&](int64_t r, int k) {
                const char* src = xb + r * row_bytes + static_cast<int64_t>(k) * CB;
                const int len = ring.chunk_len(k);
                if (!is_res(k)) {
                    ring_push(p, ring, c, src, len, keep, kSiteStagedEmpty);
                    return;
                }
                // resident slot i takes one chunk per row: row r's phase of
                // rfull[i] has parity r & 1, and it waits for row r - 1's
                // release of the slot
                const int i = k - D;
                if (c.abort) return;
                if (r > 0 && !mbar_wait_bounded<false>(smem_addr(&rempty[i]),
                                                       static_cast<uint32_t>(r - 1) & 1u,
                                                       p.timeout_ns)) {
                    report_timeout(p.status, kSiteStagedEmpty);
                    c.abort = true;
                    return;
                }
                const uint32_t fb = smem_addr(&rfull[i]);
                if (len > 0) {
                    mbar_arrive_expect_tx(fb, static_cast<uint32_t>(len));
                    bulk_g2s(smem_addr(rslots + static_cast<int64_t>(i) * CB), src,
                             static_cast<uint32_t>(len), fb, keep);
                } else {
                    mbar_arrive(fb);
                }
                res_last[i] = r;
            };
            for (int k = 0; k < NCH; ++k) first(0, k);
            if (rows > 1)
                for (int k = 0; k < D; ++k) first(1, k);
            for (int64_t r = 0; r < rows && !c.abort; ++r) {
                for (int kk = 0; kk < NCH; ++kk) {
                    const int k = b_chunk(kk);
                    const int64_t off = static_cast<int64_t>(k) * CB;
                    const int len = ring.chunk_len(k);
                    if (!is_res(k))
                        ring_push(p, ring, c, xb + r * row_bytes + off, len, done,
                                  kSiteStagedEmpty);
                    if (!kSm) ring_push(p, ring, c, wsrc + off, len, wpol, kSiteStagedEmpty);
                    if (sched == kGridInterleaved && r + 1 < rows && kk + D < NCH) first(r + 1, kk + D);
                }
                if (sched != kGridInterleaved && r + 1 < rows)
                    for (int k = D; k < NCH; ++k) first(r + 1, k);
                if (r + 2 < rows)
                    for (int k = 0; k < D; ++k) first(r + 2, k);
            }
            ring_drain(p, ring, c);
            // no resident copy may still be in flight when the CTA leaves
            for (int i = 0; i < R; ++i)
                if (res_last[i] >= 0)
                    mbar_wait_bounded<false>(smem_addr(&rfull[i]),
                                             static_cast<uint32_t>(res_last[i]) & 1u, p.timeout_ns);
        }
        __syncwarp();
        return;
    }

    if (warp == NCW + 1) {
        // ---------------------------------------------------------- exchange --
        for (int64_t r = 0; r < rows; ++r) {
            const uint32_t it = static_cast<uint32_t>(r), b = it & 1u;
            if (!mbar_wait_bounded<false>(smem_addr(&xbar[b]), (it >> 1) & 1u, p.timeout_ns)) {
                if (lane == 0) report_timeout(p.status, kSiteClusterExchange);
                return;
            }
            float m = -INFINITY, s = 0.f;
            for (int w = 0; w < NCW; ++w) {
                if constexpr (kSm) {
                    pair_fold(m, s, red[b * 32 + w].x, red[b * 32 + w].y);
                } else {
                    s += red[b * 32 + w].y;
                }
            }
            float M, Ssum;
            if (!grid_exchange<kSm>(p.scratch, G, g, it, m, s, p, M, Ssum)) return;
            if (lane == 0) {
                xres[b] = make_float2(M, Ssum);
                mbar_arrive(smem_addr(&xbar[2 + b]));
                if (r + 1 < rows) grid_clear_next(p.scratch, G, g, it);
            }
        }
        return;
    }

    // ------------------------------------------------------------ consumers --
    const int ct = tid - 32;
    const int cw = warp - 1;
    int slot = 0;
    uint32_t lap = 0;
    bool ok = true;          // warp-uniform; false once a bounded wait expired
    auto acquire = [&]() {
        ok = __all_sync(0xffffffffu, ok && mbar_wait_bounded<false>(smem_addr(&full[slot]), lap,
                                                                    p.timeout_ns));
        return ok;
    };
    auto release = [&]() {
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[slot]));
        if (++slot == S) {
            slot = 0;
            lap ^= 1u;
        }
    };
    auto slot_base = [&]() {
        return ring.slots + static_cast<int64_t>(slot) * CB + static_cast<int64_t>(ct) * 16;
    };
    auto res_base = [&](int i) {
        return rslots + static_cast<int64_t>(i) * CB + static_cast<int64_t>(ct) * 16;
    };
    const int64_t vstride = static_cast<int64_t>(NC) * 16;

    // Fold this thread's vectors of one chunk into the running statistic.
    auto fold_chunk = [&](const Vec<16> (&raw)[V], int nv, GridStat<OP>& st) {
        if constexpr (kSm) {
            const float2 ms = stream_fold<T, V, false>(raw, ct, NC, nv, make_float2(st.bm, st.b0));
            st.bm = ms.x;
            st.b0 = ms.y;
        } else {
#pragma unroll
            for (int i = 0; i < V; ++i) {
                if (ct + i * NC < nv) {
#pragma unroll
                    for (int e = 0; e < EPV; ++e) {
                        const float f = get<T, 16>(raw[i], e);
                        if (e & 1) st.b1 = fmaf(f, f, st.b1); else st.b0 = fmaf(f, f, st.b0);
                    }
                }
            }
        }
        st.end_chunk();
    };
    // First read of chunk k of row r into the running statistic: a ring
    // chunk (acquired, released), or a resident one (waited for, kept).
    // False (uniform over the warp) once a wait ran out.
    auto first_read = [&](int64_t r, int k, GridStat<OP>& st) {
        const int nv = ring.chunk_len(k) >> 4;
        Vec<16> raw[V];
        if (is_res(k)) {
            ok = __all_sync(0xffffffffu,
                            ok && mbar_wait_bounded<false>(smem_addr(&rfull[k - D]),
                                                           static_cast<uint32_t>(r) & 1u,
                                                           p.timeout_ns));
            if (!ok) return false;
            stream_load<V, false>(raw, res_base(k - D), vstride, ct, NC, nv);
        } else {
            if (!acquire()) return false;
            stream_load<V, false>(raw, slot_base(), vstride, ct, NC, nv);
            release();
        }
        fold_chunk(raw, nv, st);
        return true;
    };
    // Hand this warp's part of exchange `it` to the exchange warp: warp
    // butterfly, one slot per warp, an arrival on xbar[it & 1].
    auto post = [&](GridStat<OP>& st, uint32_t it) {
        st.close_block();
        float m = st.m, s = st.s;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float so = __shfl_xor_sync(0xffffffffu, s, o);
            if constexpr (kSm) {
                const float mo = __shfl_xor_sync(0xffffffffu, m, o);
                pair_fold(m, s, mo, so);
            } else {
                s += so;
            }
        }
        if (lane == 0) {
            red[(it & 1u) * 32 + cw] = make_float2(m, s);
            mbar_arrive(smem_addr(&xbar[it & 1u]));
        }
    };
    // The result of exchange `it` (bounded wait); false once a wait ran out.
    auto result = [&](uint32_t it, float& M, float& Ssum) {
        ok = __all_sync(0xffffffffu,
                        ok && mbar_wait_bounded<false>(smem_addr(&xbar[2 + (it & 1u)]),
                                                       (it >> 1) & 1u, p.timeout_ns));
        if (!ok) {
            if (lane == 0) report_timeout(p.status, kSiteClusterExchange);
            return false;
        }
        const float2 v = xres[it & 1u];
        M = v.x;
        Ssum = v.y;
        return true;
    };

    // row 0's first read and result
    GridStat<OP> st;
#pragma unroll 1
    for (int k = 0; k < NCH && first_read(0, k, st); ++k) {
    }
    if (!ok) return;
    post(st, 0);
    GridStat<OP> nst;
    if (rows > 1)
        for (int k = 0; k < D && first_read(1, k, nst); ++k) {
        }
    float M, Ssum;
    if (!result(0, M, Ssum)) return;

    char* ybase = static_cast<char*>(p.y) + sbeg + static_cast<int64_t>(ct) * 16;
    for (int64_t r = 0; r < rows; ++r) {
        const bool next = r + 1 < rows;
        // the outputs' scale: RMSNorm rstd; softmax 1 / S with the row's
        // offset, fused where row_exp_offset_ok allows, else exact
        const float rstd = kSm ? 0.f : rsqrtf(fmaf(Ssum, p.inv_hidden, p.eps));
        const bool fast = kSm && row_exp_offset_ok(M);
        const float c = row_exp_bias<T>() - M * kLog2e;
        const float Mu = M == -INFINITY ? 0.f : M;
        const float inv = kSm ? (fast ? slice_offset_correction<T>(M, c) : 1.0f) / Ssum : 0.f;
        const float ms = fast ? 0.f : Mu, cs = fast ? c : row_exp_bias<T>();
        char* dst = ybase + r * row_bytes;
#pragma unroll 1
        for (int kk = 0; kk < NCH; ++kk) {
            const int k = b_chunk(kk);
            const int nv = ring.chunk_len(k) >> 4;
            // second read of row r, chunk k: the outputs
            Vec<16> xr[V];
            if (is_res(k)) {
                stream_load<V, false>(xr, res_base(k - D), vstride, ct, NC, nv);
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&rempty[k - D]));
            } else {
                if (!acquire()) break;
                stream_load<V, false>(xr, slot_base(), vstride, ct, NC, nv);
                release();
            }
            Vec<16> wr[V];
            if constexpr (!kSm) {
                if (!acquire()) break;
                stream_load<V, false>(wr, slot_base(), vstride, ct, NC, nv);
                release();
            }
            char* cdst = dst + static_cast<int64_t>(k) * CB;
#pragma unroll
            for (int i = 0; i < V; ++i) {
                if (ct + i * NC < nv) {
                    if constexpr (kSm) {
                        RowVec<T, 16> e;
                        e.widen(xr[i]);
                        st_stream<16>(cdst + i * vstride, e.exp_shift_scaled(ms, cs, inv));
                    } else {
                        float o[EPV];
#pragma unroll
                        for (int j = 0; j < EPV; ++j)
                            o[j] = epilogue<EPI>((get<T, 16>(xr[i], j) * rstd) *
                                                     get<T, 16>(wr[i], j),
                                                 p.alpha);
                        st_stream<16>(cdst + i * vstride, pack<T, 16>(o));
                    }
                }
            }
            // first read of row r + 1, chunk k + D
            if (sched == kGridInterleaved && next && kk + D < NCH && !first_read(r + 1, kk + D, nst))
                break;
        }
        if (!next || !ok) break;
        if (sched != kGridInterleaved)
            for (int k = D; k < NCH && first_read(r + 1, k, nst); ++k) {
            }
        if (!ok) break;
        const uint32_t it = static_cast<uint32_t>(r + 1);
        post(nst, it);
        nst = GridStat<OP>{};
        if (r + 2 < rows)
            for (int k = 0; k < D && first_read(r + 2, k, nst); ++k) {
            }
        if (!result(it, M, Ssum)) break;
    }
}

}  // namespace rmsnorm
