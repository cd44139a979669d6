// k_exchange.cuh -- the grid-wide exchange through global scratch, and a
// producer helper for chunk streams of any order, for the kernels that split
// every row over the whole grid (k_grid.cuh: few rows, each too wide for any
// one cluster to keep on chip).
//
// The exchange.  The scratch area holds an arrival counter (its own 128-byte
// line) and two sets of G partials (G = CTAs in the grid), used by alternate
// exchanges.  For exchange `it`, CTA g's exchange warp adds the CTA's partial
// into slot g of set it & 1 (which reads zero) and 1 to the counter, both
// relaxed reductions (gpu scope): a release, or a plain store, would wait
// behind every output store the SM still has in flight, microseconds on the
// critical path.  It then reads the
// counter with acquire loads until it reaches G * (it + 1) (bounded by
// %globaltimer), and its 32 lanes read the G partials (relaxed, gpu scope:
// not from L1), each slot again until it is non-zero -- a partial's bits
// never are, and the arrival may be seen first -- and fold them in a fixed
// order, so every CTA computes the bitwise same result.  A slot must read
// zero, or the new partial, until it is rewritten: the host clears the
// scratch before each launch, and after exchange it (which showed that every
// CTA has read exchange it - 1's partials) each CTA clears its slot of the
// set exchange it + 1 reuses, then issues a release fence; its next arrival
// comes after that fence, so a CTA that sees it also sees the slot cleared.
// The launch is cooperative, so all G CTAs are resident at once and every
// wait can end.
#pragma once
#include "k_softmax.cuh"

namespace rmsnorm {

constexpr int kGridMaxCtas = 1024;
constexpr int kGridCounterBytes = 128;
constexpr int kGridScratchBytes = kGridCounterBytes + 2 * kGridMaxCtas * 8;
// Chunks a thread sums into fresh accumulators before folding them into its
// running total: no fp32 chain grows with the row (slices of millions of
// elements in the grid kernels).
constexpr int kSumBlockChunks = 32;

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_relaxed_add_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void red_relaxed_add(unsigned* p, unsigned v) {
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_acq_rel_gpu() {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// grid_post (one thread): this CTA's partial (a, b) for exchange `it`.
__device__ __forceinline__ void grid_post(void* scratch, int G, int g, uint32_t it, float a,
                                          float b, const Params& p) {
    unsigned* counter = static_cast<unsigned*>(scratch);
    unsigned long long* set = reinterpret_cast<unsigned long long*>(
                                  static_cast<char*>(scratch) + kGridCounterBytes) +
                              (it & 1u) * G;
#if RMSNORM_FAULT_INJECT
    // Test build: CTA 0 withholds its first partial; every wait must run out.
    if (p.fault == kFaultClusterWithholdPartial && g == 0 && it == 0) return;
#else
    (void)p;
#endif
    // the slot reads zero here: adding the partial writes it, by a reduction
    // rather than a store, which would queue behind the SM's output stores
    red_relaxed_add_u64(&set[g], (static_cast<unsigned long long>(__float_as_uint(b)) << 32) |
                                     __float_as_uint(a));
    red_relaxed_add(counter, 1u);
}

// After exchange `it` (one thread of the exchange warp): clear this CTA's
// slot in the set that exchange it + 1 reuses (it holds exchange it - 1's
// partial, which every CTA has read: all of them posted exchange it), then a
// release fence, so that a CTA that sees exchange it + 1's arrivals also sees
// the slot cleared or rewritten, never the old partial.
__device__ __forceinline__ void grid_clear_next(void* scratch, int G, int g, uint32_t it) {
    unsigned long long* set = reinterpret_cast<unsigned long long*>(
                                  static_cast<char*>(scratch) + kGridCounterBytes) +
                              ((it + 1u) & 1u) * G;
    if (it > 0) st_relaxed_u64(&set[g], 0ull);
    fence_acq_rel_gpu();
}

// grid_exchange (the CTA's exchange warp, all 32 lanes; it issues no global
// stores but these, so the release in grid_post waits for nothing else):
// post this CTA's partial (a, b) for exchange `it`, wait until every CTA has
// posted, then fold the G partials -- each lane the slots j = lane (mod 32)
// in order, then a butterfly, lane 0's result taken -- so every CTA computes
// the bitwise same (M, S).  kPair: (maximum, sum) pairs folded with pair_fold
// (the online-softmax combine); else the sums b are added.  Returns false
// (uniform over the warp) if the wait ran out (the status word records it).
template <bool kPair>
__device__ __forceinline__ bool grid_exchange(void* scratch, int G, int g, uint32_t it, float a,
                                              float b, const Params& p, float& M, float& S) {
    const int lane = threadIdx.x & 31;
    const unsigned* counter = static_cast<const unsigned*>(scratch);
    const unsigned long long* set = reinterpret_cast<const unsigned long long*>(
                                        static_cast<const char*>(scratch) + kGridCounterBytes) +
                                    (it & 1u) * G;
    int ok = 1;
    if (lane == 0) {
        grid_post(scratch, G, g, it, a, b, p);
        const unsigned target = static_cast<unsigned>(G) * (it + 1u);
        if (static_cast<int>(ld_acquire_u32(counter) - target) < 0) {
            const uint64_t t0 = global_timer_ns();
            while (static_cast<int>(ld_acquire_u32(counter) - target) < 0) {
                if (global_timer_ns() - t0 > p.timeout_ns) {
                    ok = 0;
                    report_timeout(p.status, kSiteClusterExchange);
                    break;
                }
            }
        }
    }
    // lane 0's acquire, then the warp barrier, orders every lane's reads of
    // the partials after the other CTAs' posts
    __syncwarp();
    if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
    float m = -INFINITY, s = 0.f;
    // the lane's slots j = lane (mod 32), eight loads in flight at a time,
    // folded in slot order
    constexpr int kBatch = 8;
    for (int j0 = lane; j0 < G && ok; j0 += 32 * kBatch) {
        unsigned long long d[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int j = j0 + 32 * u;
            d[u] = j < G ? ld_relaxed_u64(&set[j]) : 0ull;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int j = j0 + 32 * u;
            if (j >= G || !ok) continue;
            // the arrival can be seen before the partial: wait (bounded) for
            // the slot to be written (a partial is never all-zero bits)
            if (d[u] == 0ull) {
                const uint64_t t0 = global_timer_ns();
                while ((d[u] = ld_relaxed_u64(&set[j])) == 0ull) {
                    if (global_timer_ns() - t0 > p.timeout_ns) {
                        ok = 0;
                        report_timeout(p.status, kSiteClusterExchange);
                        break;
                    }
                }
            }
            const float ra = __uint_as_float(static_cast<uint32_t>(d[u]));
            const float rb = __uint_as_float(static_cast<uint32_t>(d[u] >> 32));
            if constexpr (kPair) {
                pair_fold(m, s, ra, rb);
            } else {
                s += rb;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float so = __shfl_xor_sync(0xffffffffu, s, o);
        if constexpr (kPair) {
            const float mo = __shfl_xor_sync(0xffffffffu, m, o);
            pair_fold(m, s, mo, so);
        } else {
            s += so;
        }
    }
    M = __shfl_sync(0xffffffffu, m, 0);
    S = __shfl_sync(0xffffffffu, s, 0);
    return __all_sync(0xffffffffu, ok);
}

// A producer lane's position in its CTA's chunk stream.
struct RingCursorSeq {
    int64_t seq = 0;       // chunks issued so far
    int slot = 0;          // seq % S
    uint32_t lap = 0;      // (seq / S) & 1
    bool reuse = false;    // seq >= S: the slot held an earlier chunk
    bool abort = false;    // a release wait ran out: issue nothing more
};

// Issue one chunk of `len` bytes (a multiple of 16; 0 = an empty chunk, which
// completes its slot's phase with a plain arrive) from `src` into the next
// slot, after (bounded) waiting for the slot's release when it is reused.
// Returns false, issuing nothing, once a wait has run out.
__device__ __forceinline__ bool ring_push(const Params& p, const SlotRing& r, RingCursorSeq& c,
                                          const char* src, int len, uint64_t policy,
                                          unsigned site) {
    if (c.abort) return false;
    if (c.reuse &&
        !mbar_wait_bounded<false>(smem_addr(&r.empty[c.slot]), c.lap ^ 1u, p.timeout_ns)) {
        report_timeout(p.status, site);
        c.abort = true;
        return false;
    }
    const uint32_t fb = smem_addr(&r.full[c.slot]);
    bool issue = true;
#if RMSNORM_FAULT_INJECT
    if (p.fault == kFaultStagedWithholdCopy && c.seq == 0 && len > 0) {
        mbar_arrive_expect_tx(fb, static_cast<uint32_t>(len));   // bytes that never come
        issue = false;
    }
#endif
    if (issue) {
        if (len > 0) {
            mbar_arrive_expect_tx(fb, static_cast<uint32_t>(len));
            bulk_g2s(smem_addr(r.slots + static_cast<int64_t>(c.slot) * r.CB), src,
                     static_cast<uint32_t>(len), fb, policy);
        } else {
            mbar_arrive(fb);
        }
    }
    ++c.seq;
    if (++c.slot == r.S) {
        c.slot = 0;
        c.lap ^= 1u;
        c.reuse = true;
    }
    return true;
}

// Wait (bounded) until the last S chunks issued have landed, so that no copy
// is in flight when the CTA leaves.
__device__ __forceinline__ void ring_drain(const Params& p, const SlotRing& r,
                                           const RingCursorSeq& c) {
    const int64_t first = c.seq > r.S ? c.seq - r.S : 0;
    for (int64_t n = first; n < c.seq; ++n) ring_wait_full(r, n, p.timeout_ns);
}

}  // namespace rmsnorm
