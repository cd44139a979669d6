// k_exchange.cuh -- the grid-wide exchange through global scratch, and a
// producer helper for chunk streams of any order, for the kernels that split
// every row over the whole grid (k_grid.cuh: few rows, each too wide for any
// one cluster to keep on chip).
//
// The exchange.  The scratch area holds an arrival counter (its own 128-byte
// line) and two sets of G partials (G = CTAs in the grid), used by alternate
// exchanges.  For exchange `it`, CTA g writes its partial into slot g of set
// it & 1 with a relaxed store and then adds 1 to the counter with a release
// reduction (gpu scope), which orders the partial before the arrival.  One
// thread of every CTA then reads the counter with acquire loads until it
// reaches G * (it + 1) (bounded by %globaltimer), fences, and passes a block
// barrier; the CTA's threads read the G partials (relaxed, gpu scope: not
// from L1) and fold them in slot order -- a butterfly in each warp, then the
// warps in order -- so every CTA computes the bitwise same result.  A CTA
// writes exchange it + 2's partial into a set only after the counter showed
// that every CTA arrived at exchange it + 1, which each did only after
// reading all of exchange it's partials: two sets suffice.  The host clears
// the scratch before each launch, and the launch is cooperative, so all G
// CTAs are resident at once and every wait can end.
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
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// The exchange in two halves, so that a CTA can keep streaming while the
// others arrive.  grid_post (one thread): this CTA's partial (a, b) for
// exchange `it`.
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
    st_relaxed_u64(&set[g], (static_cast<unsigned long long>(__float_as_uint(b)) << 32) |
                                __float_as_uint(a));
    red_release_add(counter, 1u);
}

// grid_wait_fold (all NC consumer threads, warps 1.. of the CTA, named
// barrier 1): wait until every CTA posted exchange `it`, then fold the G
// partials.  kPair: (maximum, sum) pairs folded with pair_fold (the
// online-softmax combine); else the sums b are added.  `wpart` is shared
// memory for 2 x 32 warp slots.  Returns false (uniform over the consumers)
// if the wait ran out (the status word then records it).
template <bool kPair>
__device__ __forceinline__ bool grid_wait_fold(void* scratch, int G, uint32_t it, float2* wpart,
                                               int ct, int NC, const Params& p, float& M,
                                               float& S) {
    const unsigned* counter = static_cast<const unsigned*>(scratch);
    const unsigned long long* set = reinterpret_cast<const unsigned long long*>(
                                        static_cast<const char*>(scratch) + kGridCounterBytes) +
                                    (it & 1u) * G;
    bool ok = true;
    if (ct == 0) {
        const unsigned target = static_cast<unsigned>(G) * (it + 1u);
        if (static_cast<int>(ld_acquire_u32(counter) - target) < 0) {
            const uint64_t t0 = global_timer_ns();
            while (static_cast<int>(ld_acquire_u32(counter) - target) < 0) {
                if (global_timer_ns() - t0 > p.timeout_ns) {
                    ok = false;
                    report_timeout(p.status, kSiteClusterExchange);
                    break;
                }
                __nanosleep(64);
            }
        }
        __threadfence();
    }
    if (named_bar_or(1, NC, !ok)) return false;
    float m = -INFINITY, s = 0.f;
    for (int j = ct; j < G; j += NC) {
        const unsigned long long d = ld_relaxed_u64(&set[j]);
        const float ra = __uint_as_float(static_cast<uint32_t>(d));
        const float rb = __uint_as_float(static_cast<uint32_t>(d >> 32));
        if constexpr (kPair) {
            pair_fold(m, s, ra, rb);
        } else {
            s += rb;
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
    const int NCW = NC >> 5;
    float2* slots = wpart + (it & 1u) * 32;
    if ((ct & 31) == 0) slots[ct >> 5] = make_float2(m, s);
    named_bar_sync(1, NC);
    m = -INFINITY;
    s = 0.f;
    for (int w = 0; w < NCW; ++w) {
        if constexpr (kPair) {
            pair_fold(m, s, slots[w].x, slots[w].y);
        } else {
            s += slots[w].y;
        }
    }
    M = m;
    S = s;
    return true;
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
