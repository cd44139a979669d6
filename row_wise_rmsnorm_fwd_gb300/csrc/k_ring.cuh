// k_ring.cuh -- a ring of shared-memory chunk slots fed by 1-D bulk copies
// (cp.async.bulk, async proxy) completing on mbarriers, shared by the staged
// RMSNorm kernel and the staged row-softmax kernel.
//
// A CTA streams the rows unit, unit + nunits, ... (or one slice [sbeg,
// sbeg + my_bytes) of each); every row slice is cut into NCH chunks of CB
// bytes (the last one shorter) that flow through S >= NCH slots.  Chunk
// number n of the CTA's stream (row n / NCH, chunk n % NCH) lives in slot
// n % S on that slot's (n / S)-th use.  Each slot has a "full" mbarrier
// (producer arrive + transaction bytes; its phase n / S completes when the
// chunk has landed).  Slots are handed back in one of two ways:
//   - ring_produce: a producer lane waits on each slot's "empty" mbarrier
//     (one arrive per consumer warp once the slot's data is no longer needed)
//     and refills it with the next chunk, running up to S - NCH chunks ahead
//     into the following rows;
//   - ring_issue_next: a kernel whose threads all pass a block barrier after
//     reading a row's slots lets one thread refill them right after that
//     barrier (no empty barriers).
// Either way this is the multi-stage prefetch loop of the CuTe DSL page (a
// prologue fills the stages; the steady state consumes stage i while stage
// i + S is in flight).
//
// Proxy rule (TileLang InjectFenceProxy page): shared memory written by the
// async proxy is read by the generic proxy only after the mbarrier wait, which
// orders it; no thread writes a slot with generic stores, so a refill needs no
// fence.proxy.async (generic reads followed by an async-proxy overwrite are
// ordered through the empty-barrier release and the producer's acquire, or
// through the block barrier).
#pragma once
#include "common.cuh"

namespace rmsnorm {

constexpr int kStagedMaxSlots = 32;
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

__device__ __forceinline__ Vec<16> as_vec(const uint4& q) {
    Vec<16> v;
    v.u[0] = q.x; v.u[1] = q.y; v.u[2] = q.z; v.u[3] = q.w;
    return v;
}

struct SlotRing {
    uint64_t* full;          // [S]
    uint64_t* empty;         // [S]
    unsigned char* slots;    // S * CB bytes
    int S;                   // slots
    int NCH;                 // chunks per row slice
    int CB;                  // bytes per chunk
    int64_t my_bytes;        // bytes of this CTA's slice of a row

    __device__ __forceinline__ int chunk_len(int k) const {
        const int64_t rem = my_bytes - static_cast<int64_t>(k) * CB;
        return rem <= 0 ? 0 : static_cast<int>(rem < CB ? rem : CB);
    }
    __device__ __forceinline__ const uint4* slot_vecs(int slot) const {
        return reinterpret_cast<const uint4*>(slots + static_cast<int64_t>(slot) * CB);
    }
};

// Initialise the ring's barriers (one thread; the caller fences and syncs).
__device__ __forceinline__ void ring_init(const SlotRing& r, int consumer_warps) {
    for (int k = 0; k < r.S; ++k) {
        mbar_init(smem_addr(&r.full[k]), 1);
        mbar_init(smem_addr(&r.empty[k]), consumer_warps);
    }
}

// Wait (bounded) until chunk n of the stream has landed in its slot.
__device__ __forceinline__ bool ring_wait_full(const SlotRing& r, int64_t n, uint64_t timeout_ns) {
    return mbar_wait_bounded<false>(smem_addr(&r.full[n % r.S]),
                                    static_cast<uint32_t>(n / r.S) & 1u, timeout_ns);
}

// Position of the next chunk to issue in a CTA's stream of whole rows: the
// row, the chunk within it and its slot, advanced with 32-bit steps (a 64-bit
// division per chunk costs more than the copy's bookkeeping should).
struct RingCursor {
    int64_t row;
    int k;
    int slot;
};

// Issue the chunk at `c` (byte range [sbeg, sbeg + my_bytes) of row c.row,
// chunk c.k; number `seq` of the CTA's stream) into its slot and advance `c`.
// A chunk past the end of a short slice completes its slot's phase with a
// plain arrive and no copy.  The caller guarantees that the slot's previous
// chunk has been read by every thread.  Returns false, issuing nothing, when
// the stream has no more rows.
__device__ __forceinline__ bool ring_issue_next(const Params& p, const SlotRing& r, RingCursor& c,
                                               int64_t nunits, int64_t row_bytes, int64_t sbeg,
                                               uint64_t policy, int64_t seq) {
    if (c.row >= p.rows) return false;
    const int len = r.chunk_len(c.k);
    const uint32_t fb = smem_addr(&r.full[c.slot]);
#if RMSNORM_FAULT_INJECT
    // Test build: the first copy is withheld, its barrier armed for bytes
    // that never come, so every wait on that phase must run out.
    const bool withhold = p.fault == kFaultStagedWithholdCopy && seq == 0;
#else
    const bool withhold = false;
    (void)seq;
#endif
    if (len > 0) {
        mbar_arrive_expect_tx(fb, static_cast<uint32_t>(len));
        if (!withhold)
            bulk_g2s(smem_addr(r.slots + static_cast<int64_t>(c.slot) * r.CB),
                     static_cast<const char*>(p.x) + c.row * row_bytes + sbeg +
                         static_cast<int64_t>(c.k) * r.CB,
                     static_cast<uint32_t>(len), fb, policy);
    } else {
        mbar_arrive(fb);
    }
    if (++c.k == r.NCH) {
        c.k = 0;
        c.row += nunits;
    }
    if (++c.slot == r.S) c.slot = 0;
    return true;
}

// The producer lane: issue the CTA's chunk stream for rows unit, unit +
// nunits, ... (byte range [sbeg, sbeg + my_bytes) of each row of row_bytes),
// then wait (bounded) until every copy it issued has landed, so that no copy
// is in flight when the CTA leaves.  A refill waits for its slot's release;
// if that wait runs out the status word records `site` and no more copies
// are issued.  `passes` > 1 streams each row that many times in a row (the
// row's chunks again after its last one), the first time with `policy`, the
// later ones with `policy2`.
__device__ __forceinline__ void ring_produce(const Params& p, const SlotRing& r, int64_t unit,
                                             int64_t nunits, int64_t row_bytes, int64_t sbeg,
                                             uint64_t policy, unsigned site, int passes = 1,
                                             uint64_t policy2 = 0) {
    const char* xb = static_cast<const char*>(p.x);
    int64_t seq = 0;       // chunks issued so far
    int slot = 0;          // seq % S
    uint32_t lap = 0;      // (seq / S) & 1
    bool reuse = false;    // seq >= S: the slot held an earlier chunk
    bool abort = false;
    for (int64_t rb = unit; rb < p.rows && !abort; rb += nunits)
    for (int ps = 0; ps < passes && !abort; ++ps) {
        const char* src = xb + rb * row_bytes + sbeg;
        const uint64_t pol = ps == 0 ? policy : policy2;
        for (int k = 0; k < r.NCH; ++k, ++seq) {
            if (reuse && !mbar_wait_bounded<false>(smem_addr(&r.empty[slot]), lap ^ 1u,
                                                   p.timeout_ns)) {
                report_timeout(p.status, site);
                abort = true;
                break;
            }
            const int len = r.chunk_len(k);
            const uint32_t fb = smem_addr(&r.full[slot]);
            bool issue = true;
#if RMSNORM_FAULT_INJECT
            if (p.fault == kFaultStagedWithholdCopy && seq == 0 && len > 0) {
                // Arm the barrier for bytes that never come: every wait on
                // this phase must run out, nothing is in flight.
                mbar_arrive_expect_tx(fb, static_cast<uint32_t>(len));
                issue = false;
            }
#endif
            if (issue) {
                if (len > 0) {
                    mbar_arrive_expect_tx(fb, static_cast<uint32_t>(len));
                    bulk_g2s(smem_addr(r.slots + static_cast<int64_t>(slot) * r.CB),
                             src + static_cast<int64_t>(k) * r.CB, static_cast<uint32_t>(len),
                             fb, pol);
                } else {
                    mbar_arrive(fb);
                }
            }
            if (++slot == r.S) {
                slot = 0;
                lap ^= 1u;
                reuse = true;
            }
        }
    }
    // Every copy issued must have landed before this CTA may leave (normally
    // it has: the consumers waited for all of them).
    const int64_t first = seq > r.S ? seq - r.S : 0;
    for (int64_t n = first; n < seq; ++n) ring_wait_full(r, n, p.timeout_ns);
}

}  // namespace rmsnorm
