// k_ringreg.cuh -- RMSNorm forward for wide rows (above 32 KB, up to 128
// KB): each row streams through the slot ring of k_ring.cuh in chunks and is
// held in registers; the weight row sits in shared memory for the CTA's
// lifetime.
//
// Warp 0 is the producer (one lane: the weight row once, then ring_produce).
// The other NT = blockDim.x - 32 threads are consumers; thread ct owns the
// NV 16-byte vectors ct, ct + NT, ... of a row.  A chunk is M vectors per
// consumer thread (CB = M * NT * 16 bytes), so vector i of every thread lies
// in chunk i / M and a warp's 32 vectors never straddle two chunks.  Per row:
//   - for each chunk: wait for it, copy this thread's M vectors into
//     registers, add their squares to the fp32 sum, and release the slot
//     (one arrive per warp) -- the producer refills it with later chunks of
//     the stream at once, so the following rows load while this row is
//     reduced and written;
//   - the sum is combined over the consumer warps (one named barrier);
//   - y = (x * rstd) * w from registers and the shared weight row, streaming
//     16-byte stores.
// The row never has to fit the ring (S slots may be fewer than a row's
// chunks): it is a pipe, and the registers hold the row.  Compared with the
// shared-memory staged kernel this frees the ring for the next rows and the
// weight row; compared with the two-pass kernel x is read from DRAM once and
// never again from L2.
//
// Every wait is bounded (wall clock); on expiry the kernel records a status
// code, stops, waits (bounded) for the copies it issued and returns.
#pragma once
#include "k_ring.cuh"

namespace rmsnorm {

constexpr int kRingregMaxConsumers = 512;   // 16 consumer warps + the producer warp

// 17 warps: ptxas caps registers at 96 so that the warps fit the register
// files of the SM sub-partitions; NV = 16 packed vectors take 64 of them.
template <typename T, int NV, int M, int EPI>
__global__ void __launch_bounds__(32 + kRingregMaxConsumers) ringreg_kernel(const Params p) {
    pdl_trigger();
    pdl_wait();
    constexpr int EPV = 16 / static_cast<int>(sizeof(T));
    constexpr int NCHMAX = NV / M;                        // chunks a thread's vectors span
    static_assert(NV % M == 0, "M must divide NV");
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kStagedMaxSlots;
    uint64_t* wbar = empty + kStagedMaxSlots;
    float* red = reinterpret_cast<float*>(smem + 16 * kStagedMaxSlots + 16);   // [2][32]

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int NT = blockDim.x - 32;
    const int NW = NT >> 5;
    const int S = p.nslots;
    const int NCH = p.nchunks;
    const int64_t row_bytes = static_cast<int64_t>(p.hidden) * sizeof(T);
    unsigned char* wsm = smem + kStagedHeader;
    const int64_t wres = (row_bytes + 127) / 128 * 128;
    const SlotRing ring{full, empty, wsm + wres, S, NCH, p.chunk_bytes, row_bytes};

    if (tid == 0) {
        ring_init(ring, NW);
        mbar_init(smem_addr(wbar), 1);
        fence_mbarrier_init_cluster();
    }
    __syncthreads();

    if (warp == 0) {
        if (lane == 0) {
            const uint32_t wb = smem_addr(wbar);
            mbar_arrive_expect_tx(wb, static_cast<uint32_t>(row_bytes));
            bulk_g2s_plain(smem_addr(wsm), p.w, static_cast<uint32_t>(row_bytes), wb);
            ring_produce(p, ring, blockIdx.x, gridDim.x, row_bytes, 0, policy_evict_first(),
                         kSiteStagedEmpty);
            mbar_wait_bounded<false>(wb, 0u, p.timeout_ns);
        }
        __syncwarp();
        return;
    }

    const int ct = tid - 32;
    bool ok = mbar_wait_bounded<false>(smem_addr(wbar), 0u, p.timeout_ns);
    char* yb = static_cast<char*>(p.y);
    uint32_t it = 0;
    int64_t base = 0;              // stream index of this row's chunk 0
    for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x, ++it, base += NCH) {
        Vec<16> xv[NV];
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int k = 0; k < NCHMAX; ++k) {
            if (k < NCH && ok) {
                const int64_t n = base + k;
                const int slot = static_cast<int>(n % S);
                if (!ring_wait_full(ring, n, p.timeout_ns)) {
                    ok = false;
                } else {
                    const unsigned char* c = ring.slots + static_cast<int64_t>(slot) * p.chunk_bytes;
#pragma unroll
                    for (int j = 0; j < M; ++j) {
                        const int i = k * M + j;
                        const int v = i * NT + ct;
                        if (v < p.nvec) {
                            xv[i] = as_vec(*reinterpret_cast<const uint4*>(
                                c + static_cast<int64_t>(j * NT + ct) * 16));
#pragma unroll
                            for (int e = 0; e < EPV; ++e) {
                                const float f = get<T, 16>(xv[i], e);
                                if (e & 1) s1 = fmaf(f, f, s1); else s0 = fmaf(f, f, s0);
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_addr(&empty[slot]));
                }
            }
        }
        float ss = warp_allreduce_sum(s0 + s1);
        const int b = it & 1;
        if (lane == 0) red[b * 32 + (warp - 1)] = ss;
        if (named_bar_or(1, NT, !ok)) {
            if (ct == 0) report_timeout(p.status, kSiteStagedFull);
            break;
        }
        ss = 0.f;
        for (int k = 0; k < NW; ++k) ss += red[b * 32 + k];
        const float rstd = rsqrtf(fmaf(ss, p.inv_hidden, p.eps));
        char* dst = yb + row * row_bytes;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int v = i * NT + ct;
            if (v < p.nvec) {
                const int64_t off = static_cast<int64_t>(v) * 16;
                const Vec<16> wv = as_vec(*reinterpret_cast<const uint4*>(wsm + off));
                float o[EPV];
#pragma unroll
                for (int e = 0; e < EPV; ++e)
                    o[e] = epilogue<EPI>((get<T, 16>(xv[i], e) * rstd) * get<T, 16>(wv, e),
                                         p.alpha);
                st_stream<16>(dst + off, pack<T, 16>(o));
            }
        }
    }
}

}  // namespace rmsnorm
