// k_twopass.cuh -- generic RMSNorm forward for any row width and alignment.
//
// One CTA per row (persistent grid-stride over rows).  Pass 1 streams the
// row and accumulates the fp32 sum of squares; the CTA combines it with a
// warp butterfly plus one shared-memory slot per warp; pass 2 reads the row
// again (usually from L2), scales and stores.  It holds nothing in registers
// across the passes, so it serves widths beyond what the register-resident
// and the shared-memory-staged kernels can hold, at the cost of a second read.
#pragma once
#include "common.cuh"

namespace rmsnorm {

constexpr int kTwoPassThreads = 1024;

template <typename T, int VB, int EPI>
__global__ void __launch_bounds__(kTwoPassThreads) twopass_kernel(const Params p) {
    pdl_trigger();
    pdl_wait();
    constexpr int EPV = VecTraits<T, VB>::kElems;
    __shared__ float red[2][32];
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int nwarps = nthr >> 5;

    const char* xb = static_cast<const char*>(p.x);
    const char* wb = static_cast<const char*>(p.w);
    char* yb = static_cast<char*>(p.y);
    const int64_t row_bytes = static_cast<int64_t>(p.hidden) * sizeof(T);

    uint32_t it = 0;
    for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x, ++it) {
        const char* src = xb + row * row_bytes;
        float s0 = 0.f, s1 = 0.f;
        for (int v = tid; v < p.nvec; v += nthr) {
            const Vec<VB> xv = ld_plain<VB>(src + static_cast<int64_t>(v) * VB);
#pragma unroll
            for (int k = 0; k < EPV; ++k) {
                const float f = get<T, VB>(xv, k);
                if (k & 1) s1 = fmaf(f, f, s1); else s0 = fmaf(f, f, s0);
            }
        }
        float ss = warp_allreduce_sum(s0 + s1);
        const int b = it & 1;
        if (lane == 0) red[b][warp] = ss;
        __syncthreads();
        ss = 0.f;
        for (int k = 0; k < nwarps; ++k) ss += red[b][k];
        const float rstd = rsqrtf(fmaf(ss, p.inv_hidden, p.eps));

        char* dst = yb + row * row_bytes;
        for (int v = tid; v < p.nvec; v += nthr) {
            const int64_t off = static_cast<int64_t>(v) * VB;
            const Vec<VB> xv = ld_stream<VB>(src + off);
            const Vec<VB> wv = ld_ro<VB>(wb + off);
            float o[EPV];
#pragma unroll
            for (int k = 0; k < EPV; ++k)
                o[k] = epilogue<EPI>((get<T, VB>(xv, k) * rstd) * get<T, VB>(wv, k), p.alpha);
            st_stream<VB>(dst + off, pack<T, VB>(o));
        }
    }
}

}  // namespace rmsnorm
