// softmax.cu -- instances of the row-softmax kernels (both dtypes).
#include "k_softmax.cuh"
#include "launch.h"

namespace rmsnorm {

// Rows of up to four vectors per thread prefetch the next row into a second
// register copy (measured, % of the HBM roofline, bf16 rows of 1024 / 2048 /
// 4096 / 8192 elements: 70 / 56 / 58 / 58 without, 80 / 68 / 74 / 74 with;
// fp32 rows of 8192: 83 without, 89 with).  Eight vectors leave no room.
template <typename T, int VB, bool CL>
static KernelFn softmax_pick_nv(int nv) {
    if constexpr (VB < static_cast<int>(sizeof(T))) {
        return nullptr;
    } else {
        switch (nv) {
            case 1: return softmax_rowreg_kernel<T, VB, 1, true, CL>;
            case 2: return softmax_rowreg_kernel<T, VB, 2, true, CL>;
            case 4: return softmax_rowreg_kernel<T, VB, 4, true, CL>;
            case 8: return softmax_rowreg_kernel<T, VB, 8, false, CL>;
            default: return nullptr;
        }
    }
}

template <typename T, bool CL>
static KernelFn softmax_pick(int vb, int nv) {
    switch (vb) {
        case 16: return softmax_pick_nv<T, 16, CL>(nv);
        case 8: return softmax_pick_nv<T, 8, CL>(nv);
        case 4: return softmax_pick_nv<T, 4, CL>(nv);
        case 2: return softmax_pick_nv<T, 2, CL>(nv);
        default: return nullptr;
    }
}

KernelFn softmax_rowreg_ptr(int dtype, int vb, int nv, bool cluster) {
    if (cluster)
        return dtype == 0 ? softmax_pick<float, true>(vb, nv)
                          : softmax_pick<__nv_bfloat16, true>(vb, nv);
    return dtype == 0 ? softmax_pick<float, false>(vb, nv)
                      : softmax_pick<__nv_bfloat16, false>(vb, nv);
}

int softmax_rowreg_max_block(int nv) { return nv >= 4 ? 512 : 1024; }

template <typename T>
static KernelFn softmax_wide_pick(int vb) {
    switch (vb) {
        case 16: return softmax_threepass_kernel<T, 16>;
        case 8: return softmax_threepass_kernel<T, 8>;
        case 4: return softmax_threepass_kernel<T, 4>;
        case 2:
            if constexpr (sizeof(T) == 2) return softmax_threepass_kernel<T, 2>;
            return nullptr;
        default: return nullptr;
    }
}

KernelFn softmax_threepass_ptr(int dtype, int vb) {
    return dtype == 0 ? softmax_wide_pick<float>(vb) : softmax_wide_pick<__nv_bfloat16>(vb);
}

int softmax_threepass_block() { return kSoftmaxWideThreads; }

static_assert(8 * kStagedMaxSlots + 4 * 16 * sizeof(float) + sizeof(PairExchange) <= kStagedHeader,
              "staged softmax header overflows");

// Vectors per thread: up to 64 fp32 values of a row (or slice) in registers.
template <bool CL>
static KernelFn softmax_staged_pick(int dtype, int nv) {
    if (dtype == 0) {
        switch (nv) {
            case 4: return softmax_staged_kernel<float, 4, CL>;
            case 8: return softmax_staged_kernel<float, 8, CL>;
            case 16: return softmax_staged_kernel<float, 16, CL>;
            default: return nullptr;
        }
    }
    switch (nv) {
        case 2: return softmax_staged_kernel<__nv_bfloat16, 2, CL>;
        case 4: return softmax_staged_kernel<__nv_bfloat16, 4, CL>;
        case 8: return softmax_staged_kernel<__nv_bfloat16, 8, CL>;
        default: return nullptr;
    }
}

KernelFn softmax_staged_ptr(int dtype, int nv, bool cluster) {
    return cluster ? softmax_staged_pick<true>(dtype, nv) : softmax_staged_pick<false>(dtype, nv);
}

int softmax_staged_max_threads() { return kSoftmaxStagedMaxThreads; }

}  // namespace rmsnorm
