// softmax.cu -- instances of the row-softmax kernels (both dtypes).
#include "k_softmax.cuh"
#include "launch.h"

namespace rmsnorm {

// Rows of up to two vectors per thread prefetch the next row (cheap in
// registers, and narrow rows are where a warp has too few bytes in flight).
template <typename T, int VB>
static KernelFn softmax_pick_nv(int nv) {
    if constexpr (VB < static_cast<int>(sizeof(T))) {
        return nullptr;
    } else {
        switch (nv) {
            case 1: return softmax_rowreg_kernel<T, VB, 1, true>;
            case 2: return softmax_rowreg_kernel<T, VB, 2, true>;
            case 4: return softmax_rowreg_kernel<T, VB, 4, false>;
            case 8: return softmax_rowreg_kernel<T, VB, 8, false>;
            default: return nullptr;
        }
    }
}

template <typename T>
static KernelFn softmax_pick(int vb, int nv) {
    switch (vb) {
        case 16: return softmax_pick_nv<T, 16>(nv);
        case 8: return softmax_pick_nv<T, 8>(nv);
        case 4: return softmax_pick_nv<T, 4>(nv);
        case 2: return softmax_pick_nv<T, 2>(nv);
        default: return nullptr;
    }
}

KernelFn softmax_rowreg_ptr(int dtype, int vb, int nv) {
    return dtype == 0 ? softmax_pick<float>(vb, nv) : softmax_pick<__nv_bfloat16>(vb, nv);
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

}  // namespace rmsnorm
