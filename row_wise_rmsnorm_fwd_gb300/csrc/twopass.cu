// twopass.cu -- instances of the generic two-pass kernel (both dtypes).
#include "k_twopass.cuh"
#include "launch.h"

namespace rmsnorm {

template <typename T>
static KernelFn twopass_pick(int vb) {
    switch (vb) {
        case 16: return twopass_kernel<T, 16>;
        case 8: return twopass_kernel<T, 8>;
        case 4: return twopass_kernel<T, 4>;
        case 2:
            if constexpr (sizeof(T) == 2) return twopass_kernel<T, 2>;
            return nullptr;
        default: return nullptr;
    }
}

KernelFn twopass_kernel_ptr(int dtype, int vb) {
    return dtype == 0 ? twopass_pick<float>(vb) : twopass_pick<__nv_bfloat16>(vb);
}

int twopass_block() { return kTwoPassThreads; }

}  // namespace rmsnorm
