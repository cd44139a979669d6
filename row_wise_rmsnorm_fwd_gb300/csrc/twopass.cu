// twopass.cu -- instances of the generic two-pass kernel (both dtypes).
#include "k_twopass.cuh"
#include "launch.h"

namespace rmsnorm {

template <typename T, int EPI>
static KernelFn twopass_pick(int vb) {
    switch (vb) {
        case 16: return twopass_kernel<T, 16, EPI>;
        case 8: return twopass_kernel<T, 8, EPI>;
        case 4: return twopass_kernel<T, 4, EPI>;
        case 2:
            if constexpr (sizeof(T) == 2) return twopass_kernel<T, 2, EPI>;
            return nullptr;
        default: return nullptr;
    }
}

template <typename T>
static KernelFn twopass_pick_epi(int vb, int epi) {
    switch (epi) {
        case kEpiNone: return twopass_pick<T, kEpiNone>(vb);
        case kEpiScale: return twopass_pick<T, kEpiScale>(vb);
        case kEpiRelu: return twopass_pick<T, kEpiRelu>(vb);
        default: return nullptr;
    }
}

KernelFn twopass_kernel_ptr(int dtype, int vb, int epi) {
    return dtype == 0 ? twopass_pick_epi<float>(vb, epi)
                      : twopass_pick_epi<__nv_bfloat16>(vb, epi);
}

int twopass_block() { return kTwoPassThreads; }

}  // namespace rmsnorm
