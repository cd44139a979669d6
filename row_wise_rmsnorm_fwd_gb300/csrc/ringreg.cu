// ringreg.cu -- instances of the ring-to-register wide-row kernel (both dtypes).
#include "k_ringreg.cuh"
#include "launch.h"

namespace rmsnorm {

static_assert(16 * kStagedMaxSlots + 16 + 256 <= kStagedHeader, "ringreg header overflows");

template <typename T, int EPI>
static KernelFn ringreg_pick(int nv, int m) {
    if (nv == 8 && m == 2) return ringreg_kernel<T, 8, 2, EPI>;
    if (nv == 8 && m == 4) return ringreg_kernel<T, 8, 4, EPI>;
    if (nv == 16 && m == 2) return ringreg_kernel<T, 16, 2, EPI>;
    if (nv == 16 && m == 4) return ringreg_kernel<T, 16, 4, EPI>;
    return nullptr;
}

template <int EPI>
static KernelFn ringreg_pick_dtype(int dtype, int nv, int m) {
    return dtype == 0 ? ringreg_pick<float, EPI>(nv, m) : ringreg_pick<__nv_bfloat16, EPI>(nv, m);
}

KernelFn ringreg_kernel_ptr(int dtype, int nv, int m, int epi) {
    switch (epi) {
        case kEpiNone: return ringreg_pick_dtype<kEpiNone>(dtype, nv, m);
        case kEpiScale: return ringreg_pick_dtype<kEpiScale>(dtype, nv, m);
        case kEpiRelu: return ringreg_pick_dtype<kEpiRelu>(dtype, nv, m);
        default: return nullptr;
    }
}

int ringreg_max_consumers() { return kRingregMaxConsumers; }

}  // namespace rmsnorm
