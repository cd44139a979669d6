// split.cu -- instances of the cluster-split two-pass (RMSNorm) and
// three-pass (softmax) kernels, both dtypes.
#include "k_split.cuh"
#include "launch.h"

namespace rmsnorm {

template <typename T, int EPI>
static KernelFn twopass_cluster_pick(int vb) {
    switch (vb) {
        case 16: return twopass_cluster_kernel<T, 16, EPI>;
        case 8: return twopass_cluster_kernel<T, 8, EPI>;
        case 4: return twopass_cluster_kernel<T, 4, EPI>;
        case 2:
            if constexpr (sizeof(T) == 2) return twopass_cluster_kernel<T, 2, EPI>;
            return nullptr;
        default: return nullptr;
    }
}

template <typename T>
static KernelFn twopass_cluster_pick_epi(int vb, int epi) {
    switch (epi) {
        case kEpiNone: return twopass_cluster_pick<T, kEpiNone>(vb);
        case kEpiScale: return twopass_cluster_pick<T, kEpiScale>(vb);
        case kEpiRelu: return twopass_cluster_pick<T, kEpiRelu>(vb);
        default: return nullptr;
    }
}

KernelFn twopass_cluster_kernel_ptr(int dtype, int vb, int epi) {
    return dtype == 0 ? twopass_cluster_pick_epi<float>(vb, epi)
                      : twopass_cluster_pick_epi<__nv_bfloat16>(vb, epi);
}

template <typename T>
static KernelFn softmax_split_pick(int vb) {
    switch (vb) {
        case 16: return softmax_threepass_cluster_kernel<T, 16>;
        case 8: return softmax_threepass_cluster_kernel<T, 8>;
        case 4: return softmax_threepass_cluster_kernel<T, 4>;
        case 2:
            if constexpr (sizeof(T) == 2) return softmax_threepass_cluster_kernel<T, 2>;
            return nullptr;
        default: return nullptr;
    }
}

KernelFn softmax_threepass_cluster_ptr(int dtype, int vb) {
    return dtype == 0 ? softmax_split_pick<float>(vb) : softmax_split_pick<__nv_bfloat16>(vb);
}

int split_block() { return kSplitThreads; }

}  // namespace rmsnorm
