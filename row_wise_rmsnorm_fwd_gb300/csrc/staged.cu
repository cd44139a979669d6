// staged.cu -- instances of the bulk-copy staged kernel (both dtypes).
#include "k_staged.cuh"
#include "launch.h"

namespace rmsnorm {

static_assert(16 * kStagedMaxSlots + 16 + 256 + sizeof(ClusterExchange) <= kStagedHeader,
              "staged header overflows");
static_assert(kStagedMaxSlots == kStagedMaxSlotsHost, "staged slot limit mismatch");
static_assert(kStagedHeader == kStagedHeaderHost, "staged header size mismatch");

template <int EPI>
static KernelFn staged_pick(int dtype, int consumer_warps) {
    if (consumer_warps == 4)
        return dtype == 0 ? staged_kernel<float, 4, EPI> : staged_kernel<__nv_bfloat16, 4, EPI>;
    if (consumer_warps == 8)
        return dtype == 0 ? staged_kernel<float, 8, EPI> : staged_kernel<__nv_bfloat16, 8, EPI>;
    return nullptr;
}

KernelFn staged_kernel_ptr(int dtype, int consumer_warps, int epi) {
    switch (epi) {
        case kEpiNone: return staged_pick<kEpiNone>(dtype, consumer_warps);
        case kEpiScale: return staged_pick<kEpiScale>(dtype, consumer_warps);
        case kEpiRelu: return staged_pick<kEpiRelu>(dtype, consumer_warps);
        default: return nullptr;
    }
}

int64_t staged_smem_bytes(int64_t chunk_bytes, int nslots, int64_t w_bytes) {
    if (nslots < 1 || nslots > kStagedMaxSlots) return -1;
    return kStagedHeader + w_bytes + chunk_bytes * nslots;
}

}  // namespace rmsnorm
