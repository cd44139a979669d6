// staged.cu -- instances of the bulk-copy staged kernel (both dtypes).
#include "k_staged.cuh"
#include "launch.h"

namespace rmsnorm {

static_assert(kStagedBlock == kStagedThreads, "staged block size mismatch");
static_assert(kStagedConsumers == kStagedConsumerWarps, "staged warp count mismatch");
static_assert(16 * kStagedMaxChunks + 256 + sizeof(ClusterExchange) <= kStagedHeader,
              "staged header overflows");

KernelFn staged_kernel_ptr(int dtype) {
    return dtype == 0 ? staged_kernel<float> : staged_kernel<__nv_bfloat16>;
}

int staged_smem_bytes(int chunk_bytes, int nchunks) {
    if (nchunks < 1 || nchunks > kStagedMaxChunks) return -1;
    return kStagedHeader + chunk_bytes * nchunks;
}

}  // namespace rmsnorm
