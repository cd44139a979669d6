// stream.cu -- instances of the two-read streamed row-softmax kernel.
#include "k_stream.cuh"
#include "launch.h"

namespace rmsnorm {

static_assert(16 * kStagedMaxSlots + 2 * 32 * sizeof(float2) + sizeof(PairExchange) <=
                  kStreamHeader,
              "streamed softmax header overflows");
static_assert(kStreamHeader == kStreamHeaderHost, "host and device header sizes differ");

// 2 or 4 vectors per consumer thread and chunk (8 spills; measured on fp32
// prefill logits with 61440-byte chunks and three slots it was slower too:
// 72% of the HBM roofline against 78% with 4).
template <typename T, int SPLIT>
static KernelFn softmax_stream_pick(int v) {
    switch (v) {
        case 2: return softmax_stream_kernel<T, 2, SPLIT>;
        case 4: return softmax_stream_kernel<T, 4, SPLIT>;
        default: return nullptr;
    }
}

KernelFn softmax_stream_ptr(int dtype, int v, bool cluster) {
    if (cluster)
        return dtype == 0 ? softmax_stream_pick<float, kSplitCluster>(v)
                          : softmax_stream_pick<__nv_bfloat16, kSplitCluster>(v);
    return dtype == 0 ? softmax_stream_pick<float, kSplitNone>(v)
                      : softmax_stream_pick<__nv_bfloat16, kSplitNone>(v);
}

int softmax_stream_max_threads() { return kStreamMaxThreads; }

}  // namespace rmsnorm
