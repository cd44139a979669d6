// grid.cu -- instances of the kernels that split every row over the whole
// grid (RMSNorm with every fused epilogue, row softmax; both dtypes).
#include "k_grid.cuh"
#include "launch.h"

namespace rmsnorm {

static_assert(16 * kStagedMaxSlots + 2 * 32 * sizeof(float2) + 4 * 8 + 2 * sizeof(float2) <=
                      kGridResBarOffset &&
                  kGridResBarOffset + 2 * 8 * kGridMaxResident <= kStreamHeader,
              "grid kernel header overflows");
static_assert(kGridMaxResident == kGridMaxResidentHost, "host and device resident limits differ");
static_assert(kGridMaxCtas == kGridMaxCtasHost && kGridScratchBytes == kGridScratchBytesHost &&
                  kGridCounterBytes == kGridCounterBytesHost,
              "host and device grid scratch sizes differ");

template <int OP, typename T, int EPI>
static KernelFn grid_pick(int v) {
    switch (v) {
        case 2: return grid_kernel<OP, T, 2, EPI>;
        case 4: return grid_kernel<OP, T, 4, EPI>;
        default: return nullptr;
    }
}

template <typename T>
static KernelFn rmsnorm_grid_pick_epi(int v, int epi) {
    switch (epi) {
        case kEpiNone: return grid_pick<kGridOpRmsNorm, T, kEpiNone>(v);
        case kEpiScale: return grid_pick<kGridOpRmsNorm, T, kEpiScale>(v);
        case kEpiRelu: return grid_pick<kGridOpRmsNorm, T, kEpiRelu>(v);
        default: return nullptr;
    }
}

KernelFn rmsnorm_grid_kernel_ptr(int dtype, int v, int epi) {
    return dtype == 0 ? rmsnorm_grid_pick_epi<float>(v, epi)
                      : rmsnorm_grid_pick_epi<__nv_bfloat16>(v, epi);
}

KernelFn softmax_grid_ptr(int dtype, int v) {
    return dtype == 0 ? grid_pick<kGridOpSoftmax, float, kEpiNone>(v)
                      : grid_pick<kGridOpSoftmax, __nv_bfloat16, kEpiNone>(v);
}

}  // namespace rmsnorm
