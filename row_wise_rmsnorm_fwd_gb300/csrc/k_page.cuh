// k_page.cuh -- the schedule of the generated kernel in the compiler write-up
// ("A hackable Python ML compiler, part 2": the Tile IR after stage_inputs and
// the CUDA kernel it emits for torch.nn.RMSNorm(2048)), rebuilt from its
// description as an in-library comparison point.  It is never chosen
// automatically; it exists to measure what the other kernels' design choices buy.
//
// The schedule, as the page describes it:
//   - one CTA per row, 256 threads (Tile axes a0:256=THREAD, a1:rows=BLOCK);
//   - stage_inputs: the whole row is copied once from global memory into
//     shared memory, element by element (4-byte accesses, stride 256), then a
//     barrier;
//   - each thread sums the squares of its strided elements from shared memory;
//   - a butterfly shuffle reduces each warp; lane 0 of each of the 8 warps
//     writes its sum to shared memory; a tree halves the 8 partials in three
//     levels (4, 2, 1) with a barrier per level; every thread reads slot 0;
//   - rstd = rsqrt(sum * (1/H) + eps);
//   - each thread normalises its strided elements from shared memory, reads
//     the weight from global memory and stores, element by element.
// Generalised only as far as needed to run on any H that fits shared memory
// (the page hard-codes H = 2048 and has no tail) and on bf16 (widened on load).
#pragma once
#include "common.cuh"

namespace rmsnorm {

constexpr int kPageThreads = 256;

template <typename T>
__device__ __forceinline__ float load_elem(const T* p) {
    if constexpr (sizeof(T) == 4) {
        return *reinterpret_cast<const float*>(p);
    } else {
        return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
    }
}

template <typename T>
__device__ __forceinline__ void store_elem(T* p, float v) {
    if constexpr (sizeof(T) == 4) {
        *reinterpret_cast<float*>(p) = v;
    } else {
        *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(v);
    }
}

template <typename T>
__global__ void __launch_bounds__(kPageThreads) page_kernel(const Params p) {
    extern __shared__ float x_smem[];            // the staged row (fp32)
    __shared__ float acc_smem[kPageThreads / 32];
    const int a0 = threadIdx.x;
    const int lane = a0 & 31, warp = a0 >> 5;
    const int H = p.hidden;
    const int64_t row = blockIdx.x;
    const T* x = static_cast<const T*>(p.x) + row * H;
    const T* w = static_cast<const T*>(p.w);
    T* y = static_cast<T*>(p.y) + row * H;

    for (int j = a0; j < H; j += kPageThreads) x_smem[j] = load_elem(x + j);
    __syncthreads();

    float acc = 0.f;
    for (int j = a0; j < H; j += kPageThreads) acc += x_smem[j] * x_smem[j];
    acc = warp_allreduce_sum(acc);
    if (lane == 0) acc_smem[warp] = acc;
    __syncthreads();
    for (int s = kPageThreads / 64; s > 0; s >>= 1) {
        if (warp < s && lane == 0) acc_smem[warp] = acc_smem[warp] + acc_smem[warp + s];
        __syncthreads();
    }
    const float rstd = rsqrtf(acc_smem[0] * p.inv_hidden + p.eps);

    for (int j = a0; j < H; j += kPageThreads)
        store_elem(y + j, (x_smem[j] * rstd) * load_elem(w + j));
}

}  // namespace rmsnorm
