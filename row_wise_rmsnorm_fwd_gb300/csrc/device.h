// device.h -- per-device state shared by the C-ABI translation units:
// device attributes, the status word's address, one-time kernel preparation,
// cached occupancy answers and the per-thread record of the last CUDA error.
// Internal to the library.
#pragma once
#include <cuda_runtime.h>
#include "launch.h"

namespace rmsnorm {

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;   // 2 s per bounded wait

struct DeviceInfo;

// Keep `e` as the calling thread's last CUDA error if it is one; returns e.
cudaError_t note(cudaError_t e);
// The calling thread's last CUDA error (cudaSuccess if none); clears it.
cudaError_t take_last_cuda_error();

struct DeviceView {
    int dev;
    int sms;
    int smem_optin;
    unsigned* status;     // device address of this device's status word
};

// Set up the current device once (attributes, status-word address).
cudaError_t current_device(DeviceView* out);
// Allow the kernel its dynamic shared memory and non-portable clusters (once).
cudaError_t ensure_prepared(int dev, KernelFn fn, int smem_optin);
// Resident CTAs per SM (cluster == 1) or resident clusters (cluster > 1);
// 0 when the shape cannot launch.  Cached per device and shape.
cudaError_t cached_occupancy(int dev, int smem_optin, KernelFn fn, int block, int smem,
                             int cluster, int* out);
// Launch a grid-split kernel with a scratch area of `bytes` zeroed bytes in
// p.scratch: taken from the current device's default memory pool in stream
// order on `stream` (cudaMallocAsync), cleared there (cudaMemsetAsync), and
// handed back after the launch (cudaFreeAsync).
cudaError_t launch_with_pool_scratch(KernelFn fn, const LaunchShape& s, cudaStream_t stream,
                                     Params p, size_t bytes);

}  // namespace rmsnorm
