// device.cu -- per-device state of the library (see device.h).
#include "device.h"

#include <map>
#include <mutex>
#include <tuple>

// The device status word: written only by a kernel whose bounded wait
// expired; read and cleared by rmsnorm_last_device_status.  Kernels get its
// address through their parameters.
__device__ unsigned g_rmsnorm_status = 0u;

namespace rmsnorm {
namespace {

constexpr int kMaxDevices = 64;

struct Dev {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    int sms = 0;
    int smem_optin = 0;
    unsigned* status = nullptr;
};
Dev g_dev[kMaxDevices];

// The CUDA runtime is linked statically, so its error state is private to
// this library; the last failing call's error is kept per host thread.
thread_local cudaError_t t_last_cuda_error = cudaSuccess;

std::mutex g_occ_mu;
std::map<std::tuple<int, KernelFn, int, int, int>, int> g_occ;
std::map<std::pair<int, KernelFn>, cudaError_t> g_prepared;

cudaError_t init_device(Dev& d, int dev) {
    cudaError_t e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess)
        e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_rmsnorm_status);
    return e;
}

}  // namespace

cudaError_t note(cudaError_t e) {
    if (e != cudaSuccess) t_last_cuda_error = e;
    return e;
}

cudaError_t take_last_cuda_error() {
    const cudaError_t e = t_last_cuda_error;
    t_last_cuda_error = cudaSuccess;
    return e;
}

cudaError_t current_device(DeviceView* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return note(e);
    if (dev < 0 || dev >= kMaxDevices) return note(cudaErrorInvalidDevice);
    Dev& d = g_dev[dev];
    std::call_once(d.once, [&] { d.err = init_device(d, dev); });
    out->dev = dev;
    out->sms = d.sms;
    out->smem_optin = d.smem_optin;
    out->status = d.status;
    return note(d.err);
}

cudaError_t ensure_prepared(int dev, KernelFn fn, int smem_optin) {
    std::lock_guard<std::mutex> lk(g_occ_mu);
    const auto key = std::make_pair(dev, fn);
    auto it = g_prepared.find(key);
    if (it != g_prepared.end()) return it->second;
    const cudaError_t e = prepare_kernel(fn, smem_optin);
    g_prepared[key] = e;
    return note(e);
}

cudaError_t cached_occupancy(int dev, int smem_optin, KernelFn fn, int block, int smem,
                             int cluster, int* out) {
    const auto key = std::make_tuple(dev, fn, block, smem, cluster);
    {
        std::lock_guard<std::mutex> lk(g_occ_mu);
        auto it = g_occ.find(key);
        if (it != g_occ.end()) { *out = it->second; return cudaSuccess; }
    }
    int v = 0;
    cudaError_t e = ensure_prepared(dev, fn, smem_optin);
    if (e == cudaSuccess) {
        if (cluster > 1) {
            e = max_active_clusters(fn, block, smem, cluster, &v);
        } else {
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &v, reinterpret_cast<const void*>(fn), block, static_cast<size_t>(smem));
        }
    }
    if (e != cudaSuccess) {
        // A cluster shape the device cannot run is "zero clusters", not an error.
        if (cluster > 1) { cudaGetLastError(); v = 0; e = cudaSuccess; }
        else return note(e);
    }
    std::lock_guard<std::mutex> lk(g_occ_mu);
    g_occ[key] = v;
    *out = v;
    return cudaSuccess;
}

cudaError_t launch_with_pool_scratch(KernelFn fn, const LaunchShape& s, cudaStream_t stream,
                                     Params p, size_t bytes) {
    void* scratch = nullptr;
    cudaError_t e = cudaMallocAsync(&scratch, bytes, stream);
    if (e != cudaSuccess) return note(e);
    e = cudaMemsetAsync(scratch, 0, bytes, stream);
    if (e == cudaSuccess) {
        p.scratch = scratch;
        e = launch_ex(fn, s, stream, p);
    }
    const cudaError_t f = cudaFreeAsync(scratch, stream);
    return note(e != cudaSuccess ? e : f);
}

}  // namespace rmsnorm
