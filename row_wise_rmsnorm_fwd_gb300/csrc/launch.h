// launch.h -- host-side interface between the C ABI (api.cu) and the
// translation units that instantiate the kernels.  Internal to the library.
#pragma once
#include <cuda_runtime.h>
#include "common.cuh"

namespace rmsnorm {

using KernelFn = void (*)(Params);

struct LaunchShape {
    int grid;       // CTAs
    int block;      // threads per CTA
    int cluster;    // CTAs per cluster (1 = plain launch)
    int smem;       // dynamic shared memory bytes
    bool cooperative = false;   // all CTAs resident at once (grid-split kernels)
};

// Kernel instances; nullptr when the combination is not compiled.
// dtype: 0 = fp32, 1 = bf16.  vb = bytes per vector, nv = vectors per thread.
// pf = register prefetch of the next row (used by the cluster split-row path);
// epi = fused epilogue (kEpiNone / kEpiScale / kEpiRelu).
KernelFn rowreg_kernel_f32_e0(int vb, int nv, bool pf);
KernelFn rowreg_kernel_f32_e1(int vb, int nv, bool pf);
KernelFn rowreg_kernel_f32_e2(int vb, int nv, bool pf);
KernelFn rowreg_kernel_bf16_e0(int vb, int nv, bool pf);
KernelFn rowreg_kernel_bf16_e1(int vb, int nv, bool pf);
KernelFn rowreg_kernel_bf16_e2(int vb, int nv, bool pf);
KernelFn rowreg_kernel_ptr(int dtype, int vb, int nv, bool pf, int epi);
int rowreg_max_block(int nv);
KernelFn twopass_kernel_ptr(int dtype, int vb, int epi);
int twopass_block();
// Row softmax: register-resident kernel (cluster = rows split over a
// thread-block cluster) and the three-pass wide-row kernel.
KernelFn softmax_rowreg_ptr(int dtype, int vb, int nv, bool cluster);
int softmax_rowreg_max_block(int nv);
KernelFn softmax_threepass_ptr(int dtype, int vb);
int softmax_threepass_block();
// Few rows too wide for every other kernel: the two-pass (RMSNorm) and
// three-pass (softmax) kernels with each row split over a thread-block
// cluster of 2..16 CTAs (slices of Params.slice_vecs vectors, totals combined
// through DSMEM); up to split_block() threads per CTA.
KernelFn twopass_cluster_kernel_ptr(int dtype, int vb, int epi);
KernelFn softmax_threepass_cluster_ptr(int dtype, int vb);
int split_block();
// Row softmax staged in shared memory and held in registers: up to 512
// threads of nv 16-byte vectors each (fp32: 4, 8 or 16; bf16: 2, 4 or 8);
// cluster = rows split over a thread-block cluster; dynamic shared memory =
// kStagedHeaderHost + nslots * chunk bytes.
KernelFn softmax_staged_ptr(int dtype, int nv, bool cluster);
int softmax_staged_max_threads();
// Row softmax streamed twice through the bulk-copy ring (online maximum and
// sum, then the outputs): one producer warp plus consumer threads of v (2 or
// 4) 16-byte vectors per chunk; dynamic shared memory = kStreamHeaderHost +
// nslots * chunk bytes, chunk = 16 * v * consumer threads; cluster = rows
// split over a thread-block cluster (slices of Params.slice_vecs vectors).
constexpr int kStreamHeaderHost = 2048;
KernelFn softmax_stream_ptr(int dtype, int v, bool cluster);
int softmax_stream_max_threads();
// RMSNorm and row softmax with every row over the whole grid (few rows of
// tens of MB): the streamed kernel's launch shape (producer warp + consumers
// of v 16-byte vectors per chunk), cooperative, at most kGridMaxCtasHost
// CTAs; Params.scratch = grid_scratch_bytes(grid) cleared bytes.
KernelFn rmsnorm_grid_kernel_ptr(int dtype, int v, int epi);
KernelFn softmax_grid_ptr(int dtype, int v);
constexpr int kGridMaxCtasHost = 1024;
constexpr int kGridCounterBytesHost = 128;
constexpr int kGridScratchBytesHost = kGridCounterBytesHost + 2 * kGridMaxCtasHost * 8;
constexpr int kGridMaxResidentHost = 16;   // grid kernels: resident chunks per slice, at most
constexpr int kGridMinRingSlots = 4;       // grid kernels: ring slots kept beside resident ones

// Chunks of each slice the whole-grid kernel keeps in shared memory between a
// row's two reads (phased schedule only): what the ring's `slots` can spare
// beyond kGridMinRingSlots, within the slice less its read-ahead.
inline int grid_resident_chunks(int schedule, int slots, int64_t nchunks, int read_ahead,
                                bool stages_forced) {
    if (schedule != 1 || stages_forced) return 0;
    int64_t r = slots - kGridMinRingSlots;
    if (r > nchunks - read_ahead) r = nchunks - read_ahead;
    if (r > kGridMaxResidentHost) r = kGridMaxResidentHost;
    return r > 0 ? static_cast<int>(r) : 0;
}
inline int grid_scratch_bytes(int grid) { return kGridCounterBytesHost + 2 * grid * 8; }

// Comparison kernel with the compiler write-up's schedule (one CTA per row).
KernelFn page_kernel_ptr(int dtype);
int page_block();

// Ring-to-register wide-row kernel: one producer warp plus up to 512 consumer
// threads of nv (8 or 16) vectors each; a chunk is m (2 or 4) vectors per
// consumer thread.  Dynamic shared memory = kStagedHeaderHost + the weight row
// rounded up to 128 bytes + nslots * chunk bytes.
KernelFn ringreg_kernel_ptr(int dtype, int nv, int m, int epi);
int ringreg_max_consumers();

// Staged kernel: one producer warp plus 4 or 8 consumer warps.
KernelFn staged_kernel_ptr(int dtype, int consumer_warps, int epi);
constexpr int kStagedMaxSlotsHost = 32;
constexpr int kStagedHeaderHost = 1024;
// Dynamic shared memory of the staged kernel: header + weight slice (0 if the
// weights come through L1/L2) + nslots chunk slots (-1 if nslots is out of range).
int64_t staged_smem_bytes(int64_t chunk_bytes, int nslots, int64_t w_bytes);

// cudaLaunchKernelEx with an optional cluster shape.
inline cudaError_t launch_ex(KernelFn kernel, const LaunchShape& s, cudaStream_t stream,
                             const Params& p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(s.grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(s.block), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(s.smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[3];
    unsigned n = 0;
    if (s.cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(s.cluster);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (s.cooperative) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    } else {
        // may start before the previous kernel in the stream ends: its CTAs
        // are placed and set up, then wait (pdl_wait) for that kernel's memory
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = n ? attr : nullptr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

// One-time kernel set-up: allow dynamic shared memory up to the per-block
// opt-in limit `smem_optin` minus the kernel's static shared memory, and
// clusters above the portable size of 8.
inline cudaError_t prepare_kernel(KernelFn kernel, int smem_optin) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(kernel));
    const int dyn_limit = smem_optin - static_cast<int>(fa.sharedSizeBytes);
    if (e == cudaSuccess && dyn_limit > 48 * 1024)
        e = cudaFuncSetAttribute(reinterpret_cast<const void*>(kernel),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_limit);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(reinterpret_cast<const void*>(kernel),
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

// How many clusters of `cluster` CTAs can be resident at once (0 = cannot launch).
inline cudaError_t max_active_clusters(KernelFn kernel, int block, int smem, int cluster,
                                       int* clusters) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cluster), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(block), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(clusters, kernel, &cfg);
}

}  // namespace rmsnorm
