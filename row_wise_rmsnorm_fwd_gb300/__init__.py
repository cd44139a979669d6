"""librmsnorm: fused row-wise RMSNorm forward (and row softmax) for NVIDIA GB300.

``y[r, j] = (x[r, j] * rsqrt(mean_j x[r, j]^2 + eps)) * w[j]`` computed by
hand-written CUDA kernels behind a C ABI (``include/rmsnorm.h``).  This package
holds the CUDA sources (``csrc/``), their in-tree build (``build.py``), the
ctypes binding (``binding.py``) and the seeded workload generators
(``workloads.py``).  The binding is imported lazily so that the generators
can be used without the compiled library.
"""

_BINDING_NAMES = {
    "rmsnorm_fwd_f32", "rmsnorm_fwd_bf16", "rmsnorm_fwd_ex", "rmsnorm_plan",
    "rmsnorm_last_device_status", "rmsnorm_status_string", "rmsnorm_abi_version",
    "rmsnorm_last_cuda_error", "rowsoftmax_fwd_f32", "rowsoftmax_fwd_bf16",
    "rowsoftmax_fwd_ex", "rowsoftmax_plan",
    "make_options", "RmsnormError", "raw", "load",
}


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
