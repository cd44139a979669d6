// rowreg_bf16_e0.cu -- bf16 instances of the register-resident kernel, epilogue kEpiNone.
#include "rowreg_instances.cuh"

namespace rmsnorm {
KernelFn rowreg_kernel_bf16_e0(int vb, int nv, bool pf) {
    return rowreg_pick<__nv_bfloat16, kEpiNone>(vb, nv, pf);
}
}  // namespace rmsnorm
