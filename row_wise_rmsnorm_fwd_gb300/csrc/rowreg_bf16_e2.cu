// rowreg_bf16_e2.cu -- bf16 instances of the register-resident kernel, epilogue kEpiRelu.
#include "rowreg_instances.cuh"

namespace rmsnorm {
KernelFn rowreg_kernel_bf16_e2(int vb, int nv, bool pf) {
    return rowreg_pick<__nv_bfloat16, kEpiRelu>(vb, nv, pf);
}
}  // namespace rmsnorm
