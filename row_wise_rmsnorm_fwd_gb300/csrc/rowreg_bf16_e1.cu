// rowreg_bf16_e1.cu -- bf16 instances of the register-resident kernel, epilogue kEpiScale.
#include "rowreg_instances.cuh"

namespace rmsnorm {
KernelFn rowreg_kernel_bf16_e1(int vb, int nv, bool pf) {
    return rowreg_pick<__nv_bfloat16, kEpiScale>(vb, nv, pf);
}
}  // namespace rmsnorm
