// rowreg_bf16.cu -- bf16 instances of the register-resident kernel.
#include "rowreg_instances.cuh"

namespace rmsnorm {
KernelFn rowreg_kernel_bf16(int vb, int nv, bool pf) {
    return rowreg_pick<__nv_bfloat16>(vb, nv, pf);
}
}  // namespace rmsnorm
