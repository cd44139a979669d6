// rowreg_f32.cu -- fp32 instances of the register-resident kernel.
#include "rowreg_instances.cuh"

namespace rmsnorm {
KernelFn rowreg_kernel_f32(int vb, int nv, bool pf) {
    return rowreg_pick<float>(vb, nv, pf);
}
}  // namespace rmsnorm
