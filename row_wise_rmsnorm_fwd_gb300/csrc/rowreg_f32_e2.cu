// rowreg_f32_e2.cu -- f32 instances of the register-resident kernel, epilogue kEpiRelu.
#include "rowreg_instances.cuh"

namespace rmsnorm {
KernelFn rowreg_kernel_f32_e2(int vb, int nv, bool pf) {
    return rowreg_pick<float, kEpiRelu>(vb, nv, pf);
}
}  // namespace rmsnorm
