// rowreg_f32_e0.cu -- f32 instances of the register-resident kernel, epilogue kEpiNone.
#include "rowreg_instances.cuh"

namespace rmsnorm {
KernelFn rowreg_kernel_f32_e0(int vb, int nv, bool pf) {
    return rowreg_pick<float, kEpiNone>(vb, nv, pf);
}
}  // namespace rmsnorm
