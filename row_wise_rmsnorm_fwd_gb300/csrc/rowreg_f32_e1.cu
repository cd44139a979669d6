// rowreg_f32_e1.cu -- f32 instances of the register-resident kernel, epilogue kEpiScale.
#include "rowreg_instances.cuh"

namespace rmsnorm {
KernelFn rowreg_kernel_f32_e1(int vb, int nv, bool pf) {
    return rowreg_pick<float, kEpiScale>(vb, nv, pf);
}
}  // namespace rmsnorm
