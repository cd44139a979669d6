// rowreg_instances.cuh -- the compiled (vector bytes x vectors per thread)
// instances of the register-resident kernel for one element type.
#pragma once
#include "k_rowreg.cuh"
#include "launch.h"

namespace rmsnorm {

template <typename T, int VB>
KernelFn rowreg_pick_nv(int nv) {
    if constexpr (VB < static_cast<int>(sizeof(T))) {
        return nullptr;
    } else {
        switch (nv) {
            case 1: return rowreg_kernel<T, VB, 1, true>;
            case 2: return rowreg_kernel<T, VB, 2, true>;
            case 4: return rowreg_kernel<T, VB, 4, true>;
            case 8: return rowreg_kernel<T, VB, 8, false>;
            default: return nullptr;
        }
    }
}

template <typename T>
KernelFn rowreg_pick(int vb, int nv) {
    switch (vb) {
        case 16: return rowreg_pick_nv<T, 16>(nv);
        case 8: return rowreg_pick_nv<T, 8>(nv);
        case 4: return rowreg_pick_nv<T, 4>(nv);
        case 2: return rowreg_pick_nv<T, 2>(nv);
        default: return nullptr;
    }
}

}  // namespace rmsnorm
