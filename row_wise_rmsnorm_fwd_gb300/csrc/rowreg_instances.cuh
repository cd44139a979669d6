// rowreg_instances.cuh -- the compiled (vector bytes x vectors per thread)
// instances of the register-resident kernel for one element type.
#pragma once
#include "k_rowreg.cuh"
#include "launch.h"

// Compile-time policy of the instances (overridable for tuning builds):
// prefetch, weights in registers, x-load and y-store cache policies.
#ifndef RMSNORM_ROWREG_PF
#define RMSNORM_ROWREG_PF 0
#endif
#ifndef RMSNORM_ROWREG_WREG
#define RMSNORM_ROWREG_WREG 1
#endif
#ifndef RMSNORM_ROWREG_LD
#define RMSNORM_ROWREG_LD 0
#endif
#ifndef RMSNORM_ROWREG_ST
#define RMSNORM_ROWREG_ST 0
#endif

namespace rmsnorm {

template <typename T, int VB, int NV, bool PF>
KernelFn rowreg_instance() {
    return rowreg_kernel<T, VB, NV, PF, RMSNORM_ROWREG_WREG != 0, RMSNORM_ROWREG_LD,
                         RMSNORM_ROWREG_ST>;
}

// `pf` asks for the register-prefetch instance (used when a cluster splits
// rows: the next row's loads then overlap the cross-CTA exchange).  Eight
// vectors per thread never prefetch (the register budget holds one row).
template <typename T, int VB>
KernelFn rowreg_pick_nv(int nv, bool pf) {
    constexpr bool kPF = RMSNORM_ROWREG_PF != 0;
    if constexpr (VB < static_cast<int>(sizeof(T))) {
        return nullptr;
    } else if (pf) {
        switch (nv) {
            case 1: return rowreg_instance<T, VB, 1, true>();
            case 2: return rowreg_instance<T, VB, 2, true>();
            case 4: return rowreg_instance<T, VB, 4, true>();
            case 8: return rowreg_instance<T, VB, 8, false>();
            default: return nullptr;
        }
    } else {
        switch (nv) {
            case 1: return rowreg_instance<T, VB, 1, kPF>();
            case 2: return rowreg_instance<T, VB, 2, kPF>();
            case 4: return rowreg_instance<T, VB, 4, kPF>();
            case 8: return rowreg_instance<T, VB, 8, false>();
            default: return nullptr;
        }
    }
}

template <typename T>
KernelFn rowreg_pick(int vb, int nv, bool pf) {
    switch (vb) {
        case 16: return rowreg_pick_nv<T, 16>(nv, pf);
        case 8: return rowreg_pick_nv<T, 8>(nv, pf);
        case 4: return rowreg_pick_nv<T, 4>(nv, pf);
        case 2: return rowreg_pick_nv<T, 2>(nv, pf);
        default: return nullptr;
    }
}

}  // namespace rmsnorm
