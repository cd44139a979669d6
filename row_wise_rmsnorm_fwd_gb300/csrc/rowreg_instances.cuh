// rowreg_instances.cuh -- the compiled (vector bytes x vectors per thread)
// instances of the register-resident kernel for one element type.
#pragma once
#include "k_rowreg.cuh"
#include "launch.h"

// Compile-time policy of the instances (overridable for tuning builds):
// prefetch, weights in registers, x-load and y-store cache policies.
#ifndef RMSNORM_ROWREG_PF
#define RMSNORM_ROWREG_PF 1
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

template <typename T, int VB, int NV, bool PF, int EPI>
KernelFn rowreg_instance() {
    return rowreg_kernel<T, VB, NV, PF, RMSNORM_ROWREG_WREG != 0, RMSNORM_ROWREG_LD,
                         RMSNORM_ROWREG_ST, EPI>;
}

// `pf` asks for the register-prefetch instance (used when a cluster splits
// rows: the next row's loads then overlap the cross-CTA exchange).  Only the
// 16-byte-vector instances have it (split rows are wide, hence aligned in
// practice); eight vectors per thread never prefetch (the register budget
// holds one row).
template <typename T, int VB, int EPI>
KernelFn rowreg_pick_nv(int nv, bool pf) {
    constexpr bool kPF = RMSNORM_ROWREG_PF != 0;
    if constexpr (VB < static_cast<int>(sizeof(T))) {
        return nullptr;
    } else {
        if constexpr (VB == 16) {
            if (pf) {
                switch (nv) {
                    case 1: return rowreg_instance<T, VB, 1, true, EPI>();
                    case 2: return rowreg_instance<T, VB, 2, true, EPI>();
                    case 4: return rowreg_instance<T, VB, 4, true, EPI>();
                    default: break;
                }
            }
        }
        if constexpr (VB == 16) {
            // 3 vectors per thread fit rows of 3 x 32k vectors without the idle
            // lanes 4 would leave (16-byte vectors only)
            if (nv == 3) return rowreg_instance<T, VB, 3, kPF, EPI>();
        }
        switch (nv) {
            case 1: return rowreg_instance<T, VB, 1, kPF, EPI>();
            case 2: return rowreg_instance<T, VB, 2, kPF, EPI>();
            case 4: return rowreg_instance<T, VB, 4, kPF, EPI>();
            case 8: return rowreg_instance<T, VB, 8, false, EPI>();
            default: return nullptr;
        }
    }
}

template <typename T, int EPI>
KernelFn rowreg_pick(int vb, int nv, bool pf) {
    switch (vb) {
        case 16: return rowreg_pick_nv<T, 16, EPI>(nv, pf);
        case 8: return rowreg_pick_nv<T, 8, EPI>(nv, pf);
        case 4: return rowreg_pick_nv<T, 4, EPI>(nv, pf);
        case 2: return rowreg_pick_nv<T, 2, EPI>(nv, pf);
        default: return nullptr;
    }
}

}  // namespace rmsnorm
