// rows_shift_cs.cuh -- the shifted kernel's form with per-column copies
// (rows_shift_kernel<C, VPT, true>), included only by the rows_shift_cs_*.cu
// units, which instantiate shift_cs_fn for each chain with per-column arrays.
#pragma once

#include "chains.cuh"

namespace mb {

template <class C> const void *shift_cs_fn(int vpt) {
    switch (vpt) {
        case 1: return (const void *)rows_shift_kernel<C, 1, true>;
        case 2: return (const void *)rows_shift_kernel<C, 2, true>;
        case 4: return (const void *)rows_shift_kernel<C, 4, true>;
        case 8: if constexpr (C::kVec == 4) return (const void *)rows_shift_kernel<C, 8, true>;
                break;
    }
    return nullptr;
}

}  // namespace mb
