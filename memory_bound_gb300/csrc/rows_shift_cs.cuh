// rows_shift_cs.cuh -- the shifted kernel's forms with per-column copies and
// the staged ring (rows_shift_kernel<C, VPT, true, STG>), included only by
// the rows_shift_cs_*.cu units, which instantiate shift_cs_fn for each chain
// with per-column arrays or a staged form.
#pragma once

#include "chains.cuh"

namespace mb {

template <class C, bool STG> const void *shift_cs_form(int vpt) {
    switch (vpt) {
        case 1: return (const void *)rows_shift_kernel<C, 1, true, STG>;
        case 2: return (const void *)rows_shift_kernel<C, 2, true, STG>;
        case 4: return (const void *)rows_shift_kernel<C, 4, true, STG>;
        case 8: if constexpr (C::kVec == 4) return (const void *)rows_shift_kernel<C, 8, true, STG>;
                break;
    }
    return nullptr;
}

template <class C> const void *shift_cs_fn(int vpt, bool stg) {
    if constexpr (C::kShiftStaged) {
        if (stg) return shift_cs_form<C, true>(vpt);
    }
    if constexpr (C::kColArrays > 0) return shift_cs_form<C, false>(vpt);
    return nullptr;
}

}  // namespace mb
