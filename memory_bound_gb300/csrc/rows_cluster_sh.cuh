// rows_cluster_sh.cuh -- the cluster kernel's form for rows off the 16-byte
// grid (rows_cluster_kernel<C, VPT, VEC, STAGED, MAXT, true>), included only
// by the rows_cluster_sh_*.cu units, which instantiate cluster_sh_fn for each
// chain that reads whole rows and takes shifted vectors.
#pragma once

#include "chains.cuh"

namespace mb {

// The 512-thread form for 32 or more values per thread when the CTA fits it,
// else the 1024-thread form (as for aligned rows).
template <class C, int VPT, bool STAGED> const void *cluster_sh_form(int threads) {
    if constexpr (VPT * C::kVec >= 32) {
        if (threads <= kWideThreads)
            return (const void *)rows_cluster_kernel<C, VPT, C::kVec, STAGED, kWideThreads, true>;
    }
    return (const void *)rows_cluster_kernel<C, VPT, C::kVec, STAGED, kCtaMaxThreads, true>;
}

template <class C, bool STAGED> const void *cluster_sh_vpt(int vpt, int threads) {
    switch (vpt) {
        case 1: return cluster_sh_form<C, 1, STAGED>(threads);
        case 2: return cluster_sh_form<C, 2, STAGED>(threads);
        case 4: return cluster_sh_form<C, 4, STAGED>(threads);
        case 8: if constexpr (C::kVec == 4) return cluster_sh_form<C, 8, STAGED>(threads);
                break;
    }
    return nullptr;
}

template <class C> const void *cluster_sh_fn(int vpt, bool staged, int threads) {
    return staged ? cluster_sh_vpt<C, true>(vpt, threads) : cluster_sh_vpt<C, false>(vpt, threads);
}

}  // namespace mb
