// rows_cluster_sh_drop.cu -- rows longer than a CTA and off the 16-byte
// grid: the LayerNorm family with dropout, fp32 and bf16.
#include "rows_cluster_sh.cuh"

namespace mb {

template const void *cluster_sh_fn<LnActChain<float, false, true>>(int, bool, int);
template const void *cluster_sh_fn<LnActChain<float, true, true>>(int, bool, int);
template const void *cluster_sh_fn<LnActChain<uint16_t, false, true>>(int, bool, int);
template const void *cluster_sh_fn<LnActChain<uint16_t, true, true>>(int, bool, int);

}  // namespace mb
