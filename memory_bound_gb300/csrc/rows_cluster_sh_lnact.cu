// rows_cluster_sh_lnact.cu -- rows longer than a CTA and off the 16-byte
// grid: the LayerNorm family without dropout, fp32 and bf16.
#include "rows_cluster_sh.cuh"

namespace mb {

template const void *cluster_sh_fn<LnActChain<float, false, false>>(int, bool, int);
template const void *cluster_sh_fn<LnActChain<float, true, false>>(int, bool, int);
template const void *cluster_sh_fn<LnActChain<uint16_t, false, false>>(int, bool, int);
template const void *cluster_sh_fn<LnActChain<uint16_t, true, false>>(int, bool, int);

}  // namespace mb
