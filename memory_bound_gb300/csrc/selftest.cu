// selftest.cu -- kernels whose barrier waits are never satisfied, to check on
// a live GPU that the library's bounded waits end and are reported (the
// failure paths of the staged row kernels and of the cluster exchange,
// without a real failure).
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace mb {
namespace {

// One thread initialises an mbarrier that expects one arrival, never arrives,
// and waits on it with the given limit; the wait runs out, the thread records
// kDevErrWaitTimeout and the kernel ends normally.
__global__ void wait_timeout_kernel(unsigned long long limit_ns, unsigned *err) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_addr(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    if (!mbar_wait_bounded(b, 0, limit_ns)) atomicOr(err, kDevErrWaitTimeout);
}

// The cluster exchange's failure path: a cluster of two CTAs in which one
// partial is never pushed.  Each CTA arms its exchange mbarrier for two
// 4-byte pushes (st.async completing on the barrier, as the cluster row
// kernel does); rank 0 pushes to both CTAs, rank 1 only to itself.  Rank 1's
// wait completes; rank 0's runs out, records kDevErrWaitTimeout, and both CTAs
// meet at the closing cluster barrier with no push in flight.
__global__ void __cluster_dims__(2, 1, 1)
exchange_timeout_kernel(unsigned long long limit_ns, unsigned *err) {
    namespace cg = cooperative_groups;
    __shared__ float slot[2];
    __shared__ __align__(8) uint64_t bar;
    cg::cluster_group cl = cg::this_cluster();
    const unsigned rank = cl.block_rank();
    const uint32_t b = smem_addr(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_mbar_init();
    }
    cl.sync();
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx_relaxed(b, 8u);
        const uint32_t mine = smem_addr(&slot[rank]);
        for (unsigned j = 0; j < 2; ++j)
            if (rank == 0 || j == rank) st_async_f32(map_cluster(mine, j), 1.0f, map_cluster(b, j));
    }
    if (!mbar_wait_bounded(b, 0, limit_ns) && threadIdx.x == 0) atomicOr(err, kDevErrWaitTimeout);
    cl.sync();
}

}  // namespace

mb_status selftest_exchange_timeout(const LaunchCtx &ctx, uint32_t limit_us) {
    const unsigned long long ns = (unsigned long long)limit_us * 1000ull;
    unsigned *err = ctx.dev_err;
    void *args[] = {(void *)&ns, &err};
    cudaError_t e = cudaLaunchKernel((const void *)exchange_timeout_kernel, dim3(2), dim3(32), args,
                                     0, ctx.stream);
    if (e != cudaSuccess) return cuda_fail(e);
    return MB_OK;
}

mb_status selftest_wait_timeout(const LaunchCtx &ctx, uint32_t limit_us) {
    const unsigned long long ns = (unsigned long long)limit_us * 1000ull;
    unsigned *err = ctx.dev_err;
    void *args[] = {(void *)&ns, &err};
    cudaError_t e = cudaLaunchKernel((const void *)wait_timeout_kernel, dim3(1), dim3(1), args, 0,
                                     ctx.stream);
    if (e != cudaSuccess) return cuda_fail(e);
    return MB_OK;
}

}  // namespace mb
