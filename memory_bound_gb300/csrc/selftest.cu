// selftest.cu -- a kernel whose barrier wait is never satisfied, to check on
// a live GPU that the library's bounded waits end and are reported (the
// failure path of the staged row kernels, without a real failure).
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

}  // namespace

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
