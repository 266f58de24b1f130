// kda_selftest.cu -- exercises the bounded-wait path the kernels rely on: one CTA waits on an mbarrier
// that nothing ever completes, gives up after the limit, reports KDA_DEV_TIMEOUT and returns, leaving the
// context usable.  No counterpart in the pages; it is the library's own failure-detection check.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"
#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {

__global__ void __launch_bounds__(32) kda_selftest_wait_kernel(uint64_t limit_ns, int32_t *status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // one arrival expected; none is ever made
        fence_mbar_init();
    }
    __syncwarp();
    if (!mbar_wait(&bar, 0, limit_ns) && threadIdx.x == 0) set_status(status, KDA_DEV_TIMEOUT);
}

}  // namespace kda

extern "C" KDA_API int kda_selftest_wait_timeout(int64_t limit_ns, int32_t *dev_status, kda_stream_t stream) {
    kda::clear_error();
    if (!dev_status || (reinterpret_cast<uintptr_t>(dev_status) & 3u))
        return kda::fail(KDA_ERR_INVALID_ARG, "selftest: dev_status NULL or misaligned");
    if (limit_ns < 1000000) limit_ns = 1000000;
    if (limit_ns > (int64_t)kda::kWaitLimitNs) limit_ns = (int64_t)kda::kWaitLimitNs;
    kda::kda_selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>((uint64_t)limit_ns,
                                                                                       dev_status);
    return kda::launch_result("kda_selftest_wait_kernel launch");
}
