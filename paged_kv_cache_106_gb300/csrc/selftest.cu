// Diagnostic for the bounded waits every kernel of this library uses: one
// thread waits, through the same bounded-wait helper, for an mbarrier phase
// that nothing completes (no thread ever arrives).  The wait gives up after
// its limit and the thread reports PA_ERR_TIMEOUT, as a kernel whose
// producer never arrives would; nothing faults and the context stays usable.
#include <cuda_runtime.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pagedkv {

namespace {

__global__ void bounded_wait_kernel(int32_t *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(smem_addr(&bar), 1);
    fence_barrier_init();
    // phase 0 needs one arrival, and none comes
    if (!mbar_wait_bounded(smem_addr(&bar), 0, status, false)) report(status, PA_ERR_TIMEOUT);
}

}  // namespace

int launch_selftest_bounded_wait(int32_t *status, void *stream) {
    if (!status) return fail(PA_ERR_INVALID_ARG, "pa_selftest_bounded_wait: status is NULL");
    bounded_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "pa_selftest_bounded_wait: launch: %s", cudaGetErrorString(e));
    return PA_OK;
}

}  // namespace pagedkv
