// zccl_selftest.cu -- a diagnostic for the library's bounded device waits.
//
// The codec kernels wait only on mbarriers that their own TMA bulk copies
// complete.  Each such wait gives up after a time limit and reports
// ZCCL_ERR_TIMEOUT instead of hanging.  This kernel lets a test show that
// path works without faulting anything: one CTA waits, with the very same
// routine, on a barrier phase that nothing ever completes.
#include <cstdint>

#include "zccl_common.cuh"
#include "zccl_internal.h"

namespace zccl {

namespace {

__global__ void wait_check_kernel(uint64_t limit_ns, uint32_t* status)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    // nothing arrives on `bar`: its phase 0 never completes
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0, limit_ns)) report(status, ZCCL_ERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_check(uint64_t limit_ns, uint32_t* status, cudaStream_t stream)
{
    wait_check_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
    return cudaGetLastError();
}

}  // namespace zccl
