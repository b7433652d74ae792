// zccl_selftest.cu -- diagnostics for the library's bounded device waits.
//
// The codec kernels wait on two kinds of things: mbarriers that their own
// TMA bulk copies complete, and -- inside the cooperative compress and
// decompress launches and the escape scan -- counters and flag words that
// other CTAs of the same launch write (the call's done counter, the run
// totals, the per-chunk entry words and the per-range look-back words).  Every such wait gives up after a time limit and
// reports ZCCL_ERR_TIMEOUT instead of hanging.  These kernels let a test
// show that each path works without faulting anything: one thread waits,
// with the very same routine, on something that never completes.
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

// kind 1: the done-counter wait (wait_count) for *word to reach 1;
// kind 2: the flag-word poll (poll_u64) for the valid bit of *word.
// The caller keeps *word at zero, so neither ever completes.
__global__ void poll_check_kernel(int kind, uint64_t limit_ns, const void* word, uint32_t* status)
{
    if (threadIdx.x != 0) return;
    bool ok = true;
    if (kind == 1) {
        ok = wait_count(reinterpret_cast<const uint32_t*>(word), 1u, limit_ns);
    } else {
        poll_u64(reinterpret_cast<const uint64_t*>(word), [](uint64_t v) { return (v & kValid) != 0; }, &ok,
                 limit_ns);
    }
    if (!ok) report(status, ZCCL_ERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_check(uint64_t limit_ns, uint32_t* status, cudaStream_t stream)
{
    wait_check_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
    return cudaGetLastError();
}

cudaError_t launch_poll_check(int kind, uint64_t limit_ns, const void* word, uint32_t* status, cudaStream_t stream)
{
    poll_check_kernel<<<1, 32, 0, stream>>>(kind, limit_ns, word, status);
    return cudaGetLastError();
}

}  // namespace zccl
