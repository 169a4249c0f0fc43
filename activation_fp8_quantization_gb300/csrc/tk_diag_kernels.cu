// The failure path of the bounded waits, exercised on purpose: one thread
// waits on a shared-memory mbarrier that nothing arrives at, gives up after a
// given number of tries exactly as the library's kernels do (mbar_wait_tries,
// the helper behind mbar_wait_bounded), sets bit 0 of the fault word and
// returns. Nothing is in flight when it returns, so the context stays usable.
#include "tk_internal.h"

namespace tk {

namespace {

__global__ void __launch_bounds__(32) unanswered_wait_kernel(unsigned *fault, uint32_t tries)
{
    __shared__ uint64_t bar;
    if (threadIdx.x != 0)
        return;
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait_tries(&bar, 0u, tries))   // phase 0 never completes
        atomicOr(fault, 1u);
}

}  // namespace

cudaError_t launch_unanswered_wait(unsigned *fault, uint32_t tries, cudaStream_t stream)
{
    unanswered_wait_kernel<<<1, 32, 0, stream>>>(fault, tries);
    return cudaGetLastError();
}

}  // namespace tk
