// selftest.cu -- exercises the bounded mbarrier wait every pipeline kernel relies on: one
// CTA waits on an mbarrier phase that nothing will complete.  The wait must give up after
// its limit, record PKM_ERR_TIMEOUT in the status word and return, leaving the context
// usable.  Failure detection is tested this way, without any fault, trap or hang.
#include "pkm_device.cuh"
#include "pkm_internal.h"

namespace pkm {
namespace {

__global__ void wait_timeout_kernel(int32_t* status, uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const WaitCtl wc{&abort_flag, status, timeout_ns};
    if (threadIdx.x == 0) {
        // no thread ever arrives on `bar`: phase 0 never completes
        const bool ok = mbar_wait(&bar, 0, wc);
        if (ok) report(status, PKM_ERR_INVALID_ARG);  // would mean the barrier lied
    }
    __syncthreads();
}

}  // namespace

cudaError_t launch_wait_timeout_check(int32_t* status, uint64_t timeout_ns, cudaStream_t stream) {
    wait_timeout_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace pkm
