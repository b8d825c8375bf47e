// selftest.cu -- the failure path of the library's bounded waits, exercised without a fault: one
// thread waits on an mbarrier that nothing completes.  The wait gives up after its poll limit
// and the kernel raises the timeout bit in the device error word, as a stalled pipeline inside
// any of the attention kernels would; then it returns, and the context stays usable.
#include "args_common.h"
#include "ptx.cuh"

namespace sinkattn {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(unsigned* err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // one arrival expected, none ever made
        fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0)) atomicOr(err, kErrTimeout);
}

}  // namespace

cudaError_t wait_timeout_selftest_launch(unsigned* err, cudaStream_t stream) {
    wait_timeout_kernel<<<1, 32, 0, stream>>>(err);
    return cudaGetLastError();
}

}  // namespace sinkattn
