// selftest.cu -- exercises the kernels' bounded-wait failure path on the
// device without faulting it: one CTA waits, through the same mbar_wait the
// decode kernels use, on an mbarrier that nothing ever arrives at.  The wait
// must give up after its cycle limit (about a second), OR its code into the
// error word and return, leaving the context usable.
#include "internal.h"
#include "ptx.cuh"

namespace gqa {
namespace {

__global__ void wait_timeout_kernel(unsigned *err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_barrier_init();
    }
    __syncthreads();
    // phase 0 of `bar` never completes: nobody arrives
    mbar_wait(smem_u32(&bar), 0, err, kErrSelfTestBit);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(unsigned *err, cudaStream_t stream) {
    wait_timeout_kernel<<<1, 32, 0, stream>>>(err);
    return cudaGetLastError();
}

}  // namespace gqa
