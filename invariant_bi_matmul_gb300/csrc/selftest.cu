// selftest.cu -- failure-detection self-test: one CTA waits on an mbarrier that nothing
// ever arrives at, bounded by a caller-chosen timeout.  The wait runs out, the kernel
// latches kErrTimeout in the device error word and returns normally, so the context
// stays usable.  This exercises the same bounded-wait routine the production kernels use.
#include "common.cuh"
#include "launch.h"

namespace bi {
namespace {

__global__ void selftest_wait_kernel(unsigned long long timeout_ns, unsigned int* err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // phase 0 never completes: nobody arrives
        if (!mbar_wait(&bar, 0, nullptr, timeout_ns)) latch_error(err, kErrTimeout);
    }
}

}  // namespace

cudaError_t launch_selftest_wait(const DeviceInfo& dev, unsigned long long timeout_ns,
                                 cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(timeout_ns, dev.err_word);
    return cudaGetLastError();
}

}  // namespace bi
