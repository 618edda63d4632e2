// kda_selftest.cu -- a self-test of the bounded device waits every kernel here uses (no
// counterpart in the pages).  One thread waits on a shared-memory mbarrier that nothing arrives
// on; the bounded wait gives up after its limit (about a second), raises the device error word
// and returns, so the kernel ends normally and the host reads the failure through
// kda_device_status.  Nothing faults and nothing hangs.
#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {

__global__ void kda_wait_selftest_kernel(int* err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);       // one arrival expected, none ever made
        fence_mbar_init();
        mbar_wait_bounded(&bar, 0, err);
    }
}

cudaError_t launch_wait_selftest(int* err, cudaStream_t s) {
    kda_wait_selftest_kernel<<<1, 32, 0, s>>>(err);
    return cudaGetLastError();
}

}  // namespace kda
