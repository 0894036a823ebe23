// selftest.cu -- exercises the failure path of the bounded device waits without a fault.
//
// Every wait in the library's kernels (an mbarrier phase for a copy or an MMA) gives up
// after a time limit, sets the timeout bit of the device error word and lets the kernel
// return, so that a lost arrival never hangs the GPU; kda_device_status() then reports
// KDA_ERR_TIMEOUT.  This kernel runs the same wait on an mbarrier that nothing ever arrives
// on, with a caller-chosen limit, so that a test can check the whole chain (bit set, status
// reported once and cleared, context still usable) with no trap, bad address or endless loop.
#include "kda_common.cuh"
#include "kda_internal.h"
#include "tc_util.cuh"

namespace kda {
namespace {

using namespace tc;

__global__ void selftest_wait_kernel(uint64_t limit_ns, unsigned* err) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);  // expects one arrival, which never comes
    fence_mbar_init();
    const uint32_t addr = smem_u32(&bar);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(addr, 0)) {
        if (globaltimer() - t0 > limit_ns) {
            atomicOr(err, kDevErrTimeout);
            return;
        }
    }
}

}  // namespace

cudaError_t launch_selftest_timeout(uint64_t limit_ns, unsigned* err, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(limit_ns, err);
    return cudaGetLastError();
}

}  // namespace kda
