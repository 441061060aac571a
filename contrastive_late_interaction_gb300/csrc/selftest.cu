// cli_selftest_bounded_wait: a check of the library's failure detection that
// faults nothing.
//
// Every wait of the tcgen05 kernels is bounded (cli_device.cuh, mbar_wait):
// a waiter that sees no progress for the limit raises its CTA's abort flag and
// writes CLI_INTERNAL to the device status, the CTA's other waiters see the
// flag and give up, and the kernel returns with the context intact.  In normal
// operation no wait comes near the limit, so that path would otherwise never
// run.  This entry point runs it on purpose: one CTA whose threads all wait on
// an mbarrier that nothing arrives at, with a short limit.  The host then
// reads CLI_INTERNAL from the status word and the number of threads that gave
// up, and the next call on the stream runs normally.

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/cli.h"
#include "cli_device.cuh"
#include "cli_internal.h"

namespace cli {
namespace {

constexpr int kSelftestThreads = 64;

__global__ void __launch_bounds__(kSelftestThreads) bounded_wait_selftest_kernel(int32_t *status, int32_t *gave_up,
                                                                                uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);   // one arrival would complete the phase; none comes
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const bool completed = mbar_wait(&bar, 0, &abort_flag, status, 0, limit_ns);
    if (!completed && gave_up) atomicAdd(gave_up, 1);
}

}  // namespace
}  // namespace cli

extern "C" cli_status_t cli_selftest_bounded_wait(int32_t *device_status, int32_t *gave_up, uint32_t limit_us,
                                                  void *stream) {
    using namespace cli;
    if (!device_status || limit_us == 0 || limit_us > 2000000u) return CLI_INVALID_ARGUMENT;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(device_status, 0, sizeof(int32_t), s) != cudaSuccess) return CLI_DEVICE;
    if (gave_up && cudaMemsetAsync(gave_up, 0, sizeof(int32_t), s) != cudaSuccess) return CLI_DEVICE;
    bounded_wait_selftest_kernel<<<1, kSelftestThreads, 0, s>>>(device_status, gave_up,
                                                                 static_cast<uint64_t>(limit_us) * 1000ull);
    return cudaGetLastError() == cudaSuccess ? CLI_OK : CLI_DEVICE;
}
