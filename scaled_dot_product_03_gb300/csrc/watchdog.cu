// watchdog.cu -- self-test of the bounded device-side waits.
#include "ptx.cuh"
#include "tc.h"

namespace gbattn {
namespace {

// Waits on a barrier whose single expected arrival never happens; the
// bounded wait gives up after the limit, records the timeout and returns.
__global__ void watchdog_selftest_kernel(unsigned *err, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        ptx::mbar_init(&bar, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    ptx::Watchdog wd{limit_ns, err, &abort_flag};
    if (threadIdx.x == 0) ptx::mbar_wait(&bar, 0, wd, 0x1u);
    __syncthreads();
}

}  // namespace

cudaError_t launch_watchdog_selftest(unsigned *err, uint64_t limit_ns, cudaStream_t st) {
    watchdog_selftest_kernel<<<1, 32, 0, st>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace gbattn
