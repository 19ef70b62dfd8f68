// A check of the bounded waits of bulkcopy.cuh, for tests of the failure path:
// one warp waits on an mbarrier whose phase nothing completes, through the same
// wait the bulk-copy kernels use.  The wait gives up after its cycle budget,
// the warp ORs DSV4_DEVERR_TIMEOUT into the error word and returns, and the
// context stays usable.  Nothing faults, traps or waits without a bound.

#include <cuda_runtime.h>
#include <stdint.h>

#include "bulkcopy.cuh"
#include "launch.h"
#include "launch_status.h"
#include "ops.h"

namespace dsv4 {
namespace {

struct WaitCheckParams {
    int32_t *err;
    long long max_cycles;
};

__global__ void __launch_bounds__(32) bounded_wait_check_kernel(const WaitCheckParams p)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // one arrival expected; none comes
        mbar_init_fence();
    }
    __syncwarp();
    // phase 0 of a fresh barrier is the current, incomplete one
    const bool done = mbar_wait(&bar, 0u, p.max_cycles);
    if (threadIdx.x == 0 && !done && p.err != nullptr)
        atomicOr(p.err, DSV4_DEVERR_TIMEOUT);
}

}  // namespace

int launch_wait_check(int64_t max_cycles, int32_t *err, cudaStream_t stream)
{
    WaitCheckParams p;
    p.err = err;
    p.max_cycles = max_cycles > 0 && max_cycles < kWaitCycles ? max_cycles : kWaitCycles;
    return launch_kernel(bounded_wait_check_kernel, dim3(1), dim3(32), 0, stream, p);
}

}  // namespace dsv4
