// mbarriers and bulk copies (cp.async.bulk) from global to shared memory, for
// the kernel that stages rows through shared memory (kv_rows.cu) and the check
// of its bounded wait (wait_check.cu).
//
// Every wait is bounded: it polls the barrier with try_wait (which blocks
// for a short, system-defined time per try) and gives up after kWaitCycles SM
// clock cycles (about one second at 2 GHz), returning false so that the
// caller can flag the error, let its copies in flight land and leave.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dsv4 {
namespace {

constexpr long long kWaitCycles = 1ll << 31;

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

// make initialised mbarriers visible to the other threads and to the bulk-copy unit
__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// one try_wait on the phase with the given parity: true once it has completed
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done)
                 : "r"(smem_addr(bar)), "r"(parity)
                 : "memory");
    return done != 0;
}

// wait for the completion of the phase with the given parity; false once
// max_cycles SM clock cycles have passed without it (the clock is read only
// when the first try does not succeed)
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          long long max_cycles = kWaitCycles)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (clock64() - t0 > max_cycles)
            return false;
    }
}

// global -> shared, completing `bytes` of the transaction count of *bar;
// both addresses 16-byte aligned, bytes a multiple of 16
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// order this thread's earlier generic-proxy accesses to shared memory before
// later bulk copies (the async proxy) that overwrite it
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace
}  // namespace dsv4
