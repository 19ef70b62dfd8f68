// Debug bounds checks.  Every global load and store of the kernels names the
// buffer it falls in (a Span: base and size in bytes).  In the checked build
// (compiled with -DDSV4_CHECK_BOUNDS: libdsv4kv_checked.so) each access first
// tests that all the bytes it touches lie inside that buffer; an access that
// would leave it is skipped (a load gives zeros) and DSV4_DEVERR_BOUNDS is
// OR-ed into the caller's error word.  In the release build the test is the
// constant true, so the spans and checks compile to nothing.
//
// The pages record two faults of this operator on other hardware, both
// address faults: a 32-bit index that wrapped past 2^31 q elements and a KV
// store that wrote into the rope region of the row (FlagGems-vllm PR #684,
// "Performance against a baseline").  The checked build holds every computed
// address against its buffer while the GPU tests run, with no memory checker
// needed.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "bounds_range.h"
#include "dsv4kv.h"

namespace dsv4 {
namespace {

struct Span {
    const void *base;
    uint64_t bytes;
};

#ifdef DSV4_CHECK_BOUNDS
// this translation unit's record of skipped accesses (read by its
// DSV4_BOUNDS_FLAG_READER function; one per file, as this namespace is unnamed)
__device__ int32_t g_bounds_flag;
#endif

// true when [p, p + n) lies inside s (always true in the release build)
__device__ __forceinline__ bool in_span(const void *p, uint32_t n, Span s, int32_t *err)
{
#ifdef DSV4_CHECK_BOUNDS
    if (range_inside(reinterpret_cast<uintptr_t>(p), n, reinterpret_cast<uintptr_t>(s.base),
                     s.bytes))
        return true;
    atomicOr(&g_bounds_flag, DSV4_DEVERR_BOUNDS);
    if (err != nullptr)
        atomicOr(err, DSV4_DEVERR_BOUNDS);
    return false;
#else
    (void)p;
    (void)n;
    (void)s;
    (void)err;
    return true;
#endif
}

// checked forms of the accesses the kernels make
__device__ __forceinline__ uint4 ld_stream16_in(const void *p, Span s, int32_t *err)
{
    return in_span(p, 16, s, err) ? __ldcs(reinterpret_cast<const uint4 *>(p))
                                  : make_uint4(0u, 0u, 0u, 0u);
}

__device__ __forceinline__ uint2 ld_stream8_in(const void *p, Span s, int32_t *err)
{
    return in_span(p, 8, s, err) ? __ldcs(reinterpret_cast<const uint2 *>(p)) : make_uint2(0u, 0u);
}

__device__ __forceinline__ uint4 ldg16_in(const void *p, Span s, int32_t *err)
{
    return in_span(p, 16, s, err) ? __ldg(reinterpret_cast<const uint4 *>(p))
                                  : make_uint4(0u, 0u, 0u, 0u);
}

__device__ __forceinline__ uint2 ldg8_in(const void *p, Span s, int32_t *err)
{
    return in_span(p, 8, s, err) ? __ldg(reinterpret_cast<const uint2 *>(p)) : make_uint2(0u, 0u);
}

__device__ __forceinline__ float4 ldg_f4_in(const float *p, Span s, int32_t *err)
{
    return in_span(p, 16, s, err) ? __ldg(reinterpret_cast<const float4 *>(p))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
}

__device__ __forceinline__ int64_t ldg_i64_in(const int64_t *p, Span s, int32_t *err)
{
    return in_span(p, 8, s, err) ? __ldg(p) : 0;
}

__device__ __forceinline__ void st_stream16_in(void *p, uint4 v, Span s, int32_t *err)
{
    if (in_span(p, 16, s, err))
        __stcs(reinterpret_cast<uint4 *>(p), v);
}

__device__ __forceinline__ void st16_in(void *p, uint4 v, Span s, int32_t *err)
{
    if (in_span(p, 16, s, err))
        *reinterpret_cast<uint4 *>(p) = v;
}

__device__ __forceinline__ void st_stream8_in(void *p, uint2 v, Span s, int32_t *err)
{
    if (in_span(p, 8, s, err))
        __stcs(reinterpret_cast<uint2 *>(p), v);
}

__device__ __forceinline__ void st_stream4_in(void *p, uint32_t v, Span s, int32_t *err)
{
    if (in_span(p, 4, s, err))
        __stcs(reinterpret_cast<unsigned int *>(p), v);
}

__device__ __forceinline__ void st_byte_in(uint8_t *p, uint8_t v, Span s, int32_t *err)
{
    if (in_span(p, 1, s, err))
        *p = v;
}

}  // namespace
}  // namespace dsv4

// Defines dsv4::name(int reset): this file's flag of skipped accesses (0 or
// DSV4_DEVERR_BOUNDS) after synchronising the current device, cleared when reset
// is nonzero; -DSV4_ERR_CUDA if the runtime fails; -1 in the release build.
#ifdef DSV4_CHECK_BOUNDS
#define DSV4_BOUNDS_FLAG_READER(name)                                                         \
    namespace dsv4 {                                                                          \
    int name(int reset)                                                                       \
    {                                                                                         \
        int32_t v = 0;                                                                        \
        if (cudaDeviceSynchronize() != cudaSuccess ||                                         \
            cudaMemcpyFromSymbol(&v, g_bounds_flag, sizeof v) != cudaSuccess)                 \
            return -DSV4_ERR_CUDA;                                                            \
        const int32_t zero = 0;                                                               \
        if (reset && cudaMemcpyToSymbol(g_bounds_flag, &zero, sizeof zero) != cudaSuccess)    \
            return -DSV4_ERR_CUDA;                                                            \
        return v;                                                                             \
    }                                                                                         \
    }
#else
#define DSV4_BOUNDS_FLAG_READER(name)                                                         \
    namespace dsv4 {                                                                          \
    int name(int) { return -1; }                                                              \
    }
#endif
