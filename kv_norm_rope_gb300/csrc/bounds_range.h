// The range test of the debug bounds checks (bounds.cuh), in plain C++ so that
// a host program can test it too.
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define DSV4_HD __host__ __device__
#else
#define DSV4_HD
#endif

namespace dsv4 {

// true when the n bytes at address p lie inside the buffer [base, base + size).
// No sum is formed that could wrap: p - base is taken only once p >= base.
DSV4_HD inline bool range_inside(uintptr_t p, uint64_t n, uintptr_t base, uint64_t size)
{
    return p >= base && uint64_t(p - base) <= size && n <= size - uint64_t(p - base);
}

}  // namespace dsv4
