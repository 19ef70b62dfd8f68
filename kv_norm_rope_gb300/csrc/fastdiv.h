// Exact division of a 32-bit unsigned value by a divisor fixed for a launch,
// with one 64 x 64 -> high-64 multiply instead of a 64-bit division.
//
// For d in [1, 2^32) let M = ceil(2^64 / d).  Then for every n in [0, 2^32),
// n / d = floor(M * n / 2^64) (Lemire, Kaser and Kurz, "Faster remainder by
// direct computation: applications to compilers and software libraries",
// Software: Practice and Experience 49(6), 2019, Theorem 1 with N = L = 32:
// 2^64 <= M * d < 2^64 + d <= 2^64 + 2^32).  M = floor((2^64 - 1) / d) + 1,
// which needs 65 bits for d = 1 only; d = 1 is stored as M = 0 and the
// quotient is then n itself.
#pragma once

#include <stdint.h>

namespace dsv4 {

inline uint64_t fastdiv_magic(uint32_t d)
{
    return d <= 1u ? 0u : UINT64_MAX / d + 1u;
}

#ifdef __CUDACC__
// The high word of magic * n for n < 2^32, from 32-bit halves: with magic =
// mh * 2^32 + ml and ml * n = a * 2^32 + b (b < 2^32), magic * n = (mh * n + a) *
// 2^32 + b, so its high 64 bits are (mh * n + a) >> 32; mh * n + a < 2^64.
__device__ __forceinline__ uint32_t fastdiv(uint32_t n, uint64_t magic)
{
    if (magic == 0u)
        return n;
    const uint64_t t = uint64_t(static_cast<uint32_t>(magic >> 32)) * n +
                       __umulhi(static_cast<uint32_t>(magic), n);
    return static_cast<uint32_t>(t >> 32);
}
#endif

}  // namespace dsv4
