// Vector loads and stores with streaming hints, and the bf16 / E4M3
// conversions every kernel of the library uses: one definition of each.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dsv4 {
namespace {

// 16 or 8 bytes touched once: evict-first (.cs) loads and stores
__device__ __forceinline__ uint4 ld_stream16(const void *p)
{
    return __ldcs(reinterpret_cast<const uint4 *>(p));
}

__device__ __forceinline__ void st_stream16(void *p, uint4 v)
{
    __stcs(reinterpret_cast<uint4 *>(p), v);
}

__device__ __forceinline__ void st_stream8(void *p, uint2 v)
{
    __stcs(reinterpret_cast<uint2 *>(p), v);
}

// 8 bf16 (one 16-byte vector) -> 8 fp32, exact
__device__ __forceinline__ void widen8(uint4 u, float *f)
{
    f[0] = __uint_as_float(u.x << 16);
    f[1] = __uint_as_float(u.x & 0xffff0000u);
    f[2] = __uint_as_float(u.y << 16);
    f[3] = __uint_as_float(u.y & 0xffff0000u);
    f[4] = __uint_as_float(u.z << 16);
    f[5] = __uint_as_float(u.z & 0xffff0000u);
    f[6] = __uint_as_float(u.w << 16);
    f[7] = __uint_as_float(u.w & 0xffff0000u);
}

// element k (0..7) of 8 bf16 in one 16-byte vector as fp32, exact (selects,
// so a run-time k stays in registers too)
__device__ __forceinline__ float bf16_at(uint4 u, int k)
{
    const uint32_t w = k < 2 ? u.x : k < 4 ? u.y : k < 6 ? u.z : u.w;
    return __uint_as_float((k & 1) ? (w & 0xffff0000u) : (w << 16));
}

// two fp32 -> bf16x2 (round to nearest even), `lo` in the low half
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint4 bf16x8_rn(const float *y)
{
    return make_uint4(bf16x2_rn(y[0], y[1]), bf16x2_rn(y[2], y[3]), bf16x2_rn(y[4], y[5]),
                      bf16x2_rn(y[6], y[7]));
}

// four fp32 -> four E4M3 bytes (round to nearest even, saturating at +-448),
// element 0 in the lowest byte.  The cvt instruction packs its first source
// into the upper byte of each 16-bit half.
__device__ __forceinline__ uint32_t e4m3x4_rn(float e0, float e1, float e2, float e3)
{
    uint32_t r;
    asm("{\n\t"
        ".reg .b16 p01, p23;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 p01, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 p23, %4, %3;\n\t"
        "mov.b32 %0, {p01, p23};\n\t"
        "}"
        : "=r"(r)
        : "f"(e0), "f"(e1), "f"(e2), "f"(e3));
    return r;
}

// two E4M3 codes (low byte first) -> two fp32, exact
__device__ __forceinline__ float2 e4m3x2_to_f32(uint32_t two_codes)
{
    uint32_t h2;
    const unsigned short c = static_cast<unsigned short>(two_codes);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
    float2 f;
    asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "cvt.f32.f16 %0, lo;\n\tcvt.f32.f16 %1, hi;\n\t}"
        : "=f"(f.x), "=f"(f.y)
        : "r"(h2));
    return f;
}

}  // namespace
}  // namespace dsv4
