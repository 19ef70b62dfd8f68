// Residual add + Gemma RMSNorm + MXFP8 quantisation of activation rows: the
// single-GPU part of the vLLM minimax_m3 finalize_allreduce_norm page
// (_LamportGemmaRMSNormMxfp8Kernel with one rank, so no all-reduce):
//   prenorm  = bf16(x + residual)                  -> residual_out
//   r        = 1 / sqrt(mean(prenorm^2) + eps)
//   normed   = bf16(prenorm * r * (1 + gamma))     (Gemma scale 1 + w)
//   per 32 normed values: e = UE8M0 of fp32(amax * fp32(1/448)), rounded up to
//   a power of two; codes = E4M3_rn_satfinite(normed * 2^(127 - e)), with the
//   page's inverse 0 for e = 0 and e = 254; e in the 128x4 swizzled layout,
//   the scales of the padding rows up to a multiple of 128 rows zeroed.
//
// HBM-bound: per element 2 + 2 bytes read, 2 + 1 written.  One CTA per row;
// thread t owns 16-byte fragments t, t + threads, ... of the row, keeps the
// prenorm values in registers across the block reduction, and the 4 adjacent
// lanes that hold one 32-element block reduce its amax with two shuffles.
// Every operation is an explicit round-to-nearest intrinsic; the block sum is
// a fixed tree, so results are reproducible run to run.

#include <cuda_runtime.h>
#include <stdint.h>

#include "bounds.cuh"
#include "convert.cuh"
#include "launch_status.h"
#include "ops.h"

namespace dsv4 {
namespace {

constexpr unsigned kFull = 0xffffffffu;

struct MParams {
    const uint16_t *x;
    const uint16_t *residual;
    const uint16_t *gamma;
    uint16_t *residual_out;
    uint8_t *codes;
    uint8_t *scales;
    int64_t m;
    int32_t n;
    int32_t padded_cols;
    float eps;
};

// the buffers of a launch, for the checked build's bounds tests (bounds.cuh);
// this entry point has no error word, so only the library's flag records a hit
__device__ __forceinline__ Span rows_span(const void *a, const MParams &p, uint32_t elem)
{
    return Span{a, uint64_t(p.m) * uint64_t(p.n) * elem};
}
__device__ __forceinline__ Span scales_span(const MParams &p)
{
    return Span{p.scales, uint64_t((p.m + 127) / 128) * 128u * uint64_t(p.padded_cols)};
}

// 8 bf16 times 2^64, exact (the rescaling of rows with a tiny mean square)
__device__ __forceinline__ uint4 bf16x8_times_2p64(uint4 x)
{
    const uint32_t k = 0x5F805F80u;  // bf16x2 (2^64, 2^64)
    uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(w[i]) : "r"(w[i]), "r"(k));
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ float bf16_round(float v)
{
    return __uint_as_float(bf16x2_rn(v, 0.0f) << 16);
}

// the exponent of the next power of two at or above x > 0, biased by 127 and
// clamped to [0, 254]; 0 for x <= 0
__device__ __forceinline__ uint32_t ue8m0_round_up(float x)
{
    if (!(x > 0.0f))
        return 0u;
    const uint32_t bits = __float_as_uint(x);
    const uint32_t ef = bits >> 23, mant = bits & 0x7fffffu;
    uint32_t e;
    if (ef == 0u)
        e = mant > 0x400000u ? 1u : 0u;  // subnormal: above 2^-127 rounds up to 2^-126
    else
        e = ef + (mant != 0u ? 1u : 0u);
    return e > 254u ? 254u : e;
}

// the inverse scale 2^(127 - e); 0 for e = 0 and for e = 254
__device__ __forceinline__ float ue8m0_inverse(uint32_t e)
{
    return (e == 0u || e >= 254u) ? 0.0f : __uint_as_float((254u - e) << 23);
}

__device__ __forceinline__ int64_t swizzled(int64_t row, int64_t col, int64_t padded_cols)
{
    return (row / 128) * 128 * padded_cols + (col / 4) * 512 + (row % 32) * 16 +
           ((row % 128) / 32) * 4 + col % 4;
}

template <int kThreads, int kTrips>
__global__ void __launch_bounds__(kThreads) gemma_rmsnorm_mxfp8_kernel(const MParams p)
{
    __shared__ float warp_sums[kThreads / 32];
    const int64_t row = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int fragments = p.n / 8;
    const int cols = p.n / 32;
    if (row >= p.m) {
        // padding row of the last 128-row scale tile: zero scales
        for (int c = tid; c < cols; c += kThreads)
            st_byte_in(p.scales + swizzled(row, c, p.padded_cols), 0, scales_span(p), nullptr);
        return;
    }
    const uint16_t *xr = p.x + row * p.n;
    const uint16_t *rr = p.residual + row * p.n;
    uint4 pre[kTrips];  // prenorm is bf16 by definition: keep it packed
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < kTrips; ++k) {
        const int f = tid + k * kThreads;
        if (f < fragments) {
            float a[8], b[8];
            widen8(ld_stream16_in(reinterpret_cast<const uint4 *>(xr) + f, rows_span(p.x, p, 2), nullptr),
                   a);
            widen8(ld_stream16_in(reinterpret_cast<const uint4 *>(rr) + f,
                                  rows_span(p.residual, p, 2), nullptr),
                   b);
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                o[i] = bf16x2_rn(__fadd_rn(a[2 * i], b[2 * i]), __fadd_rn(a[2 * i + 1], b[2 * i + 1]));
            pre[k] = make_uint4(o[0], o[1], o[2], o[3]);
            st_stream16_in(reinterpret_cast<uint4 *>(p.residual_out + row * p.n) + f, pre[k],
                           rows_span(p.residual_out, p, 2), nullptr);
            float w[8];
            widen8(pre[k], w);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                ss = __fmaf_rn(w[i], w[i], ss);
        } else {
            pre[k] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    // block sum: xor tree inside each warp, then the warps' sums in warp order
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1)
        ss = __fadd_rn(ss, __shfl_xor_sync(kFull, ss, m));
    if (lane == 0)
        warp_sums[warp] = ss;
    __syncthreads();
    float total = warp_sums[0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w)
        total = __fadd_rn(total, warp_sums[w]);
    float m = __fadd_rn(__fdiv_rn(total, float(p.n)), p.eps);
    // A mean square below 2^-100 (only with a tiny eps) may rest on subnormal fp32
    // squares: the row's prenorm is then scaled by 2^64 (exact, twice at most) and
    // summed again, which leaves prenorm * r unchanged and r accurate.  Every
    // thread holds the same total, so the branch and its barriers are block-uniform.
    float e = p.eps;
#pragma unroll 1
    for (int i = 0; i < 2 && m < 0x1p-100f; ++i) {
        float s2 = 0.0f;
#pragma unroll
        for (int k = 0; k < kTrips; ++k) {
            pre[k] = bf16x8_times_2p64(pre[k]);
            float w[8];
            widen8(pre[k], w);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                s2 = __fmaf_rn(w[j], w[j], s2);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1)
            s2 = __fadd_rn(s2, __shfl_xor_sync(kFull, s2, o));
        __syncthreads();  // every thread has read the previous sums
        if (lane == 0)
            warp_sums[warp] = s2;
        __syncthreads();
        total = warp_sums[0];
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w)
            total = __fadd_rn(total, warp_sums[w]);
        e = __fmul_rn(__fmul_rn(e, 0x1p64f), 0x1p64f);
        m = __fadd_rn(__fdiv_rn(total, float(p.n)), e);
    }
    const float r = __frcp_rn(__fsqrt_rn(m));
    const float inv448 = 1.0f / 448.0f;

#pragma unroll
    for (int k = 0; k < kTrips; ++k) {
        const int f = tid + k * kThreads;
        const bool valid = f < fragments;  // 4-lane groups are all valid or all not
        float g[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (valid)
            widen8(ldg16_in(reinterpret_cast<const uint4 *>(p.gamma) + f,
                            Span{p.gamma, uint64_t(p.n) * 2u}, nullptr),
                   g);
        float v[8];
        widen8(pre[k], v);
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[i] = bf16_round(__fmul_rn(__fmul_rn(v[i], r), __fadd_rn(g[i], 1.0f)));
            amax = fmaxf(amax, fabsf(v[i]));
        }
        amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
        const uint32_t e = ue8m0_round_up(__fmul_rn(amax, inv448));
        const float inv = ue8m0_inverse(e);
        if (valid) {
            st_stream8_in(reinterpret_cast<uint2 *>(p.codes + row * p.n) + f,
                          make_uint2(e4m3x4_rn(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv),
                                               __fmul_rn(v[2], inv), __fmul_rn(v[3], inv)),
                                     e4m3x4_rn(__fmul_rn(v[4], inv), __fmul_rn(v[5], inv),
                                               __fmul_rn(v[6], inv), __fmul_rn(v[7], inv))),
                          rows_span(p.codes, p, 1), nullptr);
            if ((lane & 3) == 0)
                st_byte_in(p.scales + swizzled(row, f / 4, p.padded_cols), uint8_t(e),
                           scales_span(p), nullptr);
        }
    }
}

template <int kThreads, int kTrips>
int launch_rows(int64_t grid, cudaStream_t stream, const MParams &p)
{
    return launch_kernel(gemma_rmsnorm_mxfp8_kernel<kThreads, kTrips>, dim3(unsigned(grid)),
                         dim3(kThreads), 0, stream, p);
}

}  // namespace

int launch_gemma_rmsnorm_mxfp8(const uint16_t *x, const uint16_t *residual, const uint16_t *gamma,
                               int64_t m, int32_t n, float eps, uint16_t *residual_out,
                               uint8_t *codes, uint8_t *scales, cudaStream_t stream)
{
    MParams p;
    p.x = x;
    p.residual = residual;
    p.gamma = gamma;
    p.residual_out = residual_out;
    p.codes = codes;
    p.scales = scales;
    p.m = m;
    p.n = n;
    p.padded_cols = ((n / 32) + 3) / 4 * 4;
    p.eps = eps;
    const int64_t grid = (m + 127) / 128 * 128;  // padding rows zero their scales
    // threads x fragments per thread covering the row, from sweeps on GB300: 8
    // warps per row (16 for the widest) with 2-4 fragments per thread; more warps
    // shorten the row's load-reduce-store chain.  Hidden 7168: 8 x 4 beat 4 x 8 by
    // 3-4% (and 7, 12, 14, 16, 28 warps); 16384: 16 x 4 beat 8 x 8 by 8%; 4096:
    // 8 x 2 beat 4 x 4 by 1%; 2048: 4 x 2 beat 8 x 1 by 11%.
    const int fragments = n / 8;
    if (fragments <= 128)
        return launch_rows<128, 1>(grid, stream, p);
    if (fragments <= 256)
        return launch_rows<128, 2>(grid, stream, p);
    if (fragments <= 512)
        return launch_rows<256, 2>(grid, stream, p);
    if (fragments <= 1024)
        return launch_rows<256, 4>(grid, stream, p);
    return launch_rows<512, 4>(grid, stream, p);
}

}  // namespace dsv4

DSV4_BOUNDS_FLAG_READER(bounds_flag_mxfp8)
