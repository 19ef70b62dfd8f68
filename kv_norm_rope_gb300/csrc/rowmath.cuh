// Row arithmetic of the whole-warp layout, shared by the fused kernels (and
// the scale helpers the half-warp layout of halfrow.cuh builds on).
//
// One warp owns one 512-wide row; lane l holds dims [8l, 8l+8) and
// [256+8l, 256+8l+8) as two 16-byte vectors.  Every operation is pinned with
// explicit round-to-nearest intrinsics, so a row's bits do not depend on which
// kernel, warp or CTA computed it (SGLang PR #33358, "Modifications", items
// 3-4: the token grouping must not change a token's output bits).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "bounds.cuh"
#include "convert.cuh"
#include "launch.h"

namespace dsv4 {
namespace {

// The buffers of a launch, for the checked build's bounds tests (bounds.cuh).
__device__ __forceinline__ Span q_span(const KParams &p)
{
    return Span{p.q, uint64_t(p.num_tokens) * uint64_t(p.num_heads) * 1024u};
}
__device__ __forceinline__ Span kv_span(const KParams &p)
{
    return Span{p.kv, uint64_t(p.num_tokens) * 1024u};
}
__device__ __forceinline__ Span w_span(const KParams &p)
{
    return Span{p.w, 1024u};
}

// What the exact scale decision reads, passed by value to its out-of-line
// routines: a reference to the launch's KParams there would make every thread
// copy the whole parameter block to its stack at the start of the kernel (a
// kernel parameter has no generic address).
struct KvSrc {
    const uint16_t *kv;
    const uint16_t *w;
    int64_t num_tokens;
    float eps;
    int32_t *err;
};
__device__ __forceinline__ KvSrc kv_src(const KParams &p)
{
    return KvSrc{p.kv, p.w, p.num_tokens, p.eps, p.err};
}
__device__ __forceinline__ Span kv_span(const KvSrc &p)
{
    return Span{p.kv, uint64_t(p.num_tokens) * 1024u};
}
__device__ __forceinline__ Span w_span(const KvSrc &p)
{
    return Span{p.w, 1024u};
}
__device__ __forceinline__ Span pos_span(const KParams &p)
{
    return Span{p.pos, uint64_t(p.num_tokens) * 8u};
}
__device__ __forceinline__ Span slot_span(const KParams &p)
{
    return Span{p.slot, uint64_t(p.num_tokens) * 8u};
}
__device__ __forceinline__ Span cs_span(const KParams &p)
{
    return Span{p.cs, uint64_t(p.max_pos) * 256u};
}
template <int kStore>
__device__ __forceinline__ Span cache_span(const KParams &p)
{
    return Span{p.cache, uint64_t(p.num_slots) *
                             (kStore == DSV4_STORE_BF16 ? DSV4_BF16_SLOT_BYTES : DSV4_FP8_SLOT_BYTES)};
}


constexpr int kHead = DSV4_HEAD_DIM;
constexpr unsigned kFull = 0xffffffffu;
constexpr uint32_t kMant1p75 = 0x600000u;  // mantissa field of 1.75 (448 = 1.75 * 2^8)
// Half-width of the fp32 "too close to call" band around a boundary, in units
// of the fp32 mantissa field: 2^9 / 2^23 = 2^-14 relative.  The fp32 value of
// an element is within ~14 ulp (2^-20) of its exact value: 16 sequential fmas
// and a 5-level tree for the sum (<= 21 ulp, halved by the root), one ulp each
// for the add of eps, the reciprocal root and two products.
constexpr uint32_t kNearBand = 512u;



__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1)
        v = __fadd_rn(v, __shfl_xor_sync(kFull, v, m));
    return v;
}

__device__ __forceinline__ double warp_sum(double v)
{
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1)
        v = __dadd_rn(v, __shfl_xor_sync(kFull, v, m));
    return v;
}

// max over the 8 lanes that hold one 64-dim block
__device__ __forceinline__ float group8_max(float v)
{
#pragma unroll
    for (int m = 1; m <= 4; m <<= 1)
        v = fmaxf(v, __shfl_xor_sync(kFull, v, m));
    return v;
}

__device__ __forceinline__ bool group8_any(bool b)
{
    unsigned v = b ? 1u : 0u;
#pragma unroll
    for (int m = 1; m <= 4; m <<= 1)
        v |= __shfl_xor_sync(kFull, v, m);
    return v != 0u;
}

// a*c - b*s with one rounding error relative to the result, however much the
// two products cancel: Kahan's algorithm for a 2x2 determinant (the fma
// recovers the rounding error of b*s exactly), relative error at most 2^-23
// (Jeannerod, Louvet and Muller, "Further analysis of Kahan's algorithm for
// the accurate computation of 2x2 determinants", Math. Comp. 2013).
__device__ __forceinline__ float det2(float a, float c, float b, float s)
{
    const float p = __fmul_rn(b, s);
    const float e = __fmaf_rn(b, s, -p);  // b*s == p + e exactly
    return __fsub_rn(__fmaf_rn(a, c, -p), e);
}

// The 8 rope dims 448+8j .. 455+8j held by lane 24+j (pairs 4j .. 4j+3):
// out = r * rot(u), i.e. each pair (a, b) -> r * (a*c - b*s, b*c + a*s).
// Rotating the unscaled inputs first keeps the result accurate when a pair
// nearly cancels; the common factor r then costs one more rounding.
__device__ __forceinline__ void rope8_scaled(const float *u, float4 c, float4 s, float r, float *out)
{
    const float cc[4] = {c.x, c.y, c.z, c.w};
    const float ss[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float a = u[2 * i], b = u[2 * i + 1];
        out[2 * i] = __fmul_rn(det2(a, cc[i], b, ss[i]), r);
        out[2 * i + 1] = __fmul_rn(det2(b, cc[i], -a, ss[i]), r);
    }
}

// 1 / sqrt(sum/512 + eps): the mean and the sum correctly rounded, then one
// correctly rounded reciprocal square root
__device__ __forceinline__ float mean_sq(float sum_sq, float eps)
{
    return __fadd_rn(__fmul_rn(sum_sq, 1.0f / 512.0f), eps);
}

__device__ __forceinline__ float inv_rms(float sum_sq, float eps)
{
    return __frsqrt_rn(mean_sq(sum_sq, eps));
}

// Rows whose mean square (eps included) is below 2^-100 are normalised on a
// copy scaled by 2^64, twice at most.  In fp32 the square of an element below
// 2^-63 is subnormal and keeps fewer bits than its exact 16; that error is
// negligible beside a sum of 2^-100 or more, but decides r when such elements
// make up the whole sum and eps is tiny too (eps = 0).  Scaling by 2^64 is
// exact and commutes with every rounding while nothing is subnormal, so the
// scaled row gives (2^64 x) * (2^-64 r) = x * r with r as accurate as for any
// other row; the second step (by 2^128 in all) makes every nonzero bf16
// element's square a normal fp32 number.  2^64 x stays below 2^19 because
// the mean square was below 2^-100.
constexpr float kTinyMeanSq = 0x1p-100f;

// r = 1 / sqrt(sum(x^2)/512 + eps) of the row held in part by this lane.
// sum() returns the row's sum of squares in the layout's fixed order (the same
// bits on every lane of the row; every lane of the warp calls it together, so
// it may shuffle); scale() multiplies this lane's elements of the row (and
// anything derived from them linearly) by 2^64.  On return those may have been
// scaled by 2^64 or 2^128, and r by the inverse, so that (element * r) is
// unchanged.  Rows of normal size take one compare and one vote more than
// inv_rms.  rescale_tiny is the rare part: given m = mean_sq of the row, it
// rescales the rows whose m is below kTinyMeanSq and returns their new m.
template <typename Sum, typename Scale>
__device__ __forceinline__ float rescale_tiny(float eps, float m, Sum sum, Scale scale)
{
    bool tiny = m < kTinyMeanSq;
    float e = eps;
#pragma unroll 1
    for (int i = 0; i < 2; ++i) {
        if (tiny) {
            scale();
            e = __fmul_rn(__fmul_rn(e, 0x1p64f), 0x1p64f);
        }
        const float s = sum();
        if (tiny)
            m = mean_sq(s, e);
        tiny = tiny && m < kTinyMeanSq;
        if (!__any_sync(kFull, tiny))
            break;
    }
    return m;
}

template <typename Sum, typename Scale>
__device__ __forceinline__ float row_inv_rms(float eps, Sum sum, Scale scale)
{
    float m = mean_sq(sum(), eps);
    if (__any_sync(kFull, m < kTinyMeanSq))
        m = rescale_tiny(eps, m, sum, scale);
    return __frsqrt_rn(m);
}

// 2^-s as fp32 for s in [-127, 127]
__device__ __forceinline__ float pow2_neg(int s)
{
    return s == 127 ? __uint_as_float(0x00400000u) : __uint_as_float(uint32_t(127 - s) << 23);
}

// First guess of a block's UE8M0 exponent from its fp32 amax (>= 0).  With
// amax = M * 2^E, M in [1, 2): the smallest s with amax <= 448 * 2^s is
// E - 8 when M <= 1.75 and E - 7 otherwise.  `near` marks amax within the
// fp32 error band of 1.75 * 2^E, where the exact value must decide.
struct ScaleGuess {
    int s;
    int e;
    bool near;
};

__device__ __forceinline__ ScaleGuess ue8m0_guess(float amax)
{
    // amax below 2^-126 (biased exponent 0) lands on -127 through the clamp; the
    // band test is one unsigned compare; with biased exponent <= 7 both
    // candidates clamp to -127, so the exact path has nothing to decide
    const uint32_t bits = __float_as_uint(amax);
    const int ef = int(bits >> 23);
    const uint32_t m = bits & 0x7fffffu;
    ScaleGuess g;
    g.e = ef - 127;
    g.s = min(max(ef - 135 + (m > kMant1p75 ? 1 : 0), -127), 127);
    g.near = (m - (kMant1p75 - kNearBand)) <= 2u * kNearBand && ef > 7;
    return g;
}

// ---- Exact scale decisions in fp32 (float-float arithmetic)
//
// A block whose fp32 amax lies within the near band of a boundary B = 1.75 * 2^e
// needs the exact answer to "does some |x * r * w| of the block exceed B", where
// r = 1 / sqrt(sum(x^2) / 512 + eps) in exact arithmetic.  As r > 0 that is
// "max |x * w| * r > B", and |x * w| is exact in fp32 (two 8-bit significands),
// so the block's question is one comparison.  GB300's fp64 units run at a small
// fraction of its fp32 rate, so it is first answered in fp32 with error-free
// transformations, and fp64 is kept for what that cannot settle:
//   * x^2 of a bf16 value is exact in fp32 when 2^-63 <= |x| < 2^59; the sum of
//     the squares is accumulated as an unevaluated pair hi + lo (Knuth's
//     TwoSum, Dekker's Fast2Sum), relative error below 2^-41 for 512 positive
//     terms;
//   * r = r0 + r1: r0 = rsqrtf(m), then one Newton step for 1/sqrt(m) with the
//     residual m * r0^2 - 1 formed exactly by fma (Dekker's TwoProd) and the
//     series 1 - h/2 + 3h^2/8, relative error below 2^-44 beyond that of m;
//   * t * r - B, t = max |x * w|, is formed as (t * r0 - B) + (err(t * r0) +
//     t * r1), where t * r0 - B is exact (Sterbenz) once t * r0 is in [B/2, 2B].
// Its sign decides when |t * r - B| > 2^-38 B, far above the errors above and
// those of the fp64 evaluation (about 2^-44), so both give the same answer
// there.  Anything closer, or any value outside the ranges where the steps are
// exact, makes the whole warp take the fp64 routine.  Kernels that lay rows out
// otherwise hand a row with a near block to the whole warp in this layout, so
// every kernel decides with the same code.

struct FF {
    float hi, lo;  // value hi + lo, |lo| <= ulp(hi) / 2 after renormalisation
};

__device__ __forceinline__ FF two_sum(float a, float b)
{
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    return FF{s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}

// requires |a| >= |b| (or a == 0)
__device__ __forceinline__ FF fast_two_sum(float a, float b)
{
    const float s = __fadd_rn(a, b);
    return FF{s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ FF ff_add(FF a, float y)
{
    const FF s = two_sum(a.hi, y);
    return fast_two_sum(s.hi, __fadd_rn(s.lo, a.lo));
}

__device__ __forceinline__ FF ff_add(FF a, FF b)
{
    const FF s = two_sum(a.hi, b.hi);
    return fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}

__device__ __forceinline__ FF ff_add_xor(FF a, int m)
{
    return ff_add(a, FF{__shfl_xor_sync(kFull, a.hi, m), __shfl_xor_sync(kFull, a.lo, m)});
}

// x^2 exact in fp32 and the sum of 512 of them finite: x = 0 or 2^-63 <= |x| < 2^59
__device__ __forceinline__ bool square_exact(float x)
{
    const uint32_t b = __float_as_uint(x) & 0x7fffffffu;
    return b == 0u || b - 0x20000000u < 0x3D000000u;
}

// r = 1 / sqrt(s / 512 + eps) as r.hi + r.lo
__device__ __forceinline__ FF ff_inv_rms(FF s, float eps, bool &ok)
{
    const FF m = ff_add(FF{s.hi * 0x1p-9f, s.lo * 0x1p-9f}, eps);
    ok = ok && m.hi >= 0x1p-120f && m.hi <= 0x1p120f;
    const float r0 = rsqrtf(m.hi);
    const float a = __fmul_rn(r0, r0), b = __fmaf_rn(r0, r0, -a);  // r0^2 = a + b
    const float c = __fmul_rn(m.hi, a), d = __fmaf_rn(m.hi, a, -c);  // m.hi * a = c + d
    // h = m * r0^2 - 1 (c - 1 is exact: c is within 2^-20 of 1)
    const float h = __fadd_rn(__fsub_rn(c, 1.0f), __fadd_rn(d, __fmaf_rn(m.hi, b, __fmul_rn(m.lo, a))));
    return FF{r0, __fmul_rn(r0, __fmaf_rn(__fmul_rn(0.375f, h), h, __fmul_rn(-0.5f, h)))};
}

// t * r against B = 1.75 * 2^e for t = max |x * w| of a block (exact in fp32):
// 1 above, 0 not above, -1 too close to call in fp32 (or outside the ranges
// where the steps are exact)
__device__ __forceinline__ int ff_exceeds(float t, FF r, float B)
{
    if (!(B >= 0x1p-80f))
        return -1;
    if (t == 0.0f)
        return 0;
    if (!(t >= 0x1p-100f && t <= 0x1p120f))
        return -1;
    const float p = __fmul_rn(t, r.hi);
    if (p > 2.0f * B)
        return 1;
    if (p < 0.5f * B)
        return 0;
    const float tail = __fmaf_rn(t, r.lo, __fmaf_rn(t, r.hi, -p));
    const float d = __fadd_rn(__fsub_rn(p, B), tail);
    if (fabsf(d) <= B * 0x1p-38f)
        return -1;
    return d > 0.0f ? 1 : 0;
}

// 1.75 * 2^e as fp32 (e is a block amax exponent of a near block, -119..127)
__device__ __forceinline__ float boundary_f32(int e)
{
    return __uint_as_float((uint32_t(e + 127) << 23) | kMant1p75);
}

// The fp64 decision for near blocks (the fallback of exact_scale_bumps): the
// norm recomputed in fp64 in the whole-warp order and each element evaluated
// in the order of the definition, (x * r) * w, against the boundary 1.75 * 2^e
// of its block.  Same arguments and result as exact_scale_bumps.
__device__ __noinline__ int exact_scale_bumps_fp64(KvSrc p, int lane, int64_t t, int e0,
                                              bool near0, int e1, bool near1)
{
    const uint4 *row = reinterpret_cast<const uint4 *>(p.kv + t * kHead);
    const uint4 *wv = reinterpret_cast<const uint4 *>(p.w);
    const uint4 xa = ldg16_in(row + lane, kv_span(p), p.err);
    const uint4 xb = ldg16_in(row + 32 + lane, kv_span(p), p.err);
    const uint4 wa = ldg16_in(wv + lane, w_span(p), p.err);
    const uint4 wb = ldg16_in(wv + 32 + lane, w_span(p), p.err);
    // rolled loops: this path is rare, its registers are not
    double ss = 0.0;
#pragma unroll 1
    for (int k = 0; k < 16; ++k) {
        const double x = double(bf16_at(k < 8 ? xa : xb, k & 7));
        ss = __fma_rn(x, x, ss);
    }
    ss = warp_sum(ss);
    const double r = 1.0 / sqrt(ss / 512.0 + double(p.eps));
    bool up0 = false, up1 = false;
#pragma unroll 1
    for (int k = 0; k < 16; ++k) {
        const bool second = k >= 8;
        if (!(second ? near1 : near0))
            continue;
        const double v = __dmul_rn(__dmul_rn(double(bf16_at(second ? xb : xa, k & 7)), r),
                                   double(bf16_at(second ? wb : wa, k & 7)));
        const int e = second ? e1 : e0;
        const double bound = __hiloint2double(int(uint32_t(1023 + e) << 20) | 0x000C0000, 0);
        if (fabs(v) > bound) {
            if (second)
                up1 = true;
            else
                up0 = true;
        }
    }
    return (group8_any(up0) ? 1 : 0) | (group8_any(up1) ? 2 : 0);
}

// Exact decision for near blocks, taken by the whole warp when any block of
// the KV row of token t is too close to call in fp32 (lane l holds dims
// [8l, 8l+8) and [256+8l, 256+8l+8) of the row).  It reloads the lane's two
// vectors of the row and of the weight (16-byte loads, issued together; the
// row was just read and is normally still in L2) rather than keep them live
// in registers, and decides each near block in fp32 float-float arithmetic
// (above); what that cannot settle goes to the fp64 routine.  Returns bit 0:
// the lane's half-0 block exceeds its boundary; bit 1: the half-1 block does
// (the same in the block's 8 lanes).
__device__ __noinline__ int exact_scale_bumps(KvSrc p, int lane, int64_t t, int e0,
                                              bool near0, int e1, bool near1)
{
    const uint4 *row = reinterpret_cast<const uint4 *>(p.kv + t * kHead);
    const uint4 *wv = reinterpret_cast<const uint4 *>(p.w);
    const uint4 xa = ldg16_in(row + lane, kv_span(p), p.err);
    const uint4 xb = ldg16_in(row + 32 + lane, kv_span(p), p.err);
    const uint4 wa = ldg16_in(wv + lane, w_span(p), p.err);
    const uint4 wb = ldg16_in(wv + 32 + lane, w_span(p), p.err);
    float x[16];
    widen8(xa, x);
    widen8(xb, x + 8);
    // four interleaved chains (the order of a float-float sum only moves its
    // error, which the margin covers)
    bool ok = true;
    FF s4[4] = {FF{0.0f, 0.0f}, FF{0.0f, 0.0f}, FF{0.0f, 0.0f}, FF{0.0f, 0.0f}};
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        ok = ok && square_exact(x[k]);
        s4[k & 3] = ff_add(s4[k & 3], __fmul_rn(x[k], x[k]));
    }
    FF s = ff_add(ff_add(s4[0], s4[1]), ff_add(s4[2], s4[3]));
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1)
        s = ff_add_xor(s, m);
    const FF r = ff_inv_rms(s, p.eps, ok);
    float w[16];
    widen8(wa, w);
    widen8(wb, w + 8);
    float t0 = 0.0f, t1 = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        t0 = fmaxf(t0, fabsf(__fmul_rn(x[k], w[k])));
        t1 = fmaxf(t1, fabsf(__fmul_rn(x[8 + k], w[8 + k])));
    }
    t0 = group8_max(t0);
    t1 = group8_max(t1);
    const int res0 = near0 ? ff_exceeds(t0, r, boundary_f32(e0)) : 0;
    const int res1 = near1 ? ff_exceeds(t1, r, boundary_f32(e1)) : 0;
    if (__any_sync(kFull, !ok || res0 < 0 || res1 < 0))
        return exact_scale_bumps_fp64(p, lane, t, e0, near0, e1, near1);
    return (res0 > 0 ? 1 : 0) | (res1 > 0 ? 2 : 0);
}

__device__ __forceinline__ int clamp_s(int s)
{
    return min(max(s, -127), 127);
}

__device__ __forceinline__ void flag_error(int32_t *err, int bit)
{
    if (err != nullptr)
        atomicOr(err, bit);
}

// ---- KV row values, shared by every layout
//
// For a normalised KV row the kernels form, per element,
//   xw = x * w                        exact: the product of two bf16 values fits fp32
//                                     (for weights 0 or 2^-9 <= |w| < 2^64)
//   v  = fp32(xw * r)                 one rounding of x * w * r
// and for the FP8 store, per 64-dim block b with t_b = max |xw| (exact),
//   amax_b    = fp32(t_b * r)         = max |v| over the block (rounding is monotone)
//   payload   = E4M3(fp32(xw * k_b)), k_b = r * 2^-s_b (exact)
// which is E4M3(v * 2^-s_b): scaling by a power of two commutes with the
// rounding.  When s_b < -64, r * 2^-s_b could overflow, and the two steps
// E4M3(fp32(xw * r) * 2^-s_b) are taken instead (blocks whose amax is below
// 2^-55: all-zero blocks, or blocks far below the rest of their row).  The
// products x * w and x * x read the bf16 inputs directly (fma.rn.f32.bf16), so
// no element is widened first.  Every layout evaluates exactly these steps, so
// a row's bytes do not depend on the kernel that wrote them.

constexpr int kTwoStepBelow = -64;

// x * y + c for bf16 half kHalf (0: low, 1: high) of two packed words: one
// rounding (x * y is exact in fp32)
template <int kHalf>
__device__ __forceinline__ float fma_bf16(uint32_t x, uint32_t y, float c)
{
    float d;
    if (kHalf == 0)
        asm("{\n\t.reg .b16 xl, xh, yl, yh;\n\tmov.b32 {xl, xh}, %1;\n\tmov.b32 {yl, yh}, %2;\n\t"
            "fma.rn.f32.bf16 %0, xl, yl, %3;\n\t}"
            : "=f"(d)
            : "r"(x), "r"(y), "f"(c));
    else
        asm("{\n\t.reg .b16 xl, xh, yl, yh;\n\tmov.b32 {xl, xh}, %1;\n\tmov.b32 {yl, yh}, %2;\n\t"
            "fma.rn.f32.bf16 %0, xh, yh, %3;\n\t}"
            : "=f"(d)
            : "r"(x), "r"(y), "f"(c));
    return d;
}

// x_0^2 + ... + x_7^2 of one 16-byte vector, accumulated in element order
__device__ __forceinline__ float sumsq8(uint4 x)
{
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    float acc = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc = fma_bf16<0>(w[i], w[i], acc);
        acc = fma_bf16<1>(w[i], w[i], acc);
    }
    return acc;
}

// The fixed order of every row's sum of squares, in every layout: whole-warp
// lane l's partial is (its first vector's sum) + (its second vector's sum),
// each vector summed in element order; the 32 partials are then added by the
// xor butterfly (16, 8, 4, 2, 1).  Two chains of 8 per partial keep the
// dependency chains short.
__device__ __forceinline__ float lane_sumsq(uint4 first, uint4 second)
{
    return __fadd_rn(sumsq8(first), sumsq8(second));
}

// out[k] = x_k * w_k, exact
__device__ __forceinline__ void prod8(uint4 x, uint4 w, float *out)
{
    const uint32_t a[4] = {x.x, x.y, x.z, x.w}, b[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        out[2 * i] = fma_bf16<0>(a[i], b[i], -0.0f);
        out[2 * i + 1] = fma_bf16<1>(a[i], b[i], -0.0f);
    }
}

// 8 bf16 times 2^64, exact (the tiny-row rescaling of row_inv_rms)
__device__ __forceinline__ uint4 scale8_2p64(uint4 x)
{
    const uint32_t k = 0x5F805F80u;  // bf16x2 (2^64, 2^64)
    uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(w[i]) : "r"(w[i]), "r"(k));
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// out[k] = in[k] * k for 8 values, two at a time with the packed fp32 multiply
// (mul.rn.f32x2): each half is the correctly rounded scalar product, so the
// bits are those of 8 scalar multiplies.  kPacked = false takes 8 scalar
// multiplies instead, for code at its register limit (a packed operand must sit
// in an aligned register pair, which can cost copies there).
template <bool kPacked = true>
__device__ __forceinline__ void scale8(const float *in, float k, float *out)
{
    if constexpr (!kPacked) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            out[i] = __fmul_rn(in[i], k);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %4};\n\t"
                "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
                : "=f"(out[2 * i]), "=f"(out[2 * i + 1])
                : "f"(in[2 * i]), "f"(in[2 * i + 1]), "f"(k));
    }
}

// E4M3 of the payload of 8 values of one block: xw * k in one rounding, or for
// two_step (s < kTwoStepBelow) fp32(xw * r) * k2 with k2 = 2^-s
template <bool kPacked = true>
__device__ __forceinline__ uint2 e4m3x8_of(const float *xw, float k)
{
    float v[8];
    scale8<kPacked>(xw, k, v);
    return make_uint2(e4m3x4_rn(v[0], v[1], v[2], v[3]), e4m3x4_rn(v[4], v[5], v[6], v[7]));
}

template <bool kPacked = true>
__device__ __forceinline__ uint2 e4m3x8_two_step(const float *xw, float r, float k2)
{
    float v[8];
    scale8<kPacked>(xw, r, v);
    scale8<kPacked>(v, k2, v);
    return make_uint2(e4m3x4_rn(v[0], v[1], v[2], v[3]), e4m3x4_rn(v[4], v[5], v[6], v[7]));
}

// the payload of a block, either form (callers take this path only when some
// lane of the warp has a block below kTwoStepBelow; the others use e4m3x8_of
// with r * 2^-s directly, so the common path carries no select)
template <bool kPacked = true>
__device__ __forceinline__ uint2 e4m3x8_block(const float *xw, float r, int s)
{
    return s < kTwoStepBelow ? e4m3x8_two_step<kPacked>(xw, r, pow2_neg(s))
                             : e4m3x8_of<kPacked>(xw, __fmul_rn(r, pow2_neg(s)));
}

// bf16 of fp32(xw * r) for 8 values
__device__ __forceinline__ uint4 bf16x8_scaled(const float *xw, float r)
{
    float v[8];
    scale8(xw, r, v);
    return bf16x8_rn(v);
}

// max(|a|, |b|, |c|) in one three-input max (sm_100 and later)
__device__ __forceinline__ float max3_abs(float a, float b, float c)
{
    float d;
    asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// max |xw| of 8 values (+0 when all are zeros)
__device__ __forceinline__ float absmax8(const float *xw)
{
    const float a = max3_abs(xw[0], xw[1], xw[2]);
    const float b = max3_abs(xw[3], xw[4], xw[5]);
    const float c = max3_abs(xw[6], xw[7], a);
    return fmaxf(fabsf(b), fabsf(c));
}

// The lane's products for the KV row of token tok in the whole-warp layout
// (lane l: dims [8l, 8l+8) in xw[0..7], [256+8l, 256+8l+8) in xw[8..15]), their
// lane-local maxima t[0] = max |xw[0..7]|, t[1] = max |xw[8..15]| (0 on rope
// lanes), and the row's r.  Rope lanes (24..31) get their dims 448.. final in
// xw[8..15]: x * w rotated (compensated), then scaled by r.  The partial sums,
// products and maxima do not depend on r and come first, so they overlap the
// reduction and x dies early; a tiny row (rare) reloads x from p.kv and scales
// the products and maxima with it.  With no norm, xw = x and r = 1.
template <bool kSmemW, bool kKvNorm>
__device__ __forceinline__ float kv_products(const KParams &p, int lane, int64_t tok, uint4 xa,
                                             uint4 xb, float4 cv, float4 sv, const uint4 *w_smem,
                                             float *xw, float *t)
{
    const bool rope_lane = lane >= 24;
    float r = 1.0f;
    float part = 0.0f;
    if (!kKvNorm) {
        // the row arrives normalised: v = x (exact), only the rope dims turn
        widen8(xa, xw);
        widen8(xb, xw + 8);
    } else {
        const uint4 wa = kSmemW
                             ? w_smem[lane]
                             : ldg16_in(reinterpret_cast<const uint4 *>(p.w) + lane, w_span(p), p.err);
        const uint4 wb =
            kSmemW ? w_smem[32 + lane]
                   : ldg16_in(reinterpret_cast<const uint4 *>(p.w) + 32 + lane, w_span(p), p.err);
        part = lane_sumsq(xa, xb);
        prod8(xa, wa, xw);
        prod8(xb, wb, xw + 8);
    }
    t[0] = absmax8(xw);
    t[1] = rope_lane ? 0.0f : absmax8(xw + 8);
    if (kKvNorm) {
        float m = mean_sq(warp_sum(part), p.eps);
        if (__any_sync(kFull, m < kTinyMeanSq)) {
            const uint4 *row = reinterpret_cast<const uint4 *>(p.kv + tok * kHead);
            uint4 ya = ldg16_in(row + lane, kv_span(p), p.err);
            uint4 yb = ldg16_in(row + 32 + lane, kv_span(p), p.err);
            m = rescale_tiny(p.eps, m, [&] { return warp_sum(lane_sumsq(ya, yb)); }, [&] {
                ya = scale8_2p64(ya);
                yb = scale8_2p64(yb);
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    xw[k] = __fmul_rn(xw[k], 0x1p64f);
                t[0] = __fmul_rn(t[0], 0x1p64f);
                t[1] = __fmul_rn(t[1], 0x1p64f);
            });
        }
        r = __frsqrt_rn(m);
    }
    if (rope_lane) {
        float u[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            u[k] = xw[8 + k];
        rope8_scaled(u, cv, sv, r, xw + 8);
    }
    return r;
}

// The KV row of token t: v = x*w*r (or v = x when the row arrives normalised),
// rotate, store into the paged cache.  xa, xb: the row's two 16-byte vectors of
// this lane (from global memory or a shared-memory stage); pos, slot: the
// token's metadata.  The rare exact-scale path reloads the row from p.kv.
template <int kStore, bool kSmemW, bool kKvNorm>
__device__ __forceinline__ void kv_row(const KParams &p, int lane, int64_t t, int64_t pos,
                                       int64_t slot, uint4 xa, uint4 xb, const uint4 *w_smem)
{
    const uint16_t *src = p.kv + t * kHead;
    if (pos < 0 || pos >= p.max_pos) {
        if (lane == 0)
            flag_error(p.err, DSV4_DEVERR_POS_RANGE);
        return;
    }
    if (slot < 0)
        return;
    if (slot >= p.num_slots) {
        if (lane == 0)
            flag_error(p.err, DSV4_DEVERR_SLOT_RANGE);
        return;
    }
    const bool rope_lane = lane >= 24;
    float4 cv = make_float4(0.f, 0.f, 0.f, 0.f), sv = cv;
    if (rope_lane) {
        const float *cs = p.cs + pos * DSV4_ROPE_DIM + 4 * (lane - 24);
        cv = ldg_f4_in(cs, cs_span(p), p.err);
        sv = ldg_f4_in(cs + DSV4_ROPE_DIM / 2, cs_span(p), p.err);
    }
    float xw[16], tmax[2];
    float r = kv_products<kSmemW, kKvNorm>(p, lane, t, xa, xb, cv, sv, w_smem, xw, tmax);

    if (kStore == DSV4_STORE_BF16) {
        uint16_t *row = reinterpret_cast<uint16_t *>(p.cache) + slot * kHead;
        st_stream16_in(row + 8 * lane, bf16x8_scaled(xw, r), cache_span<kStore>(p), p.err);
        st_stream16_in(row + 256 + 8 * lane, rope_lane ? bf16x8_rn(xw + 8) : bf16x8_scaled(xw + 8, r),
                       cache_span<kStore>(p), p.err);
        return;
    }

    // block amax: half 0 -> blocks 0..3 (lane / 8), half 1 -> blocks 4..6 (lanes 0..23)
    ScaleGuess g0 = ue8m0_guess(__fmul_rn(group8_max(tmax[0]), r));
    ScaleGuess g1 = ue8m0_guess(__fmul_rn(group8_max(tmax[1]), r));  // lanes 24..31: never near
    // with no norm, v = x exactly and the guess is already exact
    if (kKvNorm && __any_sync(kFull, g0.near || g1.near)) {
        const int bumps = exact_scale_bumps(kv_src(p), lane, t, g0.e, g0.near, g1.e, g1.near);
        if (g0.near)
            g0.s = clamp_s(g0.e - 8 + (bumps & 1));
        if (g1.near)
            g1.s = clamp_s(g1.e - 8 + ((bumps >> 1) & 1));
        // recompute the products (same bits) instead of keeping them live across the call
        r = kv_products<kSmemW, kKvNorm>(
            p, lane, t, ldg16_in(reinterpret_cast<const uint4 *>(src) + lane, kv_span(p), p.err),
            ldg16_in(reinterpret_cast<const uint4 *>(src) + 32 + lane, kv_span(p), p.err), cv, sv,
            w_smem, xw, tmax);
    }

    // 0 <= slot < num_slots <= 2^32 here, so the quotient is a 32-bit one
    const int64_t blk = fastdiv(static_cast<uint32_t>(slot), p.slot_div);
    const int64_t off = slot - blk * p.block_size;
    uint8_t *base = p.cache + blk * int64_t(p.block_size) * DSV4_FP8_SLOT_BYTES;
    uint8_t *data = base + off * DSV4_FP8_DATA_BYTES;

    const Span cspan = cache_span<kStore>(p);
    if (__any_sync(kFull, g0.s < kTwoStepBelow || (!rope_lane && g1.s < kTwoStepBelow))) {
        st_stream8_in(data + 8 * lane, e4m3x8_block(xw, r, g0.s), cspan, p.err);
        if (!rope_lane)
            st_stream8_in(data + 256 + 8 * lane, e4m3x8_block(xw + 8, r, g1.s), cspan, p.err);
    } else {
        st_stream8_in(data + 8 * lane, e4m3x8_of(xw, __fmul_rn(r, pow2_neg(g0.s))), cspan, p.err);
        if (!rope_lane)
            st_stream8_in(data + 256 + 8 * lane, e4m3x8_of(xw + 8, __fmul_rn(r, pow2_neg(g1.s))),
                          cspan, p.err);
    }
    if (rope_lane) {
        // rope dims stay bf16; 8-byte stores keep any block_size legal
        uint8_t *tail = data + DSV4_NOPE_DIM + 16 * (lane - 24);
        st_stream8_in(tail, make_uint2(bf16x2_rn(xw[8], xw[9]), bf16x2_rn(xw[10], xw[11])), cspan,
                      p.err);
        st_stream8_in(tail + 8, make_uint2(bf16x2_rn(xw[12], xw[13]), bf16x2_rn(xw[14], xw[15])),
                      cspan, p.err);
    }

    // scale word: byte b is the exponent of block b, held by lane 8*(b%4) of
    // half b/4; each of those lanes ORs its byte into place (byte 7 stays 0)
    const bool leader = (lane & 7) == 0;
    const uint32_t shift = 8u * uint32_t(lane >> 3);
    const uint32_t lo = __reduce_or_sync(kFull, leader ? uint32_t(g0.s + 127) << shift : 0u);
    const uint32_t hi =
        __reduce_or_sync(kFull, leader && !rope_lane ? uint32_t(g1.s + 127) << shift : 0u);
    if (lane == 0)
        st_stream8_in(base + int64_t(p.block_size) * DSV4_FP8_DATA_BYTES + off * DSV4_FP8_SCALE_BYTES,
                      make_uint2(lo, hi), cspan, p.err);
}


// r of kRows q head rows held in the whole-warp layout (a[j], b[j]: lane l's
// two vectors of row j), with one tiny-row vote for the whole group, so the
// rows' arithmetic stays straight-line and interleaved; a row that needs the
// rare rescaling gets it as in row_inv_rms (a[j], b[j] scaled with it).
template <int kRows>
__device__ __forceinline__ void q_rows_inv_rms(float eps, uint4 *a, uint4 *b, float *r)
{
    float m[kRows];
    bool tiny = false;
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
        m[j] = mean_sq(warp_sum(lane_sumsq(a[j], b[j])), eps);
        tiny = tiny || m[j] < kTinyMeanSq;
    }
    if (__any_sync(kFull, tiny)) {
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
            if (__any_sync(kFull, m[j] < kTinyMeanSq))
                m[j] = rescale_tiny(
                    eps, m[j], [&] { return warp_sum(lane_sumsq(a[j], b[j])); },
                    [&] {
                        a[j] = scale8_2p64(a[j]);
                        b[j] = scale8_2p64(b[j]);
                    });
        }
    }
#pragma unroll
    for (int j = 0; j < kRows; ++j)
        r[j] = __frsqrt_rn(m[j]);
}

// One q head row with its r: y = x * r with the rope dims rotated first
// (compensated) and then scaled; returns the lane's two output vectors (bf16,
// round to nearest).
__device__ __forceinline__ void q_row_out(int lane, uint4 a, uint4 b, float r, float4 cv,
                                          float4 sv, uint4 &out_a, uint4 &out_b)
{
    float y[16];
    widen8(a, y);
    widen8(b, y + 8);
    scale8(y, r, y);
    if (lane < 24) {
        scale8(y + 8, r, y + 8);
    } else {
        float u[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            u[k] = y[8 + k];
        rope8_scaled(u, cv, sv, r, y + 8);
    }
    out_a = bf16x8_rn(y);
    out_b = bf16x8_rn(y + 8);
}

// cos and sin of the 4 pairs held by a rope lane (lanes 24..31) at row pos
__device__ __forceinline__ void load_cs(const KParams &p, int lane, int64_t pos, float4 &cv,
                                        float4 &sv)
{
    cv = make_float4(0.f, 0.f, 0.f, 0.f);
    sv = cv;
    if (lane >= 24) {
        const float *cs = p.cs + pos * DSV4_ROPE_DIM + 4 * (lane - 24);
        cv = ldg_f4_in(cs, cs_span(p), p.err);
        sv = ldg_f4_in(cs + DSV4_ROPE_DIM / 2, cs_span(p), p.err);
    }
}

}  // namespace
}  // namespace dsv4
