// Row arithmetic of the half-warp layout: each 512-wide row takes half a warp
// (qnorm_rope_kv_insert_half.cu).
//
// Lane h = lane % 16 of half r = lane / 16 holds dims [128v + 8h, 128v + 8h + 8)
// of its row for v = 0..3: four 16-byte vectors, so one warp-wide load covers
// 256 contiguous bytes of each of two rows.  Vector v of lane h lies in
// quantisation block 2v + h/8; dims 448..511 (vector 3, h >= 8) are the rope
// dims, the same 4 pairs per lane as lane 24 + (h - 8) of a whole-warp row.
//
// Every value is bit-identical to the whole-warp helpers in rowmath.cuh:
// lane h's partial sums over vectors (0, 2) and (1, 3) are exactly the
// partials of whole-warp lanes h and h + 16, their sum is the first level of
// the whole-warp butterfly (xor 16) and the remaining levels (xor 8, 4, 2, 1)
// are the same; the elementwise operations, the rotation and the block
// maxima are the same operations on the same values, and a row with a block
// too close to a scale boundary is handed to the whole warp, which decides it
// in the whole-warp layout with the code every kernel uses.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "rowmath.cuh"

namespace dsv4 {
namespace {

__device__ __forceinline__ float half_sum(float v)
{
#pragma unroll
    for (int m = 8; m >= 1; m >>= 1)
        v = __fadd_rn(v, __shfl_xor_sync(kFull, v, m));
    return v;
}

// The row's sum of squares in the whole-warp order: lane h's vectors (0, 2)
// are whole-warp lane h's, its vectors (1, 3) whole-warp lane h + 16's; their
// sum is the butterfly's xor-16 level, then xor 8, 4, 2, 1 inside the half.
__device__ __forceinline__ float half_sumsq(const uint4 *x)
{
    return half_sum(__fadd_rn(lane_sumsq(x[0], x[2]), lane_sumsq(x[1], x[3])));
}

__device__ __forceinline__ void half_scale(uint4 *x)
{
#pragma unroll
    for (int j = 0; j < 4; ++j)
        x[j] = scale8_2p64(x[j]);
}

// cos and sin of the 4 pairs held by a rope lane (h >= 8) at row pos; zeros
// elsewhere and for rows that are not written
__device__ __forceinline__ void half_load_cs(const KParams &p, int h, bool active, int64_t pos,
                                             float4 &cv, float4 &sv)
{
    cv = make_float4(0.f, 0.f, 0.f, 0.f);
    sv = cv;
    if (active && h >= 8) {
        const float *cs = p.cs + pos * DSV4_ROPE_DIM + 4 * (h - 8);
        cv = ldg_f4_in(cs, cs_span(p), p.err);
        sv = ldg_f4_in(cs + DSV4_ROPE_DIM / 2, cs_span(p), p.err);
    }
}

// Vector j of the lane's row as xw = x * w (or x with no norm).  w: the weight
// (global, packed bf16 in dim order; lane h reads vector j at 16j + h).
template <bool kKvNorm>
__device__ __forceinline__ void half_vec(const KParams &p, int h, const uint4 *x, const uint4 *w,
                                         int j, float *xw)
{
    if (kKvNorm)
        prod8(x[j], ldg16_in(w + 16 * j + h, w_span(p), p.err), xw);
    else
        widen8(x[j], xw);
}

// Pass 1 of a half-warp KV row (vector j: dims [128j + 8h, 128j + 8h + 8)): the
// row's r, the maxima t[j] = max |xw[j]| (0 for the rope vector of rope lanes,
// h >= 8) and, on rope lanes, the final rope dims 448.. (x * w rotated, then
// scaled by r).  The products are dropped once their maxima are taken and formed
// again where they are stored, so a lane holds x (16 registers) rather than 32
// products.  A tiny row rescales x in place first.  With no norm, xw = x and
// r = 1.  The steps of kv_products, so the same bits.
template <bool kKvNorm>
__device__ __forceinline__ float half_pass1(const KParams &p, int h, uint4 *x, float4 cv,
                                            float4 sv, const uint4 *w, float *t, float *rope)
{
    const bool rope_lane = h >= 8;
    float r = 1.0f;
    if (kKvNorm)
        r = row_inv_rms(p.eps, [&] { return half_sumsq(x); }, [&] { half_scale(x); });
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        float xw[8];
        half_vec<kKvNorm>(p, h, x, w, j, xw);
        t[j] = absmax8(xw);
    }
    float u[8];
    half_vec<kKvNorm>(p, h, x, w, 3, u);
    t[3] = rope_lane ? 0.0f : absmax8(u);
    if (rope_lane)
        rope8_scaled(u, cv, sv, r, rope);
    return r;
}

// The exact decision for blocks too close to a boundary in fp32 (rare), for
// the row of each half that has one: the whole warp decides it in the
// whole-warp layout (exact_scale_bumps), the same code as every other kernel.
// Lane h of half r holds block 2j + h/8 in vector j, with its exponent e_j
// and near flag (bit j of near_bits); whole-warp lane l asks for blocks l/8
// and 4 + l/8.  Returns bit j set when the lane's block of vector j exceeds
// its boundary.
__device__ __noinline__ int half_exact_bumps(KvSrc p, int lane, int64_t t, int e0, int e1,
                                             int e2, int e3, int near_bits)
{
    const unsigned halves = __ballot_sync(kFull, near_bits != 0);
    const int h = lane & 15;
    int bits = 0;
#pragma unroll 1
    for (int r = 0; r < 2; ++r) {
        if (((halves >> (16 * r)) & 0xffffu) == 0u)
            continue;
        const int64_t tr = __shfl_sync(kFull, t, 16 * r);
        // blocks b = lane/8 and 4 + lane/8 of half r: vector b/2 of lane 16r + 8(b%2)
        const int b0 = lane >> 3, b1 = 4 + (lane >> 3);
        const int s0 = 16 * r + 8 * (b0 & 1), s1 = 16 * r + 8 * (b1 & 1);
        const int a0 = __shfl_sync(kFull, e0, s0), a1 = __shfl_sync(kFull, e1, s0);
        const int a2 = __shfl_sync(kFull, e2, s0), a3 = __shfl_sync(kFull, e3, s0);
        const int c0 = __shfl_sync(kFull, e0, s1), c1 = __shfl_sync(kFull, e1, s1);
        const int c2 = __shfl_sync(kFull, e2, s1), c3 = __shfl_sync(kFull, e3, s1);
        const int n0 = __shfl_sync(kFull, near_bits, s0), n1 = __shfl_sync(kFull, near_bits, s1);
        const int j0 = b0 >> 1, j1 = b1 >> 1;
        const int eb0 = j0 == 0 ? a0 : j0 == 1 ? a1 : j0 == 2 ? a2 : a3;
        const int eb1 = j1 == 0 ? c0 : j1 == 1 ? c1 : j1 == 2 ? c2 : c3;
        const int res = exact_scale_bumps(p, lane, tr, eb0, ((n0 >> j0) & 1) != 0, eb1,
                                          ((n1 >> j1) & 1) != 0);
        // block b's answer: bit 0 of lane 8b (b < 4), bit 1 of lane 8(b - 4)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int b = 2 * j + (h >> 3);
            const int got = __shfl_sync(kFull, res, 8 * (b & 3));
            if ((lane >> 4) == r && ((got >> (b >> 2)) & 1))
                bits |= 1 << j;
        }
    }
    return bits;
}

// The FP8 store of a half-warp row: block scales, E4M3 payload, bf16 rope
// tail and the scale word.  x, tmax, r, rope: as left by half_pass1.
template <bool kKvNorm>
__device__ __forceinline__ void half_row_fp8(const KParams &p, int h, bool active, int64_t t,
                                             int64_t slot, const uint4 *x, const uint4 *w,
                                             const float *tmax, float r, const float *rope)
{
    const bool rope_lane = h >= 8;

    ScaleGuess g[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        g[j] = ue8m0_guess(__fmul_rn(group8_max(tmax[j]), r));  // rope lanes: amax 0, never near
        g[j].near = g[j].near && active;
    }
    if (kKvNorm && __any_sync(kFull, g[0].near || g[1].near || g[2].near || g[3].near)) {
        const int nb = (g[0].near ? 1 : 0) | (g[1].near ? 2 : 0) | (g[2].near ? 4 : 0) |
                       (g[3].near ? 8 : 0);
        const int bumps = half_exact_bumps(kv_src(p), threadIdx.x & 31, active ? t : 0, g[0].e, g[1].e,
                                           g[2].e, g[3].e, nb);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (g[j].near)
                g[j].s = clamp_s(g[j].e - 8 + ((bumps >> j) & 1));
    }

    // scale word of each half: lane h = 0 leads blocks 0, 2, 4, 6 and lane
    // h = 8 blocks 1, 3, 5; bytes land at 8 * block, byte 7 stays 0
    const uint32_t b0 = uint32_t(g[0].s + 127), b1 = uint32_t(g[1].s + 127);
    const uint32_t b2 = uint32_t(g[2].s + 127), b3 = uint32_t(g[3].s + 127);
    const uint32_t lo_part = h == 0 ? (b0 | (b1 << 16)) : (b0 << 8) | (b1 << 24);
    const uint32_t hi_part = h == 0 ? (b2 | (b3 << 16)) : (b2 << 8);
    const uint32_t lo = lo_part | __shfl_xor_sync(kFull, lo_part, 8);
    const uint32_t hi = hi_part | __shfl_xor_sync(kFull, hi_part, 8);
    // a block below kTwoStepBelow anywhere in the warp: the two-step payload form
    // (voted by every lane before the inactive ones leave)
    bool slow = false;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        slow = slow || ((j < 3 || !rope_lane) && g[j].s < kTwoStepBelow);
    slow = __any_sync(kFull, active && slow);

    if (!active)
        return;
    const int64_t blk = fastdiv(static_cast<uint32_t>(slot), p.slot_div);
    const int64_t off = slot - blk * p.block_size;
    uint8_t *base = p.cache + blk * int64_t(p.block_size) * DSV4_FP8_SLOT_BYTES;
    uint8_t *data = base + off * DSV4_FP8_DATA_BYTES;
    const Span cspan = cache_span<DSV4_STORE_FP8>(p);
    if (slow) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (j == 3 && rope_lane)
                break;
            float xw[8];
            half_vec<kKvNorm>(p, h, x, w, j, xw);
            st_stream8_in(data + 128 * j + 8 * h, e4m3x8_block(xw, r, g[j].s), cspan, p.err);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (j == 3 && rope_lane)
                break;
            float xw[8];
            half_vec<kKvNorm>(p, h, x, w, j, xw);
            st_stream8_in(data + 128 * j + 8 * h, e4m3x8_of(xw, __fmul_rn(r, pow2_neg(g[j].s))),
                          cspan, p.err);
        }
    }
    if (rope_lane) {
        // rope dims stay bf16; 8-byte stores keep any block_size legal
        uint8_t *tail = data + DSV4_NOPE_DIM + 16 * (h - 8);
        st_stream8_in(tail, make_uint2(bf16x2_rn(rope[0], rope[1]), bf16x2_rn(rope[2], rope[3])),
                      cspan, p.err);
        st_stream8_in(tail + 8, make_uint2(bf16x2_rn(rope[4], rope[5]), bf16x2_rn(rope[6], rope[7])),
                      cspan, p.err);
    }
    if (h == 0)
        st_stream8_in(base + int64_t(p.block_size) * DSV4_FP8_DATA_BYTES + off * DSV4_FP8_SCALE_BYTES,
                      make_uint2(lo, hi), cspan, p.err);
}

// One row per half-warp.  active: this half's row is written (valid token,
// position and slot); inactive halves still take part in every shuffle.
template <int kStore, bool kKvNorm>
__device__ __forceinline__ void half_row(const KParams &p, int h, bool active, int64_t t,
                                         int64_t pos, int64_t slot, uint4 *x, const uint4 *w)
{
    float4 cv, sv;
    half_load_cs(p, h, active, pos, cv, sv);
    float tmax[4], rope[8];
    const float r = half_pass1<kKvNorm>(p, h, x, cv, sv, w, tmax, rope);

    if constexpr (kStore == DSV4_STORE_BF16) {
        if (active) {
            uint16_t *row = reinterpret_cast<uint16_t *>(p.cache) + slot * kHead;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float xw[8];
                half_vec<kKvNorm>(p, h, x, w, j, xw);
                st_stream16_in(row + 128 * j + 8 * h,
                               (j == 3 && h >= 8) ? bf16x8_rn(rope) : bf16x8_scaled(xw, r),
                               cache_span<kStore>(p), p.err);
            }
        }
    } else {
        half_row_fp8<kKvNorm>(p, h, active, t, slot, x, w, tmax, r, rope);
    }
}

// One KV row per half-warp: this half takes token t (idle when t >= T).  It
// loads the token's metadata and row, flags an out-of-range position or slot,
// and writes the cache row when both are in range.  Both halves reach every
// shuffle; a pair with no row to write skips the arithmetic (warp-uniform).
template <int kStore, bool kKvNorm>
__device__ __forceinline__ void kv_pair_item(const KParams &p, int h, int64_t t, const uint4 *w)
{
    const bool live = t < p.num_tokens;
    const int64_t pos = live ? ldg_i64_in(p.pos + t, pos_span(p), p.err) : 0;
    const int64_t slot = live ? ldg_i64_in(p.slot + t, slot_span(p), p.err) : -1;
    uint4 x[4];
#pragma unroll
    for (int v = 0; v < 4; ++v)
        x[v] = live ? ld_stream16_in(p.kv + t * kHead + 128 * v + 8 * h, kv_span(p), p.err)
                    : make_uint4(0u, 0u, 0u, 0u);
    const bool pos_ok = pos >= 0 && pos < p.max_pos;
    if (live && h == 0) {
        if (!pos_ok)
            flag_error(p.err, DSV4_DEVERR_POS_RANGE);
        else if (slot >= p.num_slots)
            flag_error(p.err, DSV4_DEVERR_SLOT_RANGE);
    }
    const bool active = live && pos_ok && slot >= 0 && slot < p.num_slots;
    if (__any_sync(kFull, active))
        half_row<kStore, kKvNorm>(p, h, active, t, pos, slot, x, w);
}

// r of the kPairs q rows of this half (x[j]: the lane's vectors of row j), one
// tiny-row vote for the group as in q_rows_inv_rms.
template <int kPairs>
__device__ __forceinline__ void q_half_rows_inv_rms(float eps, uint4 (*x)[4], float *r)
{
    float m[kPairs];
    bool tiny = false;
#pragma unroll
    for (int j = 0; j < kPairs; ++j) {
        m[j] = mean_sq(half_sumsq(x[j]), eps);
        tiny = tiny || m[j] < kTinyMeanSq;
    }
    if (__any_sync(kFull, tiny)) {
#pragma unroll
        for (int j = 0; j < kPairs; ++j) {
            if (__any_sync(kFull, m[j] < kTinyMeanSq))
                m[j] = rescale_tiny(
                    eps, m[j], [&] { return half_sumsq(x[j]); }, [&] { half_scale(x[j]); });
        }
    }
#pragma unroll
    for (int j = 0; j < kPairs; ++j)
        r[j] = __frsqrt_rn(m[j]);
}

// One q head row with its r: y = x * r with the rope dims rotated first
// (compensated) and then scaled, the operations of q_row_out on the same
// values; returns the lane's four output vectors (bf16, round to nearest).
__device__ __forceinline__ void q_half_out(int h, const uint4 *x, float r, float4 cv, float4 sv,
                                           uint4 *out)
{
    float y[4][8];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        widen8(x[j], y[j]);
#pragma unroll
    for (int j = 0; j < 3; ++j)
        scale8<false>(y[j], r, y[j]);
    if (h < 8) {
        scale8<false>(y[3], r, y[3]);
    } else {
        float u[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            u[k] = y[3][k];
        rope8_scaled(u, cv, sv, r, y[3]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
        out[j] = bf16x8_rn(y[j]);
}

}  // namespace
}  // namespace dsv4
