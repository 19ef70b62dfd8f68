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

// The weight in shared memory as fp32 (exact), laid out so that the 16 lanes
// of a half-warp read 16 consecutive float4: lane h's 8 weights of vector j
// are float4s (2j) * 16 + h and (2j + 1) * 16 + h.
__device__ __forceinline__ int w_index(int j, int part, int h)
{
    return (2 * j + part) * 16 + h;
}

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
__device__ __forceinline__ float half_sumsq(const float (*v)[8])
{
    float sa = 0.0f, sb = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k)
        sa = __fmaf_rn(v[0][k], v[0][k], sa);
#pragma unroll
    for (int k = 0; k < 8; ++k)
        sa = __fmaf_rn(v[2][k], v[2][k], sa);
#pragma unroll
    for (int k = 0; k < 8; ++k)
        sb = __fmaf_rn(v[1][k], v[1][k], sb);
#pragma unroll
    for (int k = 0; k < 8; ++k)
        sb = __fmaf_rn(v[3][k], v[3][k], sb);
    return half_sum(__fadd_rn(sa, sb));
}

__device__ __forceinline__ void half_scale(float (*v)[8])
{
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int k = 0; k < 8; ++k)
            v[j][k] = __fmul_rn(v[j][k], 0x1p64f);
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

// v = x * r * w (or x) for the lane's 32 dims of its row, rope dims rotated
template <bool kKvNorm>
__device__ __forceinline__ void half_row_values(const KParams &p, int h, const uint4 *x, float4 cv,
                                                float4 sv, const float4 *w_smem, float (*v)[8])
{
#pragma unroll
    for (int j = 0; j < 4; ++j)
        widen8(x[j], v[j]);
    const bool rope_lane = h >= 8;
    if (!kKvNorm) {
        if (rope_lane) {
            float u[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                u[k] = v[3][k];
            rope8_scaled(u, cv, sv, 1.0f, v[3]);
        }
        return;
    }
    const float r = row_inv_rms(p.eps, [&] { return half_sumsq(v); }, [&] { half_scale(v); });
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const float4 wa = w_smem[w_index(j, 0, h)], wb = w_smem[w_index(j, 1, h)];
        const float w[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
        for (int k = 0; k < 8; ++k)
            v[j][k] = __fmul_rn(__fmul_rn(v[j][k], r), w[k]);
    }
    const float4 wa = w_smem[w_index(3, 0, h)], wb = w_smem[w_index(3, 1, h)];
    const float w[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
    if (!rope_lane) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            v[3][k] = __fmul_rn(__fmul_rn(v[3][k], r), w[k]);
    } else {
        // x*w is exact in fp32; rotate, then scale
        float u[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            u[k] = __fmul_rn(v[3][k], w[k]);
        rope8_scaled(u, cv, sv, r, v[3]);
    }
}

// The exact decision for blocks too close to a boundary in fp32 (rare), for
// the row of each half that has one: the whole warp decides it in the
// whole-warp layout (exact_scale_bumps), the same code as every other kernel.
// Lane h of half r holds block 2j + h/8 in vector j, with its exponent e_j
// and near flag (bit j of near_bits); whole-warp lane l asks for blocks l/8
// and 4 + l/8.  Returns bit j set when the lane's block of vector j exceeds
// its boundary.
__device__ __noinline__ int half_exact_bumps(const KParams &p, int lane, int64_t t, int e0, int e1,
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
// tail and the scale word.
template <bool kKvNorm>
__device__ __forceinline__ void half_row_fp8(const KParams &p, int h, bool active, int64_t t,
                                             int64_t slot, float (*v)[8])
{
    const bool rope_lane = h >= 8;

    ScaleGuess g[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float am = 0.0f;
        if (j < 3 || !rope_lane) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                am = fmaxf(am, fabsf(v[j][k]));
        }
        g[j] = ue8m0_guess(group8_max(am));  // rope lanes: amax 0, never near
        g[j].near = g[j].near && active;
    }
    if (kKvNorm && __any_sync(kFull, g[0].near || g[1].near || g[2].near || g[3].near)) {
        const int nb = (g[0].near ? 1 : 0) | (g[1].near ? 2 : 0) | (g[2].near ? 4 : 0) |
                       (g[3].near ? 8 : 0);
        const int bumps = half_exact_bumps(p, threadIdx.x & 31, active ? t : 0, g[0].e, g[1].e,
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

    if (!active)
        return;
    const int64_t blk = fastdiv(static_cast<uint32_t>(slot), p.slot_div);
    const int64_t off = slot - blk * p.block_size;
    uint8_t *base = p.cache + blk * int64_t(p.block_size) * DSV4_FP8_SLOT_BYTES;
    uint8_t *data = base + off * DSV4_FP8_DATA_BYTES;
    const Span cspan = cache_span<DSV4_STORE_FP8>(p);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (j == 3 && rope_lane)
            break;
        const float kj = pow2_neg(g[j].s);
        st_stream8_in(data + 128 * j + 8 * h,
                      make_uint2(e4m3x4_rn(v[j][0] * kj, v[j][1] * kj, v[j][2] * kj, v[j][3] * kj),
                                 e4m3x4_rn(v[j][4] * kj, v[j][5] * kj, v[j][6] * kj, v[j][7] * kj)),
                      cspan, p.err);
    }
    if (rope_lane) {
        // rope dims stay bf16; 8-byte stores keep any block_size legal
        uint8_t *tail = data + DSV4_NOPE_DIM + 16 * (h - 8);
        st_stream8_in(tail, make_uint2(bf16x2_rn(v[3][0], v[3][1]), bf16x2_rn(v[3][2], v[3][3])),
                      cspan, p.err);
        st_stream8_in(tail + 8, make_uint2(bf16x2_rn(v[3][4], v[3][5]), bf16x2_rn(v[3][6], v[3][7])),
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
                                         int64_t pos, int64_t slot, const uint4 *x,
                                         const float4 *w_smem)
{
    float4 cv, sv;
    half_load_cs(p, h, active, pos, cv, sv);
    float v[4][8];
    half_row_values<kKvNorm>(p, h, x, cv, sv, w_smem, v);

    if constexpr (kStore == DSV4_STORE_BF16) {
        if (active) {
            uint16_t *row = reinterpret_cast<uint16_t *>(p.cache) + slot * kHead;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                st_stream16_in(row + 128 * j + 8 * h, bf16x8_rn(v[j]), cache_span<kStore>(p), p.err);
        }
    } else {
        half_row_fp8<kKvNorm>(p, h, active, t, slot, v);
    }
}

// thread i < 64 widens the 8 weights of dims [8i, 8i + 8): j = i / 16, h = i % 16
__device__ __forceinline__ void stage_weight(const KParams &p, int i, float4 *w_smem)
{
    float f[8];
    widen8(ldg16_in(reinterpret_cast<const uint4 *>(p.w) + i, w_span(p), p.err), f);
    const int j = i >> 4, h = i & 15;
    w_smem[w_index(j, 0, h)] = make_float4(f[0], f[1], f[2], f[3]);
    w_smem[w_index(j, 1, h)] = make_float4(f[4], f[5], f[6], f[7]);
}


// One KV row per half-warp: this half takes token t (idle when t >= T).  It
// loads the token's metadata and row, flags an out-of-range position or slot,
// and writes the cache row when both are in range.  Both halves reach every
// shuffle; a pair with no row to write skips the arithmetic (warp-uniform).
template <int kStore, bool kKvNorm>
__device__ __forceinline__ void kv_pair_item(const KParams &p, int h, int64_t t,
                                             const float4 *w_smem)
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
        half_row<kStore, kKvNorm>(p, h, active, t, pos, slot, x, w_smem);
}

// One q head row: y = x * r with the rope dims rotated first (compensated)
// and then scaled, the operations of q_row on the same values; returns the
// lane's four output vectors (bf16, round to nearest).
__device__ __forceinline__ void q_half_row(const KParams &p, int h, const uint4 *x, float4 cv,
                                           float4 sv, uint4 *out)
{
    float y[4][8];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        widen8(x[j], y[j]);
    const float r = row_inv_rms(p.eps, [&] { return half_sumsq(y); }, [&] { half_scale(y); });
#pragma unroll
    for (int j = 0; j < 3; ++j) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            y[j][k] = __fmul_rn(y[j][k], r);
    }
    if (h < 8) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            y[3][k] = __fmul_rn(y[3][k], r);
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
