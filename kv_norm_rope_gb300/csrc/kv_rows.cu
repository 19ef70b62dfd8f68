// KV rows with no q (SGLang PR #33358, "Motivation": fused_norm_rope_flashmla,
// the RMSNorm + RoPE + paged-cache store of the latent KV row alone): the same
// arithmetic as the KV rows of the fused kernel, laid out for rows that carry
// all the work.
//
// In the fused kernel a KV row is one of H + 1 rows of a token and takes a
// whole warp.  Alone, such rows are issue-bound: ~390 warp instructions per
// row in that layout, much of it per-row overhead (reductions over 32 lanes,
// both sides of the rope branch, the scale guesses and word, address
// arithmetic) rather than per-element work.  Here a quarter-warp owns a row,
// so each of those instructions serves four rows:
//
//   lane g = lane % 8 of quarter c = lane / 8 holds dims [64u + 8g, 64u + 8g + 8)
//   of token 4i + c for u = 0..7 (warp item i).
//
// Vector u of every lane lies in quantisation block u, and vector 7 holds the
// rope dims 448 + 8g .. 455 + 8g (pairs 4g .. 4g + 3) on every lane, so the
// rope takes no branch.  The block maxima are reduce-scattered over the
// quarter (lane g ends with block g's), each lane derives one block's scale
// and the quarter shares them back.
//
// Every value is bit-identical to the fused kernel's: vectors u and u + 4 of
// lane g are the two vectors of whole-warp lane 8u + g, so lane g's partial
// sums over (u, u + 4), u = 0..3, are those of whole-warp lanes g, 8 + g,
// 16 + g and 24 + g; (p0 + p2) + (p1 + p3) is the whole-warp butterfly's xor-16
// and xor-8 levels and xor 4, 2, 1 are the same shuffles.  The elementwise
// operations, the rotation and the block maxima (max is exact) are the same
// operations on the same values, and a row with a block too close to a scale
// boundary is handed to the whole warp, which decides it in the whole-warp
// layout with the code every kernel uses (exact_scale_bumps).

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "bulkcopy.cuh"
#include "launch_status.h"
#include "ops.h"
#include "rowmath.cuh"

namespace dsv4 {
namespace {

constexpr int kKvThreads = 256;
constexpr int kKvCtasPerSm = 2;

// The weight as packed bf16 in dim order (thread i < 64 copies dims
// [8i, 8i + 8)): lane g of a quarter reads vector u at 8u + g, 8 consecutive
// 16-byte words (the four quarters read the same ones).
__device__ __forceinline__ void stage_weight_q(const KParams &p, int i, uint4 *w_smem)
{
    w_smem[i] = ldg16_in(reinterpret_cast<const uint4 *>(p.w) + i, w_span(p), p.err);
}

__device__ __forceinline__ float quarter_sum(float v)
{
#pragma unroll
    for (int m = 4; m >= 1; m >>= 1)
        v = __fadd_rn(v, __shfl_xor_sync(kFull, v, m));
    return v;
}

// The row's sum of squares in the whole-warp order: the partials of whole-warp
// lanes 8u + g (their vectors u and u + 4), the xor-16 and xor-8 levels as
// (p0 + p2) + (p1 + p3), then xor 4, 2, 1 inside the quarter.
__device__ __forceinline__ float quarter_sumsq(const uint4 *x)
{
    float ps[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
        ps[u] = lane_sumsq(x[u], x[u + 4]);
    return quarter_sum(__fadd_rn(__fadd_rn(ps[0], ps[2]), __fadd_rn(ps[1], ps[3])));
}

// max |x_k * w_k| over one 16-byte vector (the products are exact and then
// dropped: the second pass forms them again where they are quantised)
__device__ __forceinline__ float absmax_prod8(uint4 x, uint4 w)
{
    float xw[8];
    prod8(x, w, xw);
    return absmax8(xw);
}

// Pass 1 of a quarter-warp row (vector u of lane g: dims [64u + 8g, 64u + 8g + 8)):
// the block maxima t[u] = max |x * w| over the lane's dims of block u (u < 7;
// t[7] = 0, the rope dims are not quantised) and the row's r.  Only the packed
// row x is held: the products are formed again by the second pass, which keeps
// the registers of a row to x plus one vector at a time.  A tiny row rescales x
// (in place) and t with it.  With no norm, t[u] = max |x| and r = 1.  The values
// are those of kv_products (exact products and maxima, the same sum order).
template <bool kKvNorm>
__device__ __forceinline__ float quarter_pass1(const KParams &p, int g, uint4 *x,
                                               const uint4 *w_smem, float *t)
{
    t[7] = 0.0f;
    if constexpr (!kKvNorm) {
#pragma unroll
        for (int u = 0; u < 7; ++u) {
            float f[8];
            widen8(x[u], f);
            t[u] = absmax8(f);
        }
        return 1.0f;
    } else {
        const float sum = quarter_sumsq(x);
#pragma unroll
        for (int u = 0; u < 7; ++u)
            t[u] = absmax_prod8(x[u], w_smem[8 * u + g]);
        float m = mean_sq(sum, p.eps);
        if (__any_sync(kFull, m < kTinyMeanSq))
            m = rescale_tiny(p.eps, m, [&] { return quarter_sumsq(x); }, [&] {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    x[u] = scale8_2p64(x[u]);
                    t[u] = __fmul_rn(t[u], 0x1p64f);
                }
            });
        return __frsqrt_rn(m);
    }
}

// Pass 2, vector u: xw = x * w (or x with no norm), formed again
template <bool kKvNorm>
__device__ __forceinline__ void quarter_vec(const uint4 *x, const uint4 *w_smem, int g, int u,
                                            float *xw)
{
    if (kKvNorm)
        prod8(x[u], w_smem[8 * u + g], xw);
    else
        widen8(x[u], xw);
}

// Max of each of 8 values over the 8 lanes of a quarter, scattered: lane g
// returns the max of a[g].  Three halving steps: at mask m a lane keeps the
// half of its values whose index bit matches its own lane bit and takes the
// partner's copy of that half.
__device__ __forceinline__ float quarter_max_scatter(const float *a, int g)
{
    float b[4], c[2];
    const bool b2 = (g & 4) != 0, b1 = (g & 2) != 0, b0 = (g & 1) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float keep = b2 ? a[i + 4] : a[i];
        const float send = b2 ? a[i] : a[i + 4];
        b[i] = fmaxf(keep, __shfl_xor_sync(kFull, send, 4));
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float keep = b1 ? b[i + 2] : b[i];
        const float send = b1 ? b[i] : b[i + 2];
        c[i] = fmaxf(keep, __shfl_xor_sync(kFull, send, 2));
    }
    const float keep = b0 ? c[1] : c[0];
    const float send = b0 ? c[0] : c[1];
    return fmaxf(keep, __shfl_xor_sync(kFull, send, 1));
}

// The exact decision for blocks too close to a boundary in fp32 (rare), for
// the row of each quarter that has one: the whole warp decides it in the
// whole-warp layout (exact_scale_bumps), the same code as every other kernel.
// Lane g of quarter c holds block g's exponent e and near flag; whole-warp
// lane l asks for blocks l/8 and 4 + l/8.  Returns, to lane g of each
// quarter, whether block g exceeds its boundary.
__device__ __noinline__ bool quarter_exact_bump(KvSrc p, int lane, int64_t t, int e,
                                                bool near)
{
    const unsigned quarters = __ballot_sync(kFull, near);
    const int g = lane & 7;
    bool mine = false;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        if (((quarters >> (8 * c)) & 0xffu) == 0u)
            continue;
        const int64_t tc = __shfl_sync(kFull, t, 8 * c);
        const int s0 = 8 * c + (lane >> 3), s1 = 8 * c + 4 + (lane >> 3);
        const int res = exact_scale_bumps(p, lane, tc, __shfl_sync(kFull, e, s0),
                                          ((quarters >> s0) & 1u) != 0u,
                                          __shfl_sync(kFull, e, s1),
                                          ((quarters >> s1) & 1u) != 0u);
        // block g's answer: bit 0 of lane 8g (g < 4), bit 1 of lane 8(g - 4)
        const int got = __shfl_sync(kFull, res, 8 * (g & 3));
        if ((lane >> 3) == c)
            mine = ((got >> (g >> 2)) & 1) != 0;
    }
    return mine;
}

// The FP8 store of a quarter-warp row: block scales, E4M3 payload, bf16 rope
// tail and the scale word.  x: the row (as scaled by pass 1), tmax and r: from
// pass 1, rope: the lane's rope dims, final.
template <bool kKvNorm>
__device__ __forceinline__ void quarter_row_fp8(const KParams &p, int lane, bool active, int64_t t,
                                                int64_t slot, const uint4 *x, const uint4 *w_smem,
                                                const float *tmax, float r, const float *rope)
{
    const int g = lane & 7, base = lane & ~7;
    // tmax[7] = 0: the rope dims are not quantised, lane 7 leads no block
    ScaleGuess sg = ue8m0_guess(__fmul_rn(quarter_max_scatter(tmax, g), r));
    sg.near = sg.near && active;
    // with no norm, v = x exactly and the guess is already exact
    if (kKvNorm && __any_sync(kFull, sg.near)) {
        const bool up = quarter_exact_bump(kv_src(p), lane, active ? t : 0, sg.e, sg.near);
        if (sg.near)
            sg.s = clamp_s(sg.e - 8 + (up ? 1 : 0));
    }
    int s[7];
#pragma unroll
    for (int u = 0; u < 7; ++u)
        s[u] = __shfl_sync(kFull, sg.s, base + u);
    // a block below kTwoStepBelow anywhere in the warp: the two-step payload form
    // (voted by every lane before the inactive ones leave)
    bool slow = false;
#pragma unroll
    for (int u = 0; u < 7; ++u)
        slow = slow || s[u] < kTwoStepBelow;
    slow = __any_sync(kFull, active && slow);
    if (!active)
        return;

    const int64_t blk = fastdiv(static_cast<uint32_t>(slot), p.slot_div);
    const int64_t off = slot - blk * p.block_size;
    uint8_t *cbase = p.cache + blk * int64_t(p.block_size) * DSV4_FP8_SLOT_BYTES;
    uint8_t *data = cbase + off * DSV4_FP8_DATA_BYTES;
    const Span cspan = cache_span<DSV4_STORE_FP8>(p);
    if (slow) {
#pragma unroll
        for (int u = 0; u < 7; ++u) {
            float xw[8];
            quarter_vec<kKvNorm>(x, w_smem, g, u, xw);
            st_stream8_in(data + 64 * u + 8 * g, e4m3x8_block(xw, r, s[u]), cspan, p.err);
        }
    } else {
#pragma unroll
        for (int u = 0; u < 7; ++u) {
            float xw[8];
            quarter_vec<kKvNorm>(x, w_smem, g, u, xw);
            st_stream8_in(data + 64 * u + 8 * g, e4m3x8_of(xw, __fmul_rn(r, pow2_neg(s[u]))), cspan,
                          p.err);
        }
    }
    // rope dims stay bf16; 8-byte stores keep any block_size legal
    uint8_t *tail = data + DSV4_NOPE_DIM + 16 * g;
    st_stream8_in(tail, make_uint2(bf16x2_rn(rope[0], rope[1]), bf16x2_rn(rope[2], rope[3])), cspan,
                  p.err);
    st_stream8_in(tail + 8, make_uint2(bf16x2_rn(rope[4], rope[5]), bf16x2_rn(rope[6], rope[7])),
                  cspan, p.err);
    if (g == 0) {
        // byte b of the scale word is block b's exponent; byte 7 stays 0
        const uint32_t lo = uint32_t(s[0] + 127) | (uint32_t(s[1] + 127) << 8) |
                            (uint32_t(s[2] + 127) << 16) | (uint32_t(s[3] + 127) << 24);
        const uint32_t hi =
            uint32_t(s[4] + 127) | (uint32_t(s[5] + 127) << 8) | (uint32_t(s[6] + 127) << 16);
        st_stream8_in(cbase + int64_t(p.block_size) * DSV4_FP8_DATA_BYTES + off * DSV4_FP8_SCALE_BYTES,
                      make_uint2(lo, hi), cspan, p.err);
    }
}

// One KV row per quarter-warp: this quarter holds token t's row in x (zeros
// when t >= T) with its metadata pos and slot.  It flags an out-of-range
// position or slot and writes the cache row when both are in range.  All
// quarters reach every shuffle; a warp with no row to write skips the
// arithmetic.
template <int kStore, bool kKvNorm>
__device__ __forceinline__ void kv_quad_row(const KParams &p, int lane, int64_t t, int64_t pos,
                                            int64_t slot, uint4 *x, const uint4 *w_smem, float4 cv,
                                            float4 sv)
{
    const int g = lane & 7;
    const bool live = t < p.num_tokens;
    const bool pos_ok = pos >= 0 && pos < p.max_pos;
    if (live && g == 0) {
        if (!pos_ok)
            flag_error(p.err, DSV4_DEVERR_POS_RANGE);
        else if (slot >= p.num_slots)
            flag_error(p.err, DSV4_DEVERR_SLOT_RANGE);
    }
    const bool active = live && pos_ok && slot >= 0 && slot < p.num_slots;
    if (!__any_sync(kFull, active))
        return;
    if constexpr (kStore == DSV4_STORE_FP8) {
        // (the bf16 kernel has its cos/sin from the caller, loaded before the kv wait)
        if (active) {
            const float *cs = p.cs + pos * DSV4_ROPE_DIM + 4 * g;
            cv = ldg_f4_in(cs, cs_span(p), p.err);
            sv = ldg_f4_in(cs + DSV4_ROPE_DIM / 2, cs_span(p), p.err);
        }
    }
    float tmax[8];
    const float r = quarter_pass1<kKvNorm>(p, g, x, w_smem, tmax);
    // the rope dims (vector 7 on every lane): x * w rotated, then scaled by r
    float rope[8];
    {
        float u7[8];
        quarter_vec<kKvNorm>(x, w_smem, g, 7, u7);
        rope8_scaled(u7, cv, sv, r, rope);
    }
    if constexpr (kStore == DSV4_STORE_BF16) {
        if (active) {
            uint16_t *row = reinterpret_cast<uint16_t *>(p.cache) + slot * kHead;
#pragma unroll
            for (int u = 0; u < 7; ++u) {
                float xw[8];
                quarter_vec<kKvNorm>(x, w_smem, g, u, xw);
                st16_in(row + 64 * u + 8 * g, bf16x8_scaled(xw, r), cache_span<kStore>(p), p.err);
            }
            st16_in(row + 64 * 7 + 8 * g, bf16x8_rn(rope), cache_span<kStore>(p), p.err);
        }
    } else {
        quarter_row_fp8<kKvNorm>(p, lane, active, t, slot, x, w_smem, tmax, r, rope);
    }
}

// Shared memory: per warp kKvStages mbarriers, the weight (packed bf16), then per
// warp kKvStages stages of one item (4 rows, 4 KB) each.
constexpr int kKvWarps = kKvThreads / 32;
constexpr int kKvStages = 2;
constexpr uint32_t kItemBytes = 4 * DSV4_HEAD_DIM * 2;
constexpr int kKvWeightOffset = 256;
constexpr int kKvStageOffset = kKvWeightOffset + 1024;
constexpr size_t kKvSmemBytes = size_t(kKvStageOffset) + size_t(kKvWarps) * kKvStages * kItemBytes;
static_assert(kKvWarps * kKvStages * 8 <= kKvWeightOffset, "barriers overlap the weight");
static_assert(kKvStageOffset % 128 == 0, "stages must be 16-byte aligned");

// Each warp takes items first, first + W, first + 2W, ... (W = warps in the
// grid); item i is tokens 4i .. 4i + 3, one 4 KB block of kv.  Lane 0 keeps
// the warp's next kKvStages items in flight as bulk copies into the warp's
// stages, so the loads of the next items overlap the arithmetic of this one.
// The metadata of the next item is loaded one item ahead.  A wait that runs
// out sets DSV4_DEVERR_TIMEOUT; the warp then lets its copies land and leaves.
template <int kStore, bool kKvNorm>
__global__ void __launch_bounds__(kKvThreads, kKvCtasPerSm) kv_rows_kernel(const KParams p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, c = lane >> 3, g = lane & 7;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem) + warp * kKvStages;
    uint4 *w_smem = reinterpret_cast<uint4 *>(smem + kKvWeightOffset);
    uint8_t *stages = smem + kKvStageOffset + size_t(warp) * kKvStages * kItemBytes;
    if (lane == 0) {
        for (int s = 0; s < kKvStages; ++s)
            mbar_init(&bars[s], 1);
        mbar_init_fence();
    }

    const int64_t T = p.num_tokens;
    const int64_t items = (T + 3) / 4;
    const int64_t total = int64_t(gridDim.x) * kKvWarps;
    const int64_t first = int64_t(blockIdx.x) * kKvWarps + warp;
    const int64_t mine = items > first ? (items - first + total - 1) / total : 0;
    // lane 0: item j of this warp into stage j % kKvStages
    auto issue = [&](int64_t j) {
        const int64_t t0 = 4 * (first + j * total);
        const uint32_t bytes = uint32_t(T - t0 < 4 ? T - t0 : 4) * (DSV4_HEAD_DIM * 2);
        uint64_t *bar = &bars[j % kKvStages];
        if (in_span(p.kv + t0 * kHead, bytes, kv_span(p), p.err)) {
            mbar_arrive_expect_tx(bar, bytes);
            bulk_load(stages + (j % kKvStages) * kItemBytes, p.kv + t0 * kHead, bytes, bar);
        } else {
            mbar_arrive(bar);  // checked build: the copy is skipped, its phase completes empty
        }
    };
    int64_t issued = mine < kKvStages ? mine : kKvStages;
    if (lane == 0)
        for (int64_t j = 0; j < issued; ++j)
            issue(j);

    int64_t t = 4 * first + c;
    int64_t pos = t < T ? ldg_i64_in(p.pos + t, pos_span(p), p.err) : 0;
    int64_t slot = t < T ? ldg_i64_in(p.slot + t, slot_span(p), p.err) : -1;
    // the first copies and metadata are in flight while the CTA stages the
    // weight; the barriers' other lanes and the weight wait for the CTA barrier
    if (kKvNorm) {
        for (int i = threadIdx.x; i < 64; i += kKvThreads)
            stage_weight_q(p, i, w_smem);
    }
    __syncthreads();
    for (int64_t j = 0; j < mine; ++j) {
        // the next item's metadata, one item ahead
        const int64_t tn = t + 4 * total;
        const bool next_live = j + 1 < mine && tn < T;
        const int64_t pos_n = next_live ? ldg_i64_in(p.pos + tn, pos_span(p), p.err) : 0;
        const int64_t slot_n = next_live ? ldg_i64_in(p.slot + tn, slot_span(p), p.err) : -1;

        // the bf16 kernel, with registers to spare, issues this item's cos/sin loads
        // before the wait for its kv (the position is known an item ahead); the FP8
        // kernel, at its register limit, loads them after (measured faster each way)
        float4 cv = make_float4(0.f, 0.f, 0.f, 0.f), sv = cv;
        if constexpr (kStore == DSV4_STORE_BF16) {
            if (t < T && pos >= 0 && pos < p.max_pos && slot >= 0 && slot < p.num_slots) {
                const float *cs = p.cs + pos * DSV4_ROPE_DIM + 4 * g;
                cv = ldg_f4_in(cs, cs_span(p), p.err);
                sv = ldg_f4_in(cs + DSV4_ROPE_DIM / 2, cs_span(p), p.err);
            }
        }
        const int s = int(j % kKvStages);
        if (!mbar_wait(&bars[s], uint32_t(j / kKvStages) & 1)) {
            if (lane == 0)
                flag_error(p.err, DSV4_DEVERR_TIMEOUT);
            // copies in flight, this item's included, land before the warp leaves
            for (int64_t k = j; k < issued; ++k)
                (void)mbar_wait(&bars[k % kKvStages], uint32_t(k / kKvStages) & 1);
            return;
        }
        const uint4 *row = reinterpret_cast<const uint4 *>(stages + s * kItemBytes) + c * 64;
        uint4 x[8];
        if (t - c + 4 <= T) {  // the whole item is live (warp-uniform): no selects
#pragma unroll
            for (int u = 0; u < 8; ++u)
                x[u] = row[8 * u + g];
        } else {
#pragma unroll
            for (int u = 0; u < 8; ++u)
                x[u] = t < T ? row[8 * u + g] : make_uint4(0u, 0u, 0u, 0u);
        }
        // every lane has read the stage: it may be refilled
        fence_proxy_async_smem();
        __syncwarp();
        if (issued < mine) {
            if (lane == 0)
                issue(issued);
            ++issued;
        }
        kv_quad_row<kStore, kKvNorm>(p, lane, t, pos, slot, x, w_smem, cv, sv);
        t = tn;
        pos = pos_n;
        slot = slot_n;
    }
}

// the opt-in to more than 48 KB of dynamic shared memory for each kernel of
// this file, once per device (bit d of `configured` for device d < 64; other
// devices set it every call)
int configure_smem()
{
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return DSV4_ERR_CUDA;
    const uint64_t bit = dev >= 0 && dev < 64 ? uint64_t(1) << dev : 0;
    if (bit != 0 && (configured.load(std::memory_order_relaxed) & bit) != 0)
        return DSV4_OK;
    const void *kernels[4] = {reinterpret_cast<const void *>(kv_rows_kernel<DSV4_STORE_FP8, true>),
                              reinterpret_cast<const void *>(kv_rows_kernel<DSV4_STORE_FP8, false>),
                              reinterpret_cast<const void *>(kv_rows_kernel<DSV4_STORE_BF16, true>),
                              reinterpret_cast<const void *>(kv_rows_kernel<DSV4_STORE_BF16, false>)};
    for (const void *k : kernels)
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kKvSmemBytes)) !=
            cudaSuccess)
            return DSV4_ERR_CUDA;
    configured.fetch_or(bit, std::memory_order_relaxed);
    return DSV4_OK;
}

template <int kStore>
int launch_store(bool kv_norm, unsigned grid, cudaStream_t stream, const KParams &p)
{
    return launch_kernel(kv_norm ? kv_rows_kernel<kStore, true> : kv_rows_kernel<kStore, false>,
                         dim3(grid), dim3(kKvThreads), kKvSmemBytes, stream, p);
}

}  // namespace

int kv_rows_ctas_per_sm(int *ctas_per_sm)
{
    if (configure_smem() != DSV4_OK)
        return DSV4_ERR_CUDA;
    // the normalising FP8 kernel is the largest of the four
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm,
                                                         kv_rows_kernel<DSV4_STORE_FP8, true>,
                                                         kKvThreads, kKvSmemBytes) == cudaSuccess
               ? DSV4_OK
               : DSV4_ERR_CUDA;
}

int kv_rows_per_warp()
{
    return 4;
}

int launch_kv_rows(int store_mode, const LaunchArgs &a, int64_t max_ctas, cudaStream_t stream)
{
    KParams p;
    p.q = nullptr;
    p.kv = a.kv;
    p.w = a.w;
    p.pos = a.pos;
    p.cs = a.cs;
    p.max_pos = a.max_pos;
    p.slot = a.slot;
    p.cache = a.cache;
    p.num_slots = a.num_slots;
    p.num_tokens = a.num_tokens;
    p.block_size = a.block_size;
    p.num_heads = 0;
    p.eps = a.eps;
    p.err = a.err;
    p.slot_div = fastdiv_magic(static_cast<uint32_t>(a.block_size));
    if (configure_smem() != DSV4_OK)
        return DSV4_ERR_CUDA;
    const int64_t quads = (a.num_tokens + 3) / 4;
    const int64_t need = quads > 0 ? (quads + kKvWarps - 1) / kKvWarps : 1;
    const unsigned grid = static_cast<unsigned>(need < max_ctas ? need : max_ctas);
    return store_mode == DSV4_STORE_BF16 ? launch_store<DSV4_STORE_BF16>(a.kv_norm, grid, stream, p)
                                         : launch_store<DSV4_STORE_FP8>(a.kv_norm, grid, stream, p);
}

}  // namespace dsv4

DSV4_BOUNDS_FLAG_READER(bounds_flag_kv_rows)
