// Fused DeepSeek-V4 attention-input step for GB300 (sm_103a).
//
// Per token t:
//   q rows  (H of them):  y = x / rms(x); rotate the trailing 64 dims; q <- bf16(y)
//   KV row  (one):        v = x / rms(x) * w; rotate the trailing 64 dims;
//                         FP8 path: 7 UE8M0 exponents + 448 E4M3 + 64 bf16 into
//                         the paged cache at slot_mapping[t]; bf16 path: 512 bf16.
// (FlagGems-vllm PR #684, sections "Ascend 910B" and "T-Head PPU-ZW810E";
//  SGLang PR #33358, sections "Motivation" and "Modifications".)
//
// The operation is HBM-bound: at 64-128 heads, 98.6-99.3% of the bytes are the
// in-place read and write of q.  Design for the GB300 memory system:
//  * One warp owns one 512-wide row.  Lane l holds dims [8l, 8l+8) and
//    [256+8l, 256+8l+8), so each 16-byte vector instruction of the warp covers
//    512 contiguous bytes (four full 128-byte lines) and every byte is read and
//    written exactly once, with evict-first (.cs) hints: q and kv are touched
//    once, so they should not push the cos/sin rows out of L1/L2.
//  * Work items: the T KV rows (one per item) and the T*H q rows in memory
//    order in groups of kRows (rows t*H .. t*H+H-1 are token t's heads),
//    interleaved so that each KV row runs among its own token's q groups: the
//    heavier KV rows then run under the q stream, not ahead of it.  A warp is
//    uniformly on a KV row or a q group at any moment (no divergence inside a
//    row); the KV rows stay out of the q loop's register budget; neighbouring
//    warps share a token's 256-byte cos/sin row in L1 (the 910B section:
//    re-gathering cos/sin per head cost 2.8x there).
//  * The streaming variant runs persistent CTAs sized to the SM count and each
//    warp issues the loads of several rows before it uses any of them, so
//    enough bytes stay in flight per SM to cover DRAM latency (the SGLang
//    section "Modifications": the one-token layout stalled on
//    long_scoreboard with DRAM at 5-7% of peak).  The small variant, for tiny
//    batches, gives every row its own warp in one wave.  (Two more layouts live
//    in their own files: one row per half-warp, and one KV row per quarter-warp
//    fed by bulk copies when there are no q heads.)
//  * Sums of squares are a fixed per-lane sequence followed by a fixed xor
//    butterfly, and the rotation is pinned to explicit fma/mul intrinsics, so
//    a row's bits do not depend on which warp, CTA or variant ran it (the
//    SGLang section "Modifications", item 4).  The rotation is applied to the
//    unscaled inputs with a compensated a*c - b*s and the norm factor after
//    it, so a pair that nearly cancels still lands within a bf16 ulp.
//  * The UE8M0 exponent must agree with an exact evaluation.  fp32 is enough
//    except when a block's amax lies within a relative 2^-14 of a boundary
//    448*2^k; only then does the warp settle it (exact_scale_bumps): in fp32
//    float-float arithmetic, and in fp64 for the values it cannot settle
//    (GB300's fp64 rate is low; about 3e-4 of KV rows take the path on
//    Gaussian data).
//  * Nothing here waits, spins or traps.  Out-of-range positions or slots set
//    a bit in the caller's error word and the affected writes are skipped.

#include <cuda_runtime.h>
#include <stdint.h>

#include "launch_status.h"
#include "rowmath.cuh"

namespace dsv4 {
namespace {

// Work items, handed out round-robin over all warps of the grid: the KV row
// of each token t and ceil(T*H/R) groups of R consecutive q rows (memory
// order), interleaved as described at the loop.
template <int kStore, int kRows, bool kSmemW, bool kKvNorm>
__global__ void __launch_bounds__(256, 3) qnorm_rope_kv_insert_kernel(const KParams p)
{
    __shared__ uint4 w_smem[kSmemW ? 64 : 1];
    const int lane = threadIdx.x & 31;
    const int warps_per_cta = blockDim.x >> 5;
    if (kSmemW && kKvNorm) {
        for (int i = threadIdx.x; i < 64; i += blockDim.x)
            w_smem[i] = ldg16_in(reinterpret_cast<const uint4 *>(p.w) + i, w_span(p), p.err);
        __syncthreads();
    }
    const int64_t H = p.num_heads;
    const int64_t T = p.num_tokens;
    const int64_t q_rows = T * H;
    const int64_t groups = (q_rows + kRows - 1) / kRows;
    const int64_t items = T + groups;
    const int64_t stride = int64_t(gridDim.x) * warps_per_cta;
    // KV rows interleaved with the q groups: period k (k < T) is KV row k then q
    // groups [k*G, k*G + G); the q groups past T*G follow.  The heavier KV rows
    // then run under the q stream instead of ahead of it, next to their token's q.
    const int64_t G = T > 0 ? groups / T : 0;
    const int64_t P = G + 1;

    for (int64_t it = int64_t(blockIdx.x) * warps_per_cta + (threadIdx.x >> 5); it < items;
         it += stride) {
        const int64_t period = it / P;
        const int64_t o = it - period * P;
        if (period < T && o == 0) {
            const int64_t t = period;
            const int64_t pos = ldg_i64_in(p.pos + t, pos_span(p), p.err);
            const int64_t slot = ldg_i64_in(p.slot + t, slot_span(p), p.err);
            const uint16_t *src = p.kv + t * kHead;
            const uint4 xa = ld_stream16_in(src + 8 * lane, kv_span(p), p.err);
            const uint4 xb = ld_stream16_in(src + 256 + 8 * lane, kv_span(p), p.err);
            kv_row<kStore, kSmemW, kKvNorm>(p, lane, t, pos, slot, xa, xb, w_smem);
            continue;
        }
        const int64_t group = period < T ? period * G + (o - 1) : T * G + (it - T * P);
        const int64_t r0 = group * kRows;
        // token of each row, and its position (tiny, cached loads first)
        int64_t t[kRows], pos[kRows];
        t[0] = r0 / H;
        int64_t h = r0 - t[0] * H;
#pragma unroll
        for (int j = 1; j < kRows; ++j) {
            t[j] = t[j - 1];
            if (++h == H) {
                h = 0;
                ++t[j];
            }
        }
#pragma unroll
        for (int j = 0; j < kRows; ++j)
            pos[j] = r0 + j < q_rows ? ldg_i64_in(p.pos + t[j], pos_span(p), p.err) : 0;
        // all row loads back to back: no dependency between them
        uint4 a[kRows], b[kRows];
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
            if (r0 + j < q_rows) {
                const uint16_t *src = p.q + (r0 + j) * kHead;
                a[j] = ld_stream16_in(src + 8 * lane, q_span(p), p.err);
                b[j] = ld_stream16_in(src + 256 + 8 * lane, q_span(p), p.err);
            } else {
                a[j] = make_uint4(0u, 0u, 0u, 0u);
                b[j] = a[j];
            }
        }
        // every row's r at once (rows past the end or with a position outside the
        // table are computed too and not stored)
        float r[kRows];
        q_rows_inv_rms<kRows>(p.eps, a, b, r);
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
            if (r0 + j >= q_rows)
                break;
            if (pos[j] < 0 || pos[j] >= p.max_pos)
                continue;  // flagged once per token by its KV row
            float4 cv, sv;
            load_cs(p, lane, pos[j], cv, sv);
            uint4 out_a, out_b;
            q_row_out(lane, a[j], b[j], r[j], cv, sv, out_a, out_b);
            uint16_t *dst = p.q + (r0 + j) * kHead;
            st_stream16_in(dst + 8 * lane, out_a, q_span(p), p.err);
            st_stream16_in(dst + 256 + 8 * lane, out_b, q_span(p), p.err);
        }
    }
}

template <int kStore, bool kKvNorm>
struct Kernels {
    static constexpr auto small = qnorm_rope_kv_insert_kernel<kStore, 1, false, kKvNorm>;
    static constexpr auto stream =
        qnorm_rope_kv_insert_kernel<kStore, kStreamRowsPerWarp, true, kKvNorm>;
};

template <int kStore, bool kKvNorm>
int launch_one(bool small, dim3 grid, dim3 block, cudaStream_t stream, const KParams &p)
{
    return launch_kernel(small ? Kernels<kStore, kKvNorm>::small : Kernels<kStore, kKvNorm>::stream,
                         grid, block, 0, stream, p);
}

}  // namespace

int stream_ctas_per_sm(int store_mode, int *ctas_per_sm)
{
    // the normalising FP8 kernel is the largest; every streaming kernel shares
    // its launch bounds, so its occupancy is the one used for all of them
    cudaError_t e;
    if (store_mode == DSV4_STORE_BF16)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            ctas_per_sm, Kernels<DSV4_STORE_BF16, true>::stream, kStreamThreads, 0);
    else
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            ctas_per_sm, Kernels<DSV4_STORE_FP8, true>::stream, kStreamThreads, 0);
    return e == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}

int launch(int store_mode, const dsv4_plan &plan, const LaunchArgs &a, cudaStream_t stream)
{
    KParams p;
    p.q = a.q;
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
    p.num_heads = a.num_heads;
    p.eps = a.eps;
    p.err = a.err;
    p.slot_div = fastdiv_magic(static_cast<uint32_t>(a.block_size));
    const dim3 grid(unsigned(plan.ctas)), block(unsigned(plan.threads));
    const bool small = plan.variant == DSV4_VARIANT_SMALL;
    if (store_mode == DSV4_STORE_BF16)
        return a.kv_norm ? launch_one<DSV4_STORE_BF16, true>(small, grid, block, stream, p)
                         : launch_one<DSV4_STORE_BF16, false>(small, grid, block, stream, p);
    return a.kv_norm ? launch_one<DSV4_STORE_FP8, true>(small, grid, block, stream, p)
                     : launch_one<DSV4_STORE_FP8, false>(small, grid, block, stream, p);
}

}  // namespace dsv4

DSV4_BOUNDS_FLAG_READER(bounds_flag_fused)
