// The fused step with one row per half-warp (DSV4_VARIANT_HALF): q heads and
// KV rows both in the half-warp layout of halfrow.cuh.
//
// The whole-warp streaming kernel is DRAM-bound on large batches but spends
// ~195 warp instructions per q row, a good part of it per-row overhead: the
// 32-lane butterfly, the reciprocal root, both sides of the rope branch,
// metadata and address arithmetic.  On small batches (decode) those
// instructions, issued by every warp at the same moment after its loads land,
// are what the launch waits on.  With half a warp per row each of them serves
// two rows.  The values are bit-identical to the other variants (the sums keep
// the whole-warp order; the same operations on the same values).
//
// Work items, handed out round-robin over all warps of the grid:
//   items [0, ceil(T/2))          : KV rows 2i and 2i + 1 (one per half)
//   then groups of 2*kQPairs q rows in memory order; half r of the warp takes
//   rows r0 + 2j + r, j < kQPairs, and loads all of them before computing any.

#include <cuda_runtime.h>
#include <stdint.h>

#include "halfrow.cuh"
#include "launch_status.h"
#include "ops.h"

namespace dsv4 {
namespace {

constexpr int kHalfThreads = 256;
constexpr int kQPairs = 2;  // q row pairs per warp item (4 rows)

template <int kStore, bool kKvNorm>
__global__ void __launch_bounds__(kHalfThreads, 3) qnorm_rope_kv_insert_half_kernel(const KParams p)
{
    // the weight (1 KB, packed bf16) is read by KV rows through the read-only
    // cache: no CTA-wide staging barrier in front of the first loads
    const uint4 *w = reinterpret_cast<const uint4 *>(p.w);
    const int lane = threadIdx.x & 31, h = lane & 15, half = lane >> 4;
    const int64_t H = p.num_heads;
    const int64_t T = p.num_tokens;
    const int64_t q_rows = T * H;
    const int64_t kv_items = (T + 1) / 2;
    const int64_t items = kv_items + (q_rows + 2 * kQPairs - 1) / (2 * kQPairs);
    const int64_t stride = int64_t(gridDim.x) * (kHalfThreads / 32);

    for (int64_t it = int64_t(blockIdx.x) * (kHalfThreads / 32) + (threadIdx.x >> 5); it < items;
         it += stride) {
        if (it < kv_items) {
            kv_pair_item<kStore, kKvNorm>(p, h, 2 * it + half, w);
            continue;
        }
        const int64_t r0 = (it - kv_items) * 2 * kQPairs;
        // token of this half's rows r0 + 2j + half: r0 = t0 * H + head0, and a
        // row d past r0 is d heads further on
        const int64_t t0 = r0 / H, head0 = r0 - t0 * H;
        int64_t pos[kQPairs];
        bool live[kQPairs];
#pragma unroll
        for (int j = 0; j < kQPairs; ++j) {
            int64_t hd = head0 + 2 * j + half, tok = t0;
            while (hd >= H) {  // at most 2 * kQPairs steps
                hd -= H;
                ++tok;
            }
            live[j] = r0 + 2 * j + half < q_rows;
            pos[j] = live[j] ? ldg_i64_in(p.pos + tok, pos_span(p), p.err) : 0;
        }
        // all row loads back to back: no dependency between them
        uint4 x[kQPairs][4];
#pragma unroll
        for (int j = 0; j < kQPairs; ++j) {
            const uint16_t *src = p.q + (r0 + 2 * j + half) * kHead + 8 * h;
#pragma unroll
            for (int v = 0; v < 4; ++v)
                x[j][v] = live[j] ? ld_stream16_in(src + 128 * v, q_span(p), p.err)
                                  : make_uint4(0u, 0u, 0u, 0u);
        }
        // every row's r at once (rows that are not written are computed too)
        float r[kQPairs];
        q_half_rows_inv_rms<kQPairs>(p.eps, x, r);
#pragma unroll
        for (int j = 0; j < kQPairs; ++j) {
            // rows past the end or with a position outside the table are not
            // written (the KV row of the token flags the position)
            const bool active = live[j] && pos[j] >= 0 && pos[j] < p.max_pos;
            if (!__any_sync(kFull, active))
                continue;
            float4 cv, sv;
            half_load_cs(p, h, active, pos[j], cv, sv);
            uint4 out[4];
            q_half_out(h, x[j], r[j], cv, sv, out);
            if (active) {
                uint16_t *dst = p.q + (r0 + 2 * j + half) * kHead + 8 * h;
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    st_stream16_in(dst + 128 * v, out[v], q_span(p), p.err);
            }
        }
    }
}

template <int kStore>
int launch_store(bool kv_norm, unsigned grid, cudaStream_t stream, const KParams &p)
{
    return launch_kernel(kv_norm ? qnorm_rope_kv_insert_half_kernel<kStore, true>
                                 : qnorm_rope_kv_insert_half_kernel<kStore, false>,
                         dim3(grid), dim3(kHalfThreads), 0, stream, p);
}

}  // namespace

int half_ctas_per_sm(int *ctas_per_sm)
{
    // the normalising FP8 kernel is the largest of the four
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
               ctas_per_sm, qnorm_rope_kv_insert_half_kernel<DSV4_STORE_FP8, true>, kHalfThreads,
               0) == cudaSuccess
               ? DSV4_OK
               : DSV4_ERR_CUDA;
}

int half_q_rows_per_warp()
{
    return 2 * kQPairs;
}

int launch_half(int store_mode, const LaunchArgs &a, int64_t ctas, cudaStream_t stream)
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
    const unsigned grid = static_cast<unsigned>(ctas);
    return store_mode == DSV4_STORE_BF16 ? launch_store<DSV4_STORE_BF16>(a.kv_norm, grid, stream, p)
                                         : launch_store<DSV4_STORE_FP8>(a.kv_norm, grid, stream, p);
}

}  // namespace dsv4

DSV4_BOUNDS_FLAG_READER(bounds_flag_half)
