// KV rows with no q (SGLang PR #33358, "Motivation": fused_norm_rope_flashmla,
// the RMSNorm + RoPE + paged-cache store of the latent KV row alone): the same
// arithmetic as the KV rows of the fused kernel, laid out for rows that carry
// all the work.
//
// In the fused kernel a KV row is one of H + 1 rows of a token and takes a
// whole warp.  Alone, such rows are issue-bound: ~390 warp instructions per
// row, much of it per-row overhead (reductions over 32 lanes, both sides of
// the rope branch, the scale word, address arithmetic) rather than per-element
// work.  Here half a warp owns a row (the layout of halfrow.cuh), so every warp
// instruction serves two rows, and the cache bytes stay identical to the
// fused kernel's.  A warp item is one row pair; 2-8 rows per warp, and 2-4 CTAs
// per SM, measured within 5% of this.

#include <cuda_runtime.h>
#include <stdint.h>

#include "halfrow.cuh"
#include "launch_status.h"
#include "ops.h"

namespace dsv4 {
namespace {

constexpr int kKvThreads = 256;

template <int kStore, bool kKvNorm>
__global__ void __launch_bounds__(kKvThreads, 3) kv_rows_kernel(const KParams p)
{
    __shared__ float4 w_smem[128];
    if (kKvNorm) {
        for (int i = threadIdx.x; i < 64; i += kKvThreads)
            stage_weight(p.w, i, w_smem);
        __syncthreads();
    }
    const int lane = threadIdx.x & 31, h = lane & 15, half = lane >> 4;
    const int64_t pairs = (p.num_tokens + 1) / 2;
    const int64_t stride = int64_t(gridDim.x) * (kKvThreads / 32);
    for (int64_t g = int64_t(blockIdx.x) * (kKvThreads / 32) + (threadIdx.x >> 5); g < pairs;
         g += stride)
        kv_pair_item<kStore, kKvNorm>(p, h, 2 * g + half, w_smem);
}

template <int kStore>
int launch_store(bool kv_norm, unsigned grid, cudaStream_t stream, const KParams &p)
{
    return launch_kernel(kv_norm ? kv_rows_kernel<kStore, true> : kv_rows_kernel<kStore, false>,
                         dim3(grid), dim3(kKvThreads), 0, stream, p);
}

}  // namespace

int kv_rows_ctas_per_sm(int *ctas_per_sm)
{
    // the normalising FP8 kernel is the largest of the four
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
               ctas_per_sm, kv_rows_kernel<DSV4_STORE_FP8, true>, kKvThreads, 0) == cudaSuccess
               ? DSV4_OK
               : DSV4_ERR_CUDA;
}

int kv_rows_per_warp()
{
    return 2;
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
    const int64_t pairs = (a.num_tokens + 1) / 2;
    const int64_t need = (pairs + kKvThreads / 32 - 1) / (kKvThreads / 32);
    const unsigned grid = static_cast<unsigned>(need < max_ctas ? need : max_ctas);
    return store_mode == DSV4_STORE_BF16 ? launch_store<DSV4_STORE_BF16>(a.kv_norm, grid, stream, p)
                                         : launch_store<DSV4_STORE_FP8>(a.kv_norm, grid, stream, p);
}

}  // namespace dsv4
