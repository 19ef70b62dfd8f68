// Internal interface between the C-ABI layer (api.cpp) and the kernels of the
// operations beside the whole-warp fused kernels: the half-warp fused kernel
// (qnorm_rope_kv_insert_half.cu), the KV-row kernel for calls with no q
// (kv_rows.cu), the MXFP8 activation quantiser (gemma_rmsnorm_mxfp8.cu), the
// indexer-K insert and gather (indexer_k.cu) and the check of the bounded waits
// (wait_check.cu).
// Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "dsv4kv.h"
#include "launch.h"

namespace dsv4 {

// KV rows with no q, one row per quarter-warp (kv_rows.cu); the grid is capped at max_ctas.
int kv_rows_ctas_per_sm(int *ctas_per_sm);
int kv_rows_per_warp();
int launch_kv_rows(int store_mode, const LaunchArgs &a, int64_t max_ctas, cudaStream_t stream);

// Warps per CTA of the FP8 cache reader (dequant_gather.cu; its other entry points
// are in launch.h).
int gather_warps_per_cta();

// The fused step with one row per half-warp (qnorm_rope_kv_insert_half.cu).
int half_ctas_per_sm(int *ctas_per_sm);
int half_q_rows_per_warp();
int launch_half(int store_mode, const LaunchArgs &a, int64_t ctas, cudaStream_t stream);

// Residual add + Gemma RMSNorm + MXFP8 rows.
int launch_gemma_rmsnorm_mxfp8(const uint16_t *x, const uint16_t *residual, const uint16_t *gamma,
                               int64_t m, int32_t n, float eps, uint16_t *residual_out,
                               uint8_t *codes, uint8_t *scales, cudaStream_t stream);

// Indexer-K quant-insert and gather; grids are capped at max_ctas.
int indexer_ctas_per_sm(int *ctas_per_sm, bool gather);
int launch_indexer_insert(const uint16_t *k, const int64_t *slots, uint8_t *cache,
                          int64_t num_blocks, int32_t block_size, int64_t rows, int32_t *err,
                          int64_t max_ctas, cudaStream_t stream);
int launch_indexer_gather(const uint8_t *cache, int64_t num_blocks, int32_t block_size,
                          const int64_t *slots, int64_t rows, uint8_t *k_out, float *scale_out,
                          int32_t *err, int64_t max_ctas, cudaStream_t stream);

// One warp waits on an mbarrier nothing completes, for at most max_cycles SM
// cycles (clamped to the kernels' own limit), then flags DSV4_DEVERR_TIMEOUT.
int launch_wait_check(int64_t max_cycles, int32_t *err, cudaStream_t stream);

// The checked build's record of skipped accesses, one reader per kernel file
// (DSV4_BOUNDS_FLAG_READER of bounds.cuh); -1 in the release build.
int bounds_flag_fused(int reset);
int bounds_flag_half(int reset);
int bounds_flag_kv_rows(int reset);
int bounds_flag_gather(int reset);
int bounds_flag_indexer(int reset);
int bounds_flag_mxfp8(int reset);

}  // namespace dsv4
