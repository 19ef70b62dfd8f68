// Internal interface between the C-ABI layer (api.cpp) and the whole-warp
// fused kernels (qnorm_rope_kv_insert.cu), plus
// the kernel arguments every fused kernel takes.  Not installed; not part of
// the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "dsv4kv.h"
#include "fastdiv.h"

namespace dsv4 {

// Rows each warp of the streaming variant loads before it computes any.
constexpr int kStreamRowsPerWarp = 3;
constexpr int kStreamThreads = 256;
constexpr int kSmallThreads = 64;

struct LaunchArgs {
    uint16_t *q;
    const uint16_t *kv;
    const uint16_t *w;
    const int64_t *pos;
    const float *cs;
    int64_t max_pos;
    const int64_t *slot;
    uint8_t *cache;
    int64_t num_slots;
    int32_t block_size;
    int32_t num_heads;
    int64_t num_tokens;
    float eps;
    int32_t *err;
    bool kv_norm;  // false: the KV rows arrive normalised (no norm, no weight)
};

// Kernel arguments (device pointers and sizes), shared by every kernel variant.
struct KParams {
    uint16_t *q;
    const uint16_t *kv;
    const uint16_t *w;
    const int64_t *pos;
    const float *cs;
    int64_t max_pos;
    const int64_t *slot;
    uint8_t *cache;
    int64_t num_slots;
    int64_t num_tokens;
    int32_t block_size;
    int32_t num_heads;
    float eps;
    int32_t *err;
    uint64_t slot_div;  // fastdiv_magic(block_size): slot / block_size by one multiply
};

// CTAs of the streaming kernel for `store_mode` that fit on one SM.
int stream_ctas_per_sm(int store_mode, int *ctas_per_sm);

// Enqueue the kernel described by `plan` on `stream`; returns a dsv4_status.
int launch(int store_mode, const dsv4_plan &plan, const LaunchArgs &args, cudaStream_t stream);

// The FP8 cache reader (dequant_gather.cu).
int gather_ctas_per_sm(int *ctas_per_sm);
int gather_rows_per_warp();
int launch_gather(const uint8_t *cache, int64_t num_blocks, int32_t block_size,
                  const int64_t *slots, int64_t rows, uint16_t *out, int32_t *err, int64_t ctas,
                  cudaStream_t stream);

}  // namespace dsv4
