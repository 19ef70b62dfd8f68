// C-ABI layer of libdsv4kv: argument checks, launch planning, status strings.
// Every check here runs on the host before anything is enqueued, so a rejected
// call touches no buffer.  See include/dsv4kv.h for the contract.

#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "dsv4kv.h"
#include "launch.h"
#include "ops.h"

namespace {

bool aligned(const void *p, uintptr_t a)
{
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// Caches hold at most 2^32 slots (more than any one GPU can hold at 132 bytes
// per slot), so the kernels divide 32-bit slot numbers by the block size.
constexpr int64_t kMaxSlots = int64_t(1) << 32;

bool too_many_slots(int64_t num_blocks, int32_t block_size)
{
    return num_blocks > kMaxSlots / block_size;
}

// Per-device cache of (SM count, CTAs of the streaming kernel per SM) for the
// two store modes: immutable properties, filled on first use.
constexpr int kMaxDevices = 64;
std::atomic<int32_t> g_sms[kMaxDevices];
std::atomic<int32_t> g_ctas[kMaxDevices][2];

int device_shape(int store_mode, int32_t *sms, int32_t *ctas)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return DSV4_ERR_CUDA;
    const bool cached = dev >= 0 && dev < kMaxDevices;
    if (cached) {
        *sms = g_sms[dev].load(std::memory_order_relaxed);
        *ctas = g_ctas[dev][store_mode].load(std::memory_order_relaxed);
        if (*sms > 0 && *ctas > 0)
            return DSV4_OK;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        return DSV4_ERR_CUDA;
    int c = 0;
    if (dsv4::stream_ctas_per_sm(store_mode, &c) != DSV4_OK || c < 1)
        return DSV4_ERR_CUDA;
    *sms = n;
    *ctas = c;
    if (cached) {
        g_sms[dev].store(n, std::memory_order_relaxed);
        g_ctas[dev][store_mode].store(c, std::memory_order_relaxed);
    }
    return DSV4_OK;
}

// CTAs per SM of the reader and indexer kernels, cached per device beside the
// SM count; resident = SMs x CTAs per SM, the cap of their persistent grids.
enum { kOccGather = 0, kOccIndexer = 1, kOccKvRows = 2, kOccHalf = 3, kOccIndexerGather = 4,
       kOccKinds = 5 };
std::atomic<int32_t> g_occ[kMaxDevices][kOccKinds];

int resident_ctas(int kind, int64_t *resident)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return DSV4_ERR_CUDA;
    const bool cached = dev >= 0 && dev < kMaxDevices;
    int sms = cached ? g_sms[dev].load(std::memory_order_relaxed) : 0;
    int per = cached ? g_occ[dev][kind].load(std::memory_order_relaxed) : 0;
    if (sms < 1) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            sms < 1)
            return DSV4_ERR_CUDA;
        if (cached)
            g_sms[dev].store(sms, std::memory_order_relaxed);
    }
    if (per < 1) {
        const int rc = kind == kOccGather    ? dsv4::gather_ctas_per_sm(&per)
                       : kind == kOccIndexer ? dsv4::indexer_ctas_per_sm(&per, false)
                       : kind == kOccIndexerGather ? dsv4::indexer_ctas_per_sm(&per, true)
                       : kind == kOccKvRows  ? dsv4::kv_rows_ctas_per_sm(&per)
                                             : dsv4::half_ctas_per_sm(&per);
        if (rc != DSV4_OK || per < 1)
            return DSV4_ERR_CUDA;
        if (cached)
            g_occ[dev][kind].store(per, std::memory_order_relaxed);
    }
    *resident = int64_t(sms) * per;
    return DSV4_OK;
}

// flags of insert()
constexpr int kKvNorm = 1;  // normalise the KV row with the weight
constexpr int kNoQ = 2;     // num_heads may be 0 (KV rows only)

int insert(int store_mode, int variant, int flags, void *q, const void *kv, const void *w,
           const int64_t *positions, const float *cos_sin, int64_t max_position,
           const int64_t *slot_mapping, void *cache, int64_t num_blocks, int32_t block_size,
           int64_t num_tokens, int32_t num_heads, float eps, int32_t *device_error, void *stream)
{
    const bool kv_norm = (flags & kKvNorm) != 0;
    if (store_mode != DSV4_STORE_FP8 && store_mode != DSV4_STORE_BF16)
        return DSV4_ERR_VALUE;
    if (variant != DSV4_VARIANT_AUTO && variant != DSV4_VARIANT_SMALL &&
        variant != DSV4_VARIANT_STREAM && variant != DSV4_VARIANT_HALF)
        return DSV4_ERR_VALUE;
    const int32_t min_heads = (flags & kNoQ) ? 0 : 1;
    if (num_tokens < 0 || num_heads < min_heads || num_blocks < 1 || block_size < 1 ||
        max_position < 1)
        return DSV4_ERR_SHAPE;
    // every byte offset the kernels form must fit in int64
    const int64_t lim = INT64_MAX / 4096;
    if (num_tokens > lim / (int64_t(num_heads) + 1) || too_many_slots(num_blocks, block_size) ||
        max_position > lim)
        return DSV4_ERR_SHAPE;
    if (!(eps >= 0.0f) || !std::isfinite(eps))
        return DSV4_ERR_VALUE;
    if (num_tokens == 0)
        return DSV4_OK;
    if ((num_heads > 0 && !q) || !kv || (kv_norm && !w) || !positions || !cos_sin ||
        !slot_mapping || !cache)
        return DSV4_ERR_NULL;
    const uintptr_t cache_align = store_mode == DSV4_STORE_FP8 ? 8 : 16;
    if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(w, 16) || !aligned(cos_sin, 16) ||
        !aligned(cache, cache_align) || !aligned(positions, 8) || !aligned(slot_mapping, 8) ||
        !aligned(device_error, 4))
        return DSV4_ERR_ALIGN;

    int32_t sms = 0, ctas = 0;
    int st = device_shape(store_mode, &sms, &ctas);
    if (st != DSV4_OK)
        return st;
    if (variant == DSV4_VARIANT_HALF) {
        int64_t resident = 0;
        if (resident_ctas(kOccHalf, &resident) != DSV4_OK)
            return DSV4_ERR_CUDA;
        ctas = static_cast<int32_t>(resident / sms);
    }
    dsv4_plan plan;
    st = dsv4_launch_plan(num_tokens, num_heads, sms, ctas, variant, &plan);
    if (st != DSV4_OK)
        return st;
    if (variant == DSV4_VARIANT_AUTO && plan.variant == DSV4_VARIANT_HALF) {
        // size the grid with the half-warp kernel's own occupancy
        int64_t resident = 0;
        if (resident_ctas(kOccHalf, &resident) != DSV4_OK)
            return DSV4_ERR_CUDA;
        st = dsv4_launch_plan(num_tokens, num_heads, sms, static_cast<int32_t>(resident / sms),
                              DSV4_VARIANT_HALF, &plan);
        if (st != DSV4_OK)
            return st;
    }

    dsv4::LaunchArgs a;
    a.q = static_cast<uint16_t *>(q);
    a.kv = static_cast<const uint16_t *>(kv);
    a.w = static_cast<const uint16_t *>(w);
    a.pos = positions;
    a.cs = cos_sin;
    a.max_pos = max_position;
    a.slot = slot_mapping;
    a.cache = static_cast<uint8_t *>(cache);
    a.num_slots = num_blocks * int64_t(block_size);
    a.block_size = block_size;
    a.num_heads = num_heads;
    a.num_tokens = num_tokens;
    a.eps = eps;
    a.err = device_error;
    a.kv_norm = kv_norm;
    if (plan.variant == DSV4_VARIANT_HALF)
        return dsv4::launch_half(store_mode, a, plan.ctas, static_cast<cudaStream_t>(stream));
    if (num_heads == 0 && plan.variant == DSV4_VARIANT_STREAM) {
        // KV rows only: the quarter-warp-per-row kernel
        int64_t resident = 0;
        if (resident_ctas(kOccKvRows, &resident) != DSV4_OK)
            return DSV4_ERR_CUDA;
        return dsv4::launch_kv_rows(store_mode, a, resident, static_cast<cudaStream_t>(stream));
    }
    return dsv4::launch(store_mode, plan, a, static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

int dsv4_launch_plan(int64_t num_tokens, int32_t num_heads, int32_t sm_count, int32_t ctas_per_sm,
                     int32_t variant, dsv4_plan *plan)
{
    if (!plan)
        return DSV4_ERR_NULL;
    if (num_tokens < 0 || num_heads < 0 || sm_count < 1 || ctas_per_sm < 1)
        return DSV4_ERR_SHAPE;
    if (num_tokens > (INT64_MAX / 4096) / (int64_t(num_heads) + 1))
        return DSV4_ERR_SHAPE;
    const int64_t rows = num_tokens * (int64_t(num_heads) + 1);
    const int stream_warps = dsv4::kStreamThreads / 32;
    const int64_t warp_slots = int64_t(sm_count) * ctas_per_sm * stream_warps;
    if (variant == DSV4_VARIANT_AUTO) {
        // Measured on GB300 (graph-timed, cold L2): with q heads, one row per warp
        // is fastest up to about the warp slots of the stream kernel (10-13% ahead
        // of the half-warp kernel at 0.5K-2K rows, 4% at 3.1K; 18-22% behind from
        // 4.1K); from there the half-warp kernel beats both the others up to 12
        // rounds of the stream kernel's 3-row groups (3-10% ahead of STREAM at
        // 16K-66K rows, a tie near 130K); beyond, the whole-warp stream (2-3% ahead
        // at 264K rows).  With no q heads, STREAM runs the KV-row kernel, whose
        // bulk-copy pipeline costs more to start: SMALL is 8-14% ahead at 1K-3K
        // rows, the KV-row kernel 15-33% ahead from 4K rows, so the switch is at
        // the warp slots there too.
        const int64_t round = warp_slots * dsv4::kStreamRowsPerWarp;
        const int64_t small_below = warp_slots;
        variant = rows < small_below                      ? DSV4_VARIANT_SMALL
                  : num_heads > 0 && rows < 12 * round    ? DSV4_VARIANT_HALF
                                                          : DSV4_VARIANT_STREAM;
    }
    plan->rows = rows;
    if (variant == DSV4_VARIANT_SMALL) {
        const int warps = dsv4::kSmallThreads / 32;
        plan->variant = DSV4_VARIANT_SMALL;
        plan->threads = dsv4::kSmallThreads;
        plan->rows_per_warp = 1;
        plan->ctas = rows > 0 ? (rows + warps - 1) / warps : 1;
        if (plan->ctas > INT32_MAX)
            return DSV4_ERR_SHAPE;
    } else if (variant == DSV4_VARIANT_STREAM) {
        // with no q heads the KV-row kernel runs: same CTA size, its own rows per warp
        const int per_warp = num_heads == 0 ? dsv4::kv_rows_per_warp() : dsv4::kStreamRowsPerWarp;
        const int64_t groups = (rows + per_warp - 1) / per_warp;
        const int64_t need = (groups + stream_warps - 1) / stream_warps;
        const int64_t resident = int64_t(sm_count) * ctas_per_sm;
        plan->variant = DSV4_VARIANT_STREAM;
        plan->threads = dsv4::kStreamThreads;
        plan->rows_per_warp = per_warp;
        plan->ctas = need < resident ? (need > 0 ? need : 1) : resident;
    } else if (variant == DSV4_VARIANT_HALF) {
        const int64_t per_warp = dsv4::half_q_rows_per_warp();
        const int64_t items = (num_tokens + 1) / 2 + (num_tokens * num_heads + per_warp - 1) / per_warp;
        const int64_t need = (items + stream_warps - 1) / stream_warps;
        const int64_t resident = int64_t(sm_count) * ctas_per_sm;
        plan->variant = DSV4_VARIANT_HALF;
        plan->threads = dsv4::kStreamThreads;
        plan->rows_per_warp = static_cast<int32_t>(per_warp);
        plan->ctas = need < resident ? (need > 0 ? need : 1) : resident;
    } else {
        return DSV4_ERR_VALUE;
    }
    return DSV4_OK;
}

int dsv4_qnorm_rope_kv_quant_insert(void *q, const void *kv, const void *kv_norm_weight,
                                    const int64_t *positions, const float *cos_sin_cache,
                                    int64_t max_position, const int64_t *slot_mapping,
                                    uint8_t *kv_cache, int64_t num_blocks, int32_t block_size,
                                    int64_t num_tokens, int32_t num_heads, float eps,
                                    int32_t *device_error, void *stream)
{
    return insert(DSV4_STORE_FP8, DSV4_VARIANT_AUTO, kKvNorm, q, kv, kv_norm_weight, positions,
                  cos_sin_cache, max_position, slot_mapping, kv_cache, num_blocks, block_size,
                  num_tokens, num_heads, eps, device_error, stream);
}

int dsv4_qnorm_rope_kv_bf16_insert(void *q, const void *kv, const void *kv_norm_weight,
                                   const int64_t *positions, const float *cos_sin_cache,
                                   int64_t max_position, const int64_t *slot_mapping,
                                   void *kv_cache, int64_t num_blocks, int32_t block_size,
                                   int64_t num_tokens, int32_t num_heads, float eps,
                                   int32_t *device_error, void *stream)
{
    return insert(DSV4_STORE_BF16, DSV4_VARIANT_AUTO, kKvNorm, q, kv, kv_norm_weight, positions,
                  cos_sin_cache, max_position, slot_mapping, kv_cache, num_blocks, block_size,
                  num_tokens, num_heads, eps, device_error, stream);
}

int dsv4_qnorm_rope_kv_insert_variant(int store_mode, int variant, void *q, const void *kv,
                                      const void *kv_norm_weight, const int64_t *positions,
                                      const float *cos_sin_cache, int64_t max_position,
                                      const int64_t *slot_mapping, void *kv_cache,
                                      int64_t num_blocks, int32_t block_size, int64_t num_tokens,
                                      int32_t num_heads, float eps, int32_t *device_error,
                                      void *stream)
{
    return insert(store_mode, variant, kKvNorm, q, kv, kv_norm_weight, positions, cos_sin_cache,
                  max_position, slot_mapping, kv_cache, num_blocks, block_size, num_tokens,
                  num_heads, eps, device_error, stream);
}

int dsv4_qnorm_rope_kv_rope_quant_insert(void *q, const void *kv, const int64_t *positions,
                                         const float *cos_sin_cache, int64_t max_position,
                                         const int64_t *slot_mapping, uint8_t *kv_cache,
                                         int64_t num_blocks, int32_t block_size,
                                         int64_t num_tokens, int32_t num_heads, float eps,
                                         int32_t *device_error, void *stream)
{
    return insert(DSV4_STORE_FP8, DSV4_VARIANT_AUTO, 0, q, kv, nullptr, positions,
                  cos_sin_cache, max_position, slot_mapping, kv_cache, num_blocks, block_size,
                  num_tokens, num_heads, eps, device_error, stream);
}

int dsv4_kv_norm_rope_insert(int store_mode, const void *kv, const void *kv_norm_weight,
                             const int64_t *positions, const float *cos_sin_cache,
                             int64_t max_position, const int64_t *slot_mapping, void *kv_cache,
                             int64_t num_blocks, int32_t block_size, int64_t num_tokens,
                             float eps, int32_t *device_error, void *stream)
{
    return insert(store_mode, DSV4_VARIANT_AUTO, kKvNorm | kNoQ, nullptr, kv, kv_norm_weight,
                  positions, cos_sin_cache, max_position, slot_mapping, kv_cache, num_blocks,
                  block_size, num_tokens, 0, eps, device_error, stream);
}

int dsv4_insert_ex(int store_mode, int variant, int kv_norm, void *q, const void *kv,
                   const void *kv_norm_weight, const int64_t *positions,
                   const float *cos_sin_cache, int64_t max_position, const int64_t *slot_mapping,
                   void *kv_cache, int64_t num_blocks, int32_t block_size, int64_t num_tokens,
                   int32_t num_heads, float eps, int32_t *device_error, void *stream)
{
    if (kv_norm != 0 && kv_norm != 1)
        return DSV4_ERR_VALUE;
    return insert(store_mode, variant, (kv_norm ? kKvNorm : 0) | kNoQ, q, kv, kv_norm_weight,
                  positions, cos_sin_cache, max_position, slot_mapping, kv_cache, num_blocks,
                  block_size, num_tokens, num_heads, eps, device_error, stream);
}

int dsv4_dequant_gather(const uint8_t *kv_cache, int64_t num_blocks, int32_t block_size,
                        const int64_t *slots, int64_t num_rows, void *out,
                        int32_t *device_error, void *stream)
{
    if (num_rows < 0 || num_blocks < 1 || block_size < 1)
        return DSV4_ERR_SHAPE;
    if (too_many_slots(num_blocks, block_size) || num_rows > INT64_MAX / 4096)
        return DSV4_ERR_SHAPE;
    if (num_rows == 0)
        return DSV4_OK;
    if (!kv_cache || !slots || !out)
        return DSV4_ERR_NULL;
    if (!aligned(kv_cache, 8) || !aligned(slots, 8) || !aligned(out, 16) ||
        !aligned(device_error, 4))
        return DSV4_ERR_ALIGN;
    int64_t resident = 0;
    if (resident_ctas(kOccGather, &resident) != DSV4_OK)
        return DSV4_ERR_CUDA;
    const int64_t groups = (num_rows + dsv4::gather_rows_per_warp() - 1) /
                           dsv4::gather_rows_per_warp();
    const int64_t warps = dsv4::gather_warps_per_cta();
    const int64_t need = (groups + warps - 1) / warps;
    return dsv4::launch_gather(kv_cache, num_blocks, block_size, slots, num_rows,
                               static_cast<uint16_t *>(out), device_error,
                               need < resident ? need : resident,
                               static_cast<cudaStream_t>(stream));
}

size_t dsv4_mxfp8_scale_bytes(int64_t num_rows, int32_t hidden)
{
    if (num_rows < 0 || hidden < 128 || hidden % 128 != 0)
        return 0;
    return size_t((num_rows + 127) / 128 * 128) * size_t(hidden / 32);
}

int dsv4_add_gemma_rmsnorm_mxfp8(const void *x, const void *residual, const void *gamma,
                                 int64_t num_rows, int32_t hidden, float eps, void *residual_out,
                                 uint8_t *codes, uint8_t *scales, void *stream)
{
    if (num_rows < 0 || hidden < 128 || hidden > 16384 || hidden % 128 != 0)
        return DSV4_ERR_SHAPE;
    if (num_rows > (INT64_MAX / 4096) / hidden || num_rows > INT32_MAX - 128)
        return DSV4_ERR_SHAPE;
    if (!(eps >= 0.0f) || !std::isfinite(eps))
        return DSV4_ERR_VALUE;
    if (num_rows == 0)
        return DSV4_OK;
    if (!x || !residual || !gamma || !residual_out || !codes || !scales)
        return DSV4_ERR_NULL;
    if (!aligned(x, 16) || !aligned(residual, 16) || !aligned(gamma, 16) ||
        !aligned(residual_out, 16) || !aligned(codes, 8))
        return DSV4_ERR_ALIGN;
    return dsv4::launch_gemma_rmsnorm_mxfp8(
        static_cast<const uint16_t *>(x), static_cast<const uint16_t *>(residual),
        static_cast<const uint16_t *>(gamma), num_rows, hidden, eps,
        static_cast<uint16_t *>(residual_out), codes, scales, static_cast<cudaStream_t>(stream));
}

int dsv4_indexer_k_quant_insert(const void *k, const int64_t *slot_mapping,
                                uint8_t *indexer_cache, int64_t num_blocks, int32_t block_size,
                                int64_t num_tokens, int32_t *device_error, void *stream)
{
    if (num_tokens < 0 || num_blocks < 1 || block_size < 1)
        return DSV4_ERR_SHAPE;
    if (too_many_slots(num_blocks, block_size) || num_tokens > INT64_MAX / 4096)
        return DSV4_ERR_SHAPE;
    if (num_tokens == 0)
        return DSV4_OK;
    if (!k || !slot_mapping || !indexer_cache)
        return DSV4_ERR_NULL;
    if (!aligned(k, 16) || !aligned(slot_mapping, 8) || !aligned(indexer_cache, 4) ||
        !aligned(device_error, 4))
        return DSV4_ERR_ALIGN;
    int64_t resident = 0;
    if (resident_ctas(kOccIndexer, &resident) != DSV4_OK)
        return DSV4_ERR_CUDA;
    return dsv4::launch_indexer_insert(static_cast<const uint16_t *>(k), slot_mapping,
                                       indexer_cache, num_blocks, block_size, num_tokens,
                                       device_error, resident, static_cast<cudaStream_t>(stream));
}

int dsv4_indexer_k_gather(const uint8_t *indexer_cache, int64_t num_blocks, int32_t block_size,
                          const int64_t *slots, int64_t num_rows, uint8_t *k_out,
                          float *scale_out, int32_t *device_error, void *stream)
{
    if (num_rows < 0 || num_blocks < 1 || block_size < 1)
        return DSV4_ERR_SHAPE;
    if (too_many_slots(num_blocks, block_size) || num_rows > INT64_MAX / 4096)
        return DSV4_ERR_SHAPE;
    if (num_rows == 0)
        return DSV4_OK;
    if (!indexer_cache || !slots || !k_out || !scale_out)
        return DSV4_ERR_NULL;
    if (!aligned(indexer_cache, 4) || !aligned(slots, 8) || !aligned(k_out, 8) ||
        !aligned(scale_out, 4) || !aligned(device_error, 4))
        return DSV4_ERR_ALIGN;
    int64_t resident = 0;
    if (resident_ctas(kOccIndexerGather, &resident) != DSV4_OK)
        return DSV4_ERR_CUDA;
    return dsv4::launch_indexer_gather(indexer_cache, num_blocks, block_size, slots, num_rows,
                                       k_out, scale_out, device_error, resident,
                                       static_cast<cudaStream_t>(stream));
}

size_t dsv4_indexer_cache_bytes(int64_t num_blocks, int32_t block_size)
{
    if (num_blocks < 1 || block_size < 1)
        return 0;
    return size_t(num_blocks) * size_t(block_size) * DSV4_INDEXER_SLOT_BYTES;
}

size_t dsv4_fp8_cache_bytes(int64_t num_blocks, int32_t block_size)
{
    if (num_blocks < 1 || block_size < 1)
        return 0;
    return size_t(num_blocks) * size_t(block_size) * DSV4_FP8_SLOT_BYTES;
}

size_t dsv4_bf16_cache_bytes(int64_t num_blocks, int32_t block_size)
{
    if (num_blocks < 1 || block_size < 1)
        return 0;
    return size_t(num_blocks) * size_t(block_size) * DSV4_BF16_SLOT_BYTES;
}

int dsv4_check_bounded_wait(int64_t max_cycles, int32_t *device_error, void *stream)
{
    if (max_cycles < 0)
        return DSV4_ERR_VALUE;
    return dsv4::launch_wait_check(max_cycles, device_error, static_cast<cudaStream_t>(stream));
}

int dsv4_debug_bounds_flags(int reset)
{
    int (*const readers[])(int) = {dsv4::bounds_flag_fused, dsv4::bounds_flag_half,
                                   dsv4::bounds_flag_kv_rows, dsv4::bounds_flag_gather,
                                   dsv4::bounds_flag_indexer, dsv4::bounds_flag_mxfp8};
    int flags = 0;
    for (auto read : readers) {
        const int v = read(reset);
        if (v < 0)
            return v;  // -1: the release build, which records nothing; else a CUDA failure
        flags |= v;
    }
    return flags;
}

const char *dsv4_status_string(int status)
{
    switch (status) {
    case DSV4_OK: return "ok";
    case DSV4_ERR_NULL: return "null pointer argument";
    case DSV4_ERR_SHAPE: return "size out of range";
    case DSV4_ERR_ALIGN: return "misaligned pointer argument";
    case DSV4_ERR_VALUE: return "invalid value (eps, store mode or variant)";
    case DSV4_ERR_CUDA: return "CUDA runtime error at launch";
    default: return "unknown status";
    }
}

}  // extern "C"
