// Indexer-K quant-insert and gather.  The lightning indexer scores queries
// against K rows held as E4M3 with one non-negative fp32 scale per 128-dim row
// (rocm-aiter PR #1, "Motivation": q_fp8 against k_fp8 [N, 128] with kv_scale
// [N], gathered out of the paged cache first); the norm-rope-store kernel keeps
// this indexer path beside the KV one (SGLang PR #33358, "Modifications").
//
// Insert, per token t with 0 <= slot < num_slots:
//   amax  = max |k[t, :]|                          (exact: k is bf16)
//   s     = smallest integer with amax <= 448 * 2^s, clamped to [-127, 127]
//   codes = E4M3_rn_satfinite(k[t, :] * 2^-s)      (an exact power-of-two scaling)
//   scale = 2^s as fp32 (2^-127 is the fp32 subnormal 0x00400000)
// written at block b = slot / bs, offset o: codes at b*bs*132 + o*128, scale at
// b*bs*132 + bs*128 + o*4.  A negative slot writes nothing; a slot past the
// cache writes nothing and raises DSV4_DEVERR_SLOT_RANGE.
// Gather: codes and scale of slots[n] copied to k_out[n, :] and scale_out[n];
// zeros for a negative slot, zeros and DSV4_DEVERR_SLOT_RANGE past the cache.
//
// Both are HBM-bound copies with a little integer work.  Half a warp holds one
// row (lane h: dims [8h, 8h + 8), one 16-byte load of k), so one warp-wide load
// reads two adjacent rows, 512 contiguous bytes.  The scale needs no floating
// point: for non-negative bf16 bit patterns integer order is magnitude order,
// so amax is an integer max of (bits & 0x7fff), and with amax = (1 + m/128) *
// 2^(E - 127), s = E - 135 + (m > 0x60) (the mantissa above 1.75 = 448 / 256).
// Both kernels are software-pipelined in registers: a warp's next group of
// row pairs is loaded before it stores the current one.

#include <cuda_runtime.h>
#include <stdint.h>

#include "convert.cuh"
#include "bounds.cuh"
#include "fastdiv.h"
#include "launch_status.h"
#include "ops.h"

namespace dsv4 {
namespace {

constexpr int kDim = DSV4_INDEXER_DIM;                // 128 dims, 256 bf16 bytes
constexpr int kSlotBytes = DSV4_INDEXER_SLOT_BYTES;   // 128 codes + 4 scale bytes
constexpr int kPairs = 2;  // row pairs per insert group: 1, 2, 4 measured, 2 best (48 registers)
constexpr int kThreads = 256;
constexpr unsigned kFull = 0xffffffffu;

struct IParams {
    const uint16_t *k;        // insert input, bf16 [rows, 128]
    const uint8_t *src;       // gather input: the indexer cache
    uint8_t *cache;           // insert output
    uint8_t *k_out;           // gather outputs
    float *scale_out;
    const int64_t *slots;
    int64_t rows;
    int64_t num_slots;
    int32_t block_size;
    int32_t *err;
    uint64_t slot_div;  // fastdiv_magic(block_size)
};

// the buffers of a launch, for the checked build's bounds tests (bounds.cuh)
__device__ __forceinline__ Span k_span(const IParams &p)
{
    return Span{p.k, uint64_t(p.rows) * kDim * 2u};
}
__device__ __forceinline__ Span slots_span(const IParams &p)
{
    return Span{p.slots, uint64_t(p.rows) * 8u};
}
__device__ __forceinline__ Span icache_span(const void *cache, const IParams &p)
{
    return Span{cache, uint64_t(p.num_slots) * kSlotBytes};
}
__device__ __forceinline__ Span kout_span(const IParams &p)
{
    return Span{p.k_out, uint64_t(p.rows) * kDim};
}
__device__ __forceinline__ Span sout_span(const IParams &p)
{
    return Span{p.scale_out, uint64_t(p.rows) * 4u};
}

// the 8 codes of one lane: E4M3(x * inv) for the 8 bf16 of v
__device__ __forceinline__ uint2 encode8(uint4 v, float inv)
{
    float f[8];
    widen8(v, f);
    return make_uint2(e4m3x4_rn(__fmul_rn(f[0], inv), __fmul_rn(f[1], inv), __fmul_rn(f[2], inv),
                                __fmul_rn(f[3], inv)),
                      e4m3x4_rn(__fmul_rn(f[4], inv), __fmul_rn(f[5], inv), __fmul_rn(f[6], inv),
                                __fmul_rn(f[7], inv)));
}

// the scale exponent s of a row from the bits of its amax (bf16, sign cleared)
__device__ __forceinline__ int row_exponent(uint32_t amax_bits)
{
    const int e = int(amax_bits >> 7), m = int(amax_bits & 0x7fu);
    const int s = e == 0 ? -127 : e - 135 + (m > 0x60 ? 1 : 0);
    return s < -127 ? -127 : (s > 127 ? 127 : s);
}

template <bool kWide>
__device__ __forceinline__ void store_codes(uint8_t *p, uint2 c, Span s, int32_t *err)
{
    if (!in_span(p, 8, s, err))
        return;
    if (kWide) {
        __stcs(reinterpret_cast<uint2 *>(p), c);
    } else {
        __stcs(reinterpret_cast<unsigned *>(p), c.x);
        __stcs(reinterpret_cast<unsigned *>(p + 4), c.y);
    }
}

template <bool kWide>
__device__ __forceinline__ uint2 load_codes(const uint8_t *p, Span s, int32_t *err)
{
    if (!in_span(p, 8, s, err))
        return make_uint2(0u, 0u);
    if (kWide)
        return __ldcs(reinterpret_cast<const uint2 *>(p));
    return make_uint2(__ldcs(reinterpret_cast<const unsigned *>(p)),
                      __ldcs(reinterpret_cast<const unsigned *>(p + 4)));
}

// The insert, software-pipelined in registers: a warp takes groups of kPairs
// row pairs (one row per half) and loads the next group's rows and slots
// before it quantises and stores the current one.
__device__ __forceinline__ void insert_load(const IParams &p, int64_t g, int half, int h,
                                            int64_t *slot, uint4 *x)
{
#pragma unroll
    for (int j = 0; j < kPairs; ++j) {
        const int64_t t = g * 2 * kPairs + half + 2 * j;
        slot[j] = t < p.rows ? ldg_i64_in(p.slots + t, slots_span(p), p.err) : -1;
        x[j] = t < p.rows ? ld_stream16_in(reinterpret_cast<const uint4 *>(p.k + t * kDim) + h,
                                           k_span(p), p.err)
                          : make_uint4(0u, 0u, 0u, 0u);
    }
}

// kWide: every code row starts on an 8-byte boundary (the cache is 8-byte
// aligned and the block size even), so each lane stores its 8 codes at once
template <bool kWide>
__device__ __forceinline__ void insert_store(const IParams &p, int h, const int64_t *slot,
                                             const uint4 *x)
{
#pragma unroll
    for (int j = 0; j < kPairs; ++j) {
        const uint32_t m2 = __vmaxu2(__vmaxu2(x[j].x & 0x7fff7fffu, x[j].y & 0x7fff7fffu),
                                     __vmaxu2(x[j].z & 0x7fff7fffu, x[j].w & 0x7fff7fffu));
        uint32_t amax = max(m2 & 0xffffu, m2 >> 16);
#pragma unroll
        for (int o = 1; o < 16; o <<= 1)  // xor below 16 stays inside the half-warp
            amax = max(amax, __shfl_xor_sync(kFull, amax, o));
        if (slot[j] < 0)
            continue;
        if (slot[j] >= p.num_slots) {
            if (h == 0 && p.err != nullptr)
                atomicOr(p.err, DSV4_DEVERR_SLOT_RANGE);
            continue;
        }
        const int s = row_exponent(amax);
        const float inv = __uint_as_float(uint32_t(127 - s) << 23);  // 2^-s, normal
        const int64_t blk = fastdiv(static_cast<uint32_t>(slot[j]), p.slot_div);
        const int64_t off = slot[j] - blk * p.block_size;
        uint8_t *base = p.cache + blk * int64_t(p.block_size) * kSlotBytes;
        store_codes<kWide>(base + off * kDim + 8 * h, encode8(x[j], inv), icache_span(p.cache, p),
                           p.err);
        if (h == 0)
            st_stream4_in(base + int64_t(p.block_size) * kDim + off * 4,
                          s > -127 ? uint32_t(s + 127) << 23 : 0x00400000u, icache_span(p.cache, p),
                          p.err);
    }
}

template <bool kWide>
__global__ void __launch_bounds__(kThreads) indexer_k_insert_kernel(const IParams p)
{
    const int lane = threadIdx.x & 31, half = lane >> 4, h = lane & 15;
    const int64_t warps = int64_t(gridDim.x) * (kThreads / 32);
    const int64_t groups = (p.rows + 2 * kPairs - 1) / (2 * kPairs);
    int64_t g = int64_t(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
    if (g >= groups)
        return;
    int64_t slot[kPairs];
    uint4 x[kPairs];
    insert_load(p, g, half, h, slot, x);
    for (; g < groups; g += warps) {
        int64_t slot_n[kPairs];
        uint4 x_n[kPairs];
        insert_load(p, g + warps, half, h, slot_n, x_n);  // nothing is read past the end
        insert_store<kWide>(p, h, slot, x);
#pragma unroll
        for (int j = 0; j < kPairs; ++j) {
            slot[j] = slot_n[j];
            x[j] = x_n[j];
        }
    }
}

// The gather, software-pipelined in registers: a warp takes groups of
// kGatherPairs row pairs (one row per half) and keeps the next group's loads
// in flight while it stores the current one; the slot ids are loaded two
// groups ahead, the codes and scales one group ahead.
constexpr int kGatherPairs = 2;  // 1-4 measured: 2 best (48 registers)

__device__ __forceinline__ void gather_slots(const IParams &p, int64_t g, int half, int64_t *slot)
{
#pragma unroll
    for (int j = 0; j < kGatherPairs; ++j) {
        const int64_t n = g * 2 * kGatherPairs + half + 2 * j;
        slot[j] = n < p.rows ? ldg_i64_in(p.slots + n, slots_span(p), p.err) : -1;
    }
}

template <bool kWide>
__device__ __forceinline__ void gather_load(const IParams &p, int h, const int64_t *slot, uint2 *c,
                                            unsigned *sc)
{
#pragma unroll
    for (int j = 0; j < kGatherPairs; ++j) {
        c[j] = make_uint2(0u, 0u);
        sc[j] = 0u;
        if (slot[j] >= 0 && slot[j] < p.num_slots) {
            const int64_t blk = fastdiv(static_cast<uint32_t>(slot[j]), p.slot_div);
            const int64_t off = slot[j] - blk * p.block_size;
            const uint8_t *base = p.src + blk * int64_t(p.block_size) * kSlotBytes;
            c[j] = load_codes<kWide>(base + off * kDim + 8 * h, icache_span(p.src, p), p.err);
            const uint8_t *sp = base + int64_t(p.block_size) * kDim + off * 4;
            if (h == 0 && in_span(sp, 4, icache_span(p.src, p), p.err))
                sc[j] = __ldcs(reinterpret_cast<const unsigned *>(sp));
        }
    }
}

__device__ __forceinline__ void gather_store(const IParams &p, int h, int half, int64_t g,
                                             const int64_t *slot, const uint2 *c, const unsigned *sc)
{
#pragma unroll
    for (int j = 0; j < kGatherPairs; ++j) {
        const int64_t n = g * 2 * kGatherPairs + half + 2 * j;
        if (n >= p.rows)
            continue;
        if (slot[j] >= p.num_slots && h == 0 && p.err != nullptr)
            atomicOr(p.err, DSV4_DEVERR_SLOT_RANGE);
        st_stream8_in(reinterpret_cast<uint2 *>(p.k_out + n * kDim) + h, c[j], kout_span(p), p.err);
        if (h == 0)
            st_stream4_in(reinterpret_cast<unsigned *>(p.scale_out) + n, sc[j], sout_span(p), p.err);
    }
}

template <bool kWide>
__global__ void __launch_bounds__(kThreads) indexer_k_gather_kernel(const IParams p)
{
    const int lane = threadIdx.x & 31, half = lane >> 4, h = lane & 15;
    const int64_t warps = int64_t(gridDim.x) * (kThreads / 32);
    const int64_t groups = (p.rows + 2 * kGatherPairs - 1) / (2 * kGatherPairs);
    int64_t g = int64_t(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
    if (g >= groups)
        return;
    int64_t slot[kGatherPairs], ahead[kGatherPairs];
    uint2 c[kGatherPairs];
    unsigned sc[kGatherPairs];
    gather_slots(p, g, half, slot);
    gather_load<kWide>(p, h, slot, c, sc);
    gather_slots(p, g + warps, half, ahead);
    for (; g < groups; g += warps) {
        int64_t slot_n[kGatherPairs];
        uint2 c_n[kGatherPairs];
        unsigned sc_n[kGatherPairs];
#pragma unroll
        for (int j = 0; j < kGatherPairs; ++j)
            slot_n[j] = ahead[j];
        gather_load<kWide>(p, h, slot_n, c_n, sc_n);  // nothing is read past the end
        gather_slots(p, g + 2 * warps, half, ahead);
        gather_store(p, h, half, g, slot, c, sc);
#pragma unroll
        for (int j = 0; j < kGatherPairs; ++j) {
            slot[j] = slot_n[j];
            c[j] = c_n[j];
            sc[j] = sc_n[j];
        }
    }
}

int64_t grid_for(int64_t rows, int64_t max_ctas, int pairs)
{
    const int64_t groups = (rows + 2 * pairs - 1) / (2 * pairs);
    const int64_t need = (groups + kThreads / 32 - 1) / (kThreads / 32);
    return need < max_ctas ? need : max_ctas;
}

}  // namespace

int indexer_ctas_per_sm(int *ctas_per_sm, bool gather)
{
    // each kernel's two forms use the same block size; take the smaller occupancy
    int a = 0, b = 0;
    const bool ok =
        gather ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, indexer_k_gather_kernel<true>, kThreads, 0) == cudaSuccess &&
                     cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, indexer_k_gather_kernel<false>, kThreads, 0) == cudaSuccess
               : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, indexer_k_insert_kernel<true>, kThreads, 0) == cudaSuccess &&
                     cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, indexer_k_insert_kernel<false>, kThreads, 0) == cudaSuccess;
    if (!ok)
        return DSV4_ERR_CUDA;
    *ctas_per_sm = min(a, b);
    return DSV4_OK;
}

int launch_indexer_insert(const uint16_t *k, const int64_t *slots, uint8_t *cache,
                          int64_t num_blocks, int32_t block_size, int64_t rows, int32_t *err,
                          int64_t max_ctas, cudaStream_t stream)
{
    IParams p = {};
    p.k = k;
    p.cache = cache;
    p.slots = slots;
    p.rows = rows;
    p.num_slots = num_blocks * int64_t(block_size);
    p.block_size = block_size;
    p.slot_div = fastdiv_magic(static_cast<uint32_t>(block_size));
    p.err = err;
    const unsigned grid = static_cast<unsigned>(grid_for(rows, max_ctas, kPairs));
    const bool wide = (reinterpret_cast<uintptr_t>(cache) & 7u) == 0 && block_size % 2 == 0;
    return launch_kernel(wide ? indexer_k_insert_kernel<true> : indexer_k_insert_kernel<false>,
                         dim3(grid), dim3(kThreads), 0, stream, p);
}

int launch_indexer_gather(const uint8_t *cache, int64_t num_blocks, int32_t block_size,
                          const int64_t *slots, int64_t rows, uint8_t *k_out, float *scale_out,
                          int32_t *err, int64_t max_ctas, cudaStream_t stream)
{
    IParams p = {};
    p.src = cache;
    p.k_out = k_out;
    p.scale_out = scale_out;
    p.slots = slots;
    p.rows = rows;
    p.num_slots = num_blocks * int64_t(block_size);
    p.block_size = block_size;
    p.slot_div = fastdiv_magic(static_cast<uint32_t>(block_size));
    p.err = err;
    const unsigned grid = static_cast<unsigned>(grid_for(rows, max_ctas, kGatherPairs));
    const bool wide = (reinterpret_cast<uintptr_t>(cache) & 7u) == 0 && block_size % 2 == 0;
    return launch_kernel(wide ? indexer_k_gather_kernel<true> : indexer_k_gather_kernel<false>,
                         dim3(grid), dim3(kThreads), 0, stream, p);
}

}  // namespace dsv4

DSV4_BOUNDS_FLAG_READER(bounds_flag_indexer)
