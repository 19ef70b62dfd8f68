// Reading the FP8 paged cache back out (the consumer of the insert kernels):
// out[n, :] = the 512 dims stored at slot slots[n], as bf16.  Dims 0..447 are
// E4M3 payload times 2^(e_b - 127) of their 64-dim block; dims 448..511 are
// the stored bf16 rope dims.  A negative slot gives a zero row, a slot past the
// cache a zero row and an error bit.  (1Cat-vLLM PR #1280, "Purpose": item 5,
// the dequantize-and-gather of the compressed KV cache; item 2, zeros for
// unused slots.)
//
// HBM-bound: per row 584 bytes read and 1024 written.  One warp per row with
// the insert kernels' lane layout (lane l: dims [8l, 8l+8) and [256+8l,
// 256+8l+8)), so each 8-byte load instruction covers 256 contiguous cache
// bytes and each 16-byte store 512 contiguous output bytes.  A warp takes
// groups of kGatherRows rows and keeps the next group's loads in flight
// while it converts and stores the current one (software pipelining in
// registers): the slot ids are loaded two groups ahead, the rows one group
// ahead.  Cache bytes come through the read-only path (ld.global.nc) and the
// rows go out with ordinary write-back stores: both measured ~1% faster than
// evict-first loads and stores here.  Every value is exact: an E4M3 code times
// a power of two fits fp32 for every scale the writer emits, so the one
// rounding is the final bf16 conversion.

#include <cuda_runtime.h>
#include <stdint.h>

#include "bounds.cuh"
#include "convert.cuh"
#include "fastdiv.h"
#include "launch.h"
#include "launch_status.h"
#include "ops.h"

namespace dsv4 {
namespace {

constexpr int kGatherRows = 1;  // rows per group: 1-4 measured, 1 best (40 registers)
// 4-warp CTAs, 12 per SM (48 warps): 0.1-0.8% ahead of 8-warp CTAs, 6 per SM
constexpr int kGatherThreads = 128;

struct GParams {
    const uint8_t *cache;
    int64_t num_slots;
    int32_t block_size;
    uint64_t slot_div;     // fastdiv_magic(block_size)
    uint64_t block_bytes;  // block_size * DSV4_FP8_SLOT_BYTES
    uint64_t scale_off;    // block_size * DSV4_FP8_DATA_BYTES: the scale words of a block
    const int64_t *slots;
    int64_t rows;
    uint16_t *out;
    int32_t *err;
};

// p * 2^(e - 127), exact in fp32 for every E4M3 value p and e in [0, 254]
__device__ __forceinline__ float scaled(float p, uint32_t e)
{
    if (e >= 1u && e <= 254u)
        return __fmul_rn(p, __uint_as_float(e << 23));
    if (e == 0u)  // 2^-127 in two exact steps (|p| >= 2^-9, so no bit falls below 2^-149)
        return __fmul_rn(__fmul_rn(p, 0x1p-64f), 0x1p-63f);
    return __fmul_rn(__fmul_rn(p, 0x1p64f), 0x1p64f);  // 2^128: beyond bf16, becomes inf
}

// Two bytes of w (selector sel) into the low bytes of two 16-bit halves, each
// half's high byte filled with its byte's sign bit (prmt's sign-replicating
// selector nibbles, bit 3 set).
__device__ __forceinline__ uint32_t sext_pair(uint32_t w, uint32_t sel)
{
    uint32_t h;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(h) : "r"(w), "r"(sel));
    return h;
}

// 8 payload bytes with scale byte e -> 8 bf16 by integer arithmetic, when every
// code is a normal E4M3 number (exponent field 1..15, not NaN) and 7 <= e <= 246:
// (1 + m/8) * 2^(E - 7) * 2^(e - 127) is then exactly the bf16 with exponent field
// E + e - 7 (1..254), mantissa m << 4 and the code's sign.  Returns false, leaving
// out unset, when any code or the scale is outside that range.
__device__ __forceinline__ bool dequant8_normal(uint2 codes, uint32_t e, uint4 &out)
{
    // per byte, bit 7 of (c & 0x78) + 0x78 is set when the exponent field is not 0,
    // and bit 7 of (c & 0x7f) + 1 when the low 7 bits are all ones (NaN); neither
    // sum carries out of its byte
    const uint32_t xe = (codes.x & 0x78787878u) + 0x78787878u;
    const uint32_t ye = (codes.y & 0x78787878u) + 0x78787878u;
    const uint32_t xn = (codes.x & 0x7f7f7f7fu) + 0x01010101u;
    const uint32_t yn = (codes.y & 0x7f7f7f7fu) + 0x01010101u;
    if ((xe & ~xn & ye & ~yn & 0x80808080u) != 0x80808080u || e - 7u > 239u)
        return false;
    // a half 0x00cc or 0xffcc shifted left by 4 and masked with 0x87f0 is the sign at
    // bit 15 and the code's exponent and mantissa at bits 7..10 and 4..6 (the bits
    // shifted across into the upper half are masked off there); adding e - 7 to the
    // exponent field cannot carry into the sign (E + e - 7 <= 254)
    const uint32_t off = ((e - 7u) << 7) * 0x00010001u;
    const auto pair = [off](uint32_t w, uint32_t sel) {
        return ((sext_pair(w, sel) << 4) & 0x87f087f0u) + off;
    };
    out = make_uint4(pair(codes.x, 0x9180u), pair(codes.x, 0xb3a2u), pair(codes.y, 0x9180u),
                     pair(codes.y, 0xb3a2u));
    return true;
}

// 8 payload bytes (one 64-bit word) with scale byte e -> 8 bf16 (one 16-byte vector)
__device__ __forceinline__ uint4 dequant8(uint2 codes, uint32_t e)
{
    uint4 fast;
    if (dequant8_normal(codes, e, fast))
        return fast;
    float2 f[4];
    f[0] = e4m3x2_to_f32(codes.x);
    f[1] = e4m3x2_to_f32(codes.x >> 16);
    f[2] = e4m3x2_to_f32(codes.y);
    f[3] = e4m3x2_to_f32(codes.y >> 16);
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        o[i] = bf16x2_rn(scaled(f[i].x, e), scaled(f[i].y, e));
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// the buffers of a launch, for the checked build's bounds tests (bounds.cuh)
__device__ __forceinline__ Span cache_span(const GParams &p)
{
    return Span{p.cache, uint64_t(p.num_slots) * DSV4_FP8_SLOT_BYTES};
}
__device__ __forceinline__ Span slots_span(const GParams &p)
{
    return Span{p.slots, uint64_t(p.rows) * 8u};
}
__device__ __forceinline__ Span out_span(const GParams &p)
{
    return Span{p.out, uint64_t(p.rows) * DSV4_HEAD_DIM * 2u};
}

// one group of rows as loaded by one lane
struct Group {
    int64_t slot[kGatherRows];
    uint2 lo[kGatherRows], hi0[kGatherRows], hi1[kGatherRows], sc[kGatherRows];
};

// slot ids of group g (-1 past the end, so nothing is read for them)
__device__ __forceinline__ void load_slots(const GParams &p, int64_t g, int64_t *slot)
{
#pragma unroll
    for (int j = 0; j < kGatherRows; ++j) {
        const int64_t r = g * kGatherRows + j;
        slot[j] = r < p.rows ? ldg_i64_in(p.slots + r, slots_span(p), p.err) : -1;
    }
}

// issue the lane's loads of the rows at `slot` (zeros for rows that read nothing)
__device__ __forceinline__ void load_rows(const GParams &p, int lane, Group &q)
{
    const bool rope_lane = lane >= 24;
#pragma unroll
    for (int j = 0; j < kGatherRows; ++j) {
        q.lo[j] = q.hi0[j] = q.hi1[j] = q.sc[j] = make_uint2(0u, 0u);
        const int64_t slot = q.slot[j];
        if (slot >= 0 && slot < p.num_slots) {
            // slot < 2^32: block and offset in 32-bit arithmetic
            const uint32_t s32 = static_cast<uint32_t>(slot);
            const uint32_t blk = fastdiv(s32, p.slot_div);
            const uint32_t off = s32 - blk * static_cast<uint32_t>(p.block_size);
            const uint8_t *base = p.cache + uint64_t(blk) * p.block_bytes;
            const uint8_t *data = base + uint64_t(off) * DSV4_FP8_DATA_BYTES;
            const Span cs = cache_span(p);
            q.lo[j] = ldg8_in(data + 8 * lane, cs, p.err);
            if (!rope_lane) {
                q.hi0[j] = ldg8_in(data + 256 + 8 * lane, cs, p.err);
            } else {
                q.hi0[j] = ldg8_in(data + DSV4_NOPE_DIM + 16 * (lane - 24), cs, p.err);
                q.hi1[j] = ldg8_in(data + DSV4_NOPE_DIM + 16 * (lane - 24) + 8, cs, p.err);
            }
            q.sc[j] = ldg8_in(base + p.scale_off + uint64_t(off) * DSV4_FP8_SCALE_BYTES, cs, p.err);
        }
    }
}

// convert and store group g
__device__ __forceinline__ void emit_rows(const GParams &p, int lane, int64_t g, const Group &q)
{
    const bool rope_lane = lane >= 24;
    const int64_t r0 = g * kGatherRows;
#pragma unroll
    for (int j = 0; j < kGatherRows; ++j) {
        if (r0 + j >= p.rows)
            break;
        uint16_t *row = p.out + (r0 + j) * DSV4_HEAD_DIM;
        uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;
        if (q.slot[j] >= p.num_slots) {
            if (lane == 0 && p.err != nullptr)
                atomicOr(p.err, DSV4_DEVERR_SLOT_RANGE);
        } else if (q.slot[j] >= 0) {
            // scale byte of block lane/8 (half 0) and 4 + lane/8 (half 1)
            const int b0 = lane >> 3, b1 = 4 + (lane >> 3);
            const uint32_t e0 = (q.sc[j].x >> (8 * b0)) & 0xFFu;
            const uint32_t e1 = (q.sc[j].y >> (8 * (b1 - 4))) & 0xFFu;
            a = dequant8(q.lo[j], e0);
            // the rope lanes' bytes are bf16, not codes: they convert the code of 1.0
            // (a normal code, so they never send the warp down the slow path) and keep
            // their bf16
            const uint4 d = dequant8(rope_lane ? make_uint2(0x38383838u, 0x38383838u) : q.hi0[j],
                                     rope_lane ? 127u : e1);
            b = rope_lane ? make_uint4(q.hi0[j].x, q.hi0[j].y, q.hi1[j].x, q.hi1[j].y) : d;
        }
        st16_in(row + 8 * lane, a, out_span(p), p.err);
        st16_in(row + 256 + 8 * lane, b, out_span(p), p.err);
    }
}

__global__ void __launch_bounds__(kGatherThreads, 12) dequant_gather_kernel(const GParams p)
{
    const int lane = threadIdx.x & 31;
    const int warps_per_cta = blockDim.x >> 5;
    const int64_t groups = (p.rows + kGatherRows - 1) / kGatherRows;
    const int64_t stride = int64_t(gridDim.x) * warps_per_cta;
    int64_t g = int64_t(blockIdx.x) * warps_per_cta + (threadIdx.x >> 5);
    if (g >= groups)
        return;
    Group cur;
    load_slots(p, g, cur.slot);
    load_rows(p, lane, cur);
    int64_t ahead[kGatherRows];  // slot ids of the group after the next one
    load_slots(p, g + stride, ahead);
    for (; g < groups; g += stride) {
        Group nxt;
#pragma unroll
        for (int j = 0; j < kGatherRows; ++j)
            nxt.slot[j] = ahead[j];
        load_rows(p, lane, nxt);  // nothing is read for a group past the end
        load_slots(p, g + 2 * stride, ahead);
        emit_rows(p, lane, g, cur);
        cur = nxt;
    }
}

}  // namespace

int gather_ctas_per_sm(int *ctas_per_sm)
{
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, dequant_gather_kernel, kGatherThreads,
                                                         0) == cudaSuccess
               ? DSV4_OK
               : DSV4_ERR_CUDA;
}

int launch_gather(const uint8_t *cache, int64_t num_blocks, int32_t block_size,
                  const int64_t *slots, int64_t rows, uint16_t *out, int32_t *err, int64_t ctas,
                  cudaStream_t stream)
{
    GParams p;
    p.cache = cache;
    p.num_slots = num_blocks * int64_t(block_size);
    p.block_size = block_size;
    p.slot_div = fastdiv_magic(static_cast<uint32_t>(block_size));
    p.block_bytes = uint64_t(block_size) * DSV4_FP8_SLOT_BYTES;
    p.scale_off = uint64_t(block_size) * DSV4_FP8_DATA_BYTES;
    p.slots = slots;
    p.rows = rows;
    p.out = out;
    p.err = err;
    return launch_kernel(dequant_gather_kernel, dim3(unsigned(ctas)), dim3(kGatherThreads), 0, stream,
                         p);
}

int gather_rows_per_warp()
{
    return kGatherRows;
}

int gather_warps_per_cta()
{
    return kGatherThreads / 32;
}

}  // namespace dsv4

DSV4_BOUNDS_FLAG_READER(bounds_flag_gather)
