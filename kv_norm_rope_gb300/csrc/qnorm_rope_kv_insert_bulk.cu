// The fused step with its rows staged through shared memory by the bulk-copy
// (TMA) engine: the variant for large batches.
//
// Why: the step is a read-modify-write stream of q (98.6-99.3% of its bytes).
// With plain vector loads, a warp has its loads in flight only between its
// compute phases, so the bytes in flight per SM swing with the compute.  Here
// one producer thread per CTA keeps a fixed ring of row chunks in flight with
// cp.async.bulk, independent of the compute, and writes finished q chunks back
// with bulk stores; the consumer warps only read and write shared memory.
// Measured on a plain in-place stream, this reaches the device-to-device copy
// rate, where warp-issued loads stay ~2.5% below it.  With the full row
// arithmetic it does too when the per-row metadata is held constant, but the
// dependent position -> cos/sin loads in front of each chunk still cost ~10%
// here, so this variant is opt-in; the streaming variant is the default.
//
// Layout: one CTA per SM (persistent), 16 consumer warps + 1 producer warp.
// A chunk is 32 consecutive 1 KB rows (32 KB, one bulk copy), 6 in flight:
// chunks [0, Ckv) are KV rows, chunks [Ckv, Ckv + Cq) q rows in memory order;
// CTA b takes chunks b, b + G, b + 2G, ... (G = grid size).  Consumer warp w
// handles rows w and w + 16 of every chunk, the two rows' dependency chains
// interleaved (a row's latency, not its instruction count, limits a warp),
// with the same row arithmetic as the other variants (rowmath.cuh), so
// outputs are bit-identical to them.  A KV row's cache bytes are stored
// directly; a q chunk goes back to q in one bulk store.
//
// Every wait on an mbarrier is bounded.  A wait that runs out (it never does
// unless something is broken) sets DSV4_DEVERR_TIMEOUT in the error word; the
// CTA then lets its copies in flight land and returns.

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "bulkcopy.cuh"
#include "launch_status.h"
#include "rowmath.cuh"

namespace dsv4 {
namespace {

constexpr int kConsumers = 16;
constexpr int kChunkRows = 2 * kConsumers;  // two rows per consumer warp, computed interleaved
constexpr int kStages = 6;
constexpr int kStoresInFlight = 2;  // bulk stores allowed to be still reading their stage
static_assert(kStoresInFlight < kStages, "a stage must be free before it is reloaded");
constexpr int kBulkThreadsPerCta = 32 * (kConsumers + 1);
// Waits are the bounded polls of bulkcopy.cuh.
constexpr int kWeightOffset = 256;   // after 2 * kStages mbarriers
constexpr int kStageOffset = 1280;   // after the 1 KB weight
constexpr uint32_t kChunkBytes = kChunkRows * 1024;
static_assert(2 * kStages * 8 <= kWeightOffset, "barriers overlap the weight");

__device__ __forceinline__ void bulk_store(void *dst, const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_addr(src)), "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// all but the kStoresInFlight most recent bulk store groups have finished
// reading shared memory
__device__ __forceinline__ void bulk_stores_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kStoresInFlight) : "memory");
}

__device__ __forceinline__ void bulk_stores_done()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

struct Chunk {
    bool kv;      // KV rows (else q rows)
    int64_t r0;   // first row (token for KV, q row index for q)
    int rows;     // rows in this chunk (the last one of each kind may be short)
};

__device__ __forceinline__ Chunk chunk_of(int64_t c, int64_t kv_chunks, int64_t T, int64_t q_rows)
{
    Chunk k;
    k.kv = c < kv_chunks;
    k.r0 = (k.kv ? c : c - kv_chunks) * kChunkRows;
    const int64_t end = k.kv ? T : q_rows;
    k.rows = int(end - k.r0 < kChunkRows ? end - k.r0 : kChunkRows);
    return k;
}

// A consumer warp's two rows of a chunk: token, position, slot (KV), whether
// the row exists and its position is in range, and (q) its cos/sin.
struct Meta {
    bool kv;
    bool has[2], ok[2];
    int64_t t[2], pos[2], slot[2];
    float4 cv[2], sv[2];
};

__device__ __forceinline__ void fetch_positions(const KParams &p, int lane, int warp,
                                                const Chunk &c, int64_t H, Meta &m)
{
    m.kv = c.kv;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int r = warp + kConsumers * j;
        m.has[j] = r < c.rows;
        m.t[j] = 0;
        m.pos[j] = 0;
        m.slot[j] = -1;
        if (m.has[j]) {
            m.t[j] = c.kv ? c.r0 + r : (c.r0 + r) / H;
            m.pos[j] = __ldg(p.pos + m.t[j]);
            if (c.kv)
                m.slot[j] = __ldg(p.slot + m.t[j]);
        }
    }
}

__device__ __forceinline__ void fetch_cos_sin(const KParams &p, int lane, Meta &m)
{
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        m.ok[j] = m.has[j] && m.pos[j] >= 0 && m.pos[j] < p.max_pos;
        m.cv[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        m.sv[j] = m.cv[j];
        if (!m.kv && m.ok[j])
            load_cs(p, lane, m.pos[j], m.cv[j], m.sv[j]);
    }
}

template <int kStore, bool kKvNorm>
__global__ void __launch_bounds__(kBulkThreadsPerCta, 1)
    qnorm_rope_kv_insert_bulk_kernel(const KParams p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kStages;
    uint4 *w_smem = reinterpret_cast<uint4 *>(smem + kWeightOffset);
    uint4 *stage0 = reinterpret_cast<uint4 *>(smem + kStageOffset);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumers);
        }
        mbar_init_fence();
    }
    if (kKvNorm)
        for (int i = threadIdx.x; i < 64; i += blockDim.x)
            w_smem[i] = __ldg(reinterpret_cast<const uint4 *>(p.w) + i);
    __syncthreads();

    const int64_t T = p.num_tokens, H = p.num_heads;
    const int64_t q_rows = T * H;
    const int64_t kv_chunks = (T + kChunkRows - 1) / kChunkRows;
    const int64_t chunks = kv_chunks + (q_rows + kChunkRows - 1) / kChunkRows;
    const int64_t G = gridDim.x, b = blockIdx.x;
    const int64_t mine = chunks > b ? (chunks - b + G - 1) / G : 0;

    if (warp == kConsumers) {
        // producer: one thread.  Chunk j lives on stage j % kStages.  In order:
        // load the first kStages chunks; then for each chunk j, wait until its
        // consumers release it, bulk-store it (q; one commit group per chunk,
        // empty for KV), and once the store of chunk f is kStoresInFlight
        // groups old, reload its stage with chunk f + kStages.
        if (lane != 0)
            return;
        bool ok = true;
        const int64_t first = mine < kStages ? mine : kStages;
        for (int64_t j = 0; j < first; ++j) {
            const Chunk c = chunk_of(b + j * G, kv_chunks, T, q_rows);
            mbar_arrive_expect_tx(&full[j], uint32_t(c.rows) * 1024u);
            bulk_load(stage0 + j * (kChunkBytes / 16), (c.kv ? p.kv : p.q) + c.r0 * kHead,
                      uint32_t(c.rows) * 1024u, &full[j]);
        }
        int64_t loaded = first, freed = 0;
        for (int64_t j = 0; j < mine; ++j) {
            const int s = int(j % kStages);
            if (!mbar_wait(&empty[s], uint32_t(j / kStages) & 1)) {
                ok = false;
                break;
            }
            const Chunk c = chunk_of(b + j * G, kv_chunks, T, q_rows);
            if (!c.kv)
                bulk_store(p.q + c.r0 * kHead, stage0 + s * (kChunkBytes / 16),
                           uint32_t(c.rows) * 1024u);
            else
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            // chunks up to j - kStoresInFlight have had their stages read out
            for (; freed + kStoresInFlight <= j; ++freed) {
                bulk_stores_read();
                if (loaded < mine) {
                    const int s2 = int(loaded % kStages);
                    const Chunk n = chunk_of(b + loaded * G, kv_chunks, T, q_rows);
                    mbar_arrive_expect_tx(&full[s2], uint32_t(n.rows) * 1024u);
                    bulk_load(stage0 + s2 * (kChunkBytes / 16), (n.kv ? p.kv : p.q) + n.r0 * kHead,
                              uint32_t(n.rows) * 1024u, &full[s2]);
                    ++loaded;
                }
            }
        }
        bulk_stores_done();
        if (!ok) {
            flag_error(p.err, DSV4_DEVERR_TIMEOUT);
            // let every issued load land before this CTA's shared memory is released
            for (int64_t j = loaded > kStages ? loaded - kStages : 0; j < loaded; ++j)
                (void)mbar_wait(&full[j % kStages], uint32_t(j / kStages) & 1);
        }
        return;
    }

    // consumers: warp w handles rows w and w + kConsumers of each chunk.  The
    // positions of chunk i + 1 are fetched while chunk i is computed; the
    // cos/sin rows they select are fetched at the top of iteration i + 1,
    // before the wait for the chunk, and first used by the rotation at the
    // end of the row arithmetic.  Neither load is waited on where it is issued.
    Meta cur, nxt;
    fetch_positions(p, lane, warp, chunk_of(b, kv_chunks, T, q_rows), H, cur);
    for (int64_t i = 0; i < mine; ++i) {
        const int s = int(i % kStages);
        fetch_cos_sin(p, lane, cur);
        if (i + 1 < mine)
            fetch_positions(p, lane, warp, chunk_of(b + (i + 1) * G, kv_chunks, T, q_rows), H, nxt);
        if (!mbar_wait(&full[s], uint32_t(i / kStages) & 1)) {
            if (lane == 0)
                flag_error(p.err, DSV4_DEVERR_TIMEOUT);
            return;
        }
        uint4 *rows = stage0 + s * (kChunkBytes / 16);
        if (cur.kv) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                if (cur.has[j]) {
                    const uint4 *row = rows + (warp + kConsumers * j) * 64;
                    kv_row<kStore, true, kKvNorm>(p, lane, cur.t[j], cur.pos[j], cur.slot[j],
                                                  row[lane], row[32 + lane], w_smem);
                }
            }
        } else if (cur.ok[0] && cur.ok[1]) {
            uint4 *r0 = rows + warp * 64, *r1 = rows + (warp + kConsumers) * 64;
            const uint4 in[4] = {r0[lane], r0[32 + lane], r1[lane], r1[32 + lane]};
            uint4 out[4];
            q_row2(p, lane, in, cur.cv, cur.sv, out);
            r0[lane] = out[0];
            r0[32 + lane] = out[1];
            r1[lane] = out[2];
            r1[32 + lane] = out[3];
        } else {
            // a short last chunk or an out-of-range position: one row at a time
            // (a q row whose position is out of range goes back unchanged)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                if (cur.ok[j]) {
                    uint4 *row = rows + (warp + kConsumers * j) * 64;
                    uint4 out_a, out_b;
                    q_row(p, lane, row[lane], row[32 + lane], cur.cv[j], cur.sv[j], out_a, out_b);
                    row[lane] = out_a;
                    row[32 + lane] = out_b;
                }
            }
        }
        // make this warp's shared-memory writes visible to the bulk store, then release
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[s]);
        if (i + 1 < mine)
            cur = nxt;
    }
}

template <int kStore, bool kKvNorm>
int launch_bulk_one(dim3 grid, cudaStream_t stream, const KParams &p)
{
    auto kernel = qnorm_rope_kv_insert_bulk_kernel<kStore, kKvNorm>;
    // the opt-in to more than 48 KB of dynamic shared memory, once per device
    // (bit d of `configured` for device d < 64; other devices set it every call)
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return DSV4_ERR_CUDA;
    const uint64_t bit = dev >= 0 && dev < 64 ? uint64_t(1) << dev : 0;
    if (bit == 0 || (configured.load(std::memory_order_relaxed) & bit) == 0) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(bulk_smem_bytes())) != cudaSuccess)
            return DSV4_ERR_CUDA;
        configured.fetch_or(bit, std::memory_order_relaxed);
    }
    return launch_kernel(kernel, grid, dim3(kBulkThreadsPerCta), bulk_smem_bytes(), stream, p);
}

}  // namespace

size_t bulk_smem_bytes()
{
    return size_t(kStageOffset) + size_t(kStages) * kChunkBytes;
}

int bulk_threads()
{
    return kBulkThreadsPerCta;
}

int bulk_chunk_rows()
{
    return kChunkRows;
}

int launch_bulk(int store_mode, bool kv_norm, int64_t ctas, const KParams &p, cudaStream_t stream)
{
    const dim3 grid(static_cast<unsigned>(ctas));
    if (store_mode == DSV4_STORE_BF16)
        return kv_norm ? launch_bulk_one<DSV4_STORE_BF16, true>(grid, stream, p)
                       : launch_bulk_one<DSV4_STORE_BF16, false>(grid, stream, p);
    return kv_norm ? launch_bulk_one<DSV4_STORE_FP8, true>(grid, stream, p)
                   : launch_bulk_one<DSV4_STORE_FP8, false>(grid, stream, p);
}

}  // namespace dsv4
