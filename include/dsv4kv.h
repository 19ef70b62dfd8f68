/*
 * dsv4kv.h -- C ABI of the fused DeepSeek-V4 attention-input step for GB300
 * (sm_103a): per token, RMS-normalise every 512-wide query head and rotate its
 * trailing 64 dims in place; RMS-normalise the token's 512-wide latent KV row
 * with a learned weight, rotate its trailing 64 dims, and write it into a
 * paged KV cache, either quantised (448 E4M3 + 7 UE8M0 exponents + 64 bf16)
 * or as 512 bf16.
 *
 * Sources restated here:
 *  - FlagGems-vllm PR #684, "fused_deepseek_v4_qnorm_rope_kv_rope_quant_insert
 *    backends": section "T-Head PPU-ZW810E" (the operator rewrites q in place);
 *    section "Ascend 910B" (a weightless q RMSNorm, 256 bytes of cos/sin per
 *    position shared by all heads of a token, mixed negative slots that write
 *    nothing); section 'What "as shipped" would give' (seven per-block
 *    exponents per token in the FP8 cache).
 *  - SGLang PR #33358, "DSv4 flashmla norm-rope" (section "Motivation": RMSNorm
 *    over head_dim 512 with a weight, RoPE on the trailing 64 dims, paged-cache
 *    store with an FP8-UE8M0 path and a bf16 path; section "Accuracy Tests":
 *    448 E4M3 bytes, 7 per-64-group exponents, bf16 rope tail).
 *
 * Conventions for every entry point:
 *  - Pointers marked (device) are CUDA device pointers; the caller owns all
 *    memory.  The library allocates nothing, keeps no state between calls and
 *    takes no locks.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream).  A DSV4_OK return means the launch was accepted,
 *    not that it has finished.
 *  - Host-side argument checks run before anything is enqueued; a non-OK
 *    status means nothing was launched and no buffer was touched.
 *  - Conditions that need device data (a slot or a position out of range) are
 *    reported by OR-ing DSV4_DEVERR_* bits into *device_error (device int32,
 *    may be NULL) and skipping the affected writes.  Nothing traps or asserts
 *    on the device; the one kernel that waits on its own bulk copies bounds
 *    every wait (DSV4_DEVERR_TIMEOUT).
 *  - Preconditions that are not checked: non-negative slots are distinct (if
 *    two tokens share a slot, which one's row lands is unspecified); q does
 *    not overlap kv, the cache or the metadata arrays; inputs are finite and
 *    sum(x^2) of a row stays below 3.4e38; each kv_norm_weight element is 0 or
 *    has magnitude in [2^-9, 2^64), so that every product x * w of a KV element
 *    and its weight is exact in fp32 (the kernels form v = (x * w) * r).  With
 *    eps = 0 a row of zeros has no norm: 1/sqrt(0) is infinite and its outputs
 *    are NaN, as the definition gives them; rows of tiny elements (down to
 *    bf16 subnormals) are normalised like any other row.
 *  - Every paged cache holds at most 2^32 slots (num_blocks * block_size <=
 *    2^32; larger returns DSV4_ERR_SHAPE).  At 132 bytes or more per slot such
 *    a cache exceeds one GPU's memory, and the bound lets the kernels split a
 *    slot into block and offset with a 32-bit division.
 */
#ifndef DSV4KV_H
#define DSV4KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DSV4_OK = 0,
    DSV4_ERR_NULL = 1,   /* a required pointer is NULL */
    DSV4_ERR_SHAPE = 2,  /* a size is out of range */
    DSV4_ERR_ALIGN = 3,  /* a pointer is not aligned as documented */
    DSV4_ERR_VALUE = 4,  /* eps negative or not finite; unknown store mode or variant */
    DSV4_ERR_CUDA = 5    /* the CUDA runtime reported an error while launching */
} dsv4_status;

enum {
    DSV4_HEAD_DIM = 512,        /* q head and latent KV width */
    DSV4_ROPE_DIM = 64,         /* trailing rotated dims 448..511, GPT-J interleaved pairs */
    DSV4_NOPE_DIM = 448,        /* leading dims quantised to E4M3 on the FP8 path */
    DSV4_QUANT_BLOCK = 64,      /* elements per UE8M0 exponent */
    DSV4_NUM_QUANT_BLOCKS = 7,
    DSV4_FP8_DATA_BYTES = 576,  /* 448 E4M3 + 64 bf16 */
    DSV4_FP8_SCALE_BYTES = 8,   /* 7 UE8M0 bytes + 1 zero pad byte */
    DSV4_FP8_SLOT_BYTES = 584,
    DSV4_BF16_SLOT_BYTES = 1024,
    DSV4_INDEXER_DIM = 128,        /* indexer K width: one E4M3 row with one fp32 scale */
    DSV4_INDEXER_SLOT_BYTES = 132  /* 128 E4M3 codes + 4 scale bytes per slot */
};

/* bits OR-ed into *device_error */
enum {
    DSV4_DEVERR_SLOT_RANGE = 1, /* slot_mapping[t] >= num_blocks*block_size: cache row not written */
    DSV4_DEVERR_POS_RANGE = 2,  /* positions[t] < 0 or >= max_position: token not written at all */
    DSV4_DEVERR_TIMEOUT = 4,    /* the KV-row kernel (num_heads 0, STREAM): a bounded wait on a
                                   bulk copy inside the kernel ran out (never expected); the
                                   outputs of that launch are undefined */
    DSV4_DEVERR_BOUNDS = 8      /* the checked build only (libdsv4kv_checked.so, compiled with
                                   DSV4_CHECK_BOUNDS): an access would have touched bytes outside
                                   the buffer it belongs to; it was skipped (never expected) */
};

/* store modes and launch variants of dsv4_qnorm_rope_kv_insert_variant */
enum { DSV4_STORE_FP8 = 0, DSV4_STORE_BF16 = 1 };
enum {
    DSV4_VARIANT_AUTO = 0,    /* pick from the row count and the SM count (below) */
    DSV4_VARIANT_SMALL = 1,   /* one row per warp, 2-warp CTAs, one wave: small batches */
    DSV4_VARIANT_STREAM = 2,  /* persistent CTAs sized to the SMs, several rows in flight per warp */
    /* 3 is not a variant (DSV4_ERR_VALUE) */
    DSV4_VARIANT_HALF = 4     /* persistent CTAs sized to the SMs, one row per half-warp (q and KV) */
};

/*
 * Fused q-norm + RoPE (in place) and KV norm + RoPE + FP8 quant + paged insert.
 *
 *  q              (device) bf16 [num_tokens, num_heads, 512], contiguous, read and
 *                 rewritten in place: q[t,h,:] = bf16( rot( x * r ) ), with
 *                 x = q[t,h,:], r = 1/sqrt(sum(x^2)/512 + eps), no weight.
 *                 16-byte aligned.
 *  kv             (device) bf16 [num_tokens, 512], contiguous, read only. 16-byte aligned.
 *  kv_norm_weight (device) bf16 [512].  v = x * r * w for the KV row.  16-byte aligned.
 *  positions      (device) int64 [num_tokens]: row of cos_sin_cache for token t.
 *  cos_sin_cache  (device) fp32 [max_position, 64]: columns 0..31 = cos of the 32
 *                 pair angles, 32..63 = their sin.  Pair i = dims (448+2i, 449+2i)
 *                 turns as (a, b) -> (a*cos - b*sin, b*cos + a*sin).  16-byte aligned.
 *  slot_mapping   (device) int64 [num_tokens]: slot = block*block_size + offset;
 *                 a negative slot writes no cache row (q is still rewritten).
 *  kv_cache       (device) uint8, num_blocks * block_size * 584 bytes.  Block b
 *                 occupies [b*bs*584, (b+1)*bs*584); inside it, slot offset o has
 *                   data  at b*bs*584 + o*576         : 448 E4M3 bytes of dims 0..447,
 *                                                       then dims 448..511 as 64
 *                                                       little-endian bf16,
 *                   scale at b*bs*584 + bs*576 + o*8  : UE8M0 bytes e_0..e_6 of the
 *                                                       seven 64-dim blocks, then 0.
 *                 e_b = s_b + 127 with s_b the smallest integer such that
 *                 max|v| over block b <= 448 * 2^s_b (clamped to [-127, 127]; an
 *                 all-zero block gives e_b = 0); payload = E4M3_rn(v * 2^-s_b).
 *                 8-byte aligned.  Bytes of slots that are not written keep
 *                 their previous contents.
 *  num_blocks, block_size   cache geometry (>= 1 each; num_blocks*block_size <= 2^32).
 *  num_tokens     T >= 0 (T == 0 returns DSV4_OK and launches nothing).
 *  num_heads      H >= 1.
 *  eps            >= 0 and finite; added to mean(x^2) inside the root.
 *  device_error   (device, nullable) int32; DSV4_DEVERR_* bits are OR-ed in.
 *  stream         cudaStream_t.
 * Returns a dsv4_status.
 */
int dsv4_qnorm_rope_kv_quant_insert(void *q, const void *kv, const void *kv_norm_weight,
                                    const int64_t *positions, const float *cos_sin_cache,
                                    int64_t max_position, const int64_t *slot_mapping,
                                    uint8_t *kv_cache, int64_t num_blocks, int32_t block_size,
                                    int64_t num_tokens, int32_t num_heads, float eps,
                                    int32_t *device_error, void *stream);

/*
 * As above, but the cache holds bf16 rows: kv_cache (device) bf16
 * [num_blocks, block_size, 512], 16-byte aligned; slot s gets bf16(rot(v))
 * for all 512 dims (SGLang PR #33358, "Motivation": the kBf16Store path).
 */
int dsv4_qnorm_rope_kv_bf16_insert(void *q, const void *kv, const void *kv_norm_weight,
                                   const int64_t *positions, const float *cos_sin_cache,
                                   int64_t max_position, const int64_t *slot_mapping,
                                   void *kv_cache, int64_t num_blocks, int32_t block_size,
                                   int64_t num_tokens, int32_t num_heads, float eps,
                                   int32_t *device_error, void *stream);

/*
 * Either store mode with an explicit launch variant (DSV4_VARIANT_*).  Every
 * variant computes bit-identical outputs: each token's rows depend only on
 * that token's inputs (SGLang PR #33358, "Modifications": the grouping of
 * tokens into blocks does not change a token's bits).  Used by tests that
 * exercise each variant and by benchmarks.
 */
int dsv4_qnorm_rope_kv_insert_variant(int store_mode, int variant, void *q, const void *kv,
                                      const void *kv_norm_weight, const int64_t *positions,
                                      const float *cos_sin_cache, int64_t max_position,
                                      const int64_t *slot_mapping, void *kv_cache,
                                      int64_t num_blocks, int32_t block_size, int64_t num_tokens,
                                      int32_t num_heads, float eps, int32_t *device_error,
                                      void *stream);

/*
 * The operator with the KV row already normalised (FlagGems-vllm PR #684: the
 * operator is q-norm + RoPE and KV RoPE + quant + insert; its eager baseline in
 * section "Ascend 910B" normalises q only).  As dsv4_qnorm_rope_kv_quant_insert,
 * except the KV row gets no RMSNorm and no weight: v = kv[t,:], rotated,
 * quantised and inserted.  eps applies to the q heads only.
 */
int dsv4_qnorm_rope_kv_rope_quant_insert(void *q, const void *kv, const int64_t *positions,
                                         const float *cos_sin_cache, int64_t max_position,
                                         const int64_t *slot_mapping, uint8_t *kv_cache,
                                         int64_t num_blocks, int32_t block_size,
                                         int64_t num_tokens, int32_t num_heads, float eps,
                                         int32_t *device_error, void *stream);

/*
 * KV rows only, no q (SGLang PR #33358, "Motivation": fused_norm_rope_flashmla,
 * RMSNorm over 512 with a weight, RoPE on the trailing 64 dims, paged store):
 * store_mode DSV4_STORE_FP8 (kv_cache uint8, FP8 layout above, 8-byte aligned) or
 * DSV4_STORE_BF16 (kv_cache bf16 [num_blocks, block_size, 512], 16-byte aligned).
 * Other arguments as in dsv4_qnorm_rope_kv_quant_insert.  Batches that plan as
 * STREAM run a kernel laid out for KV rows alone (one row per quarter-warp); its cache
 * bytes are identical to those the fused entry points write for the same rows.
 */
int dsv4_kv_norm_rope_insert(int store_mode, const void *kv, const void *kv_norm_weight,
                             const int64_t *positions, const float *cos_sin_cache,
                             int64_t max_position, const int64_t *slot_mapping, void *kv_cache,
                             int64_t num_blocks, int32_t block_size, int64_t num_tokens,
                             float eps, int32_t *device_error, void *stream);

/*
 * The general form behind all of the above: any store mode and launch variant;
 * kv_norm 1 normalises the KV row with kv_norm_weight, 0 takes it as already
 * normalised (kv_norm_weight may then be NULL); num_heads >= 0, and q may be
 * NULL when num_heads is 0.
 */
int dsv4_insert_ex(int store_mode, int variant, int kv_norm, void *q, const void *kv,
                   const void *kv_norm_weight, const int64_t *positions,
                   const float *cos_sin_cache, int64_t max_position, const int64_t *slot_mapping,
                   void *kv_cache, int64_t num_blocks, int32_t block_size, int64_t num_tokens,
                   int32_t num_heads, float eps, int32_t *device_error, void *stream);

/*
 * Read rows of an FP8 cache back out as bf16 (1Cat-vLLM PR #1280, "Purpose"
 * item 5: the dequantize-and-gather of the compressed KV cache; item 2: the
 * gather writes zeros for unused slots).
 *
 *  kv_cache  (device) uint8, FP8 layout of dsv4_qnorm_rope_kv_quant_insert; 8-byte aligned.
 *  slots     (device) int64 [num_rows]: slot = block*block_size + offset.
 *  out       (device) bf16 [num_rows, 512], 16-byte aligned: row n = bf16(E4M3 value *
 *            2^(e_b - 127)) for dims 0..447 (b = dim / 64) and the stored bf16 for
 *            448..511 -- exact for every row the insert kernels write.  A negative
 *            slot gives a zero row; a slot >= num_blocks*block_size gives a zero row
 *            and DSV4_DEVERR_SLOT_RANGE.
 *  num_rows >= 0 (0: no launch); num_blocks, block_size >= 1, num_blocks*block_size <= 2^32.
 * Returns a dsv4_status.
 */
int dsv4_dequant_gather(const uint8_t *kv_cache, int64_t num_blocks, int32_t block_size,
                        const int64_t *slots, int64_t num_rows, void *out,
                        int32_t *device_error, void *stream);

/*
 * Residual add + Gemma RMSNorm + MXFP8 quantisation of activation rows: the
 * single-GPU part of the vLLM minimax_m3 finalize_allreduce_norm page
 * (_LamportGemmaRMSNormMxfp8Kernel with one rank; no all-reduce).  Per row:
 *   residual_out = bf16(x + residual)                   (the new residual stream)
 *   r            = 1 / sqrt(mean(residual_out^2) + eps)
 *   normed       = bf16(residual_out * r * (1 + gamma))  (Gemma: the scale is 1 + w)
 * and per 32-element block of normed: e = the UE8M0 byte of fp32(amax * fp32(1/448))
 * rounded up to a power of two (clamped to [0, 254], 0 for amax 0); codes =
 * E4M3_rn_satfinite(normed * 2^(127 - e)) (the inverse is 0 for e = 0 and e = 254).
 *
 *  x, residual   (device) bf16 [num_rows, hidden], 16-byte aligned; residual_out may
 *                be residual itself (rewritten in place), x must not overlap an output.
 *  gamma         (device) bf16 [hidden], 16-byte aligned.
 *  residual_out  (device) bf16 [num_rows, hidden], 16-byte aligned.
 *  codes         (device) uint8 [num_rows, hidden] E4M3, 8-byte aligned.
 *  scales        (device) uint8, dsv4_mxfp8_scale_bytes(num_rows, hidden) bytes: the
 *                byte of row r, block c sits at (r/128)*128*C + (c/4)*512 + (r%32)*16
 *                + ((r%128)/32)*4 + c%4, with C = hidden/32 (the 128x4 swizzled layout);
 *                the rows past num_rows up to the next multiple of 128 get 0.
 *  hidden        a multiple of 128 in [128, 16384]; num_rows >= 0 (0: no launch).
 * Returns a dsv4_status.
 */
int dsv4_add_gemma_rmsnorm_mxfp8(const void *x, const void *residual, const void *gamma,
                                 int64_t num_rows, int32_t hidden, float eps, void *residual_out,
                                 uint8_t *codes, uint8_t *scales, void *stream);

/* Bytes of the swizzled scales of num_rows rows: ceil(num_rows/128)*128 * hidden/32
 * (0 for an invalid hidden). */
size_t dsv4_mxfp8_scale_bytes(int64_t num_rows, int32_t hidden);

/* Launch plan of a call (pure host arithmetic, no CUDA call). */
typedef struct {
    int32_t variant;        /* DSV4_VARIANT_SMALL, DSV4_VARIANT_STREAM or DSV4_VARIANT_HALF */
    int32_t threads;        /* threads per CTA */
    int64_t ctas;           /* grid size */
    int32_t rows_per_warp;  /* rows each warp loads together */
    int64_t rows;           /* num_tokens * (num_heads + 1) work rows */
} dsv4_plan;

/*
 * Fill *plan for T tokens, H heads on a GPU with sm_count SMs where
 * ctas_per_sm CTAs of the streaming kernel fit per SM.  variant AUTO picks
 * SMALL when there are fewer rows than the GPU's warp slots (sm_count x
 * ctas_per_sm x 8) (SGLang PR #33358, "Modifications" item 3: a grid-starved
 * multi-token layout loses at small N); with q heads, HALF below 12
 * rounds of the streaming kernel's groups
 * (warp slots x rows_per_warp x 12; decode- to mid-sized batches, where HALF
 * measured faster); else STREAM (for num_heads 0, the KV-row kernel).  HALF: ceil(T/2) KV row pairs and
 * groups of rows_per_warp q rows over persistent CTAs (ctas_per_sm then being
 * the HALF kernel's occupancy).  With num_heads 0, STREAM describes the
 * KV-row kernel: one row per quarter-warp, rows_per_warp 4, and ctas_per_sm should
 * then be that kernel's occupancy.  Returns a dsv4_status.
 */
int dsv4_launch_plan(int64_t num_tokens, int32_t num_heads, int32_t sm_count,
                     int32_t ctas_per_sm, int32_t variant, dsv4_plan *plan);

/* Bytes of an FP8 cache of num_blocks x block_size slots: num_blocks*block_size*584. */
size_t dsv4_fp8_cache_bytes(int64_t num_blocks, int32_t block_size);
/* Bytes of a bf16 cache: num_blocks*block_size*1024. */
size_t dsv4_bf16_cache_bytes(int64_t num_blocks, int32_t block_size);

/*
 * Indexer-K quant-insert.  The lightning indexer scores queries against K rows
 * held as E4M3 [N, 128] with one non-negative fp32 scale per row (rocm-aiter
 * PR #1, "Motivation": k_fp8 and kv_scale, gathered out of the paged cache
 * before scoring); the norm-rope-store kernel keeps this indexer path beside
 * the KV path (SGLang PR #33358, "Modifications").  Per token t with
 * 0 <= slot_mapping[t] < num_blocks*block_size:
 *   s      = the smallest integer with max|k[t,:]| <= 448 * 2^s, clamped to [-127, 127]
 *   codes  = E4M3_rn_satfinite(k[t,:] * 2^-s);   scale = 2^s (fp32, exact)
 * Cache layout: block b occupies bytes [b*bs*132, (b+1)*bs*132); slot o's 128 codes
 * sit at b*bs*132 + o*128 and its scale (fp32, little-endian) at b*bs*132 + bs*128 + o*4.
 *
 *  k              (device) bf16 [num_tokens, 128], 16-byte aligned, finite values.
 *  slot_mapping   (device) int64 [num_tokens], 8-byte aligned; < 0: the token writes
 *                 nothing; >= num_blocks*block_size: nothing written and
 *                 DSV4_DEVERR_SLOT_RANGE.  Non-negative slots are distinct.
 *  indexer_cache  (device) uint8, dsv4_indexer_cache_bytes(num_blocks, block_size)
 *                 bytes, 4-byte aligned (8-byte aligned with an even block_size
 *                 takes 8-byte stores).  Bytes of slots no token names are untouched.
 *  num_tokens >= 0 (0: no launch); num_blocks, block_size >= 1, num_blocks*block_size <= 2^32.
 * Returns a dsv4_status.
 */
int dsv4_indexer_k_quant_insert(const void *k, const int64_t *slot_mapping,
                                uint8_t *indexer_cache, int64_t num_blocks, int32_t block_size,
                                int64_t num_tokens, int32_t *device_error, void *stream);

/*
 * Indexer-K gather: for each n, the 128 codes and the fp32 scale stored at
 * slots[n] copied unchanged to k_out[n,:] and scale_out[n] -- the contiguous
 * [N, 128] E4M3 + [N] fp32 form the indexer scores against (rocm-aiter PR #1,
 * "Motivation").  A negative slot gives zero codes and scale 0; a slot
 * >= num_blocks*block_size the same and DSV4_DEVERR_SLOT_RANGE.
 *
 *  indexer_cache  (device) the layout of dsv4_indexer_k_quant_insert, 4-byte aligned.
 *  slots          (device) int64 [num_rows], 8-byte aligned.
 *  k_out          (device) uint8 [num_rows, 128], 8-byte aligned.
 *  scale_out      (device) fp32 [num_rows], 4-byte aligned.
 *  num_rows >= 0 (0: no launch); num_blocks, block_size >= 1, num_blocks*block_size <= 2^32.
 * Returns a dsv4_status.
 */
int dsv4_indexer_k_gather(const uint8_t *indexer_cache, int64_t num_blocks, int32_t block_size,
                          const int64_t *slots, int64_t num_rows, uint8_t *k_out,
                          float *scale_out, int32_t *device_error, void *stream);

/* Bytes of an indexer cache of num_blocks x block_size slots: num_blocks*block_size*132. */
size_t dsv4_indexer_cache_bytes(int64_t num_blocks, int32_t block_size);

/*
 * Check of the failure path of the bulk-copy kernel (the KV-row kernel that
 * KV-only batches run): its waits on mbarriers give up after a budget of SM clock
 * cycles instead of waiting without bound.  This launches one warp that waits,
 * through the same code, on an mbarrier whose phase nothing completes.  After
 * max_cycles cycles (0, or anything above the kernels' own limit of 2^31 cycles,
 * about one second at 2 GHz: that limit) it ORs DSV4_DEVERR_TIMEOUT into
 * *device_error (device int32, nullable) and returns; the GPU context stays
 * usable.  Asynchronous on `stream` (cudaStream_t).  Returns DSV4_ERR_VALUE for
 * max_cycles < 0, DSV4_ERR_CUDA if the launch fails, else DSV4_OK.
 */
int dsv4_check_bounded_wait(int64_t max_cycles, int32_t *device_error, void *stream);

/*
 * Debug aid of the checked build.  libdsv4kv_checked.so is the same library
 * compiled with DSV4_CHECK_BOUNDS: before every global load or store, each kernel
 * tests that the bytes it touches lie inside the buffer the access belongs to
 * (q, kv, weight, positions, slots, cos/sin, cache, outputs; extents from the
 * call's sizes).  An access that would leave its buffer is skipped and
 * DSV4_DEVERR_BOUNDS is OR-ed into *device_error (where the entry point has one)
 * and into a flag of the library.  This returns that flag, synchronising the
 * current device first, and clears it when `reset` is nonzero: 0 if no access was
 * skipped since the last reset, DSV4_DEVERR_BOUNDS if one was, DSV4_ERR_CUDA
 * negated (-5) if reading it failed.  The release library (libdsv4kv.so) records
 * nothing and returns -1.  The pages record two address faults of this operator
 * on other hardware (FlagGems-vllm PR #684, "Performance against a baseline": a
 * 32-bit index past 2^31 q elements, a KV store into the rope region).
 */
int dsv4_debug_bounds_flags(int reset);

/* Static string naming a dsv4_status value ("unknown status" otherwise). */
const char *dsv4_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* DSV4KV_H */
