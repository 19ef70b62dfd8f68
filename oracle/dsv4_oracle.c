/*
 * CPU oracle of the fused DeepSeek-V4 attention-input step: q-norm + RoPE (in
 * place), KV norm + RoPE + UE8M0/E4M3 quantisation + paged-cache insert.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline / reference arm may load this library.  The CUDA
 * library never calls it and shares no source with it.
 *
 * It is written to be checked by eye against the definition, not to be fast:
 * every value is widened exactly to double, every sum is a plain left-to-right
 * loop, and rounding happens once, at the store, with explicit
 * round-to-nearest-even encoders.  Compiled with -ffp-contract=off so that
 * a*b - c*d is two products and a difference, as written.
 *
 * Sources (pages on the operator this library restates):
 *  [FG] FlagGems-vllm PR #684, "fused_deepseek_v4_qnorm_rope_kv_rope_quant_insert
 *       backends, plus test and benchmark fixes".
 *  [SG] SGLang PR #33358, "DSv4 flashmla norm-rope: K-tokens-per-block ILP to
 *       hide load latency".
 *  [VL] vLLM API page of minimax_m3 finalize_allreduce_norm (_f32x4_to_e4m3x4,
 *       _ue8m0_ceil, _ue8m0_inverse).
 *
 * Per token t (readings of open points are listed in the design notes):
 *   Q:  for every head h, x = q[t,h,:]; r = 1/sqrt(sum(x^2)/512 + eps);
 *       y = x*r (weightless, [FG] "Ascend 910B": the eager baseline uses a
 *       weightless RMSNorm); rotate the pairs (448+2i, 449+2i) by the angle of
 *       row positions[t] of the cos/sin table (cos in columns 0..31, sin in
 *       32..63; [FG] "Ascend 910B": 256 bytes of cos/sin per position);
 *       q[t,h,:] = bf16(y).  No intermediate rounding before the rotation
 *       ([FG] "Ascend 910B": rounding the normalised value first stops matching
 *       the operator's arithmetic).
 *   KV: x = kv[t,:]; the same r; v = x*r*w with the learned weight w
 *       ([SG] "Motivation", "Modifications": RMSNorm over 512 with a weight
 *       loaded once); rotate v[448..511] as above.
 *   FP8 store ([FG] title; [SG] "Accuracy Tests": 448 E4M3 bytes, 7 UE8M0
 *       exponents per 64-element group, bf16 rope tail): for block b < 7,
 *       amax = max |v| over the block; s = the smallest integer with
 *       amax <= 448 * 2^s, clamped to [-127, 127]; scale byte s + 127
 *       ([VL] _ue8m0_inverse: the scale is 2^(byte - 127)); payload
 *       E4M3(v * 2^-s), an exact power-of-two scaling ([FG] "The seven test
 *       and benchmark fixes": build the power of two exactly, never via exp2).
 *   bf16 store ([SG] "Motivation", kBf16Store): bf16(v) for all 512 dims.
 *   slot_mapping[t] < 0: no cache write; q is still rewritten.
 *   KV already normalised (kv_norm = 0): v = x, rotated as above, with no
 *       norm and no weight.  The [FG] operator's name (qnorm + rope, kv rope +
 *       quant + insert) and its eager baseline in "Ascend 910B" (a weightless
 *       RMSNorm of q, RoPE, the FP8 encoder, a scatter into the cache) apply no
 *       norm to KV.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { HEAD = 512, ROPE = 64, NOPE = 448, QBLK = 64, NQBLK = 7 };
enum { FP8_DATA_BYTES = 576, FP8_SCALE_BYTES = 8, FP8_SLOT_BYTES = 584 };
enum { ERR_SLOT_RANGE = 1, ERR_POS_RANGE = 2 };

/* ---------------------------------------------------------------- encoders */

/* exact value of a bfloat16 bit pattern: 1 sign, 8 exponent (bias 127), 7 mantissa bits */
double oracle_bf16_value(uint16_t bits)
{
    int sign = bits >> 15;
    int ef = (bits >> 7) & 0xFF;
    int m = bits & 0x7F;
    double mag;
    if (ef == 0xFF)
        mag = m ? NAN : INFINITY;
    else if (ef == 0)
        mag = ldexp((double)m, -133);            /* subnormal: m * 2^-126 * 2^-7 */
    else
        mag = ldexp((double)(128 + m), ef - 134); /* (1 + m/128) * 2^(ef-127) */
    return sign ? -mag : mag;
}

/*
 * Round n_real = a / 2^qe (a >= 0) to the nearest integer, ties to even.
 * a / 2^qe is an exact power-of-two scaling, so scaled, its floor and the
 * remainder below are all exact in double.
 */
static uint64_t round_half_even_scaled(double a, int qe)
{
    double scaled = ldexp(a, -qe);
    double fl = floor(scaled);
    double rem = scaled - fl;
    uint64_t n = (uint64_t)fl;
    if (rem > 0.5 || (rem == 0.5 && (n & 1u)))
        n += 1;
    return n;
}

/* nearest bfloat16 to x, ties to even; overflow to +-inf as IEEE rounding does */
uint16_t oracle_bf16_rne(double x)
{
    if (isnan(x))
        return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7F80;
    int ex;
    (void)frexp(a, &ex);
    int e = ex - 1;          /* a in [2^e, 2^(e+1)) */
    if (e < -126)
        e = -126;            /* below the normal range the spacing stays 2^-133 */
    int qe = e - 7;          /* spacing of bf16 values next to a */
    uint64_t n = round_half_even_scaled(a, qe);
    if (n == 256) {          /* rounded up into the next binade */
        n = 128;
        qe += 1;
    }
    if (n < 128)             /* subnormal (qe == -133) */
        return sign | (uint16_t)n;
    int field = qe + 134;    /* exponent field of n * 2^qe, n in [128, 256) */
    if (field >= 255)
        return sign | 0x7F80;
    return sign | (uint16_t)(field << 7) | (uint16_t)(n - 128);
}

/*
 * nearest E4M3 (the "fn" variant: bias 7, no infinities, 0x7F/0xFF are NaN,
 * largest finite 448 = 1.75 * 2^8) to x, ties to even.  Subnormals are
 * m * 2^-9 for m = 1..7; exponent field 15 with mantissa 0..6 are normal
 * values (256 .. 448).  Magnitudes >= 448 saturate to 448: the quantiser
 * never produces them (|v| * 2^-s <= 448 by the choice of s).
 */
uint8_t oracle_e4m3_rne(double x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs(x);
    if (a >= 448.0)
        return sign | 0x7E;
    if (a == 0.0)
        return sign;
    int ex;
    (void)frexp(a, &ex);
    int e = ex - 1;          /* a in [2^e, 2^(e+1)) */
    if (e < -6)
        e = -6;              /* subnormal spacing 2^-9 */
    int qe = e - 3;          /* 3 mantissa bits */
    uint64_t n = round_half_even_scaled(a, qe);
    if (n == 16) {
        n = 8;
        qe += 1;
    }
    if (n < 8)               /* subnormal (qe == -9) */
        return sign | (uint8_t)n;
    int field = qe + 10;     /* n * 2^qe with n in [8, 16): exponent e = qe + 3, field e + 7 */
    return sign | (uint8_t)(field << 3) | (uint8_t)(n - 8);
}

/*
 * UE8M0 block exponent: the smallest integer s with amax <= 448 * 2^s,
 * clamped to [-127, 127].  amax = 0 gives -127 (scale byte 0).
 * The search starts at ex - 10 (raised to -127, capped at 127), where
 * amax >= 2^(ex-1) > 448 * 2^(ex-10), so the predicate is false there and
 * the first s that satisfies it is the smallest one.  ldexp(448, s) is exact.
 */
int oracle_ue8m0_exponent(double amax)
{
    int s = -127;
    if (amax > 0.0) {
        int ex;
        (void)frexp(amax, &ex);
        if (ex - 10 > s)
            s = ex - 10;
        if (s > 127)
            s = 127;
    }
    while (s < 127 && amax > ldexp(448.0, s))
        s++;
    return s;
}

/* ------------------------------------------------------------ row algebra */

/* RoPE on the trailing 64 dims of a 512-vector: GPT-J interleaved pairs */
static void rotate_tail(double *y, const float *cs)
{
    for (int i = 0; i < ROPE / 2; ++i) {
        double a = y[NOPE + 2 * i];
        double b = y[NOPE + 2 * i + 1];
        double c = (double)cs[i];
        double s = (double)cs[ROPE / 2 + i];
        y[NOPE + 2 * i] = a * c - b * s;
        y[NOPE + 2 * i + 1] = b * c + a * s;
    }
}

/* 1 / sqrt(mean(x^2) + eps) of a bf16 row, sum taken left to right in double */
static double inv_rms(const uint16_t *x, double eps)
{
    double ss = 0.0;
    for (int d = 0; d < HEAD; ++d) {
        double xd = oracle_bf16_value(x[d]);
        ss += xd * xd;
    }
    return 1.0 / sqrt(ss / (double)HEAD + eps);
}

/* normalised and rotated q head (no weight), before rounding */
void oracle_q_values(const uint16_t *x, const float *cs, float eps, double *y)
{
    double r = inv_rms(x, (double)eps);
    for (int d = 0; d < HEAD; ++d)
        y[d] = oracle_bf16_value(x[d]) * r;
    rotate_tail(y, cs);
}

/* KV row that arrives normalised: only rotated, before rounding or quantisation */
void oracle_kv_rope_values(const uint16_t *x, const float *cs, double *v)
{
    for (int d = 0; d < HEAD; ++d)
        v[d] = oracle_bf16_value(x[d]);
    rotate_tail(v, cs);
}

/* normalised, weighted and rotated KV row, before rounding or quantisation */
void oracle_kv_values(const uint16_t *x, const uint16_t *w, const float *cs, float eps, double *v)
{
    double r = inv_rms(x, (double)eps);
    for (int d = 0; d < HEAD; ++d)
        v[d] = oracle_bf16_value(x[d]) * r * oracle_bf16_value(w[d]);
    rotate_tail(v, cs);
}

static void put_bf16_le(uint8_t *p, uint16_t b)
{
    p[0] = (uint8_t)(b & 0xFF);
    p[1] = (uint8_t)(b >> 8);
}

/*
 * FP8 slot image (584 bytes of one paged-cache slot, split in two places):
 *   data  [576]: E4M3 of dims 0..447, then dims 448..511 as little-endian bf16
 *   scale [8]  : the 7 UE8M0 exponent bytes of blocks 0..6, then a 0 pad byte
 */
void oracle_fp8_slot(const double *v, uint8_t *data, uint8_t *scale)
{
    for (int b = 0; b < NQBLK; ++b) {
        double amax = 0.0;
        for (int d = b * QBLK; d < (b + 1) * QBLK; ++d)
            if (fabs(v[d]) > amax)
                amax = fabs(v[d]);
        int s = oracle_ue8m0_exponent(amax);
        scale[b] = (uint8_t)(s + 127);
        for (int d = b * QBLK; d < (b + 1) * QBLK; ++d)
            data[d] = oracle_e4m3_rne(ldexp(v[d], -s));
    }
    scale[NQBLK] = 0;
    for (int d = NOPE; d < HEAD; ++d)
        put_bf16_le(data + NOPE + 2 * (d - NOPE), oracle_bf16_rne(v[d]));
}

/* ----------------------------------------------------------------- driver */

typedef struct {
    int store_bf16;
    int kv_norm;
    uint16_t *q;
    const uint16_t *kv, *w;
    const int64_t *pos;
    const float *cs;
    int64_t max_pos;
    const int64_t *slot;
    uint8_t *cache;
    int64_t num_blocks;
    int32_t bs;
    int64_t t0, t1;
    int32_t H;
    float eps;
    int32_t err;
} job_t;

static void *run_tokens(void *arg)
{
    job_t *j = (job_t *)arg;
    double y[HEAD];
    const int64_t num_slots = j->num_blocks * (int64_t)j->bs;
    for (int64_t t = j->t0; t < j->t1; ++t) {
        int64_t p = j->pos[t];
        if (p < 0 || p >= j->max_pos) {
            j->err |= ERR_POS_RANGE; /* token skipped entirely */
            continue;
        }
        const float *cs = j->cs + p * ROPE;
        for (int32_t h = 0; h < j->H; ++h) {
            uint16_t *x = j->q + (t * j->H + h) * HEAD;
            oracle_q_values(x, cs, j->eps, y);
            for (int d = 0; d < HEAD; ++d)
                x[d] = oracle_bf16_rne(y[d]);
        }
        if (!j->kv || !j->slot)
            continue;
        int64_t slot = j->slot[t];
        if (slot < 0)
            continue;
        if (slot >= num_slots) {
            j->err |= ERR_SLOT_RANGE;
            continue;
        }
        if (j->kv_norm)
            oracle_kv_values(j->kv + t * HEAD, j->w, cs, j->eps, y);
        else
            oracle_kv_rope_values(j->kv + t * HEAD, cs, y);
        int64_t blk = slot / j->bs, off = slot % j->bs;
        if (j->store_bf16) {
            uint8_t *row = j->cache + slot * (int64_t)(HEAD * 2);
            for (int d = 0; d < HEAD; ++d)
                put_bf16_le(row + 2 * d, oracle_bf16_rne(y[d]));
        } else {
            uint8_t *base = j->cache + blk * (int64_t)j->bs * FP8_SLOT_BYTES;
            oracle_fp8_slot(y, base + off * FP8_DATA_BYTES,
                            base + (int64_t)j->bs * FP8_DATA_BYTES + off * FP8_SCALE_BYTES);
        }
    }
    return NULL;
}

/*
 * Whole-batch oracle.  q [T,H,512] bf16 is rewritten in place (H may be 0);
 * kv [T,512] (NULL: no cache writes), normalised with w when kv_norm is 1,
 * taken as already normalised when 0; cache is the poisoned pre-image, of
 * num_blocks*block_size*584 bytes (FP8) or num_blocks*block_size*1024 (bf16).
 * Returns the OR of ERR_* bits.  Tokens are independent, so threads split
 * them into contiguous ranges; the result does not depend on the split.
 */
int32_t oracle_qnorm_rope_kv_insert(int store_bf16, int kv_norm, uint16_t *q, const uint16_t *kv,
                                    const uint16_t *w, const int64_t *positions,
                                    const float *cos_sin, int64_t max_position,
                                    const int64_t *slot_mapping, uint8_t *cache,
                                    int64_t num_blocks, int32_t block_size, int64_t T,
                                    int32_t H, float eps, int n_threads)
{
    if (n_threads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        n_threads = n > 0 ? (int)n : 1;
    }
    if (n_threads > 256)
        n_threads = 256;
    if (n_threads > T)
        n_threads = T > 0 ? (int)T : 1;
    job_t jobs[256];
    pthread_t th[256];
    int64_t per = (T + n_threads - 1) / n_threads;
    for (int i = 0; i < n_threads; ++i) {
        int64_t a = i * per, b = a + per;
        if (a > T) a = T;
        if (b > T) b = T;
        jobs[i] = (job_t){store_bf16, kv_norm, q, kv, w, positions, cos_sin, max_position, slot_mapping,
                          cache, num_blocks, block_size, a, b, H, eps, 0};
    }
    for (int i = 1; i < n_threads; ++i)
        pthread_create(&th[i], NULL, run_tokens, &jobs[i]);
    run_tokens(&jobs[0]);
    int32_t err = jobs[0].err;
    for (int i = 1; i < n_threads; ++i) {
        pthread_join(th[i], NULL);
        err |= jobs[i].err;
    }
    return err;
}

/* ------------------------------------------- reading the FP8 cache back out */

/* exact value of an E4M3 ("fn") code: bias 7, subnormals m * 2^-9, 0x7F/0xFF NaN */
double oracle_e4m3_value(uint8_t code)
{
    int sign = code >> 7;
    int ef = (code >> 3) & 0xF;
    int m = code & 7;
    double mag;
    if (ef == 15 && m == 7)
        mag = NAN;
    else if (ef == 0)
        mag = ldexp((double)m, -9);
    else
        mag = ldexp((double)(8 + m), ef - 10); /* (1 + m/8) * 2^(ef-7) */
    return sign ? -mag : mag;
}

/*
 * Dequantise-and-gather: out[n, :] (bf16 [n_rows, 512]) = the row stored at
 * slots[n] of an FP8 cache (layout of oracle_fp8_slot), dims 0..447 as
 * bf16(E4M3 value * 2^(e_b - 127)), dims 448..511 copied.  A negative slot
 * gives a zero row (the sparse-attention gather of 1Cat-vLLM PR #1280,
 * "Purpose" item 2, writes zeros for unused slots); a slot past the cache
 * also gives a zero row and sets ERR_SLOT_RANGE.  The reader of the cache
 * (same PR, item 5: dequantize_and_gather_k_cache).
 */
int32_t oracle_dequant_gather(const uint8_t *cache, int64_t num_blocks, int32_t block_size,
                              const int64_t *slots, int64_t n_rows, uint16_t *out)
{
    int32_t err = 0;
    const int64_t num_slots = num_blocks * (int64_t)block_size;
    for (int64_t n = 0; n < n_rows; ++n) {
        uint16_t *row = out + n * HEAD;
        int64_t slot = slots[n];
        if (slot < 0 || slot >= num_slots) {
            if (slot >= num_slots)
                err |= ERR_SLOT_RANGE;
            memset(row, 0, HEAD * sizeof(uint16_t));
            continue;
        }
        int64_t blk = slot / block_size, off = slot % block_size;
        const uint8_t *base = cache + blk * (int64_t)block_size * FP8_SLOT_BYTES;
        const uint8_t *data = base + off * FP8_DATA_BYTES;
        const uint8_t *scale = base + (int64_t)block_size * FP8_DATA_BYTES + off * FP8_SCALE_BYTES;
        for (int d = 0; d < NOPE; ++d)
            row[d] = oracle_bf16_rne(ldexp(oracle_e4m3_value(data[d]), (int)scale[d / QBLK] - 127));
        for (int d = NOPE; d < HEAD; ++d) {
            const uint8_t *p = data + NOPE + 2 * (d - NOPE);
            row[d] = (uint16_t)(p[0] | (p[1] << 8));
        }
    }
    return err;
}

/* ------------------- residual add + Gemma RMSNorm + MXFP8 (32-element blocks) */

/*
 * The single-GPU part of the vLLM minimax_m3 finalize_allreduce_norm page
 * (_LamportGemmaRMSNormMxfp8Kernel): with one rank there is no all-reduce, so
 * for each row
 *   prenorm = bf16(x + residual)                 (also the new residual)
 *   r       = 1 / sqrt(mean(prenorm^2) + eps)
 *   normed  = bf16(prenorm * r * (1 + gamma))    (Gemma: the scale is 1 + w;
 *                                                 the page rounds to bf16 here)
 * and for each block of 32 normed values
 *   e       = UE8M0 of amax * (1/448), both factors and the product in fp32
 *             (the page's _ue8m0_ceil of amax * Float32(1.0 / 448.0))
 *   code    = E4M3_rn_satfinite(normed * 2^(127 - e))   (0 when e is 0 or 254:
 *             the page's _ue8m0_inverse)
 * Scales go to the 128x4 swizzled layout (_swizzled_scale_offset); the scales
 * of the padding rows up to the next multiple of 128 rows are zero.
 */

/* smallest e in [0, 254] with x <= 2^(e - 127) (254 if none); 0 for x <= 0.
 * For x > 0 this is ceil(log2 x) + 127, clamped: the exponent of the next
 * power of two at or above x. */
int oracle_ue8m0_of_f32(float x)
{
    if (!(x > 0.0f))
        return 0;
    for (int e = 0; e < 254; ++e)
        if ((double)x <= ldexp(1.0, e - 127))
            return e;
    return 254;
}

/* the page's inverse scale: 2^(127 - e), except 0 for e = 0 and for e = 254 */
double oracle_ue8m0_inverse(int e)
{
    if (e == 0 || e >= 254)
        return 0.0;
    return ldexp(1.0, 127 - e);
}

/* byte offset of block col of row in the 128x4 swizzled scale layout */
int64_t oracle_swizzled_scale_offset(int64_t row, int64_t col, int64_t padded_cols)
{
    int64_t tile = (row / 128) * 128 * padded_cols + (col / 4) * 512;
    return tile + (row % 32) * 16 + ((row % 128) / 32) * 4 + col % 4;
}

int64_t oracle_mxfp8_scale_bytes(int64_t m, int64_t n)
{
    int64_t rows = (m + 127) / 128 * 128;
    int64_t cols = (n / 32 + 3) / 4 * 4;
    return rows * cols;
}

/* x, residual: bf16 [m, n]; gamma bf16 [n]; n a multiple of 128.  Writes
 * residual_out bf16 [m, n], codes [m, n] (E4M3) and scales (all
 * oracle_mxfp8_scale_bytes(m, n) bytes, padding rows zeroed). */
void oracle_gemma_rmsnorm_mxfp8(const uint16_t *x, const uint16_t *residual, const uint16_t *gamma,
                                int64_t m, int64_t n, float eps, uint16_t *residual_out,
                                uint8_t *codes, uint8_t *scales)
{
    const int64_t cols = n / 32, padded_cols = (cols + 3) / 4 * 4;
    const float inv448 = (float)(1.0 / 448.0);
    memset(scales, 0, (size_t)oracle_mxfp8_scale_bytes(m, n));
    double *pre = (double *)malloc((size_t)n * sizeof(double));
    double *normed = (double *)malloc((size_t)n * sizeof(double));
    for (int64_t row = 0; row < m; ++row) {
        const uint16_t *xr = x + row * n, *rr = residual + row * n;
        double ss = 0.0;
        for (int64_t d = 0; d < n; ++d) {
            uint16_t p = oracle_bf16_rne(oracle_bf16_value(xr[d]) + oracle_bf16_value(rr[d]));
            residual_out[row * n + d] = p;
            pre[d] = oracle_bf16_value(p);
            ss += pre[d] * pre[d];
        }
        const double r = 1.0 / sqrt(ss / (double)n + (double)eps);
        for (int64_t d = 0; d < n; ++d)
            normed[d] = oracle_bf16_value(
                oracle_bf16_rne(pre[d] * r * (1.0 + oracle_bf16_value(gamma[d]))));
        for (int64_t c = 0; c < cols; ++c) {
            double amax = 0.0;
            for (int64_t d = 32 * c; d < 32 * c + 32; ++d)
                if (fabs(normed[d]) > amax)
                    amax = fabs(normed[d]);
            const float scaled = (float)amax * inv448; /* fp32 product, as on the page */
            const int e = oracle_ue8m0_of_f32(scaled);
            const double inv = oracle_ue8m0_inverse(e);
            for (int64_t d = 32 * c; d < 32 * c + 32; ++d)
                codes[row * n + d] = oracle_e4m3_rne(normed[d] * inv);
            scales[oracle_swizzled_scale_offset(row, c, padded_cols)] = (uint8_t)e;
        }
    }
    free(pre);
    free(normed);
}

/* ------------------------------------------------- array forms for the tests */

void oracle_bf16_rne_array(const double *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_rne(x[i]);
}

void oracle_e4m3_rne_array(const double *x, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_rne(x[i]);
}

void oracle_bf16_value_array(const uint16_t *b, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_value(b[i]);
}

void oracle_e4m3_value_array(const uint8_t *c, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_value(c[i]);
}

void oracle_ue8m0_exponent_array(const double *amax, int32_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_ue8m0_exponent(amax[i]);
}

/* ------------------------------------------------ indexer-K quant + insert */

/*
 * The lightning indexer scores queries against K rows that arrive as a
 * contiguous [N, 128] E4M3 buffer with one non-negative fp32 scale per row
 * (rocm-aiter PR #1, "Motivation": kv_scale[n], the K rows gathered out of the
 * paged cache beforehand), and the norm-rope-store kernel keeps a separate
 * indexer path ([SG] "Modifications").  Per token t with a valid slot:
 *   amax  = max |k[t, d]| over the 128 dims (exact: the inputs are bf16)
 *   s     = the smallest integer with amax <= 448 * 2^s, clamped to [-127, 127]
 *           (the same power-of-two rule as the 64-element blocks above)
 *   scale = 2^s as fp32 (exact, 2^-127 being an fp32 subnormal)
 *   code  = E4M3(k[t, d] * 2^-s)
 * Cache layout, chosen like the FP8 KV cache's: block b occupies
 * [b*bs*132, (b+1)*bs*132); slot o's 128 codes sit at b*bs*132 + o*128 and its
 * scale (little-endian fp32) at b*bs*132 + bs*128 + o*4.
 * slot < 0: nothing written; slot >= num_blocks * bs: nothing written and
 * error bit ERR_SLOT_RANGE.
 */
enum { IDX_DIM = 128, IDX_SLOT_BYTES = 132 };

static void put_f32_le(uint8_t *p, float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    for (int i = 0; i < 4; ++i)
        p[i] = (uint8_t)(u >> (8 * i));
}

static float get_f32_le(const uint8_t *p)
{
    uint32_t u = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) |
                 ((uint32_t)p[3] << 24);
    float f;
    memcpy(&f, &u, 4);
    return f;
}

int32_t oracle_indexer_k_quant_insert(const uint16_t *k, const int64_t *slots, uint8_t *cache,
                                      int64_t num_blocks, int32_t block_size, int64_t num_tokens)
{
    int32_t err = 0;
    const int64_t num_slots = num_blocks * (int64_t)block_size;
    for (int64_t t = 0; t < num_tokens; ++t) {
        const int64_t slot = slots[t];
        if (slot < 0)
            continue;
        if (slot >= num_slots) {
            err |= ERR_SLOT_RANGE;
            continue;
        }
        const uint16_t *row = k + t * IDX_DIM;
        double amax = 0.0;
        for (int d = 0; d < IDX_DIM; ++d) {
            double a = fabs(oracle_bf16_value(row[d]));
            if (a > amax)
                amax = a;
        }
        const int s = oracle_ue8m0_exponent(amax);
        const int64_t blk = slot / block_size, off = slot % block_size;
        uint8_t *base = cache + blk * (int64_t)block_size * IDX_SLOT_BYTES;
        uint8_t *codes = base + off * IDX_DIM;
        for (int d = 0; d < IDX_DIM; ++d)
            codes[d] = oracle_e4m3_rne(ldexp(oracle_bf16_value(row[d]), -s));
        put_f32_le(base + (int64_t)block_size * IDX_DIM + off * 4, (float)ldexp(1.0, s));
    }
    return err;
}

/*
 * The reader the indexer's prefill path calls before scoring: for each n, the
 * 128 codes and the fp32 scale stored at slots[n], copied unchanged into
 * contiguous k_out [n, 128] and scale_out [n].  A negative slot gives zero
 * codes and scale 0; a slot past the cache the same plus ERR_SLOT_RANGE.
 */
int32_t oracle_indexer_k_gather(const uint8_t *cache, int64_t num_blocks, int32_t block_size,
                                const int64_t *slots, int64_t n_rows, uint8_t *k_out,
                                float *scale_out)
{
    int32_t err = 0;
    const int64_t num_slots = num_blocks * (int64_t)block_size;
    for (int64_t n = 0; n < n_rows; ++n) {
        const int64_t slot = slots[n];
        if (slot < 0 || slot >= num_slots) {
            if (slot >= num_slots)
                err |= ERR_SLOT_RANGE;
            memset(k_out + n * IDX_DIM, 0, IDX_DIM);
            scale_out[n] = 0.0f;
            continue;
        }
        const int64_t blk = slot / block_size, off = slot % block_size;
        const uint8_t *base = cache + blk * (int64_t)block_size * IDX_SLOT_BYTES;
        memcpy(k_out + n * IDX_DIM, base + off * IDX_DIM, IDX_DIM);
        scale_out[n] = get_f32_le(base + (int64_t)block_size * IDX_DIM + off * 4);
    }
    return err;
}
