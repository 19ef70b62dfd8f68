/*
 * Seeded, counter-based synthetic input generator.
 *
 * Shared by the tests, the benchmark and the smoke check on both sides of
 * every comparison (the CPU oracle and the CUDA path).  It holds none of the
 * fused operator's arithmetic: it only draws numbers.  Every element is a pure
 * function of (seed, tensor id, element index), so any slice of a tensor can be
 * regenerated on its own, in any order, on any number of threads, and gives
 * the same bits on x86-64 and AArch64 hosts as long as the C library's log,
 * cos and sin agree there (they are only used for the Gaussian draw, never for
 * the operator itself).
 *
 *   key(seed, id, i) = splitmix64(seed * 2^40 + id * 2^36 + i)
 *
 * splitmix64 is Steele, Lea and Flood's SplitMix finaliser ("Fast splittable
 * pseudorandom number generators", OOPSLA 2014): add the golden-ratio
 * increment, then two xor-shift-multiply rounds and a final xor-shift.
 *
 * Normals come from the Box-Muller transform (Box and Muller, 1958) on two
 * uniforms in (0, 1]; element 2p takes the cosine branch of pair p and element
 * 2p+1 the sine branch.  The value mean + std * z (times `tail_mult` for the
 * elements whose tail draw falls below `tail_frac`) is rounded once, to
 * nearest-even, directly from double to bfloat16.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>
#include <unistd.h>

static uint64_t splitmix64(uint64_t x)
{
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

uint64_t synth_key(uint64_t seed, uint64_t tensor_id, uint64_t index)
{
    return splitmix64((seed << 40) + (tensor_id << 36) + index);
}

/* uniform in (0, 1]: the top 53 bits, plus one, times 2^-53 */
static double unit_open0(uint64_t bits)
{
    return ldexp((double)((bits >> 11) + 1ull), -53);
}

/* nearest bfloat16 to a finite double, ties to even (inputs only) */
static uint16_t input_to_bf16(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    int ex;
    (void)frexp(a, &ex); /* a in [2^(ex-1), 2^ex) */
    int e = ex - 1;
    if (e < -126) {
        /* subnormal range: multiples of 2^-133 */
        double m = rint(ldexp(a, 133)); /* exact scaling, then ties-to-even */
        return (uint16_t)(sign | (uint16_t)m);
    }
    double m = rint(ldexp(a, 7 - e)); /* in [128, 256] */
    if (m >= 256.0) {
        m = 128.0;
        e += 1;
    }
    if (e > 127)
        return (uint16_t)(sign | 0x7F80u);
    return (uint16_t)(sign | (uint16_t)((e + 127) << 7) | (uint16_t)((int)m - 128));
}

static double normal_at(uint64_t seed, uint64_t id, uint64_t i)
{
    uint64_t p = i >> 1;
    double u1 = unit_open0(synth_key(seed, id, 2 * p));
    double u2 = unit_open0(synth_key(seed, id, 2 * p + 1));
    double rad = sqrt(-2.0 * log(u1));
    double ang = 6.283185307179586476925286766559 * u2;
    return (i & 1) ? rad * sin(ang) : rad * cos(ang);
}

typedef struct {
    uint16_t *out;
    uint64_t seed, id, tail_id, start, begin, end;
    double mean, std, tail_frac, tail_mult;
} normal_job;

static void *normal_worker(void *arg)
{
    normal_job *j = (normal_job *)arg;
    for (uint64_t k = j->begin; k < j->end; ++k) {
        uint64_t i = j->start + k;
        double v = j->mean + j->std * normal_at(j->seed, j->id, i);
        if (j->tail_frac > 0.0 && unit_open0(synth_key(j->seed, j->tail_id, i)) <= j->tail_frac)
            v *= j->tail_mult;
        j->out[k] = input_to_bf16(v);
    }
    return NULL;
}

static int pick_threads(int n_threads, uint64_t count)
{
    if (n_threads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        n_threads = n > 0 ? (int)n : 1;
    }
    if (n_threads > 256)
        n_threads = 256;
    if ((uint64_t)n_threads > count / 65536 + 1)
        n_threads = (int)(count / 65536 + 1);
    return n_threads;
}

/*
 * Fill out[0..count) with elements start..start+count of a bf16 N(mean, std)
 * tensor.  tail_frac > 0 multiplies a tail_frac share of elements (chosen by
 * the independent stream tail_id) by tail_mult before rounding.
 */
void synth_normal_bf16(uint16_t *out, uint64_t seed, uint64_t tensor_id, uint64_t start,
                       uint64_t count, double mean, double std, double tail_frac,
                       double tail_mult, uint64_t tail_id, int n_threads)
{
    int nt = pick_threads(n_threads, count);
    normal_job jobs[256];
    pthread_t th[256];
    uint64_t per = (count + (uint64_t)nt - 1) / (uint64_t)nt;
    for (int t = 0; t < nt; ++t) {
        uint64_t b = (uint64_t)t * per, e = b + per;
        if (b > count) b = count;
        if (e > count) e = count;
        jobs[t] = (normal_job){out, seed, tensor_id, tail_id, start, b, e,
                               mean, std, tail_frac, tail_mult};
    }
    for (int t = 1; t < nt; ++t)
        pthread_create(&th[t], NULL, normal_worker, &jobs[t]);
    normal_worker(&jobs[0]);
    for (int t = 1; t < nt; ++t)
        pthread_join(th[t], NULL);
}

/* raw 64-bit draws key(seed, id, start + k) for k < count */
void synth_u64(uint64_t *out, uint64_t seed, uint64_t tensor_id, uint64_t start, uint64_t count)
{
    for (uint64_t k = 0; k < count; ++k)
        out[k] = synth_key(seed, tensor_id, start + k);
}

typedef struct {
    uint8_t *out;
    uint64_t seed, id, begin, end;
} bytes_job;

static void *bytes_worker(void *arg)
{
    bytes_job *j = (bytes_job *)arg;
    /* byte i is the low byte of key(seed, id, i / 8) shifted by 8 * (i % 8) */
    for (uint64_t i = j->begin; i < j->end; ++i)
        j->out[i] = (uint8_t)(synth_key(j->seed, j->id, i >> 3) >> (8 * (i & 7)));
    return NULL;
}

/* count pseudo-random bytes (used as a poison pre-image for output buffers) */
void synth_bytes(uint8_t *out, uint64_t seed, uint64_t tensor_id, uint64_t count, int n_threads)
{
    int nt = pick_threads(n_threads, count);
    bytes_job jobs[256];
    pthread_t th[256];
    uint64_t per = ((count + (uint64_t)nt - 1) / (uint64_t)nt + 7) & ~7ull;
    for (int t = 0; t < nt; ++t) {
        uint64_t b = (uint64_t)t * per, e = b + per;
        if (b > count) b = count;
        if (e > count) e = count;
        jobs[t] = (bytes_job){out, seed, tensor_id, b, e};
    }
    for (int t = 1; t < nt; ++t)
        pthread_create(&th[t], NULL, bytes_worker, &jobs[t]);
    bytes_worker(&jobs[0]);
    for (int t = 1; t < nt; ++t)
        pthread_join(th[t], NULL);
}
