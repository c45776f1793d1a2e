/*
 * Seeded, counter-based input generators for the feed-forward block's workloads.
 *
 * This file draws input tensors only. It holds none of the block's arithmetic (no
 * matmul, no activation, no output rounding) and is shared, as a plain input source,
 * by the test/bench harness for both the CUDA path and the oracle.
 *
 * Generator: element i of a tensor with seed s takes the 64-bit word
 *     r(s, i) = mix(mix(s) + (i + 1) * 0x9E3779B97F4A7C15)
 * where mix() is the SplitMix64 output function (Steele, Lea & Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014). A uniform double in [0,1) is
 * (r >> 11) * 2^-53. Normals use the Box-Muller transform on the word pair
 * (2p, 2p+1): element 2p takes the cosine branch, element 2p+1 the sine branch.
 * Every value is produced in double and rounded to bfloat16 with round-to-nearest-even,
 * then stored as raw 16-bit patterns. Results do not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

static const double SYNTH_TWO_PI = 6.283185307179586476925286766559;

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline uint64_t word_at(uint64_t key, uint64_t i) {
    return mix64(key + (i + 1ull) * 0x9E3779B97F4A7C15ull);
}

/* Uniform in [0, 1) with 53 random bits. */
static inline double unit_open_hi(uint64_t w) { return (double)(w >> 11) * 0x1.0p-53; }
/* Uniform in (0, 1], for the logarithm in Box-Muller. */
static inline double unit_open_lo(uint64_t w) { return (double)((w >> 11) + 1ull) * 0x1.0p-53; }

/* Round a finite double to the nearest bfloat16 (ties to even); returns the 16-bit pattern.
 * The significand is scaled to an integer with 8 significant bits and rounded with
 * nearbyint() under the default round-to-nearest-even mode, which is exact in double. */
static uint16_t to_bf16_bits(double v) {
    if (v == 0.0) return signbit(v) ? 0x8000u : 0u;
    int e;
    double m = frexp(fabs(v), &e);           /* |v| = m * 2^e, m in [0.5, 1) */
    double r = nearbyint(ldexp(m, 8));       /* 128..256 */
    double q = ldexp(r, e - 8);
    float f = (float)q;                      /* exact: q has <= 8 significant bits */
    union { float f; uint32_t u; } cv;
    cv.f = f;
    uint16_t bits = (uint16_t)(cv.u >> 16);
    if (v < 0) bits |= 0x8000u;
    return bits;
}

typedef struct {
    uint16_t* out;
    int64_t begin, end;
    uint64_t key;
    int kind;        /* 0 = normal(0,1), 1 = uniform(-bound, bound) */
    double bound;
} fill_job;

static void* fill_worker(void* arg) {
    fill_job* j = (fill_job*)arg;
    for (int64_t i = j->begin; i < j->end; ++i) {
        double v;
        if (j->kind == 0) {
            uint64_t p = (uint64_t)(i >> 1);
            double u1 = unit_open_lo(word_at(j->key, 2 * p));
            double u2 = unit_open_hi(word_at(j->key, 2 * p + 1));
            double rad = sqrt(-2.0 * log(u1));
            v = (i & 1) ? rad * sin(SYNTH_TWO_PI * u2) : rad * cos(SYNTH_TWO_PI * u2);
        } else {
            double u = unit_open_hi(word_at(j->key, (uint64_t)i));
            v = j->bound * (2.0 * u - 1.0);
        }
        j->out[i] = to_bf16_bits(v);
    }
    return NULL;
}

static int fill(uint16_t* out, int64_t n, uint64_t seed, int kind, double bound, int nthreads) {
    if (n <= 0) return 0;
    if (!out) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (n < 65536) nthreads = 1;
    uint64_t key = mix64(seed);
    fill_job jobs[256];
    pthread_t tids[256];
    int64_t chunk = (n + nthreads - 1) / nthreads;
    chunk = (chunk + 1) & ~(int64_t)1; /* keep Box-Muller pairs in one job (not required, tidy) */
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        int64_t b = (int64_t)t * chunk, e = b + chunk;
        if (b >= n) break;
        if (e > n) e = n;
        jobs[t] = (fill_job){out, b, e, key, kind, bound};
        if (t == 0) continue;
        if (pthread_create(&tids[t], NULL, fill_worker, &jobs[t]) != 0) {
            fill_worker(&jobs[t]);
            tids[t] = 0;
        }
        started = t;
    }
    fill_worker(&jobs[0]);
    for (int t = 1; t <= started; ++t)
        if (tids[t]) pthread_join(tids[t], NULL);
    return 0;
}

int synth_fill_normal_bf16(uint16_t* out, int64_t n, uint64_t seed, int nthreads) {
    return fill(out, n, seed, 0, 0.0, nthreads);
}

int synth_fill_uniform_bf16(uint16_t* out, int64_t n, uint64_t seed, double bound, int nthreads) {
    return fill(out, n, seed, 1, bound, nthreads);
}

/* Raw words, exposed so tests can check the generator against its published definition. */
uint64_t synth_word(uint64_t seed, uint64_t i) { return word_at(mix64(seed), i); }
