/*
 * fmlp oracle: a plain, slow, obviously correct CPU implementation of the transformer
 * feed-forward block, in double precision, for testing the CUDA library against.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the package's smoke check and the benchmark's
 * CPU-baseline leg load this file. It shares no code with the CUDA library.
 *
 * What it computes (source: "Profiling in PyTorch (Part 2): From nn.Linear to a Fused MLP"):
 *   Linear (section "From matmul-add to Linear"; "Why are there no separate mul and add
 *   kernels?"):                      y = x @ W^T + b,  W stored [out, in] as nn.Linear owns it.
 *   GeGLU block (section "Stacking three Linears: the MLP", the SimpleGeGLUMLP forward):
 *       g = x Wg^T, u = x Wu^T, h = gelu_tanh(g), m = h * u, y = m Wd^T, all bias-free.
 *   Linear -> GELU -> Linear with biases (ainews.cool fused-MLP article, technical deep-dive
 *   and benchmark sections):        y = W2 GELU(W1 x + b1) + b2.
 *
 * Inputs are the same bfloat16 bit patterns the GPU reads. Every product and sum is done in
 * double, in plain index order. The only roundings to bfloat16 are the ones the fused GPU
 * path performs: the intermediate (m, or h for the MLP) once, and the output once. With
 * eager_rounding != 0 the oracle instead rounds every tensor the eager PyTorch module would
 * materialise in bf16 (g, u, gelu(g), m; or W1 x + b1 and its GELU), which is the other
 * admissible reading of where rounding happens.
 *
 * GELU: the pages name only `approximate="tanh"`. The formulas are the published ones
 * (Hendrycks & Gimpel, "Gaussian Error Linear Units (GELUs)", 2016):
 *   exact  gelu(x) = 0.5 x (1 + erf(x / sqrt 2))
 *   tanh   gelu(x) = 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))
 * Build without fast-math and without floating-point contraction.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_MAX_THREADS 256

/* ---- bfloat16 <-> double ------------------------------------------------------------ */

static double bf16_value(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to bfloat16 (round to nearest, ties to even) by working on the IEEE-754
 * binary64 fields directly. NaN maps to the canonical quiet NaN 0x7FC0; overflow to +-Inf. */
uint16_t oracle_round_bf16(double v) {
    uint64_t b;
    memcpy(&b, &v, sizeof b);
    uint16_t sign = (uint16_t)((b >> 63) << 15);
    int exp = (int)((b >> 52) & 0x7FF);
    uint64_t frac = b & ((1ull << 52) - 1);
    if (exp == 0x7FF) return frac ? (uint16_t)0x7FC0 : (uint16_t)(sign | 0x7F80);
    if (exp == 0) return sign;                       /* binary64 subnormals are far below bf16's */
    uint64_t sig = frac | (1ull << 52);              /* 53-bit significand */
    int e = exp - 1023 + 127;                        /* bf16 biased exponent */
    if (e >= 1) {
        uint64_t keep = sig >> 45, rem = sig & ((1ull << 45) - 1), half = 1ull << 44;
        if (rem > half || (rem == half && (keep & 1))) ++keep;
        if (keep == (1ull << 8)) { keep >>= 1; ++e; }
        if (e >= 255) return (uint16_t)(sign | 0x7F80);
        return (uint16_t)(sign | (uint16_t)(e << 7) | (uint16_t)(keep & 0x7F));
    }
    /* bf16 subnormal: count units of 2^-133 */
    int s = 942 - exp;                               /* >= 46 here */
    if (s >= 64) return sign;
    uint64_t keep = sig >> s, rem = sig & ((1ull << s) - 1), half = 1ull << (s - 1);
    if (rem > half || (rem == half && (keep & 1))) ++keep;
    return (uint16_t)(sign | (uint16_t)keep);        /* keep == 128 encodes the least normal */
}

static double round_bf16(double v) { return bf16_value(oracle_round_bf16(v)); }

/* ---- GELU ------------------------------------------------------------------------------ */

static double gelu_tanh(double x) {
    const double k = sqrt(2.0 / 3.14159265358979323846264338327950288);
    return 0.5 * x * (1.0 + tanh(k * (x + 0.044715 * x * x * x)));
}

static double gelu_erf(double x) {
    return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));
}

/* ReLU, the hidden activation of the two-layer MLP of the ainews.cool article's technical
 * deep-dive: max(x, 0), with NaN passed through (as torch's relu does) and -0 giving +0. */
static double relu(double x) { return x > 0.0 ? x : (x != x ? x : 0.0); }

/* mode 0 = GELU tanh approximation, 1 = exact GELU (erf), 2 = ReLU */
static double gelu(double x, int mode) {
    return mode == 2 ? relu(x) : (mode == 1 ? gelu_erf(x) : gelu_tanh(x));
}

void oracle_gelu(const double* in, double* out, int64_t n, int mode) {
    for (int64_t i = 0; i < n; ++i) out[i] = gelu(in[i], mode);
}

/* ---- one dense row: out[n] = sum_k a[k] * W[n, k] ------------------------------------- */

static void row_times_wT(const double* a, const uint16_t* W, int64_t K, int64_t N, double* out) {
    for (int64_t n = 0; n < N; ++n) {
        const uint16_t* w = W + n * K;
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) acc += a[k] * bf16_value(w[k]);
        out[n] = acc;
    }
}

/* ---- the three operations, one output row at a time ----------------------------------- */

typedef struct {
    int op;                       /* 0 linear, 1 mlp, 2 geglu */
    const uint16_t *x, *W1, *W2, *W3, *b1, *b2;
    uint16_t* y;                  /* [nrows, out] */
    double* y_acc;                /* [nrows, out] or NULL: value before the final rounding */
    uint16_t* mid;                /* [nrows, hidden] or NULL: the bf16 intermediate */
    int64_t T, D, H, Dout;
    int gelu_mode, eager;
    const int64_t* rows;          /* NULL = 0..T-1 */
    int64_t nrows;
    int64_t next;                 /* work counter, guarded by lock */
    pthread_mutex_t lock;
    int failed;
} job_t;

static int64_t take_row(job_t* j) {
    pthread_mutex_lock(&j->lock);
    int64_t r = j->next < j->nrows ? j->next++ : -1;
    pthread_mutex_unlock(&j->lock);
    return r;
}

static void* worker(void* arg) {
    job_t* j = (job_t*)arg;
    int64_t hid = j->op == 0 ? 0 : j->H;
    int64_t outw = j->op == 0 ? j->H : (j->op == 1 ? j->Dout : j->D);
    int64_t inw = j->D;
    double* a = (double*)malloc(sizeof(double) * (size_t)(inw > 0 ? inw : 1));
    double* t1 = (double*)malloc(sizeof(double) * (size_t)(hid > 0 ? hid : 1));
    double* t2 = (double*)malloc(sizeof(double) * (size_t)(hid > 0 ? hid : 1));
    double* acc = (double*)malloc(sizeof(double) * (size_t)(outw > 0 ? outw : 1));
    if (!a || !t1 || !t2 || !acc) {
        j->failed = 1;
        free(a); free(t1); free(t2); free(acc);
        return NULL;
    }
    int64_t i;
    while ((i = take_row(j)) >= 0) {
        int64_t r = j->rows ? j->rows[i] : i;
        for (int64_t k = 0; k < inw; ++k) a[k] = bf16_value(j->x[r * inw + k]);
        if (j->op == 0) {
            /* y = x W^T + b */
            row_times_wT(a, j->W1, inw, outw, acc);
            if (j->b1)
                for (int64_t n = 0; n < outw; ++n) acc[n] += bf16_value(j->b1[n]);
        } else if (j->op == 1) {
            /* h = GELU(x W1^T + b1); y = h W2^T + b2 */
            row_times_wT(a, j->W1, inw, hid, t1);
            for (int64_t n = 0; n < hid; ++n) {
                double z = t1[n] + (j->b1 ? bf16_value(j->b1[n]) : 0.0);
                if (j->eager) z = round_bf16(z);
                t1[n] = round_bf16(gelu(z, j->gelu_mode));
                if (j->mid) j->mid[i * hid + n] = oracle_round_bf16(t1[n]);
            }
            row_times_wT(t1, j->W2, hid, outw, acc);
            if (j->b2)
                for (int64_t n = 0; n < outw; ++n) acc[n] += bf16_value(j->b2[n]);
        } else {
            /* g = x Wg^T, u = x Wu^T, m = gelu_tanh(g) * u, y = m Wd^T */
            row_times_wT(a, j->W1, inw, hid, t1);
            row_times_wT(a, j->W2, inw, hid, t2);
            for (int64_t n = 0; n < hid; ++n) {
                double g = t1[n], u = t2[n], m;
                if (j->eager) {
                    g = round_bf16(g);
                    u = round_bf16(u);
                    m = round_bf16(round_bf16(gelu_tanh(g)) * u);
                } else {
                    m = round_bf16(gelu_tanh(g) * u);
                }
                t1[n] = m;
                if (j->mid) j->mid[i * hid + n] = oracle_round_bf16(m);
            }
            row_times_wT(t1, j->W3, hid, outw, acc);
        }
        for (int64_t n = 0; n < outw; ++n) {
            j->y[i * outw + n] = oracle_round_bf16(acc[n]);
            if (j->y_acc) j->y_acc[i * outw + n] = acc[n];
        }
    }
    free(a); free(t1); free(t2); free(acc);
    return NULL;
}

static int run(job_t* j, int nthreads) {
    if (j->nrows <= 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > ORACLE_MAX_THREADS) nthreads = ORACLE_MAX_THREADS;
    if (nthreads > j->nrows) nthreads = (int)j->nrows;
    for (int64_t i = 0; i < j->nrows; ++i) {
        int64_t r = j->rows ? j->rows[i] : i;
        if (r < 0 || r >= j->T) return -2;
    }
    pthread_mutex_init(&j->lock, NULL);
    j->next = 0;
    j->failed = 0;
    pthread_t tids[ORACLE_MAX_THREADS];
    int started[ORACLE_MAX_THREADS] = {0};
    for (int t = 1; t < nthreads; ++t)
        started[t] = pthread_create(&tids[t], NULL, worker, j) == 0;
    worker(j);
    for (int t = 1; t < nthreads; ++t)
        if (started[t]) pthread_join(tids[t], NULL);
    pthread_mutex_destroy(&j->lock);
    return j->failed ? -1 : 0;
}

/* y[nrows, out] = bf16(x[rows] W^T + b). b may be NULL. */
int oracle_linear(const uint16_t* x, const uint16_t* W, const uint16_t* b, uint16_t* y,
                  double* y_acc, int64_t T, int64_t in, int64_t out,
                  const int64_t* rows, int64_t nrows, int nthreads) {
    job_t j;
    memset(&j, 0, sizeof j);
    j.op = 0; j.x = x; j.W1 = W; j.b1 = b; j.y = y; j.y_acc = y_acc;
    j.T = T; j.D = in; j.H = out; j.Dout = out;
    j.rows = rows; j.nrows = rows ? nrows : T;
    return run(&j, nthreads);
}

/* h = bf16(GELU(x W1^T + b1)); y = bf16(h W2^T + b2). b1, b2 may be NULL.
 * gelu_mode: 0 GELU tanh, 1 GELU erf, 2 ReLU. h_out (nullable) receives h as bf16 bits [nrows, H]. */
int oracle_mlp_gelu(const uint16_t* x, const uint16_t* W1, const uint16_t* b1,
                    const uint16_t* W2, const uint16_t* b2, uint16_t* y, double* y_acc,
                    uint16_t* h_out, int64_t T, int64_t D, int64_t H, int64_t Dout,
                    int gelu_mode, int eager_rounding,
                    const int64_t* rows, int64_t nrows, int nthreads) {
    job_t j;
    memset(&j, 0, sizeof j);
    j.op = 1; j.x = x; j.W1 = W1; j.b1 = b1; j.W2 = W2; j.b2 = b2; j.y = y; j.y_acc = y_acc;
    j.mid = h_out; j.T = T; j.D = D; j.H = H; j.Dout = Dout;
    j.gelu_mode = gelu_mode; j.eager = eager_rounding;
    j.rows = rows; j.nrows = rows ? nrows : T;
    return run(&j, nthreads);
}

/* m = bf16(gelu_tanh(x Wg^T) * (x Wu^T)); y = bf16(m Wd^T). m_out (nullable) receives m. */
int oracle_geglu(const uint16_t* x, const uint16_t* Wg, const uint16_t* Wu,
                 const uint16_t* Wd, uint16_t* y, double* y_acc, uint16_t* m_out,
                 int64_t T, int64_t D, int64_t H, int eager_rounding,
                 const int64_t* rows, int64_t nrows, int nthreads) {
    job_t j;
    memset(&j, 0, sizeof j);
    j.op = 2; j.x = x; j.W1 = Wg; j.W2 = Wu; j.W3 = Wd; j.y = y; j.y_acc = y_acc;
    j.mid = m_out; j.T = T; j.D = D; j.H = H; j.Dout = D;
    j.eager = eager_rounding;
    j.rows = rows; j.nrows = rows ? nrows : T;
    return run(&j, nthreads);
}
