/*
 * CPU oracle for the compensated-FP32 projection — TEST INFRASTRUCTURE ONLY.
 *
 * This file is the slow, plain reference that the CUDA path is checked against.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
 * load it.  It shares no code, header, table or helper with the CUDA library and
 * includes nothing from it.
 *
 * Source of the method: laya.cpp, "docs/vulkan.md" (Vulkan backend page),
 *   - compensated-FP32 paragraph: each FP32 input becomes two FP16 components,
 *     each multiplied by the exactly stored FP16 weights with FP32 accumulation,
 *     and the two results are combined in FP32;
 *   - split/merge paragraph: the split rounds to nearest, ties to even, keeping
 *     subnormal results, and the residual is multiplied by 1024;
 *   - 1024-scale paragraph: why the residual is scaled by 2^10 (so that it
 *     cannot overflow binary16 for large activations).
 * The merge formula y = acc_hi + acc_lo * 2^-10 is the plain reading of the
 * FP32 combination with the 1024 scale undone.
 *   - feed-forward paragraph: the FP32 feed-forward layers fuse the GEGLU gate
 *     activation and multiplication into one dispatch.  oracle_epilogue is that
 *     step on a projection's output, read as out = gelu(gate) * (y + bias) with
 *     the exact GELU, g * Phi(g), Phi the standard normal distribution function.
 *
 * Every floating-point step here is done in IEEE double, where each step used is
 * exact, and then rounded once to the target format.  Compile with
 * -ffp-contract=off (no fused multiply-add) and without fast-math.
 *
 * Parity pins (tests/test_oracle_*.py): fp16_rne against brute-force nearest
 * search over every binary16 value and against numpy's float16 cast; split
 * against hand-derived bits and the reconstruction bound; merge against numpy
 * float32 arithmetic and hand-derived special pairs; GEMMs against closed-form
 * special cases, numpy float64 matmul for the true product, and the split's
 * reconstruction bound.  No function here is unpinned.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------- */
/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
/* Normal values (1 + f/1024) * 2^(E)   for E = -14 .. 15;                      */
/* subnormal values f * 2^-24           for f = 1 .. 1023;                      */
/* largest finite 65504 = (2 - 2^-10) * 2^15.                                   */
/* ------------------------------------------------------------------------- */

/* Round a non-negative double t (t < 2^12) to the nearest integer, ties to the
 * even integer. */
static double round_half_even(double t)
{
    double f = floor(t);
    double d = t - f; /* exact: t < 2^12 has at most 53 significant bits */
    if (d > 0.5)
        return f + 1.0;
    if (d < 0.5)
        return f;
    return (((int64_t)f & 1) == 0) ? f : f + 1.0;
}

/* Value of a binary16 bit pattern, exactly, as a double. */
double oracle_fp16_value(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0x1f)
        v = (f == 0) ? INFINITY : NAN;
    else if (e == 0)
        v = ldexp((double)f, -24);
    else
        v = ldexp(1024.0 + (double)f, e - 25);
    return sign ? -v : v;
}

/* binary16 roundTiesToEven of the real number v (given exactly as a double),
 * with gradual underflow and overflow to infinity.
 *
 * The rounding is done on the real line: |v| lies in the binade [2^E, 2^(E+1));
 * binary16 values there are n * 2^(E-10) for integers n in [1024, 2048) (the
 * subnormal range, |v| < 2^-14, shares the spacing 2^-24 of the smallest normal
 * binade, with n < 1024).  So n = round_half_even(|v| / 2^(E-10)), an exact
 * scaling.  n = 2048 carries into the next binade; a result above 65504
 * (E = 15, n = 2048) is an overflow, which includes the tie at 65520. */
uint16_t oracle_fp16_rne(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v))
        return (uint16_t)(sign | 0x7e00u);
    double a = fabs(v);
    if (isinf(a))
        return (uint16_t)(sign | 0x7c00u);

    int e2 = 0;
    if (a != 0.0)
        (void)frexp(a, &e2); /* a in [2^(e2-1), 2^e2) */
    int E = e2 - 1;
    if (a == 0.0 || E < -14)
        E = -14;
    int n = (int)round_half_even(ldexp(a, 10 - E)); /* a / 2^(E-10), exact */
    if (n == 2048) {                                  /* carried into the next binade */
        n = 1024;
        E += 1;
    }
    if (E > 15)
        return (uint16_t)(sign | 0x7c00u); /* above 65504: overflow to infinity */
    if (n < 1024)                           /* E == -14: zero or subnormal, value n * 2^-24 */
        return (uint16_t)(sign | (uint16_t)n);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(n - 1024));
}

/* ------------------------------------------------------------------------- */
/* Split and merge (one element each).                                        */
/* ------------------------------------------------------------------------- */

/* hi = fp16_rne(x); lo = fp16_rne((x - hi) * 1024), the difference and the
 * scaling taken exactly. */
static void split_one(float x, uint16_t* hi, uint16_t* lo)
{
    uint16_t h = oracle_fp16_rne((double)x);
    double r = (double)x - oracle_fp16_value(h); /* exact in double */
    *hi = h;
    *lo = oracle_fp16_rne(r * 1024.0);
}

/* y = acc_hi + acc_lo * 2^-10 in binary32: the product rounded to binary32,
 * then the sum rounded to binary32 (two separate IEEE operations, no fused
 * multiply-add).  Each operation is done exactly in double and rounded once to
 * float; for a single +, -, * on binary32 operands this gives the correctly
 * rounded binary32 result. */
static float merge_one(float acc_hi, float acc_lo)
{
    float t = (float)((double)acc_lo * 0x1p-10);
    return (float)((double)acc_hi + (double)t);
}

/* ------------------------------------------------------------------------- */
/* Thread pool helper: run fn(lo, hi, ctx) over [0, n) in nthreads chunks.    */
/* ------------------------------------------------------------------------- */

typedef void (*range_fn)(int64_t lo, int64_t hi, void* ctx);

struct range_job {
    range_fn fn;
    void* ctx;
    int64_t lo, hi;
};

static void* range_thread(void* p)
{
    struct range_job* j = (struct range_job*)p;
    j->fn(j->lo, j->hi, j->ctx);
    return NULL;
}

int oracle_default_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static void parallel_for(int64_t n, int nthreads, range_fn fn, void* ctx)
{
    if (nthreads <= 0)
        nthreads = oracle_default_threads();
    if ((int64_t)nthreads > n)
        nthreads = (int)(n > 0 ? n : 1);
    if (nthreads <= 1) {
        fn(0, n, ctx);
        return;
    }
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int* running = (int*)malloc(sizeof(int) * (size_t)nthreads);
    struct range_job* jobs = (struct range_job*)malloc(sizeof(struct range_job) * (size_t)nthreads);
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].fn = fn;
        jobs[t].ctx = ctx;
        jobs[t].lo = n * t / nthreads;
        jobs[t].hi = n * (t + 1) / nthreads;
        running[t] = pthread_create(&th[t], NULL, range_thread, &jobs[t]) == 0;
        if (!running[t])
            fn(jobs[t].lo, jobs[t].hi, ctx); /* run inline if a thread cannot start */
    }
    for (int t = 0; t < nthreads; ++t)
        if (running[t])
            pthread_join(th[t], NULL);
    free(jobs);
    free(running);
    free(th);
}

/* ------------------------------------------------------------------------- */
/* Elementwise entry points.                                                  */
/* ------------------------------------------------------------------------- */

struct split_ctx {
    const float* x;
    uint16_t* hi;
    uint16_t* lo;
};

static void split_range(int64_t a, int64_t b, void* p)
{
    struct split_ctx* c = (struct split_ctx*)p;
    for (int64_t i = a; i < b; ++i)
        split_one(c->x[i], &c->hi[i], &c->lo[i]);
}

void oracle_split(const float* x, uint16_t* hi, uint16_t* lo, int64_t n, int nthreads)
{
    struct split_ctx c = {x, hi, lo};
    parallel_for(n, nthreads, split_range, &c);
}

struct merge_ctx {
    const float* acc_hi;
    const float* acc_lo;
    float* y;
};

static void merge_range(int64_t a, int64_t b, void* p)
{
    struct merge_ctx* c = (struct merge_ctx*)p;
    for (int64_t i = a; i < b; ++i)
        c->y[i] = merge_one(c->acc_hi[i], c->acc_lo[i]);
}

void oracle_merge(const float* acc_hi, const float* acc_lo, float* y, int64_t n, int nthreads)
{
    struct merge_ctx c = {acc_hi, acc_lo, y};
    parallel_for(n, nthreads, merge_range, &c);
}

/* ------------------------------------------------------------------------- */
/* GEMMs.  x: binary32 [M, K] row-major.  W: binary16 bits [N, K] row-major.   */
/* Output element (i, j) is a dot product of row i of x with row j of W.       */
/* If rows/cols are given, only the `count` listed elements are computed       */
/* (out[s] for pair (rows[s], cols[s])); otherwise all M*N, out[i*N + j].      */
/* Sums are taken in double, in increasing k.                                  */
/* ------------------------------------------------------------------------- */

enum gemm_kind { GEMM_COMP = 0, GEMM_TRUE = 1, GEMM_CAST = 2, GEMM_DEN = 3 };

struct gemm_ctx {
    enum gemm_kind kind;
    const float* x;
    const uint16_t* W;
    int64_t M, N, K;
    const int64_t* rows;
    const int64_t* cols;
    float* outf;
    double* outd;
    const double* wd; /* W decoded to double, [N, K], or NULL (decode per use) */
};

/* Row i of x as the doubles the kind needs: x itself (TRUE, DEN) or its split
 * components hi, lo (COMP, CAST). */
static void prepare_row(const struct gemm_ctx* c, int64_t i, double* a, double* b)
{
    const float* xr = c->x + i * c->K;
    for (int64_t k = 0; k < c->K; ++k) {
        if (c->kind == GEMM_TRUE || c->kind == GEMM_DEN) {
            a[k] = (double)xr[k];
            b[k] = 0.0;
        } else {
            uint16_t h, l;
            split_one(xr[k], &h, &l);
            a[k] = oracle_fp16_value(h);
            b[k] = oracle_fp16_value(l);
        }
    }
}

/* One output element from the prepared row (a, b) and row w of W (doubles). */
static double gemm_elem(const struct gemm_ctx* c, const double* a, const double* b, const double* w)
{
    switch (c->kind) {
    case GEMM_COMP: {
        /* the method: acc_hi = sum hi*w, acc_lo = sum lo*w, y = acc_hi + acc_lo * 2^-10 */
        double s_hi = 0.0, s_lo = 0.0;
        for (int64_t k = 0; k < c->K; ++k) {
            s_hi += a[k] * w[k];
            s_lo += b[k] * w[k];
        }
        return s_hi + s_lo * 0x1p-10;
    }
    case GEMM_TRUE:
    case GEMM_CAST: { /* CAST: a single FP16 cast of x, only the hi component */
        double s = 0.0;
        for (int64_t k = 0; k < c->K; ++k)
            s += a[k] * w[k];
        return s;
    }
    case GEMM_DEN:
    default: {
        double s = 0.0;
        for (int64_t k = 0; k < c->K; ++k)
            s += fabs(a[k]) * fabs(w[k]);
        return s;
    }
    }
}

static void gemm_store(const struct gemm_ctx* c, int64_t slot, double v)
{
    if (c->kind == GEMM_DEN)
        c->outd[slot] = v;
    else
        c->outf[slot] = (float)v;
}

static const double* w_row(const struct gemm_ctx* c, int64_t j, double* scratch)
{
    if (c->wd)
        return c->wd + j * c->K;
    for (int64_t k = 0; k < c->K; ++k)
        scratch[k] = oracle_fp16_value(c->W[j * c->K + k]);
    return scratch;
}

/* Full product: a range of rows i. */
static void gemm_rows(int64_t lo_i, int64_t hi_i, void* p)
{
    const struct gemm_ctx* c = (const struct gemm_ctx*)p;
    size_t kk = (size_t)(c->K > 0 ? c->K : 1);
    double* a = (double*)malloc(kk * sizeof(double));
    double* b = (double*)malloc(kk * sizeof(double));
    double* wsc = (double*)malloc(kk * sizeof(double));
    for (int64_t i = lo_i; i < hi_i; ++i) {
        prepare_row(c, i, a, b);
        for (int64_t j = 0; j < c->N; ++j)
            gemm_store(c, i * c->N + j, gemm_elem(c, a, b, w_row(c, j, wsc)));
    }
    free(a);
    free(b);
    free(wsc);
}

/* Sampled product: a range of listed (row, col) pairs. */
static void gemm_pairs(int64_t lo_s, int64_t hi_s, void* p)
{
    const struct gemm_ctx* c = (const struct gemm_ctx*)p;
    size_t kk = (size_t)(c->K > 0 ? c->K : 1);
    double* a = (double*)malloc(kk * sizeof(double));
    double* b = (double*)malloc(kk * sizeof(double));
    double* wsc = (double*)malloc(kk * sizeof(double));
    int64_t have = -1;
    for (int64_t s = lo_s; s < hi_s; ++s) {
        int64_t i = c->rows[s], j = c->cols[s];
        if (i != have) {
            prepare_row(c, i, a, b);
            have = i;
        }
        gemm_store(c, s, gemm_elem(c, a, b, w_row(c, j, wsc)));
    }
    free(a);
    free(b);
    free(wsc);
}

struct decode_ctx {
    const uint16_t* W;
    double* wd;
};

static void decode_range(int64_t a, int64_t b, void* p)
{
    struct decode_ctx* d = (struct decode_ctx*)p;
    for (int64_t i = a; i < b; ++i)
        d->wd[i] = oracle_fp16_value(d->W[i]);
}

static void gemm_run(enum gemm_kind kind, const float* x, const uint16_t* W, int64_t M, int64_t N, int64_t K,
                     const int64_t* rows, const int64_t* cols, int64_t count, float* outf, double* outd,
                     int nthreads)
{
    struct gemm_ctx c = {kind, x, W, M, N, K, rows, cols, outf, outd, NULL};
    if (rows && cols) {
        parallel_for(count, nthreads, gemm_pairs, &c);
        return;
    }
    /* full product: decode W once (falls back to per-row decoding without memory) */
    double* wd = (double*)malloc((size_t)(N * K > 0 ? N * K : 1) * sizeof(double));
    if (wd) {
        struct decode_ctx d = {W, wd};
        parallel_for(N * K, nthreads, decode_range, &d);
        c.wd = wd;
    }
    parallel_for(M, nthreads, gemm_rows, &c);
    free(wd);
}

/* The compensated product, following the method step by step (the gate
 * oracle): y = fp32( sum_k hi_ik w_jk + 2^-10 * sum_k lo_ik w_jk ). */
void oracle_gemm_comp(const float* x, const uint16_t* W, int64_t M, int64_t N, int64_t K,
                      const int64_t* rows, const int64_t* cols, int64_t count, float* y, int nthreads)
{
    gemm_run(GEMM_COMP, x, W, M, N, K, rows, cols, count, y, NULL, nthreads);
}

/* The true product of the FP32 input: y = fp32( sum_k x_ik w_jk ). */
void oracle_gemm_true(const float* x, const uint16_t* W, int64_t M, int64_t N, int64_t K,
                      const int64_t* rows, const int64_t* cols, int64_t count, float* y, int nthreads)
{
    gemm_run(GEMM_TRUE, x, W, M, N, K, rows, cols, count, y, NULL, nthreads);
}

/* A single FP16 cast of x (the best such a cast can do): y = fp32( sum_k fp16(x_ik) w_jk ). */
void oracle_gemm_cast(const float* x, const uint16_t* W, int64_t M, int64_t N, int64_t K,
                      const int64_t* rows, const int64_t* cols, int64_t count, float* y, int nthreads)
{
    gemm_run(GEMM_CAST, x, W, M, N, K, rows, cols, count, y, NULL, nthreads);
}

/* The error scale of a dot product: den = sum_k |x_ik| |w_jk| (double). */
void oracle_gemm_den(const float* x, const uint16_t* W, int64_t M, int64_t N, int64_t K,
                     const int64_t* rows, const int64_t* cols, int64_t count, double* den, int nthreads)
{
    gemm_run(GEMM_DEN, x, W, M, N, K, rows, cols, count, NULL, den, nthreads);
}

/* ------------------------------------------------------------------------- */
/* Epilogue of a GEGLU feed-forward step on a projection's output y [M, N]:   */
/*   out[m, n] = gelu(gate[m, n]) * (y[m, n] + bias[n]),                     */
/*   gelu(g) = g * Phi(g),  Phi(g) = erfc(-g / sqrt(2)) / 2,                 */
/* (the same function as (1 + erf(g / sqrt 2)) / 2, without its cancellation  */
/* for negative g),                                                          */
/* bias NULL: no bias; gate NULL: factor 1.  Evaluated in double from the     */
/* binary32 inputs (y + bias is exact in double) and rounded once to binary32. */
/* ------------------------------------------------------------------------- */
static double gelu_exact(double g)
{
    return 0.5 * g * erfc(-g * 0.70710678118654752440); /* 1/sqrt(2) */
}

struct epi_ctx {
    const float* y;
    const float* bias;
    const float* gate;
    float* out;
    int64_t N;
};

static void epi_range(int64_t a, int64_t b, void* p)
{
    const struct epi_ctx* c = (const struct epi_ctx*)p;
    for (int64_t i = a; i < b; ++i) {
        double v = (double)c->y[i];
        if (c->bias)
            v += (double)c->bias[i % c->N];
        if (c->gate)
            v *= gelu_exact((double)c->gate[i]);
        c->out[i] = (float)v;
    }
}

void oracle_epilogue(const float* y, const float* bias, const float* gate, float* out, int64_t M, int64_t N,
                     int nthreads)
{
    struct epi_ctx c = {y, bias, gate, out, N};
    parallel_for(M * N, nthreads, epi_range, &c);
}

double oracle_gelu(double g)
{
    return gelu_exact(g);
}

