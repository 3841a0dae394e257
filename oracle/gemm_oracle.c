/*
 * CPU oracle for the fp16 GEMM with an fp32 accumulator.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or calls
 * this file; only the tests, the package's smoke check and the benchmark's CPU
 * baseline do. It shares no code, header or constant with the CUDA library.
 *
 * What it computes (the plain definition, written out):
 *   "03: Matrix multiplication" (phobos-lang.dev tutorial: the kernel and the
 *   paragraph under it): C = A B with fp16 operands; the running sum is kept in
 *   fp32 for the whole k loop and converted to fp16 a single time, when the
 *   output tile is written (the same cast Triton's tutorial applies to its
 *   accumulator).
 *
 *   c32[i][j] = sum_{k=0}^{K-1} float(A[i][k]) * float(B[k][j])   (fp32, k ascending)
 *   C[i][j]   = fp16_round_nearest_even(c32[i][j])                 (once)
 *
 * A is [M,K] row-major, B is [K,N] row-major, both fp16 given as raw IEEE
 * binary16 bit patterns (uint16_t). Every fp16 value is exactly representable in
 * fp32, and the product of two fp16 values has at most 22 significant bits, so
 * each product is exact in fp32; only the running sum rounds.
 *
 * Readings where the pages are silent:
 *   - the summation order is not stated: this oracle sums in ascending k;
 *   - the narrowing mode is not stated beyond Triton's `.to(float16)`: this
 *     oracle uses IEEE-754 round-to-nearest, ties-to-even, keeping subnormals,
 *     with overflow to +-inf (written out below from the format's definition);
 *   - K == 0 gives the empty sum, +0.
 *
 * Loop order: for each output row i the fp32 row accumulator acc[0..N) is
 * zeroed, then for k = 0, 1, ..., K-1 the term float(A[i][k]) * float(B[k][j])
 * is added to acc[j] for every j. Each acc[j] therefore receives its K terms in
 * ascending k, exactly as the sum above is written; only the order in which
 * different, independent outputs are visited differs from an i-j-k loop.
 * Rows are split across POSIX threads; a row is never split.
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -pthread -ffp-contract=off
 *        (no -ffast-math: the fp32 sums must not be reassociated).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* IEEE-754 binary16 decoding: sign bit, 5 exponent bits (bias 15), 10
 * fraction bits. Exponent 0 is zero/subnormal (value = f * 2^-24), exponent
 * 31 is inf/NaN, otherwise value = (1024 + f) * 2^(e - 25). */
float oracle_half_to_float(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1f;
    const int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + f), e - 25);
    }
    return (float)(sign ? -v : v);
}

/* Round a non-negative double holding an exact value below 2^30 to the nearest
 * integer, ties to the even one. */
static double round_half_even(double q)
{
    const double fl = floor(q);
    const double d = q - fl;
    if (d > 0.5) return fl + 1.0;
    if (d < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* IEEE-754 binary32 -> binary16, round to nearest, ties to even.
 * Largest finite half is 65504 = (2 - 2^-10) * 2^15; the next value of the
 * format's grid would be 65536, so every |x| >= 65520 (the midpoint, which
 * ties to the even significand of 65536) overflows to infinity. Below 2^-14
 * the grid spacing is 2^-24 (subnormals). */
uint16_t oracle_float_to_half_rne(float x)
{
    const uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7e00u);
    const double a = fabs((double)x);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: value = m * 2^-24, m in [0, 1024]; m == 1024 is the
         * smallest normal, whose bit pattern is exactly 0x0400 */
        const double m = round_half_even(a * ldexp(1.0, 24));
        return (uint16_t)(sign | (uint16_t)m);
    }
    int E;
    (void)frexp(a, &E); /* a = fr * 2^E, fr in [0.5, 1): unbiased exponent E-1 */
    int ex = E - 1;
    double sig = round_half_even(ldexp(a, 10 - ex)); /* in [1024, 2048] */
    if (sig == 2048.0) {
        sig = 1024.0;
        ex += 1;
    }
    /* ex <= 15 here because a < 65520 */
    return (uint16_t)(sign | (uint16_t)((ex + 15) << 10) | (uint16_t)(sig - 1024.0));
}

/* ------------------------------------------------------------------------- */
typedef struct {
    const uint16_t* A;
    const float* Bf; /* B converted to fp32, [K,N] row-major */
    const float* lut; /* binary16 bits -> fp32 value, all 65536 patterns */
    int64_t N, K;
    const int64_t* rows;
    int64_t r_begin, r_end; /* positions in rows[] */
    uint16_t* C;            /* [nrows, N] */
    float* C32;             /* [nrows, N] or NULL */
    int status;
} oracle_job;

static void* oracle_worker(void* arg)
{
    oracle_job* job = (oracle_job*)arg;
    const int64_t N = job->N, K = job->K;
    float* acc = (float*)malloc((size_t)(N > 0 ? N : 1) * sizeof(float));
    if (!acc) {
        job->status = 1;
        return NULL;
    }
    for (int64_t r = job->r_begin; r < job->r_end; ++r) {
        const int64_t i = job->rows[r];
        for (int64_t j = 0; j < N; ++j) acc[j] = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            const float a = job->lut[job->A[i * K + k]];
            const float* brow = job->Bf + k * N;
            for (int64_t j = 0; j < N; ++j) acc[j] += a * brow[j];
        }
        for (int64_t j = 0; j < N; ++j) {
            job->C[r * N + j] = oracle_float_to_half_rne(acc[j]);
            if (job->C32) job->C32[r * N + j] = acc[j];
        }
    }
    free(acc);
    job->status = 0;
    return NULL;
}

/* Computes rows rows[0..nrows) of C. Returns 0 on success, 1 on a bad
 * argument, 2 on allocation failure. nthreads <= 0 means one thread. */
int oracle_gemm_f16_rows(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N, int64_t K,
                         const int64_t* rows, int64_t nrows, int nthreads, uint16_t* C, float* C32)
{
    if (M < 0 || N < 0 || K < 0 || nrows < 0) return 1;
    if (nrows == 0 || N == 0) return 0;
    if (!rows || !C || (K > 0 && (!A || !B))) return 1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return 1;

    float* lut = (float*)malloc(65536 * sizeof(float));
    float* Bf = (float*)malloc((size_t)(K * N > 0 ? K * N : 1) * sizeof(float));
    if (!lut || !Bf) {
        free(lut);
        free(Bf);
        return 2;
    }
    for (uint32_t h = 0; h < 65536u; ++h) lut[h] = oracle_half_to_float((uint16_t)h);
    for (int64_t t = 0; t < K * N; ++t) Bf[t] = lut[B[t]];

    if (nthreads <= 0) nthreads = 1;
    if (nthreads > nrows) nthreads = (int)nrows;
    oracle_job* jobs = (oracle_job*)calloc((size_t)nthreads, sizeof(oracle_job));
    pthread_t* tids = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    char* created = (char*)calloc((size_t)nthreads, 1);
    int rc = 0;
    if (!jobs || !tids || !created) {
        rc = 2;
    } else {
        for (int t = 0; t < nthreads; ++t) {
            oracle_job* j = &jobs[t];
            j->A = A;
            j->Bf = Bf;
            j->lut = lut;
            j->N = N;
            j->K = K;
            j->rows = rows;
            j->r_begin = nrows * t / nthreads;
            j->r_end = nrows * (t + 1) / nthreads;
            j->C = C;
            j->C32 = C32;
            j->status = 1;
            if (nthreads > 1 && pthread_create(&tids[t], NULL, oracle_worker, j) == 0)
                created[t] = 1;
            else
                oracle_worker(j); /* one thread, or a thread that could not start */
        }
        for (int t = 0; t < nthreads; ++t)
            if (created[t]) pthread_join(tids[t], NULL);
        for (int t = 0; t < nthreads; ++t)
            if (jobs[t].status != 0) rc = 2;
    }
    free(created);
    free(jobs);
    free(tids);
    free(lut);
    free(Bf);
    return rc;
}

/* Array forms of the two conversions above, for exhaustive tests. */
void oracle_half_to_float_array(const uint16_t* h, float* out, int64_t n)
{
    for (int64_t t = 0; t < n; ++t) out[t] = oracle_half_to_float(h[t]);
}

void oracle_float_to_half_rne_array(const float* x, uint16_t* out, int64_t n)
{
    for (int64_t t = 0; t < n; ++t) out[t] = oracle_float_to_half_rne(x[t]);
}
