/*
 * splitk_oracle.c -- plain, slow F64 CPU oracle for split-K GEMM with prepared,
 * transposed weights.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the package's smoke check and the
 * benchmark's CPU-baseline leg call it; the library (libsplitk) never does, and
 * this file shares no code, header, table or helper with the CUDA path.
 *
 * What is computed follows the launch contract printed on two pages:
 *   "Aligned shared rows for pipelined NAX on CUDA", section "Contract and
 *    correctness", and
 *   "Wider consecutive-weight NAX GEMM", section "Launch contract and
 *    correctness".
 * A is row-major [M,K] and B is row-major [N,K] (the prepared, transposed
 * weight).  Split s covers k in [s*kps, min((s+1)*kps, K)), so the last split is
 * clamped to K.  The pages check "every partial slab against independent F64
 * products of the actual dtype-rounded inputs", and every final output against
 * an independent F64 reference; this file is that reference:
 *
 *   P[s,m,n]  = sum_{k in split s} A[m,k]*B[n,k]     k ascending, in F64
 *   SP[s,m,n] = sum_{k in split s} |A[m,k]*B[n,k]|   error scale of P
 *   O[m,n]    = sum_{k=0}^{K-1}   A[m,k]*B[n,k]      unsplit product, in F64
 *   SO[m,n]   = sum_{k=0}^{K-1}   |A[m,k]*B[n,k]|
 *
 * Weight preparation (the pages keep the transposed weight resident, prepared
 * once outside timing: "Wider consecutive-weight NAX GEMM", section
 * "Performance method") is the plain transpose B[n,k] = W[k,n], oracle_transpose.
 *
 * Inputs arrive as the bit patterns the GPU sees (binary16, bfloat16 or
 * binary32) and are decoded here from each format's field definition
 * (sign, biased exponent, fraction), not by reinterpreting memory.
 *
 * Threads split the output rows m among themselves; every dot product is still
 * the plain ascending-k loop, so threading changes no result.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Element formats, numbered as the oracle's callers pass them. */
enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_BF16 = 2 };

/* ---------------------------------------------------------------- decoders */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);              /* subnormal: f/2^10 * 2^-14 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(1.0 + (double)f / 1024.0, e - 15);
    return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
static double decode_bf16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xFF;
    int f = h & 0x7F;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);             /* subnormal: f/2^7 * 2^-126 */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(1.0 + (double)f / 128.0, e - 127);
    return sign ? -v : v;
}

/* IEEE 754 binary32: 1 sign bit, 8 exponent bits (bias 127), 23 fraction bits. */
static double decode_f32(uint32_t u)
{
    int sign = (u >> 31) & 1;
    int e = (u >> 23) & 0xFF;
    uint32_t f = u & 0x7FFFFFu;
    double v;
    if (e == 0)
        v = ldexp((double)f, -149);             /* subnormal: f/2^23 * 2^-126 */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(1.0 + (double)f / 8388608.0, e - 127);
    return sign ? -v : v;
}

/* Decode n elements of format `dtype` at src into dst.  Returns 0, or -1 for an
 * unknown format. */
int oracle_decode(int dtype, const void *src, int64_t n, double *dst)
{
    int64_t i;
    if (dtype == ORACLE_F16) {
        const uint16_t *p = (const uint16_t *)src;
        for (i = 0; i < n; ++i) dst[i] = decode_f16(p[i]);
    } else if (dtype == ORACLE_BF16) {
        const uint16_t *p = (const uint16_t *)src;
        for (i = 0; i < n; ++i) dst[i] = decode_bf16(p[i]);
    } else if (dtype == ORACLE_F32) {
        const uint32_t *p = (const uint32_t *)src;
        for (i = 0; i < n; ++i) dst[i] = decode_f32(p[i]);
    } else {
        return -1;
    }
    return 0;
}

/* ---------------------------------------------------------------- contract */

/* The launch contract, as the pages state it:
 *   - M, K and K-per-split are positive multiples of 32; N is a positive
 *     multiple of 64                                  -> else returns 1;
 *   - every split starts below K and the splits together cover K, i.e.
 *     (splits-1)*kps < K <= splits*kps                -> else returns 2.
 * The shape rule is checked first.  Returns 0 for a legal geometry. */
int oracle_contract(int64_t M, int64_t N, int64_t K, int64_t splits, int64_t kps)
{
    if (M <= 0 || M % 32 != 0) return 1;
    if (K <= 0 || K % 32 != 0) return 1;
    if (kps <= 0 || kps % 32 != 0) return 1;
    if (N <= 0 || N % 64 != 0) return 1;
    if (splits <= 0) return 2;
    if ((splits - 1) * kps >= K) return 2;     /* the last split starts at or past K */
    if (splits * kps < K) return 2;            /* the splits leave the end of K uncovered */
    return 0;
}

/* Half-open k range of split s: [s*kps, min((s+1)*kps, K)). */
void oracle_split_range(int64_t K, int64_t kps, int64_t s, int64_t *k0, int64_t *k1)
{
    int64_t lo = s * kps, hi = (s + 1) * kps;
    if (hi > K) hi = K;
    if (lo > K) lo = K;
    *k0 = lo;
    *k1 = hi;
}

/* ------------------------------------------------------ weight preparation */

/* dst[c][r] = src[r][c] for a row-major rows x cols matrix of elem_bytes-byte
 * elements (copied as bits).  Returns 0, or -1 for an element size other than
 * 2 or 4. */
int oracle_transpose(int elem_bytes, const void *src, int64_t rows, int64_t cols, void *dst)
{
    const unsigned char *s = (const unsigned char *)src;
    unsigned char *d = (unsigned char *)dst;
    int64_t r, c;
    if (elem_bytes != 2 && elem_bytes != 4) return -1;
    for (r = 0; r < rows; ++r)
        for (c = 0; c < cols; ++c)
            memcpy(d + (size_t)(c * rows + r) * elem_bytes, s + (size_t)(r * cols + c) * elem_bytes,
                   (size_t)elem_bytes);
    return 0;
}

/* ---------------------------------------------------------------- products */

/* sum_{k=k0}^{k1-1} a[k]*b[k] and the same sum of |a[k]*b[k]|, k ascending. */
static void dot(const double *a, const double *b, int64_t k0, int64_t k1,
                double *sum, double *abs_sum)
{
    double s = 0.0, t = 0.0;
    int64_t k;
    for (k = k0; k < k1; ++k) {
        double p = a[k] * b[k];
        s += p;
        t += fabs(p);
    }
    *sum = s;
    *abs_sum = t;
}

typedef struct {
    const double *A, *B;        /* decoded operands: A[M,K], B[N,K] */
    int64_t M, N, K, splits, kps;
    double *out, *bound;        /* P/SP [splits,M,N] or O/SO [M,N] */
    int split_mode;             /* 1: per-split partials, 0: unsplit output */
    int tid, nthreads;
} job_t;

static void *run_rows(void *arg)
{
    job_t *j = (job_t *)arg;
    int64_t m, n, s;
    for (m = j->tid; m < j->M; m += j->nthreads) {
        const double *a = j->A + m * j->K;
        for (n = 0; n < j->N; ++n) {
            const double *b = j->B + n * j->K;
            if (j->split_mode) {
                for (s = 0; s < j->splits; ++s) {
                    int64_t k0, k1, idx = (s * j->M + m) * j->N + n;
                    oracle_split_range(j->K, j->kps, s, &k0, &k1);
                    dot(a, b, k0, k1, &j->out[idx], &j->bound[idx]);
                }
            } else {
                int64_t idx = m * j->N + n;
                dot(a, b, 0, j->K, &j->out[idx], &j->bound[idx]);
            }
        }
    }
    return NULL;
}

static int run_jobs(int dtype, const void *A, const void *B, int64_t M, int64_t N,
                    int64_t K, int64_t splits, int64_t kps, double *out,
                    double *bound, int split_mode, int threads)
{
    double *a = (double *)malloc(sizeof(double) * (size_t)(M * K));
    double *b = (double *)malloc(sizeof(double) * (size_t)(N * K));
    job_t *jobs;
    pthread_t *tids;
    int t;
    if (!a || !b) { free(a); free(b); return -2; }
    if (oracle_decode(dtype, A, M * K, a) || oracle_decode(dtype, B, N * K, b)) {
        free(a); free(b); return -1;
    }
    if (threads < 1) threads = 1;
    if (threads > M) threads = (int)M;
    jobs = (job_t *)calloc((size_t)threads, sizeof(job_t));
    tids = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
    if (!jobs || !tids) { free(a); free(b); free(jobs); free(tids); return -2; }
    for (t = 0; t < threads; ++t) {
        job_t j = {a, b, M, N, K, splits, kps, out, bound, split_mode, t, threads};
        jobs[t] = j;
    }
    for (t = 1; t < threads; ++t) {
        if (pthread_create(&tids[t], NULL, run_rows, &jobs[t]) != 0) {
            run_rows(&jobs[t]);           /* no thread: do its rows here */
            jobs[t].nthreads = 0;         /* marks "nothing to join" */
        }
    }
    run_rows(&jobs[0]);
    for (t = 1; t < threads; ++t)
        if (jobs[t].nthreads) pthread_join(tids[t], NULL);
    free(a); free(b); free(jobs); free(tids);
    return 0;
}

/* Every partial slab P[s,m,n] and its error scale SP, both [splits,M,N].
 * Returns 0, 1/2 for a geometry that breaks the contract, or <0 on error. */
int oracle_partials(int dtype, const void *A, const void *B, int64_t M, int64_t N,
                    int64_t K, int64_t splits, int64_t kps, double *P, double *SP,
                    int threads)
{
    int c = oracle_contract(M, N, K, splits, kps);
    if (c) return c;
    return run_jobs(dtype, A, B, M, N, K, splits, kps, P, SP, 1, threads);
}

/* The unsplit product O[m,n] and its error scale SO, both [M,N]. */
int oracle_output(int dtype, const void *A, const void *B, int64_t M, int64_t N,
                  int64_t K, double *O, double *SO, int threads)
{
    if (M <= 0 || N <= 0 || K <= 0) return 1;
    return run_jobs(dtype, A, B, M, N, K, 1, K, O, SO, 0, threads);
}

/* Selected elements only, for matrices too large to evaluate whole.  Point i is
 * (s_idx[i], m_idx[i], n_idx[i]); s_idx[i] < 0 selects the unsplit output
 * O[m,n], otherwise the partial P[s,m,n].  Writes val[i] and its scale bound[i].
 * Returns 0, or -1 for an index outside the matrices. */
int oracle_points(int dtype, const void *A, const void *B, int64_t M, int64_t N,
                  int64_t K, int64_t kps, int64_t splits, int64_t npts,
                  const int64_t *s_idx, const int64_t *m_idx, const int64_t *n_idx,
                  double *val, double *bound)
{
    double *a = (double *)malloc(sizeof(double) * (size_t)K);
    double *b = (double *)malloc(sizeof(double) * (size_t)K);
    const unsigned char *pa = (const unsigned char *)A, *pb = (const unsigned char *)B;
    size_t esz = (dtype == ORACLE_F32) ? 4 : 2;
    int64_t i;
    int rc = 0;
    if (!a || !b) { free(a); free(b); return -2; }
    for (i = 0; i < npts; ++i) {
        int64_t s = s_idx[i], m = m_idx[i], n = n_idx[i], k0 = 0, k1 = K;
        if (m < 0 || m >= M || n < 0 || n >= N || s >= splits) { rc = -1; break; }
        if (oracle_decode(dtype, pa + (size_t)(m * K) * esz, K, a) ||
            oracle_decode(dtype, pb + (size_t)(n * K) * esz, K, b)) { rc = -1; break; }
        if (s >= 0) oracle_split_range(K, kps, s, &k0, &k1);
        dot(a, b, k0, k1, &val[i], &bound[i]);
    }
    free(a);
    free(b);
    return rc;
}
