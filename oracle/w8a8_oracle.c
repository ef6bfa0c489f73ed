/*
 * CPU oracle for the W8A8 block-FP8 matmul -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the package smoke check and the benchmark's CPU-baseline
 * leg may load this library.  The product path never calls it, and it shares
 * no code, header, table or constant with the CUDA library.
 *
 * What it computes (operator definition, "feat: optimize w8a8 block fp8
 * matmul for Hopper", FlagGems-vllm PR #693, Description and Numerical
 * safety sections):
 *
 *     C[m,n] = sum_g  a_s[m,g] * b_s[n / block_n, g] * sum_{k in g} A[m,k] * B[n,k]
 *
 * with A an FP8 E4M3 [M,K] activation matrix carrying one fp32 scale per
 * token per block_k-wide K group, B an FP8 E4M3 [N,K] weight matrix carrying
 * one fp32 scale per [block_n, block_k] block, and group g covering
 * k in [g*block_k, min((g+1)*block_k, K)).  The result is kept in double; the
 * cast to the output dtype is done by the caller.
 *
 * Precision: every E4M3FN value is a multiple of 2^-9 below 2^9 in magnitude,
 * so each product is an exact multiple of 2^-18 below 2^18, and a sum of up
 * to 2^17 such products is exact in double (53-bit significand).  The
 * per-group dot is therefore exact whatever the order; the scale product
 * a_s*b_s of two floats (24+24 significant bits) is exact in double too.
 * Only the multiply by the group sum and the running sum over groups round.
 * Build with -ffp-contract=off so that no fused multiply-add changes that.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

/* OCP 8-bit floating point, E4M3 "FN" encoding: 1 sign bit, 4 exponent bits
 * (bias 7), 3 mantissa bits; no infinities; S.1111.111 is NaN; exponent 0
 * holds subnormals f * 2^-9.  Max finite 448 = 1.75 * 2^8. */
static double e4m3fn_decode(unsigned code)
{
    unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, f = code & 7u;
    double v;
    if (e == 15u && f == 7u)
        return NAN;
    if (e == 0u)
        v = ldexp((double)f, -9);
    else
        v = ldexp((double)(8u + f), (int)e - 10);
    return s ? -v : v;
}

void oracle_e4m3fn_table(double *out256)
{
    for (unsigned c = 0; c < 256u; ++c)
        out256[c] = e4m3fn_decode(c);
}

typedef struct {
    const uint8_t *A;
    const float *a_s;
    const uint8_t *B;
    const float *b_s;
    double *C;
    int64_t M, N, K, block_n, block_k;
    int64_t row_begin, row_end;
    const double *table;
    const int64_t *pairs; /* sampled mode: (m, n) pairs, else NULL */
} oracle_job;

/* One output element straight from the definition. */
static double element(const oracle_job *j, int64_t m, int64_t n)
{
    const int64_t G = (j->K + j->block_k - 1) / j->block_k;
    const uint8_t *arow = j->A + m * j->K;
    const uint8_t *brow = j->B + n * j->K;
    double acc = 0.0;
    for (int64_t g = 0; g < G; ++g) {
        int64_t k0 = g * j->block_k;
        int64_t k1 = k0 + j->block_k < j->K ? k0 + j->block_k : j->K;
        double p = 0.0;
        for (int64_t k = k0; k < k1; ++k)
            p += j->table[arow[k]] * j->table[brow[k]];
        double s = (double)j->a_s[m * G + g] * (double)j->b_s[(n / j->block_n) * G + g];
        acc += s * p;
    }
    return acc;
}

static void *run_rows(void *arg)
{
    const oracle_job *j = (const oracle_job *)arg;
    for (int64_t i = j->row_begin; i < j->row_end; ++i) {
        if (j->pairs) {
            j->C[i] = element(j, j->pairs[2 * i], j->pairs[2 * i + 1]);
        } else {
            for (int64_t n = 0; n < j->N; ++n)
                j->C[i * j->N + n] = element(j, i, n);
        }
    }
    return NULL;
}

static int launch(oracle_job base, int64_t rows, int nthreads)
{
    double table[256];
    oracle_e4m3fn_table(table);
    base.table = table;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    if ((int64_t)nthreads > rows)
        nthreads = rows > 0 ? (int)rows : 1;
    pthread_t th[256];
    int spawned[256];
    oracle_job jobs[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].row_begin = rows * t / nthreads;
        jobs[t].row_end = rows * (t + 1) / nthreads;
        spawned[t] = 0;
    }
    for (int t = 0; t < nthreads - 1; ++t)
        spawned[t] = pthread_create(&th[t], NULL, run_rows, &jobs[t]) == 0;
    for (int t = 0; t < nthreads; ++t)
        if (!spawned[t])
            run_rows(&jobs[t]); /* the last slice, and any slice whose spawn failed */
    for (int t = 0; t < nthreads - 1; ++t)
        if (spawned[t])
            pthread_join(th[t], NULL);
    return 0;
}

static int check_args(const uint8_t *A, const float *a_s, const uint8_t *B, const float *b_s,
                      const double *C, int64_t M, int64_t N, int64_t K,
                      int64_t block_n, int64_t block_k)
{
    if (M < 0 || N < 0 || K < 0 || block_n < 1 || block_k < 1)
        return 1;
    if ((M && K && !A) || (N && K && !B) || !C)
        return 1;
    if (K && ((M && !a_s) || (N && !b_s)))
        return 1;
    return 0;
}

/* Full product: C is [M, N] row-major double.  Returns 0 on success. */
int oracle_w8a8_block_fp8(const uint8_t *A, const float *a_s, const uint8_t *B, const float *b_s,
                          double *C, int64_t M, int64_t N, int64_t K,
                          int64_t block_n, int64_t block_k, int nthreads)
{
    if (check_args(A, a_s, B, b_s, C, M, N, K, block_n, block_k))
        return 1;
    oracle_job j = {A, a_s, B, b_s, C, M, N, K, block_n, block_k, 0, 0, NULL, NULL};
    return launch(j, M, nthreads);
}

/* Sampled elements: pairs holds count (m, n) index pairs; C[i] = C[m_i, n_i]. */
int oracle_w8a8_block_fp8_sampled(const uint8_t *A, const float *a_s, const uint8_t *B,
                                  const float *b_s, double *C, int64_t M, int64_t N, int64_t K,
                                  int64_t block_n, int64_t block_k, const int64_t *pairs,
                                  int64_t count, int nthreads)
{
    if (check_args(A, a_s, B, b_s, C, M, N, K, block_n, block_k) || (count > 0 && !pairs))
        return 1;
    for (int64_t i = 0; i < count; ++i)
        if (pairs[2 * i] < 0 || pairs[2 * i] >= M || pairs[2 * i + 1] < 0 || pairs[2 * i + 1] >= N)
            return 1;
    oracle_job j = {A, a_s, B, b_s, C, M, N, K, block_n, block_k, 0, 0, NULL, pairs};
    return launch(j, count, nthreads);
}
