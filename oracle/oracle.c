/*
 * oracle.c -- plain CPU oracle for the dense fp16 GEMM  C = A * B^T.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the package smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code, header, table or
 * constant with the CUDA path.
 *
 * What it computes (the plain definition, written out):
 *
 *     C[m][n] = sum_{k=0}^{K-1}  A[m][k] * B[n][k]        (fp64 accumulate)
 *
 *   - A is M x K, row-major fp16: element (m,k) at A[m*K + k].
 *   - B is N x K, "K-major" fp16: element (n,k) at B[n*K + k].  The pages load
 *     the A tile at coordinate {m,k} and the B tile at {n,k}, each BLK_x x BLK_K
 *     ("GEMM II -- pipelining with TMA", Step 4, the byte_count formula), so B
 *     holds N rows of K values and the product is A times B transposed.
 *   - C is M x N, row-major (ldc = N).  The pages do not fix C's layout; the
 *     plain reading (row-major, ldc = N) is taken.
 *   - The method accumulates in fp32 and narrows to the output type at the end
 *     ("GEMM II", the baseline paragraph: "right math, fp32 accumulate"; the
 *     TMA-store epilogue: "narrow for the output dtype").  The oracle keeps the
 *     exact-as-possible fp64 sum; the tests compare against it with a tolerance
 *     that absorbs the fp32 accumulation order.
 *
 * Every fp16 x fp16 product is exact in fp64 (11 + 11 significand bits), so the
 * only rounding here is in the fp64 running sum, taken in ascending k.
 *
 * fp16 is decoded by this file's own routine (IEEE 754 binary16: 1 sign bit,
 * 5 exponent bits with bias 15, 10 fraction bits) and rounded back with its own
 * round-to-nearest-even routine, which is how the fp16 output of the method is
 * defined (cvt.rn: round to nearest, ties to even).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- fp16 codec */

/* IEEE binary16 -> double, exact for every one of the 65536 bit patterns. */
double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        /* zero or subnormal: f * 2^-24 */
        v = ldexp((double)f, -24);
    } else if (e == 0x1f) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        /* normal: (1 + f/1024) * 2^(e-15) = (1024 + f) * 2^(e-25) */
        v = ldexp((double)(1024 + f), e - 25);
    }
    return sign ? -v : v;
}

/* Round-to-nearest-even of an integer-valued or real q >= 0 held in a double
 * whose integer part fits in 53 bits: returns the nearest integer, ties to the
 * even one.  Written out instead of relying on the FPU rounding mode. */
static double round_half_even(double q)
{
    double fl = floor(q);
    double frac = q - fl; /* exact: q and fl share the exponent range */
    if (frac > 0.5) return fl + 1.0;
    if (frac < 0.5) return fl;
    /* exact tie: pick the even neighbour */
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* double -> IEEE binary16, round to nearest, ties to even; overflow -> inf. */
uint16_t oracle_f64_to_f16(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return (uint16_t)(sign | 0x7e00);
    double a = fabs(x);
    /* 65504 is the largest finite half; 65520 lies exactly halfway to 2^16
     * and ties to the even significand, which is the overflow to infinity. */
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: quantum 2^-24; a result of 1024 is 2^-14, the
         * smallest normal, whose encoding is exactly 0x0400 */
        double q = round_half_even(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)q);
    }
    int e2;
    frexp(a, &e2);      /* a = m * 2^e2, m in [0.5, 1) */
    int E = e2 - 1;     /* a in [2^E, 2^(E+1)),  -14 <= E <= 15 */
    double q = round_half_even(ldexp(a, 10 - E)); /* in [1024, 2048] */
    if (q == 2048.0) {
        q = 1024.0;
        E += 1;
    }
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)((int)q - 1024));
}

void oracle_decode_f16(int64_t n, const uint16_t *in, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_to_f64(in[i]);
}

void oracle_encode_f16(int64_t n, const double *in, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f64_to_f16(in[i]);
}

/* ------------------------------------------------------------------- GEMM */

typedef struct {
    int64_t M, N, K;
    const double *A; /* rows [m_begin, m_end) of the M x K row-major A */
    const double *B; /* N x K, row-major */
    double *C;       /* rows [m_begin, m_end) of M x N, row-major */
    int64_t m_begin, m_end;
} rows_job;

/* The definition, one output at a time: dot product of row m of A with row n
 * of B, summed in ascending k. */
static void *rows_worker(void *arg)
{
    rows_job *j = (rows_job *)arg;
    for (int64_t m = j->m_begin; m < j->m_end; ++m) {
        const double *a = j->A + (m - j->m_begin) * j->K;
        for (int64_t n = 0; n < j->N; ++n) {
            const double *b = j->B + n * j->K;
            double acc = 0.0;
            for (int64_t k = 0; k < j->K; ++k) acc += a[k] * b[k];
            j->C[(m - j->m_begin) * j->N + n] = acc;
        }
    }
    return NULL;
}

/* Rows [m_begin, m_end) of C from already-decoded fp64 operands, split over
 * `threads` POSIX threads by contiguous row ranges.  A_rows holds only those
 * rows of A ((m_end - m_begin) x K); B is all N x K.  C receives
 * (m_end - m_begin) * N values.  Returns 0 on success. */
int oracle_gemm_rows_f64(int64_t M, int64_t N, int64_t K, const double *A_rows, const double *B,
                         double *C, int64_t m_begin, int64_t m_end, int threads)
{
    if (M < 0 || N < 0 || K < 0 || m_begin < 0 || m_end > M || m_begin > m_end) return 1;
    int64_t rows = m_end - m_begin;
    if (rows == 0 || N == 0) return 0;
    if (threads < 1) threads = 1;
    if (threads > rows) threads = (int)rows;
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)threads);
    rows_job *jobs = (rows_job *)malloc(sizeof(rows_job) * (size_t)threads);
    if (!tid || !jobs) {
        free(tid);
        free(jobs);
        return 2;
    }
    int64_t per = rows / threads, extra = rows % threads, at = m_begin;
    for (int t = 0; t < threads; ++t) {
        int64_t cnt = per + (t < extra ? 1 : 0);
        jobs[t].M = M;
        jobs[t].N = N;
        jobs[t].K = K;
        jobs[t].A = A_rows + (at - m_begin) * K;
        jobs[t].B = B;
        jobs[t].C = C + (at - m_begin) * N;
        jobs[t].m_begin = at;
        jobs[t].m_end = at + cnt;
        at += cnt;
    }
    int started = 0, rc = 0;
    for (; started < threads; ++started)
        if (pthread_create(&tid[started], NULL, rows_worker, &jobs[started]) != 0) break;
    /* Any job whose thread could not be started runs here instead. */
    for (int t = started; t < threads; ++t) rows_worker(&jobs[t]);
    for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
    free(tid);
    free(jobs);
    return rc;
}

/* Rows [m_begin, m_end) of C from fp16 operands: decodes the needed rows of A
 * and all of B to fp64, then forms the dot products. */
int oracle_gemm_rows_f16(int64_t M, int64_t N, int64_t K, const uint16_t *A16,
                         const uint16_t *B16, double *C, int64_t m_begin, int64_t m_end,
                         int threads)
{
    if (M < 0 || N < 0 || K < 0 || m_begin < 0 || m_end > M || m_begin > m_end) return 1;
    int64_t rows = m_end - m_begin;
    double *A = (double *)malloc(sizeof(double) * (size_t)(rows * K > 0 ? rows * K : 1));
    double *B = (double *)malloc(sizeof(double) * (size_t)(N * K > 0 ? N * K : 1));
    if (!A || !B) {
        free(A);
        free(B);
        return 2;
    }
    oracle_decode_f16(rows * K, A16 + m_begin * K, A);
    oracle_decode_f16(N * K, B16, B);
    int rc = oracle_gemm_rows_f64(M, N, K, A, B, C, m_begin, m_end, threads);
    free(A);
    free(B);
    return rc;
}

/* Full C (M x N, fp64) from fp16 operands. */
int oracle_gemm_f16(int64_t M, int64_t N, int64_t K, const uint16_t *A16, const uint16_t *B16,
                    double *C, int threads)
{
    return oracle_gemm_rows_f16(M, N, K, A16, B16, C, 0, M, threads);
}

/* Selected entries C[rows[i]][cols[i]], i < count, straight from fp16 operands
 * (decoded on the fly).  Returns 1 if an index is out of range. */
int oracle_gemm_entries_f16(int64_t M, int64_t N, int64_t K, const uint16_t *A16,
                            const uint16_t *B16, int64_t count, const int64_t *rows,
                            const int64_t *cols, double *out)
{
    for (int64_t i = 0; i < count; ++i) {
        int64_t m = rows[i], n = cols[i];
        if (m < 0 || m >= M || n < 0 || n >= N) return 1;
        const uint16_t *a = A16 + m * K;
        const uint16_t *b = B16 + n * K;
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) acc += oracle_f16_to_f64(a[k]) * oracle_f16_to_f64(b[k]);
        out[i] = acc;
    }
    return 0;
}
