/*
 * gemm_oracle.c -- plain CPU reference for dense GEMM. TEST INFRASTRUCTURE.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
 * load this library. The CUDA library never calls it, links it or shares code
 * with it: the two sides have separate element decoders, separate index
 * arithmetic and separate layouts, and meet only on the host buffers that
 * datagen/ writes.
 *
 * What it computes (the plain definition, no blocking, no reordering):
 *
 *     C_ref[m][n] = sum_{k=0}^{K-1} (double)A(m,k) * (double)B(n,k)
 *     S[m][n]     = sum_{k=0}^{K-1} |(double)A(m,k) * (double)B(n,k)|
 *
 * with A an M x K operand and B an N x K operand, i.e. C = A * B^T in storage
 * terms. This is the product that the CuTe DSL Ampere SGEMM example checks its
 * kernel against (its reference check in run() contracts "mk,nk->mn"), and the
 * CK Tile practice GEMM builds the same problem ("Problem Size Configuration":
 * A is M x K, B is N x K, C is M x N) and checks against a CPU GEMM ("Result
 * Verification"). The Gluon Multi-CTA tutorial (its matmul_multicta section)
 * stores B as K x N, which is the N-major B below.
 *
 * Element addressing (the major/leading-dimension model of the CuTe SGEMM
 * example's run(): a_major "k"|"m", b_major "k"|"n"):
 *     A K-major : A[m*lda + k]        A M-major : A[k*lda + m]
 *     B K-major : B[n*ldb + k]        B N-major : B[k*ldb + n]
 *
 * Element types: binary32, binary16 and bfloat16, each decoded exactly into a
 * double from its sign/exponent/fraction fields. The products of two such
 * values are exact in binary64 (at most 24+24 significand bits), so the only
 * rounding in C_ref is the fp64 accumulation in ascending k; for the integer
 * workloads every partial sum is an integer below 2^53 and C_ref is exact.
 *
 * S is the error scale of the acceptance rule |C - C_ref| <= 1e-4 * S.
 *
 * The oracle computes any block rows x cols of C (all rows/cols when the index
 * list is NULL), so a test can check sampled rows and columns of a large GEMM.
 * Rows of the block are split over POSIX threads; each output element is still
 * one sequential sum over k.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_BF16 = 2 };
enum { ORACLE_MAJOR_K = 0, ORACLE_MAJOR_MN = 1 };
enum { ORACLE_OK = 0, ORACLE_EINVAL = -1, ORACLE_ENOMEM = -2 };

/* IEEE 754 binary16: sign, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);              /* subnormal: f * 2^-14 * 2^-10 */
    else if (e == 0x1f)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(0x400 | f), e - 25); /* 1.f * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: sign, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_f64(uint16_t b) {
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);             /* subnormal: f * 2^-126 * 2^-7 */
    else if (e == 0xff)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(0x80 | f), e - 134); /* 1.f * 2^(e-127) */
    return sign ? -v : v;
}

/* IEEE 754 binary32: sign, 8 exponent bits (bias 127), 23 fraction bits. */
double oracle_f32_to_f64(uint32_t u) {
    int sign = (u >> 31) & 1;
    int e = (u >> 23) & 0xff;
    uint32_t f = u & 0x7fffff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -149);
    else if (e == 0xff)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(0x800000u | f), e - 150);
    return sign ? -v : v;
}

typedef struct {
    const void *p;
    int64_t ld;
    int major;
    int dtype;
} operand_t;

static double element(const operand_t *o, int64_t r, int64_t k) {
    int64_t idx = (o->major == ORACLE_MAJOR_K) ? r * o->ld + k : k * o->ld + r;
    switch (o->dtype) {
    case ORACLE_F32: {
        uint32_t u;
        memcpy(&u, (const char *)o->p + idx * 4, 4);
        return oracle_f32_to_f64(u);
    }
    case ORACLE_F16: {
        uint16_t h;
        memcpy(&h, (const char *)o->p + idx * 2, 2);
        return oracle_f16_to_f64(h);
    }
    default: {
        uint16_t b;
        memcpy(&b, (const char *)o->p + idx * 2, 2);
        return oracle_bf16_to_f64(b);
    }
    }
}

typedef struct {
    int64_t K, n_cols;
    const double *arows;  /* n_rows x K, decoded rows of A */
    const double *bcols;  /* n_cols x K, decoded rows of B (columns of C) */
    double *C, *S;
    int64_t r_begin, r_end;
} job_t;

static void *run_rows(void *arg) {
    job_t *j = (job_t *)arg;
    for (int64_t i = j->r_begin; i < j->r_end; ++i) {
        const double *a = j->arows + i * j->K;
        for (int64_t c = 0; c < j->n_cols; ++c) {
            const double *b = j->bcols + c * j->K;
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < j->K; ++k) {
                double p = a[k] * b[k];
                acc += p;
                mag += fabs(p);
            }
            j->C[i * j->n_cols + c] = acc;
            if (j->S) j->S[i * j->n_cols + c] = mag;
        }
    }
    return NULL;
}

int oracle_num_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * oracle_gemm: C_ref and S for the block (rows x cols) of C = A * B^T.
 *   rows/cols : index lists (NULL = all M rows / all N columns)
 *   C_out, S_out : n_rows x n_cols doubles, row-major (S_out may be NULL)
 *   n_threads : <= 0 means one thread per online core
 * Returns ORACLE_OK, ORACLE_EINVAL (bad sizes, majors, dtypes, indices or
 * leading dimensions) or ORACLE_ENOMEM.
 */
int oracle_gemm(int64_t M, int64_t N, int64_t K,
                const void *A, int64_t lda, int a_major, int a_dtype,
                const void *B, int64_t ldb, int b_major, int b_dtype,
                const int64_t *rows, int64_t n_rows,
                const int64_t *cols, int64_t n_cols,
                double *C_out, double *S_out, int n_threads) {
    if (M < 0 || N < 0 || K < 0) return ORACLE_EINVAL;
    if ((a_major != 0 && a_major != 1) || (b_major != 0 && b_major != 1)) return ORACLE_EINVAL;
    if (a_dtype < 0 || a_dtype > 2 || b_dtype < 0 || b_dtype > 2) return ORACLE_EINVAL;
    if (!rows) n_rows = M;
    if (!cols) n_cols = N;
    if (n_rows < 0 || n_cols < 0) return ORACLE_EINVAL;
    if (n_rows == 0 || n_cols == 0) return ORACLE_OK;
    if (!C_out) return ORACLE_EINVAL;
    if (K > 0) {
        if (!A || !B) return ORACLE_EINVAL;
        if (lda < (a_major == ORACLE_MAJOR_K ? K : M)) return ORACLE_EINVAL;
        if (ldb < (b_major == ORACLE_MAJOR_K ? K : N)) return ORACLE_EINVAL;
    }
    for (int64_t i = 0; rows && i < n_rows; ++i)
        if (rows[i] < 0 || rows[i] >= M) return ORACLE_EINVAL;
    for (int64_t i = 0; cols && i < n_cols; ++i)
        if (cols[i] < 0 || cols[i] >= N) return ORACLE_EINVAL;

    size_t kk = (size_t)(K > 0 ? K : 1);
    double *arows = (double *)malloc((size_t)n_rows * kk * sizeof(double));
    double *bcols = (double *)malloc((size_t)n_cols * kk * sizeof(double));
    if (!arows || !bcols) {
        free(arows);
        free(bcols);
        return ORACLE_ENOMEM;
    }
    operand_t oa = {A, lda, a_major, a_dtype};
    operand_t ob = {B, ldb, b_major, b_dtype};
    for (int64_t i = 0; i < n_rows; ++i) {
        int64_t m = rows ? rows[i] : i;
        for (int64_t k = 0; k < K; ++k) arows[i * K + k] = element(&oa, m, k);
    }
    for (int64_t c = 0; c < n_cols; ++c) {
        int64_t n = cols ? cols[c] : c;
        for (int64_t k = 0; k < K; ++k) bcols[c * K + k] = element(&ob, n, k);
    }

    if (n_threads <= 0) n_threads = oracle_num_threads();
    if (n_threads > n_rows) n_threads = (int)n_rows;
    job_t *jobs = (job_t *)calloc((size_t)n_threads, sizeof(job_t));
    pthread_t *tids = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        free(arows);
        free(bcols);
        return ORACLE_ENOMEM;
    }
    int64_t per = (n_rows + n_threads - 1) / n_threads;
    for (int t = 0; t < n_threads; ++t) {
        int64_t b = t * per, e = (t + 1) * per < n_rows ? (t + 1) * per : n_rows;
        job_t j = {K, n_cols, arows, bcols, C_out, S_out, b < e ? b : e, e};
        jobs[t] = j;
    }
    /* threads 1..T-1 in the background, job 0 on the calling thread; a job
       whose thread cannot be spawned runs inline */
    char *spawned = (char *)calloc((size_t)n_threads, 1);
    for (int t = 1; t < n_threads; ++t) {
        if (spawned && pthread_create(&tids[t], NULL, run_rows, &jobs[t]) == 0)
            spawned[t] = 1;
        else
            run_rows(&jobs[t]);
    }
    run_rows(&jobs[0]);
    for (int t = 1; t < n_threads; ++t)
        if (spawned && spawned[t]) pthread_join(tids[t], NULL);
    free(spawned);
    free(jobs);
    free(tids);
    free(arows);
    free(bcols);
    return ORACLE_OK;
}

/*
 * oracle_epilogue: D = act(alpha * C_ref + beta * C_in + bias), elementwise in
 * fp64, for the block whose C_ref was computed by oracle_gemm (n_rows x
 * n_cols, row-major; rows/cols are the same index lists, NULL = all).
 *   C_in   : the incoming C (storage of c_dtype, addressed with ldc/c_major as
 *            the C ABI does: c_major 1 = C[m*ldc+n], 0 = C[n*ldc+m]); read
 *            only when beta != 0
 *   bias   : NULL or N elements of c_dtype, bias[n] added to column n
 *   act    : 0 none, 1 ReLU max(x, 0), 2 GELU x * Phi(x) = x/2 (1 + erf(x/sqrt 2))
 * This is the fused epilogue of the CuTe DSL Ampere SGEMM example (its
 * `epilogue_op` hook, applied to the accumulator before the store) with the
 * usual GEMM scaling, bias and activation written out.
 */
int oracle_epilogue(int64_t M, int64_t N, const double *C_ref,
                    const int64_t *rows, int64_t n_rows, const int64_t *cols, int64_t n_cols,
                    double alpha, double beta, const void *C_in, int64_t ldc, int c_major,
                    int c_dtype, const void *bias, int act, double *D_out) {
    if (!rows) n_rows = M;
    if (!cols) n_cols = N;
    if (n_rows < 0 || n_cols < 0 || !C_ref || !D_out) return ORACLE_EINVAL;
    if (c_dtype < 0 || c_dtype > 2 || act < 0 || act > 2) return ORACLE_EINVAL;
    if (beta != 0.0 && !C_in) return ORACLE_EINVAL;
    /* C viewed as an operand: row-major C is "K-major" with r = m, k = n */
    operand_t oc = {C_in, ldc, c_major == 1 ? ORACLE_MAJOR_K : ORACLE_MAJOR_MN, c_dtype};
    operand_t ob = {bias, 0, ORACLE_MAJOR_MN, c_dtype};
    for (int64_t i = 0; i < n_rows; ++i) {
        int64_t m = rows ? rows[i] : i;
        if (m < 0 || m >= M) return ORACLE_EINVAL;
        for (int64_t j = 0; j < n_cols; ++j) {
            int64_t n = cols ? cols[j] : j;
            if (n < 0 || n >= N) return ORACLE_EINVAL;
            double x = alpha * C_ref[i * n_cols + j];
            if (beta != 0.0) x += beta * element(&oc, m, n);
            if (bias) x += element(&ob, n, 0); /* bias[n]: MN-major, r = n, k = 0 */
            if (act == 1) x = x > 0.0 ? x : 0.0;
            else if (act == 2) x = 0.5 * x * (1.0 + erf(x / sqrt(2.0)));
            D_out[i * n_cols + j] = x;
        }
    }
    return ORACLE_OK;
}

/*
 * oracle_softmax_rows: y[m][n] = exp(x[m][n] - mx) / sum_j exp(x[m][j] - mx),
 * mx = max_j x[m][j], per row, in fp64 (x and y fp32 storage, row pitches
 * ldx/ldy in elements). The numerically stable row softmax of the Gluon
 * Multi-CTA tutorial's multi-CTA softmax kernel: row max, exponentials of the
 * shifted row, their sum, one division. Rows are independent; each is one
 * sequential max, one sequential sum.
 */
int oracle_softmax_rows(int64_t M, int64_t N, const float *x, int64_t ldx, double *y,
                        int64_t ldy) {
    if (M < 0 || N < 0) return ORACLE_EINVAL;
    if (M == 0 || N == 0) return ORACLE_OK;
    if (!x || !y || ldx < N || ldy < N) return ORACLE_EINVAL;
    for (int64_t m = 0; m < M; ++m) {
        const float *xr = x + m * ldx;
        double *yr = y + m * ldy;
        double mx = -INFINITY;
        for (int64_t n = 0; n < N; ++n) {
            uint32_t u;
            memcpy(&u, xr + n, 4);
            double v = oracle_f32_to_f64(u);
            if (v > mx) mx = v;
        }
        double sum = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            uint32_t u;
            memcpy(&u, xr + n, 4);
            yr[n] = exp(oracle_f32_to_f64(u) - mx);
            sum += yr[n];
        }
        for (int64_t n = 0; n < N; ++n) yr[n] /= sum;
    }
    return ORACLE_OK;
}
