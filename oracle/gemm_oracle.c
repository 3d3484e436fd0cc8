/*
 * Plain CPU oracle for the pipelined tiled matrix multiply C = A * B.
 *
 * TEST INFRASTRUCTURE ONLY.  The product path (the CUDA library and its
 * Python binding) never links, loads or calls this file; only the tests,
 * the smoke check and the bench's CPU-baseline leg do.  It shares no code,
 * header or table with the CUDA path.
 *
 * What it computes (the plain definition the tiled kernel must reach):
 *   "Quickstart: GPU", section "Pipelining: a matmul kernel":
 *   matmul(a, b, out_dtype) with a:[m,k], b:[k,n] fp16, an fp32 Tensor Core
 *   accumulator (plgpu.ACC), and a final acc.astype(out_dtype).  The page
 *   "JAX Pallas Mosaic GPU 快速上手" (section "与仓库实现的对应关系") notes the
 *   pipelined kernels are checked with assert_allclose(result, a @ b), i.e.
 *   against the untiled product.
 *
 *   C_ref[i][j] = round_out( sum_{k=0..K-1} f64(A[i][k]) * f64(B[k][j]) )
 *
 *   - f64() decodes an IEEE 754 binary16 bit pattern exactly (written below
 *     from the format's definition: 1 sign bit, 5 exponent bits with bias 15,
 *     10 fraction bits, subnormals at exponent field 0, inf/NaN at 31).
 *   - Every product of two binary16 values is exact in binary64 (11 x 11
 *     significant bits), so the only roundings in the sum are the binary64
 *     additions, taken in ascending k for every element, independent of the
 *     thread count.
 *   - round_out is round-to-nearest-even to binary16 (subnormals kept,
 *     overflow to +-inf) or to binary32.  The pages do not name the rounding
 *     mode of astype; the IEEE default (nearest, ties to even) is the reading
 *     taken.
 *
 * Layouts: A is M x K, B is K x N, C is M x N, all dense row-major.
 * Nothing here is blocked, fused or reordered beyond the definition above;
 * rows are handed to threads whole.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- binary16 codec ---------------------------------------------------- */

double oracle_f16_decode(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int efield = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double mag;
    if (efield == 0) {
        /* zero or subnormal: frac * 2^-24 */
        mag = ldexp((double)frac, -24);
    } else if (efield == 31) {
        mag = frac == 0 ? INFINITY : NAN;
    } else {
        /* normal: (1024 + frac) * 2^(efield - 15 - 10) */
        mag = ldexp((double)(1024 + frac), efield - 25);
    }
    return sign ? -mag : mag;
}

/* Round a non-negative double that holds an integer plus a fraction to the
 * nearest integer, ties to the even neighbour. */
static double round_half_even(double q)
{
    double fl = floor(q);
    double rem = q - fl; /* exact: q < 2^52 in every call below */
    if (rem > 0.5) return fl + 1.0;
    if (rem < 0.5) return fl;
    return fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0;
}

uint16_t oracle_f16_round(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x)) return (uint16_t)(sign | 0x7e00);
    if (isinf(x)) return (uint16_t)(sign | 0x7c00);
    /* Largest finite binary16 is 65504 = 2047 * 2^5; the next step would be
     * 65536.  Half way is 65520, and the tie goes to the even significand,
     * which is the overflowing one, so everything >= 65520 becomes inf. */
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: value = f * 2^-24, f in [0, 1024] */
        double f = round_half_even(ldexp(a, 24));
        /* f == 1024 encodes the smallest normal, 0x0400, as required */
        return (uint16_t)(sign | (uint16_t)f);
    }
    int ex;
    (void)frexp(a, &ex);    /* a = m * 2^ex, m in [0.5, 1) */
    int e = ex - 1;         /* a = (2m) * 2^e, 2m in [1, 2) */
    double sig = round_half_even(ldexp(a, 10 - e)); /* in [1024, 2048] */
    if (sig == 2048.0) {
        sig = 1024.0;
        e += 1;
    }
    if (e + 15 >= 31) return (uint16_t)(sign | 0x7c00);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(sig - 1024.0));
}

float oracle_f32_round(double x)
{
    /* C's conversion from double to float rounds to nearest, ties to even,
     * in the default floating-point environment. */
    return (float)x;
}

void oracle_f16_decode_array(const uint16_t *h, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_decode(h[i]);
}

void oracle_f16_round_array(const double *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_round(x[i]);
}

/* ---- the product --------------------------------------------------------- */

enum { ORACLE_OUT_F16 = 0, ORACLE_OUT_F32 = 1, ORACLE_OUT_F64 = 2 };

typedef struct {
    const uint16_t *A;
    const double *Bd;   /* B decoded once, K x N */
    void *C;            /* nrows x N, output rows packed in `rows` order */
    int N, K, out_dtype;
    const int64_t *rows;
    int64_t row_begin, row_end;
    const void *Cin;    /* NULL, or the M x N values the sums start from */
    int cin_dtype;      /* 0 = binary16 bits, 1 = binary32 */
} row_job;

static void *row_worker(void *arg)
{
    row_job *job = (row_job *)arg;
    const int N = job->N, K = job->K;
    double *acc = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    if (!acc) return (void *)1;
    for (int64_t r = job->row_begin; r < job->row_end; ++r) {
        int64_t i = job->rows[r];
        if (job->Cin == NULL) {
            for (int j = 0; j < N; ++j) acc[j] = 0.0;
        } else if (job->cin_dtype == ORACLE_OUT_F16) {
            const uint16_t *cin = (const uint16_t *)job->Cin + i * (int64_t)N;
            for (int j = 0; j < N; ++j) acc[j] = oracle_f16_decode(cin[j]);
        } else {
            const float *cin = (const float *)job->Cin + i * (int64_t)N;
            for (int j = 0; j < N; ++j) acc[j] = (double)cin[j];
        }
        /* k ascending for every element of the row */
        for (int k = 0; k < K; ++k) {
            double a = oracle_f16_decode(job->A[i * (int64_t)K + k]);
            const double *brow = job->Bd + (int64_t)k * N;
            for (int j = 0; j < N; ++j) acc[j] += a * brow[j];
        }
        if (job->out_dtype == ORACLE_OUT_F16) {
            uint16_t *c = (uint16_t *)job->C + r * (int64_t)N;
            for (int j = 0; j < N; ++j) c[j] = oracle_f16_round(acc[j]);
        } else if (job->out_dtype == ORACLE_OUT_F32) {
            float *c = (float *)job->C + r * (int64_t)N;
            for (int j = 0; j < N; ++j) c[j] = oracle_f32_round(acc[j]);
        } else {
            double *c = (double *)job->C + r * (int64_t)N;
            memcpy(c, acc, sizeof(double) * (size_t)N);
        }
    }
    free(acc);
    return NULL;
}

int oracle_gemm_rows_decoded(const uint16_t *A, const double *Bd, void *C, int M, int N, int K,
                             int out_dtype, const int64_t *rows, int64_t nrows, int nthreads);

/*
 * Compute the listed rows of C.  `rows` holds nrows row indices into A;
 * output row r of C (nrows x N, packed) is row rows[r] of the product.
 * out_dtype: 0 = binary16 bits, 1 = binary32, 2 = the unrounded binary64
 * sums (for checking the summation itself).  Returns 0 on success, -1 on
 * bad arguments, -2 if memory or threads could not be had.
 */
int oracle_gemm_rows(const uint16_t *A, const uint16_t *B, void *C, int M, int N, int K,
                     int out_dtype, const int64_t *rows, int64_t nrows, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || nrows < 0) return -1;
    if (out_dtype < 0 || out_dtype > 2) return -1;
    if (nrows == 0 || N == 0) return 0;
    if (!C || !rows) return -1;
    if (K > 0 && (!A || !B)) return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nrows) nthreads = (int)nrows;

    double *Bd = (double *)malloc(sizeof(double) * (size_t)((int64_t)K * N > 0 ? (int64_t)K * N : 1));
    if (!Bd) return -2;
    if (K > 0) oracle_f16_decode_array(B, Bd, (int64_t)K * N);
    int rc = oracle_gemm_rows_decoded(A, Bd, C, M, N, K, out_dtype, rows, nrows, nthreads);
    free(Bd);
    return rc;
}

/*
 * As oracle_gemm_rows, with B already decoded to binary64 (K x N, e.g. by
 * oracle_f16_decode_array), so that a caller computing many row samples of
 * one product decodes B once.
 */
static int gemm_rows_impl(const uint16_t *A, const double *Bd, const void *Cin, int cin_dtype, void *C,
                          int M, int N, int K, int out_dtype, const int64_t *rows, int64_t nrows, int nthreads);

int oracle_gemm_rows_decoded(const uint16_t *A, const double *Bd, void *C, int M, int N, int K,
                             int out_dtype, const int64_t *rows, int64_t nrows, int nthreads)
{
    return gemm_rows_impl(A, Bd, NULL, 0, C, M, N, K, out_dtype, rows, nrows, nthreads);
}

/*
 * Accumulation into an existing output ("JAX Pallas 软件流水线 Software
 * Pipelining 完全指南", section 7.2: a sum accumulated into the output block
 * over the innermost grid axis, there initialised to zero on the first step;
 * here initialised to the values the output already holds, as an output that
 * aliases an input per section 7.1):
 *
 *   C_ref[i][j] = round_out( f64(Cin[i][j]) + sum_k f64(A[i][k]) * f64(B[k][j]) )
 *
 * The running sum starts at Cin and adds the products in ascending k.  Cin is
 * M x N, binary16 bits (cin_dtype 0) or binary32 (1).  Otherwise as
 * oracle_gemm_rows.
 */
int oracle_gemm_acc_rows(const uint16_t *A, const uint16_t *B, const void *Cin, int cin_dtype, void *C, int M,
                         int N, int K, int out_dtype, const int64_t *rows, int64_t nrows, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || nrows < 0) return -1;
    if (cin_dtype < 0 || cin_dtype > 1 || !Cin) return -1;
    if (nrows == 0 || N == 0) return 0;
    if (K > 0 && (!A || !B)) return -1;
    double *Bd = (double *)malloc(sizeof(double) * (size_t)((int64_t)K * N > 0 ? (int64_t)K * N : 1));
    if (!Bd) return -2;
    if (K > 0) oracle_f16_decode_array(B, Bd, (int64_t)K * N);
    int rc = gemm_rows_impl(A, Bd, Cin, cin_dtype, C, M, N, K, out_dtype, rows, nrows, nthreads);
    free(Bd);
    return rc;
}

static int gemm_rows_impl(const uint16_t *A, const double *Bd, const void *Cin, int cin_dtype, void *C,
                          int M, int N, int K, int out_dtype, const int64_t *rows, int64_t nrows, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || nrows < 0) return -1;
    if (out_dtype < 0 || out_dtype > 2) return -1;
    if (nrows == 0 || N == 0) return 0;
    if (!C || !rows) return -1;
    if (K > 0 && (!A || !Bd)) return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nrows) nthreads = (int)nrows;
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    row_job *jobs = (row_job *)calloc((size_t)nthreads, sizeof(row_job));
    int rc = 0;
    if (!tids || !jobs) rc = -2;
    int started = 0;
    for (int t = 0; rc == 0 && t < nthreads; ++t) {
        jobs[t].A = A;
        jobs[t].Bd = Bd;
        jobs[t].C = C;
        jobs[t].N = N;
        jobs[t].K = K;
        jobs[t].out_dtype = out_dtype;
        jobs[t].rows = rows;
        jobs[t].row_begin = nrows * t / nthreads;
        jobs[t].row_end = nrows * (t + 1) / nthreads;
        jobs[t].Cin = Cin;
        jobs[t].cin_dtype = cin_dtype;
        if (pthread_create(&tids[t], NULL, row_worker, &jobs[t]) != 0) {
            rc = -2;
            break;
        }
        ++started;
    }
    for (int t = 0; t < started; ++t) {
        void *ret = NULL;
        pthread_join(tids[t], &ret);
        if (ret) rc = -2;
    }
    free(jobs);
    free(tids);
    return rc;
}

/* Every row of C. */
int oracle_gemm(const uint16_t *A, const uint16_t *B, void *C, int M, int N, int K,
                int out_dtype, int nthreads)
{
    if (M < 0) return -1;
    if (M == 0) return 0;
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)M);
    if (!rows) return -2;
    for (int64_t i = 0; i < M; ++i) rows[i] = i;
    int rc = oracle_gemm_rows(A, B, C, M, N, K, out_dtype, rows, M, nthreads);
    free(rows);
    return rc;
}

/*
 * Single elements, one by one: out[t] = C_ref[ii[t]][jj[t]] for t < n, for
 * checking outputs of products too large to form whole.  Same definition,
 * same k order.  out_dtype as for oracle_gemm_rows.
 */
int oracle_gemm_elems(const uint16_t *A, const uint16_t *B, void *out, int M, int N, int K,
                      int out_dtype, const int64_t *ii, const int64_t *jj, int64_t n)
{
    if (M < 0 || N < 0 || K < 0 || n < 0) return -1;
    if (out_dtype < 0 || out_dtype > 2) return -1;
    for (int64_t t = 0; t < n; ++t) {
        int64_t i = ii[t], j = jj[t];
        if (i < 0 || i >= M || j < 0 || j >= N) return -1;
        double acc = 0.0;
        for (int k = 0; k < K; ++k)
            acc += oracle_f16_decode(A[i * (int64_t)K + k]) * oracle_f16_decode(B[(int64_t)k * N + j]);
        if (out_dtype == ORACLE_OUT_F16) ((uint16_t *)out)[t] = oracle_f16_round(acc);
        else if (out_dtype == ORACLE_OUT_F32) ((float *)out)[t] = oracle_f32_round(acc);
        else ((double *)out)[t] = acc;
    }
    return 0;
}

/* ---- the pipelined blocked add ------------------------------------------------ */

/*
 * Z = X + Y elementwise in binary32 ("JAX Pallas 软件流水线 Software Pipelining
 * 完全指南", section 6: two f32[4096, 4096] arrays added block by block, the
 * result checked with assert_array_equal against x + y).  The blocking does
 * not change any element, so the oracle is the plain definition: one IEEE
 * binary32 addition per element (round to nearest even, as C's float + in the
 * default floating-point environment).  n elements, any layout.
 */
void oracle_add_f32(const float *X, const float *Y, float *Z, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) Z[i] = X[i] + Y[i];
}
