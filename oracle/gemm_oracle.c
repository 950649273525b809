/*
 * gemm_oracle.c -- plain FP64 reference GEMM with the fused epilogue.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links, loads or calls
 * this file; only the test suite, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA path: the enum values below are restated from the public ABI's
 * documentation, not included from it.
 *
 * What it computes (the problem as the pages state it):
 *   - "DeepGEMM" (discosf.com), sec. 1.2 and 3.1/3.4: C = A*B with FP16/BF16
 *     (or FP32) inputs, accumulation kept in a wider type than the inputs, an
 *     operator-fusion hook for activation / residual add / scaling, and C
 *     written once.
 *   - "CUDA Tile ... GEMM" (pgsm.cn), sec. 4.1 and 5.1: A is M x K, B is K x N,
 *     C is M x N, all row-major (A[row*K+k], B[k*N+col], C[row*N+col]); the CPU
 *     check is a triple loop over i, j, k.  Here the accumulator is double,
 *     not float, so the reference is exact up to one rounding per term.
 *   - Same page, sec. 2: the FFN linear Y = X W^T + b, i.e. B handed over as
 *     W[N,K] ("NK" layout), and a batch of per-head QK^T products.
 *
 * For every batch b, row i and column j:
 *     s_ij   = sum_{k=0..K-1} double(A[i,k]) * double(Bhat[k,j])     (k ascending)
 *     Bhat[k,j] = B[k*ldb + j]   (KN layout)   or   B[j*ldb + k]   (NK layout)
 *     y_ij   = alpha * s_ij  (+ bias[j])
 *     y_ij   = act(y_ij)          none | GELU (erf form) | ReLU
 *     y_ij  += beta * R[i,j]      (if a residual is given)
 *   or, for the row softmax of the scaled scores (the attention step
 *   Softmax(QK^T) of "CUDA Tile ... GEMM", sec. 2; no residual):
 *     y_ij   = exp(t_ij - m_i) / sum_j' exp(t_ij' - m_i),
 *     t_ij   = alpha * s_ij (+ bias[j]),  m_i = max_j t_ij  (all N columns)
 *     c_ij   = y_ij rounded to the output type, round-to-nearest-even
 *     S_ij   = sum_k |A[i,k] * Bhat[k,j]|    (scale of the rounding error)
 * Readings where the pages are silent: the epilogue order (scale, bias,
 * activation, residual), the exact-erf GELU, FP32 bias and residual.
 *
 * Inputs are the exact 16-bit or 32-bit values given to the GPU; 16-bit
 * values are decoded here from their IEEE bit patterns.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Element types (values as documented for the library's public dtype enum). */
#define OR_F32 0
#define OR_F16 1
#define OR_BF16 2
/* Activations. */
#define OR_ACT_NONE 0
#define OR_ACT_GELU 1
#define OR_ACT_RELU 2
#define OR_ACT_SOFTMAX 3
/* Layout of B. */
#define OR_B_KN 0
#define OR_B_NK 1

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_decode_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 0x1f;
    int fr = h & 0x3ff;
    double v;
    if (ex == 0)
        v = ldexp((double)fr, -24);                 /* subnormal: fr * 2^-14 * 2^-10 */
    else if (ex == 31)
        v = fr ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + fr), ex - 25);    /* (1 + fr/1024) * 2^(ex-15) */
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32 pattern. */
double oracle_decode_bf16(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to a binary format with p significant bits, minimum normal
 * exponent emin and largest finite value maxfinite, ties to even.  The
 * division by a power of two is exact; nearbyint() rounds half to even in the
 * default rounding mode. */
static double round_rne(double x, int p, int emin, double maxfinite)
{
    if (x == 0.0 || !isfinite(x))
        return x;
    int e;
    frexp(x, &e);             /* |x| in [2^(e-1), 2^e) */
    int lead = e - 1;
    if (lead < emin)
        lead = emin;          /* subnormal range: fixed quantum */
    double quantum = ldexp(1.0, lead - (p - 1));
    double r = nearbyint(x / quantum) * quantum;
    if (fabs(r) > maxfinite)
        return copysign(INFINITY, x);
    return r;
}

double oracle_round_to(int out_dtype, double x)
{
    switch (out_dtype) {
    case OR_F32:  return round_rne(x, 24, -126, ldexp(16777215.0, 104));   /* (2^24-1)*2^104 */
    case OR_F16:  return round_rne(x, 11, -14, 65504.0);
    case OR_BF16: return round_rne(x, 8, -126, ldexp(255.0, 120));         /* (2^8-1)*2^120 */
    default:      return NAN;
    }
}

static double load_elem(const void* base, int dtype, int64_t idx)
{
    switch (dtype) {
    case OR_F32:  return (double)((const float*)base)[idx];
    case OR_F16:  return oracle_decode_f16(((const uint16_t*)base)[idx]);
    case OR_BF16: return oracle_decode_bf16(((const uint16_t*)base)[idx]);
    default:      return NAN;
    }
}

/* GELU, erf form: 0.5*y*(1 + erf(y/sqrt(2))). */
double oracle_act(int act, double y)
{
    switch (act) {
    case OR_ACT_GELU: return 0.5 * y * (1.0 + erf(y / sqrt(2.0)));
    case OR_ACT_RELU: return y > 0.0 ? y : 0.0;
    default:          return y;
    }
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* s = sum_k A[i,k] * Bhat[k,j] (k ascending) and sa = sum_k |A[i,k] * Bhat[k,j]|. */
static void dot_ij(int dtype, int64_t K, int64_t i, int64_t j, const void* Abat, int64_t lda,
                   const void* Bbat, int64_t ldb, int b_layout, double* s_out, double* sa_out)
{
    double s = 0.0, sa = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double a = load_elem(Abat, dtype, i * lda + k);
        double bv = load_elem(Bbat, dtype, b_layout == OR_B_KN ? k * ldb + j : j * ldb + k);
        s += a * bv;
        sa += fabs(a * bv);
    }
    *s_out = s;
    *sa_out = sa;
}

/* One output row of the row softmax (every column is needed for the
 * maximum and the sum, whichever columns are reported). */
static void softmax_row(int dtype, int64_t N, int64_t K, int64_t i, const void* Abat,
                        int64_t lda, const void* Bbat, int64_t ldb, int b_layout, double alpha,
                        const float* bias, int out_dtype, const int64_t* cols, int64_t ncols,
                        double* y_row, double* c_row, double* sabs_row, double* t, double* sa_all)
{
    for (int64_t j = 0; j < N; ++j) {
        double s, sa;
        dot_ij(dtype, K, i, j, Abat, lda, Bbat, ldb, b_layout, &s, &sa);
        t[j] = alpha * s + (bias ? (double)bias[j] : 0.0);
        sa_all[j] = sa;
    }
    double m = -INFINITY;
    for (int64_t j = 0; j < N; ++j)
        if (t[j] > m)
            m = t[j];
    double z = 0.0;
    for (int64_t j = 0; j < N; ++j)
        z += exp(t[j] - m);
    for (int64_t c = 0; c < ncols; ++c) {
        int64_t j = cols ? cols[c] : c;
        double y = exp(t[j] - m) / z;
        if (y_row)
            y_row[c] = y;
        if (c_row)
            c_row[c] = oracle_round_to(out_dtype, y);
        if (sabs_row)
            sabs_row[c] = sa_all[j];
    }
}

/*
 * Full or sampled reference.  rows/cols select which outputs to compute
 * (NULL = all M rows / all N columns); results are written densely as
 * [batch][nrows][ncols].  y_out gets the epilogue value before output
 * rounding, c_out the value rounded to out_dtype, sabs_out the sum of
 * |a*b| (each may be NULL).  Returns 0, or -1 on a bad argument (the row
 * softmax takes no residual).
 */
int oracle_gemm(int dtype, int64_t M, int64_t N, int64_t K, int64_t batch,
                const void* A, int64_t lda, int64_t stride_a,
                const void* B, int64_t ldb, int64_t stride_b, int b_layout,
                double alpha, const float* bias, int act,
                const float* R, int64_t ldr, int64_t stride_r, double beta,
                int out_dtype,
                const int64_t* rows, int64_t nrows,
                const int64_t* cols, int64_t ncols,
                double* y_out, double* c_out, double* sabs_out,
                int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || batch < 0 || !A || !B)
        return -1;
    if (dtype != OR_F32 && dtype != OR_F16 && dtype != OR_BF16)
        return -1;
    if (b_layout != OR_B_KN && b_layout != OR_B_NK)
        return -1;
    if (act == OR_ACT_SOFTMAX && R)
        return -1;
    if (!rows)
        nrows = M;
    if (!cols)
        ncols = N;
    for (int64_t r = 0; rows && r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M)
            return -1;
    for (int64_t c = 0; cols && c < ncols; ++c)
        if (cols[c] < 0 || cols[c] >= N)
            return -1;

    int64_t work = batch * nrows;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t w = 0; w < work; ++w) {
        int64_t b = w / nrows;
        int64_t r = w % nrows;
        int64_t i = rows ? rows[r] : r;
        const char* Ab = (const char*)A;
        const char* Bb = (const char*)B;
        int esz = dtype == OR_F32 ? 4 : 2;
        const void* Abat = Ab + (size_t)(b * stride_a) * esz;
        const void* Bbat = Bb + (size_t)(b * stride_b) * esz;
        if (act == OR_ACT_SOFTMAX) {
            int64_t o = (b * nrows + r) * ncols;
            double* t = (double*)malloc(sizeof(double) * (size_t)(2 * N + 1));
            if (!t)
                continue;
            softmax_row(dtype, N, K, i, Abat, lda, Bbat, ldb, b_layout, alpha, bias, out_dtype,
                        cols, ncols, y_out ? y_out + o : NULL, c_out ? c_out + o : NULL,
                        sabs_out ? sabs_out + o : NULL, t, t + N);
            free(t);
            continue;
        }
        for (int64_t c = 0; c < ncols; ++c) {
            int64_t j = cols ? cols[c] : c;
            double s, sa;
            dot_ij(dtype, K, i, j, Abat, lda, Bbat, ldb, b_layout, &s, &sa);
            double y = alpha * s;
            if (bias)
                y += (double)bias[j];
            y = oracle_act(act, y);
            if (R)
                y += beta * (double)R[b * stride_r + i * ldr + j];
            int64_t o = (b * nrows + r) * ncols + c;
            if (y_out)
                y_out[o] = y;
            if (c_out)
                c_out[o] = oracle_round_to(out_dtype, y);
            if (sabs_out)
                sabs_out[o] = sa;
        }
    }
    return 0;
}

/*
 * Freivalds-style whole-matrix check vector for a linear epilogue (no
 * activation): for x in R^N,
 *     v_i = alpha * sum_k A[i,k] * (Bhat x)_k + sum_j bias_j x_j + beta * sum_j R[i,j] x_j
 * equals (C x)_i in exact arithmetic, and
 *     w_i = sum_k |A[i,k]| * sum_j |Bhat[k,j]| |x_j|
 * bounds sum_j |x_j| * S_ij.  Outputs are [batch][M].  Returns 0 or -1.
 */
int oracle_freivalds(int dtype, int64_t M, int64_t N, int64_t K, int64_t batch,
                     const void* A, int64_t lda, int64_t stride_a,
                     const void* B, int64_t ldb, int64_t stride_b, int b_layout,
                     double alpha, const float* bias,
                     const float* R, int64_t ldr, int64_t stride_r, double beta,
                     const double* x, double* u_scratch, double* ua_scratch,
                     double* v_out, double* w_out)
{
    if (M < 0 || N < 0 || K < 0 || batch < 0 || !A || !B || !x)
        return -1;
    int esz = dtype == OR_F32 ? 4 : 2;
    double bx = 0.0;
    if (bias)
        for (int64_t j = 0; j < N; ++j)
            bx += (double)bias[j] * x[j];
    for (int64_t b = 0; b < batch; ++b) {
        const void* Abat = (const char*)A + (size_t)(b * stride_a) * esz;
        const void* Bbat = (const char*)B + (size_t)(b * stride_b) * esz;
        for (int64_t k = 0; k < K; ++k) {
            double s = 0.0, sa = 0.0;
            for (int64_t j = 0; j < N; ++j) {
                double bv = load_elem(Bbat, dtype,
                                      b_layout == OR_B_KN ? k * ldb + j : j * ldb + k);
                s += bv * x[j];
                sa += fabs(bv) * fabs(x[j]);
            }
            u_scratch[k] = s;
            ua_scratch[k] = sa;
        }
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
        for (int64_t i = 0; i < M; ++i) {
            double s = 0.0, sa = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double a = load_elem(Abat, dtype, i * lda + k);
                s += a * u_scratch[k];
                sa += fabs(a) * ua_scratch[k];
            }
            double v = alpha * s + bx;
            if (R) {
                double rx = 0.0;
                for (int64_t j = 0; j < N; ++j)
                    rx += (double)R[b * stride_r + i * ldr + j] * x[j];
                v += beta * rx;
            }
            v_out[b * M + i] = v;
            w_out[b * M + i] = sa;
        }
    }
    return 0;
}
