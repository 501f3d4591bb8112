/*
 * gemm_oracle.c -- CPU oracle for dense GEMM.  TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
 * load this code.  The product (the CUDA library) never calls it, and it
 * shares no source, header or helper with the CUDA path.
 *
 * What it computes, for every 0 <= i < M, 0 <= j < N:
 *
 *     ref(i,j) = alpha * sum_{k<K} a(i,k) * b(k,j) + beta * c(i,j)
 *
 * This is the BLAS GEMM update C <- alpha*A*B + beta*C given in
 * "AI Programming: Matrix Product" (elainafan.one), section "Dense matrix
 * multiplication" (the text after the stripped formula says that alpha and
 * beta let one call scale and accumulate).  The loop follows the CPU triple
 * loop of the same page, section "Row-major order", with two changes that
 * only widen precision: the accumulator is fp64 (int64 for INT8 inputs), and
 * every stored operand is first decoded exactly to fp64.
 *
 * Layout (same page, section "Row-major order": offset = row*ld + col):
 *   A(i,k) = A[i*lda + k]   if layout_a==0  (row-major, M x K)
 *          = A[k*lda + i]   if layout_a==1  (column-major, i.e. stored K x M)
 *   B(k,j) = B[k*ldb + j]   if layout_b==0  (row-major, K x N)
 *          = B[j*ldb + k]   if layout_b==1  (column-major, i.e. stored N x K)
 *   C(i,j) = C[i*ldc + j]                   (row-major)
 *
 * Optional bias row (the _ex entry points), the fully-connected layer of the
 * same page, section "Fully-connected layer" (Y = X W^T + b, the bias added
 * to every row):  ref(i,j) += bias[j], bias stored in the output type.  The
 * same section's bias gradient, the sum over the batch of the output
 * gradient, is oracle_sum_rows.
 *
 * BLAS conventions (readings where the pages are silent):
 *   beta == 0  -> C is not read (NaN/Inf in C do not reach the result);
 *   alpha == 0 -> A and B are not read; ref = beta*c.
 *
 * The k order of every sum is ascending, so the result does not depend on
 * the OpenMP thread count.
 *
 * Error bound returned beside ref (fp64):
 *   bound(i,j) = rel * sum_k |alpha*a(i,k)*b(k,j)| + (|beta*c(i,j)| + |bias(j)|) * 2^-22
 * with rel = 1e-4.  The output-rounding ulp terms are separate functions
 * (oracle_ulp_bf16 for bf16 output, oracle_ulp_f16 for fp16 output), and so
 * are the roundings themselves (oracle_round_bf16, oracle_round_f16).
 *
 * TF32 inputs (in_dtype OR_TF32): the operands are stored as fp32 and ref is
 * the same exact definition as for OR_F32.  "Matrix multiplication:
 * arithmetic intensity, tiling and Tensor Core" (dilfish.github.io),
 * sections 5.5 and 5.7, lists TF32 beside FP32 and says it keeps fewer
 * mantissa bits (10 instead of 23), so it is lossy; it does not say how an
 * fp32 value is reduced to TF32.  Reading: each operand may be replaced by a
 * value with 10 fraction bits, by truncation or by rounding, which changes
 * it by less than 2^-10 of its magnitude (normal numbers); a product then
 * changes by less than (1 + 2^-10)^2 - 1 = 2^-9 + 2^-20 of its magnitude.
 * rel is widened by that much: rel = 2^-9 + 2^-20 + 1e-4.
 *
 * CSR sparse matrix-vector product (oracle_spmv_csr): see its comment.
 *
 * Parity pins: every function here is pinned by tests/test_oracle.py
 * (identity, permutation, alpha/beta semantics, exact small integers against
 * Python integers, tiny shapes against exact rationals, MAC count = M*N*K,
 * bf16 and fp16 rounding against IEEE round-to-nearest-even, the sampled
 * entry points against Python integers and against the full matrix at the
 * same elements, with padded leading dimensions).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef ORACLE_COUNT_MACS
static int64_t g_mac_count = 0;
#define COUNT_MAC() __atomic_fetch_add(&g_mac_count, 1, __ATOMIC_RELAXED)
#else
#define COUNT_MAC() ((void)0)
#endif

enum { OR_F32 = 0, OR_BF16 = 1, OR_F16 = 2, OR_I8 = 3, OR_I32 = 4, OR_TF32 = 5 };
enum { OR_ROW_MAJOR = 0, OR_COL_MAJOR = 1 };

/* ---- exact decoding of stored elements ---------------------------------- */

/* bfloat16: the upper 16 bits of an IEEE binary32. */
static double decode_bf16(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);              /* subnormal: m * 2^-14 * 2^-10 */
    } else if (e == 31) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + m), e - 25);  /* (1 + m/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

static double load_fp(int dtype, const void* p, int64_t idx) {
    switch (dtype) {
    case OR_F32:
    case OR_TF32: return (double)((const float*)p)[idx];  /* TF32 operands are stored as fp32 */
    case OR_BF16: return decode_bf16(((const uint16_t*)p)[idx]);
    case OR_F16: return decode_f16(((const uint16_t*)p)[idx]);
    default: return NAN;
    }
}

static int64_t b_index(int layout_b, int64_t k, int64_t j, int64_t ldb) {
    return layout_b == OR_COL_MAJOR ? j * ldb + k : k * ldb + j;
}

static int64_t a_index(int layout_a, int64_t i, int64_t k, int64_t lda) {
    return layout_a == OR_COL_MAJOR ? k * lda + i : i * lda + k;
}

/* ---- one output element, floating point --------------------------------- */

static void fp_element(int in_dtype, int out_dtype, int layout_a, int layout_b, int64_t K,
                       double alpha, const void* A, int64_t lda, const void* B,
                       int64_t ldb, double beta, const void* C, int64_t ldc,
                       const void* bias, int64_t i, int64_t j, double* ref, double* bound) {
    double sum = 0.0, abs_sum = 0.0;
    if (alpha != 0.0) {
        for (int64_t k = 0; k < K; ++k) {
            double a = load_fp(in_dtype, A, a_index(layout_a, i, k, lda));
            double b = load_fp(in_dtype, B, b_index(layout_b, k, j, ldb));
            sum += a * b;            /* exact product for fp32/bf16/fp16 inputs */
            abs_sum += fabs(a * b);
            COUNT_MAC();
        }
    }
    double cterm = 0.0;
    if (beta != 0.0) cterm = beta * load_fp(out_dtype, C, i * ldc + j);
    double bterm = bias ? load_fp(out_dtype, bias, j) : 0.0;
    /* relative term: fp32 accumulation (1e-4), plus TF32 operand reduction */
    const double rel = in_dtype == OR_TF32 ? ldexp(1.0, -9) + ldexp(1.0, -20) + 1e-4 : 1e-4;
    *ref = alpha * sum + cterm + bterm;
    *bound = rel * fabs(alpha) * abs_sum + (fabs(cterm) + fabs(bterm)) * ldexp(1.0, -22);
}

/* ---- one output element, INT8 x INT8 -> INT32 ---------------------------- */

/* (alpha*sum + beta*c) evaluated in int64, then reduced mod 2^32 to int32
 * two's complement.  Unsigned arithmetic keeps the wrap well defined. */
static int32_t i8_element(int layout_a, int layout_b, int64_t K, int32_t alpha,
                          const int8_t* A, int64_t lda, const int8_t* B,
                          int64_t ldb, int32_t beta, const int32_t* C,
                          int64_t ldc, const int32_t* bias, int64_t i, int64_t j) {
    int64_t sum = 0;
    if (alpha != 0) {
        for (int64_t k = 0; k < K; ++k) {
            sum += (int64_t)A[a_index(layout_a, i, k, lda)] * (int64_t)B[b_index(layout_b, k, j, ldb)];
            COUNT_MAC();
        }
    }
    uint64_t r = (uint64_t)((int64_t)alpha) * (uint64_t)sum;
    if (beta != 0) r += (uint64_t)((int64_t)beta) * (uint64_t)((int64_t)C[i * ldc + j]);
    if (bias) r += (uint64_t)((int64_t)bias[j]);
    uint32_t low = (uint32_t)r;
    int32_t out;
    memcpy(&out, &low, sizeof out);
    return out;
}

/* ---- public entry points ------------------------------------------------- */

/* Full matrix, floating-point inputs, both operand layouts and an optional
 * bias row (NULL: none).  ref and bound are M x N row-major fp64 arrays with
 * leading dimension N.  Returns 0, or -1 on an unsupported dtype. */
int oracle_gemm_fp_ex(int in_dtype, int out_dtype, int layout_a, int layout_b, int64_t M,
                      int64_t N, int64_t K, double alpha, const void* A, int64_t lda,
                      const void* B, int64_t ldb, double beta, const void* C, int64_t ldc,
                      const void* bias, double* ref, double* bound) {
    if (in_dtype != OR_F32 && in_dtype != OR_BF16 && in_dtype != OR_F16 && in_dtype != OR_TF32)
        return -1;
    if (out_dtype != OR_F32 && out_dtype != OR_BF16 && out_dtype != OR_F16) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j)
            fp_element(in_dtype, out_dtype, layout_a, layout_b, K, alpha, A, lda, B, ldb,
                       beta, C, ldc, bias, i, j, &ref[i * N + j], &bound[i * N + j]);
    return 0;
}

/* The same with A row-major and no bias. */
int oracle_gemm_fp(int in_dtype, int out_dtype, int layout_b, int64_t M,
                   int64_t N, int64_t K, double alpha, const void* A,
                   int64_t lda, const void* B, int64_t ldb, double beta,
                   const void* C, int64_t ldc, double* ref, double* bound) {
    return oracle_gemm_fp_ex(in_dtype, out_dtype, OR_ROW_MAJOR, layout_b, M, N, K, alpha, A,
                             lda, B, ldb, beta, C, ldc, NULL, ref, bound);
}

/* Selected elements only: for s < n_samples, element (rows[s], cols[s]). */
int oracle_gemm_fp_sampled(int in_dtype, int out_dtype, int layout_b, int64_t K,
                           double alpha, const void* A, int64_t lda,
                           const void* B, int64_t ldb, double beta,
                           const void* C, int64_t ldc, int64_t n_samples,
                           const int64_t* rows, const int64_t* cols,
                           double* ref, double* bound) {
    if (in_dtype != OR_F32 && in_dtype != OR_BF16 && in_dtype != OR_F16 && in_dtype != OR_TF32)
        return -1;
    if (out_dtype != OR_F32 && out_dtype != OR_BF16 && out_dtype != OR_F16) return -1;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t s = 0; s < n_samples; ++s)
        fp_element(in_dtype, out_dtype, OR_ROW_MAJOR, layout_b, K, alpha, A, lda, B, ldb,
                   beta, C, ldc, NULL, rows[s], cols[s], &ref[s], &bound[s]);
    return 0;
}

/* Full matrix, INT8 inputs, INT32 output (M x N, leading dimension N), both
 * operand layouts and an optional int32 bias row. */
int oracle_gemm_i8_ex(int layout_a, int layout_b, int64_t M, int64_t N, int64_t K,
                      int32_t alpha, const int8_t* A, int64_t lda, const int8_t* B,
                      int64_t ldb, int32_t beta, const int32_t* C, int64_t ldc,
                      const int32_t* bias, int32_t* out) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j)
            out[i * N + j] = i8_element(layout_a, layout_b, K, alpha, A, lda, B, ldb, beta,
                                        C, ldc, bias, i, j);
    return 0;
}

int oracle_gemm_i8(int layout_b, int64_t M, int64_t N, int64_t K, int32_t alpha,
                   const int8_t* A, int64_t lda, const int8_t* B, int64_t ldb,
                   int32_t beta, const int32_t* C, int64_t ldc, int32_t* out) {
    return oracle_gemm_i8_ex(OR_ROW_MAJOR, layout_b, M, N, K, alpha, A, lda, B, ldb, beta, C,
                             ldc, NULL, out);
}

int oracle_gemm_i8_sampled(int layout_b, int64_t K, int32_t alpha,
                           const int8_t* A, int64_t lda, const int8_t* B,
                           int64_t ldb, int32_t beta, const int32_t* C,
                           int64_t ldc, int64_t n_samples, const int64_t* rows,
                           const int64_t* cols, int32_t* out) {
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t s = 0; s < n_samples; ++s)
        out[s] = i8_element(OR_ROW_MAJOR, layout_b, K, alpha, A, lda, B, ldb, beta, C, ldc,
                            NULL, rows[s], cols[s]);
    return 0;
}

/* out[j] = sum over i < rows of G(i, j), G row-major with leading dimension
 * ldg, in fp64 (ascending i), and bound[j] = 1e-4 * sum_i |G(i, j)|: the bias
 * gradient of "AI Programming: Matrix Product", section "Fully-connected
 * layer" (the output gradient summed over the batch). */
int oracle_sum_rows(int dtype, int64_t rows, int64_t cols, const void* G, int64_t ldg,
                    double* out, double* bound) {
    if (dtype != OR_F32 && dtype != OR_BF16 && dtype != OR_F16) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < cols; ++j) {
        double s = 0.0, a = 0.0;
        for (int64_t i = 0; i < rows; ++i) {
            double g = load_fp(dtype, G, i * ldg + j);
            s += g;
            a += fabs(g);
        }
        out[j] = s;
        bound[j] = 1e-4 * a;
    }
    return 0;
}

/* ---- CSR sparse matrix-vector product ------------------------------------ */

/* y <- alpha * A * x + beta * y for A in CSR form: the SpMV of "AI
 * Programming: Matrix Product", sections "CSR" and "SpMV".  Row i holds the
 * nonzeros p in the half-open interval [row_offsets[i], row_offsets[i+1]),
 * each with its value values[p] in column column_indices[p]; the row's
 * result is the sum of values[p] * x[column_indices[p]] over those p.  The
 * page gives y = A x; the scaling by alpha and beta is the same BLAS-style
 * update as the GEMM above (beta == 0: y is not read; alpha == 0: A and x
 * are not read).  fp64 accumulation in ascending p.  Beside ref,
 *   bound[i] = 1e-4 * |alpha| * sum_p |values[p] * x[col]| + |beta * y[i]| * 2^-22.
 * Returns -1 when the arrays are not a CSR matrix of rows x cols
 * (row_offsets[0] != 0, decreasing offsets, or a column index outside
 * [0, cols)), else 0. */
int oracle_spmv_csr(int64_t rows, int64_t cols, const int32_t* row_offsets,
                    const int32_t* column_indices, const float* values, double alpha,
                    const float* x, double beta, const float* y, double* ref, double* bound) {
    if (rows > 0 && row_offsets[0] != 0) return -1;
    for (int64_t i = 0; i < rows; ++i) {
        if (row_offsets[i + 1] < row_offsets[i]) return -1;
        for (int64_t p = row_offsets[i]; p < row_offsets[i + 1]; ++p)
            if (column_indices[p] < 0 || column_indices[p] >= cols) return -1;
    }
#pragma omp parallel for schedule(dynamic, 256)
    for (int64_t i = 0; i < rows; ++i) {
        double sum = 0.0, abs_sum = 0.0;
        if (alpha != 0.0) {
            for (int64_t p = row_offsets[i]; p < row_offsets[i + 1]; ++p) {
                double prod = (double)values[p] * (double)x[column_indices[p]];  /* exact */
                sum += prod;
                abs_sum += fabs(prod);
                COUNT_MAC();
            }
        }
        double yterm = beta != 0.0 ? beta * (double)y[i] : 0.0;
        ref[i] = alpha * sum + yterm;
        bound[i] = 1e-4 * fabs(alpha) * abs_sum + fabs(yterm) * ldexp(1.0, -22);
    }
    return 0;
}

/* ---- output rounding ----------------------------------------------------- */

/* Nearest bfloat16 to x, ties to even, per IEEE 754 round-to-nearest-even
 * applied to a format with 8 significant bits, exponent range [-126, 127]
 * and subnormal quantum 2^-133.  Returns the 16-bit encoding. */
uint16_t oracle_round_bf16(double x) {
    float f;
    uint32_t u;
    if (isnan(x)) return 0x7fc0;
    if (x == 0.0 || isinf(x)) {
        f = (float)x;                         /* exact: +-0 and +-inf */
    } else {
        int e;
        frexp(fabs(x), &e);                   /* |x| in [2^(e-1), 2^e) */
        int exp2 = e - 1;                     /* floor(log2|x|) */
        int q = exp2 < -126 ? -133 : exp2 - 7; /* quantum: 2^(exp - 7) */
        double scaled = ldexp(x, -q);         /* exact: power-of-two scaling */
        double n = nearbyint(scaled);         /* ties-to-even (default mode) */
        double r = ldexp(n, q);
        const double max_bf16 = ldexp(255.0, 120);   /* (2 - 2^-7) * 2^127 */
        if (fabs(r) > max_bf16) r = copysign(INFINITY, x);
        f = (float)r;                         /* exact: r has <= 8 bits */
    }
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* One unit in the last place of the bfloat16 value nearest x:
 * 2^(floor(log2|x|) - 7) in the normal range, 2^-133 below it. */
double oracle_ulp_bf16(double x) {
    if (x == 0.0 || !isfinite(x)) return ldexp(1.0, -133);
    int e;
    frexp(fabs(x), &e);
    int exp2 = e - 1;
    return exp2 < -126 ? ldexp(1.0, -133) : ldexp(1.0, exp2 - 7);
}

/* Nearest IEEE binary16 to x, ties to even: 11 significant bits, exponent
 * range [-14, 15], subnormal quantum 2^-24, largest finite value
 * (2 - 2^-10) * 2^15 = 65504; anything that rounds above it is infinite.
 * Returns the 16-bit encoding (sign, 5 exponent bits with bias 15, 10
 * fraction bits). */
uint16_t oracle_round_f16(double x) {
    if (isnan(x)) return 0x7e00;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double ax = fabs(x);
    if (ax == 0.0) return sign;
    if (isinf(ax)) return sign | 0x7c00;
    int e;
    frexp(ax, &e);                            /* ax in [2^(e-1), 2^e) */
    int exp2 = e - 1;                         /* floor(log2|x|) */
    int q = exp2 < -14 ? -24 : exp2 - 10;     /* quantum: 2^(exp - 10) */
    double r = ldexp(nearbyint(ldexp(ax, -q)), q);  /* ties-to-even (default mode) */
    if (r > 65504.0) return sign | 0x7c00;
    if (r < ldexp(1.0, -14))                  /* subnormal (or zero): fraction = r / 2^-24 */
        return sign | (uint16_t)ldexp(r, 24);
    frexp(r, &e);                             /* rounding may have moved r up a binade */
    exp2 = e - 1;
    uint16_t frac = (uint16_t)(ldexp(r, 10 - exp2) - 1024.0);
    return sign | (uint16_t)((exp2 + 15) << 10) | frac;
}

/* One unit in the last place of the binary16 value nearest x:
 * 2^(floor(log2|x|) - 10) in the normal range (|x| >= 2^-14), 2^-24 below it. */
double oracle_ulp_f16(double x) {
    if (x == 0.0 || !isfinite(x)) return ldexp(1.0, -24);
    int e;
    frexp(fabs(x), &e);
    int exp2 = e - 1;
    return exp2 < -14 ? ldexp(1.0, -24) : ldexp(1.0, exp2 - 10);
}

/* Exact decode, exposed so the tests can pin it. */
double oracle_decode_bf16(uint16_t h) { return decode_bf16(h); }
double oracle_decode_f16(uint16_t h) { return decode_f16(h); }

/* MAC counter of the instrumented build (-DORACLE_COUNT_MACS); -1 otherwise. */
int64_t oracle_mac_count(void) {
#ifdef ORACLE_COUNT_MACS
    return __atomic_load_n(&g_mac_count, __ATOMIC_RELAXED);
#else
    return -1;
#endif
}

void oracle_reset_mac_count(void) {
#ifdef ORACLE_COUNT_MACS
    __atomic_store_n(&g_mac_count, 0, __ATOMIC_RELAXED);
#endif
}

/* Array forms of the rounding helpers (element-wise, same definitions). */
void oracle_round_bf16_array(const double* x, uint16_t* out, int64_t n) {
#pragma omp parallel for schedule(static)
    for (int64_t s = 0; s < n; ++s) out[s] = oracle_round_bf16(x[s]);
}

void oracle_ulp_bf16_array(const double* x, double* out, int64_t n) {
#pragma omp parallel for schedule(static)
    for (int64_t s = 0; s < n; ++s) out[s] = oracle_ulp_bf16(x[s]);
}

void oracle_round_f16_array(const double* x, uint16_t* out, int64_t n) {
#pragma omp parallel for schedule(static)
    for (int64_t s = 0; s < n; ++s) out[s] = oracle_round_f16(x[s]);
}

void oracle_ulp_f16_array(const double* x, double* out, int64_t n) {
#pragma omp parallel for schedule(static)
    for (int64_t s = 0; s < n; ++s) out[s] = oracle_ulp_f16(x[s]);
}
