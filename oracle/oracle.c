/*
 * oracle.c -- plain, slow, obviously-correct CPU oracle for the mixed-precision
 * dense GEMM   C = alpha * op(A) * op(B) + beta * C.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this file: only the test-suite, the smoke check and the CPU-baseline leg
 * of the benchmark use it.  It shares no code with the CUDA library; the two
 * meet only in the 16-bit input bit patterns produced by the seeded workload
 * generator.
 *
 * What it computes, and the passage each step follows:
 *
 *   - Semantics.  Each C[i][j] sums A[i][k] * B[k][j] over k -- the naive
 *     triple loop of the SGEMM tutorial page (section 3.1) -- and the
 *     formula C = A * B + C of the CATLASS page (section 2.1).  alpha/beta scaling and op() are the
 *     BLAS reading of that formula (the pages never name alpha or beta):
 *       r_ij = alpha * sum_k op(A)_ik op(B)_kj + beta * C_ij.
 *   - Precision.  Inputs are FP16 or BF16 -- or FP32 used as TF32 (the third
 *     format of the CATLASS page, section 3.2: the mantissa is truncated to 10
 *     bits, see oracle_decode_tf32); accumulation must be wider than the
 *     inputs (DeepGEMM page, section 6.2; CATLASS page, section 3.4).  The
 *     oracle decodes every input exactly to binary64 and accumulates in
 *     binary64, so it is strictly more accurate than any FP32-accumulating
 *     kernel.  An FP16 x FP16 (or BF16 x BF16) product has at most 22
 *     significant bits and is exact in binary64.
 *   - Formats.  FP16 = 1 sign, 5 exponent, 10 mantissa bits (max 65504, min
 *     normal 2^-14 ~ 6e-5, min subnormal 2^-24 ~ 6e-8); BF16 = 1 sign, 8
 *     exponent, 7 mantissa bits (max ~3.4e38, min normal 2^-126 ~ 1e-38)
 *     (CATLASS page, section 3.2).  The decoders below follow these field
 *     splits and the IEEE-754 interpretation of each field.
 *   - Layout.  Row-major with a leading dimension: element (m, n) of a stored
 *     matrix sits at offset m * ld + n (CATLASS page, section 1.3).
 *     op(X) = X for 'N'/'n', X^T for 'T'/'t'.  A with 'N' is stored M x K,
 *     with 'T' it is stored K x M; B with 'N' is stored K x N, with 'T' it is
 *     stored N x K.  C is M x N.
 *   - Output rounding.  FP32 output is the binary64 result converted by the C
 *     language's own double -> float conversion (round to nearest even).
 *     FP16/BF16 output is rounded directly from binary64 to the 16-bit format
 *     with round-to-nearest, ties-to-even, written out below from the format
 *     definition (one rounding, never through FP32).  The pages do not state a
 *     rounding mode; round-to-nearest-even is the IEEE-754 default.
 *   - Quick returns (BLAS convention, pages silent): with K == 0 or
 *     alpha == 0 the result is beta * C and A, B are not read; with
 *     beta == 0, C is not read, so NaN/Inf already in C does not propagate.
 *
 * Alongside r_ij the oracle returns S_ij = sum_k |op(A)_ik * op(B)_kj|, the
 * scale the acceptance tolerance is expressed in.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (no fast-math, no FMA
 * contraction, so every multiply and add is a separately rounded binary64 op).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F16 = 0, OR_BF16 = 1, OR_F32 = 2 };
enum { OR_OK = 0, OR_BAD_ARG = 1, OR_NO_MEM = 2 };

/* ---------------------------------------------------------------- decoders */

/* binary16: value = (-1)^s * 2^(e-15) * 1.m  (e in 1..30),
 *                   (-1)^s * 2^-14 * 0.m     (e == 0, subnormal),
 *                   +-inf / NaN              (e == 31). */
double oracle_decode_f16(uint16_t h) {
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);           /* m * 2^-10 * 2^-14 */
    } else if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/2^10) * 2^(e-15) */
    }
    return s ? -v : v;
}

/* bfloat16: the upper half of a binary32: value = (-1)^s * 2^(e-127) * 1.m
 * (e in 1..254), (-1)^s * 2^-126 * 0.m (e == 0), +-inf / NaN (e == 255). */
double oracle_decode_bf16(uint16_t h) {
    int s = (h >> 15) & 1;
    int e = (h >> 7) & 0xFF;
    int m = h & 0x7F;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -133);           /* m * 2^-7 * 2^-126 */
    } else if (e == 255) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(128 + m), e - 134); /* (1 + m/2^7) * 2^(e-127) */
    }
    return s ? -v : v;
}

double oracle_decode_f32(uint32_t u) {
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* --------------------------------------------------------------- rounders */

/* Round a non-negative finite q (q < 2^53) to the nearest integer, ties to
 * even.  q - floor(q) is exact for such q. */
static double rne_integer(double q) {
    double fl = floor(q);
    double frac = q - fl;
    if (frac > 0.5) return fl + 1.0;
    if (frac < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/*
 * Generic direct binary64 -> small binary format rounding, round to nearest,
 * ties to even.  A format with `mbits` stored mantissa bits and exponent bias
 * `bias` (exponent field width `ebits`) has, for |x| in the binade
 * [2^e, 2^(e+1)), a grid spacing of 2^(e - mbits); below the smallest normal
 * 2^(1-bias) the spacing stays 2^(1 - bias - mbits) (subnormals).  The value is
 * scaled onto that grid (an exact power-of-two scaling), rounded to an integer
 * n, and re-encoded; a carry to n == 2^(mbits+1) moves to the next binade, and
 * an exponent field that reaches all-ones means overflow to infinity.
 */
static uint16_t round_to_small(double x, int ebits, int mbits, int bias) {
    const uint16_t sign = signbit(x) ? (uint16_t)(1u << (ebits + mbits)) : 0;
    const uint16_t exp_all_ones = (uint16_t)(((1u << ebits) - 1u) << mbits);
    if (isnan(x)) return (uint16_t)(exp_all_ones | (1u << (mbits - 1)));  /* quiet NaN */
    double a = fabs(x);
    if (isinf(a)) return sign | exp_all_ones;
    if (a == 0.0) return sign;

    int E;
    (void)frexp(a, &E);           /* a = f * 2^E, f in [0.5, 1) -> binade exponent E-1 */
    int e = E - 1;
    const int emin = 1 - bias;    /* exponent of the smallest normal */
    int ulp_exp = (e < emin ? emin : e) - mbits;
    double n = rne_integer(ldexp(a, -ulp_exp));
    const double hidden = ldexp(1.0, mbits);      /* 2^mbits */
    if (n < hidden) {
        /* subnormal (only reachable when ulp_exp is the subnormal spacing) */
        return sign | (uint16_t)n;
    }
    if (n >= 2.0 * hidden) {      /* carried into the next binade */
        n = n / 2.0;
        ulp_exp += 1;
    }
    int efield = ulp_exp + mbits + bias;
    if (efield >= (1 << ebits) - 1) return sign | exp_all_ones;   /* overflow -> inf */
    return sign | (uint16_t)((unsigned)efield << mbits) | (uint16_t)(n - hidden);
}

uint16_t oracle_round_f16(double x) { return round_to_small(x, 5, 10, 15); }
uint16_t oracle_round_bf16(double x) { return round_to_small(x, 8, 7, 127); }

/* FP32 output: the C language's double -> float conversion (round to nearest
 * even under the default floating-point environment, overflow to +-inf). */
float oracle_round_f32(double x) { return (float)x; }

/* ------------------------------------------------------------------- GEMM */

/* TF32 inputs: FP32 storage whose value enters the product with its mantissa
 * cut to the 10 bits TF32 keeps.  The CATLASS page (section 3.2) describes
 * TF32 as FP32 data that stays FP32 in memory and is cut short to a 10-bit
 * mantissa only inside the tensor core.  Reading "cut short" as truncation,
 * the low 13 mantissa bits are dropped (round toward zero); the sign, the
 * 8-bit exponent and infinities/NaNs are kept. */
double oracle_decode_tf32(uint32_t u) {
    const uint32_t e = (u >> 23) & 0xFFu;
    if (e == 0xFFu) return oracle_decode_f32(u);          /* inf / NaN unchanged */
    return oracle_decode_f32(u & 0xFFFFE000u);
}

static double decode_in(int dt, const void* p, int64_t idx) {
    if (dt == OR_F32) return oracle_decode_tf32(((const uint32_t*)p)[idx]);
    const uint16_t* h = (const uint16_t*)p;
    return dt == OR_F16 ? oracle_decode_f16(h[idx]) : oracle_decode_bf16(h[idx]);
}

static double decode_c(int dt, const void* p, int64_t idx) {
    if (dt == OR_F32) return oracle_decode_f32(((const uint32_t*)p)[idx]);
    return decode_in(dt, p, idx);
}

static int is_n(char t) { return t == 'N' || t == 'n'; }
static int is_t(char t) { return t == 'T' || t == 't'; }

static int check_args(char transA, char transB, int64_t M, int64_t N, int64_t K,
                      int64_t lda, int64_t ldb, int64_t ldc, int ab_dtype, int c_dtype) {
    if (!(is_n(transA) || is_t(transA)) || !(is_n(transB) || is_t(transB))) return OR_BAD_ARG;
    if (M < 0 || N < 0 || K < 0) return OR_BAD_ARG;
    if (ab_dtype != OR_F16 && ab_dtype != OR_BF16 && ab_dtype != OR_F32) return OR_BAD_ARG;
    if (c_dtype != OR_F16 && c_dtype != OR_BF16 && c_dtype != OR_F32) return OR_BAD_ARG;
    int64_t a_cols = is_n(transA) ? K : M;
    int64_t b_cols = is_n(transB) ? N : K;
    if (lda < (a_cols > 1 ? a_cols : 1)) return OR_BAD_ARG;
    if (ldb < (b_cols > 1 ? b_cols : 1)) return OR_BAD_ARG;
    if (ldc < (N > 1 ? N : 1)) return OR_BAD_ARG;
    return OR_OK;
}

/* op(A)_ik and op(B)_kj as stored-matrix offsets (row-major, offset = row*ld+col). */
static int64_t a_off(char transA, int64_t i, int64_t k, int64_t lda) {
    return is_n(transA) ? i * lda + k : k * lda + i;
}
static int64_t b_off(char transB, int64_t k, int64_t j, int64_t ldb) {
    return is_n(transB) ? k * ldb + j : j * ldb + k;
}

/*
 * Full oracle.  R and S are dense M x N row-major binary64 outputs.
 * A is decoded once into opA (M x K), B once into opB (K x N); then
 *   for i: for k: for j: acc[j] += opA[i][k] * opB[k][j]
 * which, for every (i, j), adds the K products in increasing k -- the same
 * sum, in the same order, as the i-j-k loop of the definition.
 */
int oracle_gemm(char transA, char transB, int64_t M, int64_t N, int64_t K,
                float alpha, const void* A, int64_t lda,
                const void* B, int64_t ldb,
                float beta, const void* C, int64_t ldc,
                int ab_dtype, int c_dtype,
                double* R, double* S, int nthreads) {
    int st = check_args(transA, transB, M, N, K, lda, ldb, ldc, ab_dtype, c_dtype);
    if (st != OR_OK) return st;
    if (M == 0 || N == 0) return OR_OK;
    const double al = (double)alpha, be = (double)beta;
    const int use_ab = (K > 0 && alpha != 0.0f);
    double* opA = NULL;
    double* opB = NULL;
    if (use_ab) {
        opA = (double*)malloc(sizeof(double) * (size_t)M * (size_t)K);
        opB = (double*)malloc(sizeof(double) * (size_t)K * (size_t)N);
        if (!opA || !opB) { free(opA); free(opB); return OR_NO_MEM; }
        for (int64_t i = 0; i < M; ++i)
            for (int64_t k = 0; k < K; ++k)
                opA[i * K + k] = decode_in(ab_dtype, A, a_off(transA, i, k, lda));
        for (int64_t k = 0; k < K; ++k)
            for (int64_t j = 0; j < N; ++j)
                opB[k * N + j] = decode_in(ab_dtype, B, b_off(transB, k, j, ldb));
    }
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < M; ++i) {
        double* acc = R + i * N;
        double* sabs = S + i * N;
        for (int64_t j = 0; j < N; ++j) { acc[j] = 0.0; sabs[j] = 0.0; }
        if (use_ab) {
            for (int64_t k = 0; k < K; ++k) {
                const double a = opA[i * K + k];
                const double* brow = opB + k * N;
                for (int64_t j = 0; j < N; ++j) {
                    double p = a * brow[j];          /* exact for 16-bit inputs */
                    acc[j] = acc[j] + p;
                    sabs[j] = sabs[j] + fabs(p);
                }
            }
        }
        for (int64_t j = 0; j < N; ++j) {
            double r = use_ab ? al * acc[j] : 0.0;
            if (be != 0.0) r = r + be * decode_c(c_dtype, C, i * ldc + j);
            acc[j] = r;
        }
    }
    free(opA);
    free(opB);
    return OR_OK;
}

/*
 * Sampled oracle: the same definition evaluated only at the listed (row, col)
 * positions, one K-long dot product each, for shapes too large for the full
 * triple loop.  R[s], S[s] receive r and S at (rows[s], cols[s]).
 */
int oracle_gemm_sampled(char transA, char transB, int64_t M, int64_t N, int64_t K,
                        float alpha, const void* A, int64_t lda,
                        const void* B, int64_t ldb,
                        float beta, const void* C, int64_t ldc,
                        int ab_dtype, int c_dtype,
                        int64_t nsamp, const int64_t* rows, const int64_t* cols,
                        double* R, double* S, int nthreads) {
    int st = check_args(transA, transB, M, N, K, lda, ldb, ldc, ab_dtype, c_dtype);
    if (st != OR_OK) return st;
    for (int64_t s = 0; s < nsamp; ++s)
        if (rows[s] < 0 || rows[s] >= M || cols[s] < 0 || cols[s] >= N) return OR_BAD_ARG;
    const double al = (double)alpha, be = (double)beta;
    const int use_ab = (K > 0 && alpha != 0.0f);
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
#endif
    for (int64_t s = 0; s < nsamp; ++s) {
        const int64_t i = rows[s], j = cols[s];
        double acc = 0.0, sabs = 0.0;
        if (use_ab) {
            for (int64_t k = 0; k < K; ++k) {
                double p = decode_in(ab_dtype, A, a_off(transA, i, k, lda)) *
                           decode_in(ab_dtype, B, b_off(transB, k, j, ldb));
                acc = acc + p;
                sabs = sabs + fabs(p);
            }
        }
        double r = use_ab ? al * acc : 0.0;
        if (be != 0.0) r = r + be * decode_c(c_dtype, C, i * ldc + j);
        R[s] = r;
        S[s] = sabs;
    }
    return OR_OK;
}

/* Round `count` binary64 results to the output type: FP32 (float, written as
 * its 32-bit pattern) or FP16/BF16 (16-bit patterns). */
int oracle_round_output(int c_dtype, int64_t count, const double* R, void* out) {
    if (c_dtype == OR_F32) {
        float* o = (float*)out;
        for (int64_t s = 0; s < count; ++s) o[s] = oracle_round_f32(R[s]);
    } else if (c_dtype == OR_F16) {
        uint16_t* o = (uint16_t*)out;
        for (int64_t s = 0; s < count; ++s) o[s] = oracle_round_f16(R[s]);
    } else if (c_dtype == OR_BF16) {
        uint16_t* o = (uint16_t*)out;
        for (int64_t s = 0; s < count; ++s) o[s] = oracle_round_bf16(R[s]);
    } else {
        return OR_BAD_ARG;
    }
    return OR_OK;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* --------------------------------------------------- fused epilogue oracle */

/*
 * Fused epilogue.  The CATLASS page (section 5.2) fuses work into the GEMM
 * by swapping in a different epilogue after an unchanged mainloop, and names
 * residual add and activations next to the linear layer; it gives no
 * formula.  Read as the usual linear-layer form
 *     r_ij = act(alpha * sum_k op(A)_ik op(B)_kj + beta * C_ij + bias_j)
 * with act one of: none, ReLU (x if x > 0, else 0; NaN stays NaN),
 * GELU in its erf form x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2)), and
 * SiLU x / (1 + exp(-x)).  bias (length N, indexed by the output column) may
 * be NULL.  The sums are the plain oracle's; the epilogue is applied to each
 * binary64 result.
 */
enum { OR_ACT_NONE = 0, OR_ACT_RELU = 1, OR_ACT_GELU = 2, OR_ACT_SILU = 3 };

double oracle_activation(int act, double x) {
    switch (act) {
        case OR_ACT_NONE: return x;
        case OR_ACT_RELU: return isnan(x) ? x : (x > 0.0 ? x : 0.0);
        /* x Phi(x) with Phi(x) = erfc(-x / sqrt 2) / 2, the same value as
           (1 + erf(x / sqrt 2)) / 2 but without its cancellation where Phi(x)
           is tiny (x well below zero): full relative precision on both tails */
        case OR_ACT_GELU: return 0.5 * x * erfc(-x / sqrt(2.0));
        case OR_ACT_SILU: return x / (1.0 + exp(-x));
    }
    return NAN;
}

static int check_epilogue(const void* bias, int bias_dtype, int act) {
    if (act < OR_ACT_NONE || act > OR_ACT_SILU) return OR_BAD_ARG;
    if (bias != NULL && bias_dtype != OR_F16 && bias_dtype != OR_BF16 && bias_dtype != OR_F32)
        return OR_BAD_ARG;
    return OR_OK;
}

int oracle_gemm_ex(char transA, char transB, int64_t M, int64_t N, int64_t K,
                   float alpha, const void* A, int64_t lda,
                   const void* B, int64_t ldb,
                   float beta, const void* C, int64_t ldc,
                   int ab_dtype, int c_dtype,
                   const void* bias, int bias_dtype, int act,
                   double* R, double* S, int nthreads) {
    int st = check_epilogue(bias, bias_dtype, act);
    if (st != OR_OK) return st;
    st = oracle_gemm(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                     ab_dtype, c_dtype, R, S, nthreads);
    if (st != OR_OK) return st;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double x = R[i * N + j];
            if (bias != NULL) x = x + decode_c(bias_dtype, bias, j);
            R[i * N + j] = oracle_activation(act, x);
        }
    return OR_OK;
}

int oracle_gemm_sampled_ex(char transA, char transB, int64_t M, int64_t N, int64_t K,
                           float alpha, const void* A, int64_t lda,
                           const void* B, int64_t ldb,
                           float beta, const void* C, int64_t ldc,
                           int ab_dtype, int c_dtype,
                           const void* bias, int bias_dtype, int act,
                           int64_t nsamp, const int64_t* rows, const int64_t* cols,
                           double* R, double* S, int nthreads) {
    int st = check_epilogue(bias, bias_dtype, act);
    if (st != OR_OK) return st;
    st = oracle_gemm_sampled(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                             ab_dtype, c_dtype, nsamp, rows, cols, R, S, nthreads);
    if (st != OR_OK) return st;
    for (int64_t s = 0; s < nsamp; ++s) {
        double x = R[s];
        if (bias != NULL) x = x + decode_c(bias_dtype, bias, cols[s]);
        R[s] = oracle_activation(act, x);
    }
    return OR_OK;
}

/* ---------------------------------------------------------- softmax oracle */

/*
 * Row softmax, the SGEMM tutorial page's memory-bound kernel (section 2):
 * for each row x_0..x_{n-1} of X,
 *     m   = max_j x_j
 *     e_j = exp(x_j - m)
 *     s   = sum_j e_j
 *     y_j = e_j / s
 * Section 2.1 gives the three steps (maximum, sum of exponentials of the
 * shifted values, division); section 2.2 derives the online rescaling
 * (m' = max(m, m_new), s' = s exp(m - m') + sum exp(x - m')) that reaches the
 * same y in one scan.  The oracle is the plain three-step definition: every
 * input decoded exactly to binary64 (FP32 exactly -- no TF32 cut here), the
 * maximum, exp from libm and the sum in binary64, in increasing j.
 *
 * Special values follow the formula as written (the pages only discuss the
 * fully masked row, section 2.5, which gives 0/0):
 *   - a row that contains NaN: m is NaN, so every y_j is NaN;
 *   - a row that contains +inf: inf - inf is NaN, so every y_j is NaN;
 *   - a row whose entries are all -inf (fully masked): -inf - (-inf) is NaN,
 *     so every y_j is NaN;
 *   - otherwise an entry of -inf gives e_j = 0 and y_j = 0.
 *
 * X is rows x cols with row pitch ldx (elements) in x_dtype (F16, BF16 or
 * F32).  row_ids (length nsel) selects the rows to evaluate; NULL means all
 * rows (nsel is then ignored).  R receives one row of cols binary64 values per
 * evaluated row, densely.
 */
int oracle_softmax(int64_t rows, int64_t cols, const void* X, int64_t ldx, int x_dtype,
                   const int64_t* row_ids, int64_t nsel, double* R, int nthreads) {
    if (rows < 0 || cols < 0 || ldx < (cols > 1 ? cols : 1)) return OR_BAD_ARG;
    if (x_dtype != OR_F16 && x_dtype != OR_BF16 && x_dtype != OR_F32) return OR_BAD_ARG;
    const int64_t n_out = row_ids ? nsel : rows;
    if (n_out < 0) return OR_BAD_ARG;
    if (cols == 0 || n_out == 0) return OR_OK;
    if (X == NULL || R == NULL) return OR_BAD_ARG;
    if (row_ids)
        for (int64_t t = 0; t < nsel; ++t)
            if (row_ids[t] < 0 || row_ids[t] >= rows) return OR_BAD_ARG;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 4)
#endif
    for (int64_t t = 0; t < n_out; ++t) {
        const int64_t i = row_ids ? row_ids[t] : t;
        double* y = R + t * cols;
        int has_nan = 0;
        double m = -INFINITY;
        for (int64_t j = 0; j < cols; ++j) {
            const double x = decode_c(x_dtype, X, i * ldx + j);
            y[j] = x;
            if (isnan(x)) has_nan = 1;
            else if (x > m) m = x;
        }
        if (has_nan) m = NAN;
        double s = 0.0;
        for (int64_t j = 0; j < cols; ++j) {
            y[j] = exp(y[j] - m);
            s = s + y[j];
        }
        for (int64_t j = 0; j < cols; ++j) y[j] = y[j] / s;
    }
    return OR_OK;
}

/* ------------------------------------------------------ convolution oracle */

/*
 * 2-D convolution, forward (CATLASS page, section 5.1: a convolution is a
 * four-deep loop that becomes a matrix product once the input windows are
 * unrolled -- im2col -- which an implicit GEMM does without materialising
 * them).  The page fixes no layout or padding rule; read as the usual deep
 * learning convolution (a cross-correlation, the filter is not flipped),
 * channels last:
 *     X  N x H x W x C      input, element (n, h, w, c) at ((n*H + h)*W + w)*C + c
 *     Wt K x R x S x C      filter, element (k, r, s, c) at ((k*R + r)*S + s)*C + c
 *     Y  N x P x Q x K      output, element (n, p, q, k) at ((n*P + p)*Q + q)*K + k
 *     P = (H + 2 pad_h - dil_h (R - 1) - 1) / stride_h + 1   (floor), Q alike
 *     y = alpha * sum_{r, s, c} x(n, p*stride_h - pad_h + r*dil_h,
 *                                   q*stride_w - pad_w + s*dil_w, c) * w(k, r, s, c)
 *         + beta * y_in
 * with x = 0 outside 0 <= h < H, 0 <= w < W (zero padding on every side).
 * As a GEMM: M = N*P*Q rows, N = K columns, and the reduction runs over
 * (r, s, c).  Inputs FP16/BF16 decoded exactly, products exact in binary64,
 * summed in the order r, s, c; S receives sum |products| for the tolerance.
 * R and S are (N*P*Q) x K row-major.  y_in (the output's own type) is read
 * only when beta != 0.
 */
static int64_t conv_out_dim(int64_t in, int64_t pad, int64_t dil, int64_t f, int64_t stride) {
    const int64_t span = in + 2 * pad - dil * (f - 1) - 1;
    return span < 0 ? 0 : span / stride + 1;
}

int oracle_conv2d_dims(int64_t H, int64_t W, int64_t R, int64_t S, int64_t pad_h, int64_t pad_w,
                       int64_t stride_h, int64_t stride_w, int64_t dil_h, int64_t dil_w,
                       int64_t* P, int64_t* Q) {
    if (H < 1 || W < 1 || R < 1 || S < 1 || pad_h < 0 || pad_w < 0 || stride_h < 1 ||
        stride_w < 1 || dil_h < 1 || dil_w < 1)
        return OR_BAD_ARG;
    *P = conv_out_dim(H, pad_h, dil_h, R, stride_h);
    *Q = conv_out_dim(W, pad_w, dil_w, S, stride_w);
    return OR_OK;
}

/* The definition at selected output pixels: rows[t] (0 <= rows[t] < N*P*Q)
 * gives row t of R and S (all K channels); nrows of them. */
static void conv2d_row(int64_t m, int64_t H, int64_t W, int64_t C, int64_t K, int64_t R,
                       int64_t S, int64_t P, int64_t Q, int64_t pad_h, int64_t pad_w,
                       int64_t stride_h, int64_t stride_w, int64_t dil_h, int64_t dil_w,
                       double al, const void* X, const void* Wt, double be, const void* Yin,
                       int x_dtype, int y_dtype, double* Rrow, double* Srow) {
    const int64_t n = m / (P * Q), p = (m / Q) % P, q = m % Q;
    for (int64_t k = 0; k < K; ++k) {
        double acc = 0.0, sabs = 0.0;
        for (int64_t r = 0; r < R; ++r) {
            const int64_t h = p * stride_h - pad_h + r * dil_h;
            if (h < 0 || h >= H) continue;
            for (int64_t s = 0; s < S; ++s) {
                const int64_t w = q * stride_w - pad_w + s * dil_w;
                if (w < 0 || w >= W) continue;
                for (int64_t c = 0; c < C; ++c) {
                    const double a = decode_in(x_dtype, X, ((n * H + h) * W + w) * C + c);
                    const double b = decode_in(x_dtype, Wt, ((k * R + r) * S + s) * C + c);
                    const double prod = a * b;
                    acc = acc + prod;
                    sabs = sabs + fabs(prod);
                }
            }
        }
        double y = al * acc;
        if (be != 0.0) y = y + be * decode_c(y_dtype, Yin, m * K + k);
        Rrow[k] = y;
        Srow[k] = sabs;
    }
}

int oracle_conv2d_sampled(int64_t N, int64_t H, int64_t W, int64_t C, int64_t K, int64_t R,
                          int64_t S, int64_t pad_h, int64_t pad_w, int64_t stride_h,
                          int64_t stride_w, int64_t dil_h, int64_t dil_w, float alpha,
                          const void* X, const void* Wt, float beta, const void* Yin,
                          int x_dtype, int y_dtype, int64_t nrows, const int64_t* rows,
                          double* Rout, double* Sout, int nthreads) {
    int64_t P, Q;
    if (N < 0 || C < 1 || K < 1 || nrows < 0) return OR_BAD_ARG;
    if (oracle_conv2d_dims(H, W, R, S, pad_h, pad_w, stride_h, stride_w, dil_h, dil_w, &P, &Q))
        return OR_BAD_ARG;
    if (x_dtype != OR_F16 && x_dtype != OR_BF16) return OR_BAD_ARG;
    if (y_dtype != OR_F16 && y_dtype != OR_BF16 && y_dtype != OR_F32) return OR_BAD_ARG;
    if (nrows == 0) return OR_OK;
    if (X == NULL || Wt == NULL || rows == NULL || Rout == NULL || Sout == NULL) return OR_BAD_ARG;
    if (beta != 0.0f && Yin == NULL) return OR_BAD_ARG;
    for (int64_t t = 0; t < nrows; ++t)
        if (rows[t] < 0 || rows[t] >= N * P * Q) return OR_BAD_ARG;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 8)
#endif
    for (int64_t t = 0; t < nrows; ++t)
        conv2d_row(rows[t], H, W, C, K, R, S, P, Q, pad_h, pad_w, stride_h, stride_w, dil_h, dil_w,
                   (double)alpha, X, Wt, (double)beta, Yin, x_dtype, y_dtype, Rout + t * K,
                   Sout + t * K);
    return OR_OK;
}

int oracle_conv2d(int64_t N, int64_t H, int64_t W, int64_t C, int64_t K, int64_t R, int64_t S,
                  int64_t pad_h, int64_t pad_w, int64_t stride_h, int64_t stride_w,
                  int64_t dil_h, int64_t dil_w, float alpha, const void* X, const void* Wt,
                  float beta, const void* Yin, int x_dtype, int y_dtype,
                  double* Rout, double* Sout, int nthreads) {
    int64_t P, Q;
    if (N < 0 || C < 1 || K < 1) return OR_BAD_ARG;
    if (oracle_conv2d_dims(H, W, R, S, pad_h, pad_w, stride_h, stride_w, dil_h, dil_w, &P, &Q))
        return OR_BAD_ARG;
    if (x_dtype != OR_F16 && x_dtype != OR_BF16) return OR_BAD_ARG;
    if (y_dtype != OR_F16 && y_dtype != OR_BF16 && y_dtype != OR_F32) return OR_BAD_ARG;
    const int64_t M = N * P * Q;
    if (M == 0) return OR_OK;
    if (X == NULL || Wt == NULL || Rout == NULL || Sout == NULL) return OR_BAD_ARG;
    if (beta != 0.0f && Yin == NULL) return OR_BAD_ARG;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 8)
#endif
    for (int64_t m = 0; m < M; ++m)
        conv2d_row(m, H, W, C, K, R, S, P, Q, pad_h, pad_w, stride_h, stride_w, dil_h, dil_w,
                   (double)alpha, X, Wt, (double)beta, Yin, x_dtype, y_dtype, Rout + m * K,
                   Sout + m * K);
    return OR_OK;
}

/* ------------------------------------------ LayerNorm-after-linear oracle */

/* A binary64 value rounded to the output type (round to nearest even) and
 * read back: the value the stored element holds. */
static double round_to_type(int dt, double x) {
    if (dt == OR_F32) return (double)oracle_round_f32(x);
    if (dt == OR_F16) return oracle_decode_f16(oracle_round_f16(x));
    return oracle_decode_bf16(oracle_round_bf16(x));
}

/*
 * A linear layer with a residual add followed by LayerNorm -- the fused layer
 * the CATLASS page sets out from (its introduction; section 4.1 adds that a
 * normalisation is usually fused into the operator before it) -- with the
 * page's mixed precision rule for normalisations (section 3.4): the data path
 * stays in the storage type, the reduction is done in a wider type.  Read as
 *     h_ij  = round_C(alpha * sum_k op(A)_ik op(B)_kj + beta * C_ij + bias_j)
 *     mu_i  = (1/N) sum_j h_ij
 *     var_i = (1/N) sum_j (h_ij - mu_i)^2          (the biased variance)
 *     y_ij  = (h_ij - mu_i) / sqrt(var_i + eps) * gamma_j + shift_j
 * round_C is the output type's round to nearest even: h is the linear
 * layer's output as the storage type holds it.  The residual is C (scaled by
 * beta, usually 1).  bias, gamma and shift have N elements each in ln_dtype
 * for gamma/shift and bias_dtype for bias; NULL bias or shift reads as 0,
 * NULL gamma as 1.  mu, var and y are evaluated in binary64 from the decoded
 * h, in increasing j; y is returned before its final rounding.
 *
 * row_ids (nsel entries) selects the rows; NULL means every row (nsel is then
 * ignored).  Y and H receive one row of N values per selected row: y, and
 * the decoded h.  S receives, per element, the sum of |products| of h's dot
 * product (the GEMM oracle's tolerance scale).
 */
int oracle_gemm_layernorm(char transA, char transB, int64_t M, int64_t N, int64_t K,
                          float alpha, const void* A, int64_t lda,
                          const void* B, int64_t ldb,
                          float beta, const void* C, int64_t ldc,
                          int ab_dtype, int c_dtype,
                          const void* bias, int bias_dtype,
                          const void* gamma, const void* shift, int ln_dtype, double eps,
                          int64_t nsel, const int64_t* row_ids,
                          double* Y, double* H, double* S, int nthreads) {
    int st = check_epilogue(bias, bias_dtype, OR_ACT_NONE);
    if (st != OR_OK) return st;
    if ((gamma != NULL || shift != NULL) && ln_dtype != OR_F16 && ln_dtype != OR_BF16 &&
        ln_dtype != OR_F32)
        return OR_BAD_ARG;
    if (!(eps >= 0.0) || N < 1) return OR_BAD_ARG;
    const int64_t nr = row_ids != NULL ? nsel : M;
    if (nr < 0) return OR_BAD_ARG;
    int64_t* rr = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nr * N + 1));
    int64_t* cc = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nr * N + 1));
    if (rr == NULL || cc == NULL) {
        free(rr);
        free(cc);
        return OR_NO_MEM;
    }
    for (int64_t s = 0; s < nr; ++s)
        for (int64_t j = 0; j < N; ++j) {
            rr[s * N + j] = row_ids != NULL ? row_ids[s] : s;
            cc[s * N + j] = j;
        }
    /* alpha * sum + beta * C for every element of the selected rows */
    st = oracle_gemm_sampled(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                             ab_dtype, c_dtype, nr * N, rr, cc, H, S, nthreads);
    free(rr);
    free(cc);
    if (st != OR_OK) return st;
    for (int64_t s = 0; s < nr; ++s) {
        double* h = H + s * N;
        for (int64_t j = 0; j < N; ++j) {
            double x = h[j];
            if (bias != NULL) x = x + decode_c(bias_dtype, bias, j);
            h[j] = round_to_type(c_dtype, x);
        }
        double sum = 0.0;
        for (int64_t j = 0; j < N; ++j) sum = sum + h[j];
        const double mu = sum / (double)N;
        double sq = 0.0;
        for (int64_t j = 0; j < N; ++j) sq = sq + (h[j] - mu) * (h[j] - mu);
        const double var = sq / (double)N;
        const double inv = 1.0 / sqrt(var + eps);
        for (int64_t j = 0; j < N; ++j) {
            const double g = gamma != NULL ? decode_c(ln_dtype, gamma, j) : 1.0;
            const double t = shift != NULL ? decode_c(ln_dtype, shift, j) : 0.0;
            Y[s * N + j] = (h[j] - mu) * inv * g + t;
        }
    }
    return OR_OK;
}
