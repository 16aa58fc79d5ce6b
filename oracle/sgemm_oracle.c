/*
 * sgemm_oracle.c -- CPU oracle for row-major SGEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / --impl reference legs of bench.py may load this code.  It
 * shares nothing (no header, helper, table or build step) with the CUDA
 * library in sgemm_row_major_gb300/.
 *
 * What it computes (BLAS SGEMM, itan.pw "CUDA NVIDIA 4090 高性能計算",
 * 概要: C = alpha * op(A) * op(B) + beta * C; element definition from
 * klklkl10086.github.io "Sgemm单精度矩阵乘法", 问题定义:
 * C_ij = sum_{k=0}^{K-1} A_ik B_kj on row-major matrices):
 *
 *   Cref_ij = fl32( alpha * sum_k op(A)_ik * op(B)_kj + beta * C_ij )
 *
 * evaluated in double.  Every product of two floats is exact in double; the
 * k-sum runs in ascending k with one double accumulator per element (the
 * i-j-k loop of the page's cpu_sgemm, 代码框架); alpha*sum and beta*C are
 * formed in double and the result is rounded to float once.
 *
 * Readings where the pages are silent (BLAS / CBLAS row-major conventions):
 *   - op(X) = X for 'N'/'n', X^T for 'T'/'t'/'C'/'c' (real data).
 *   - ld is the row stride of the STORED matrix: for 'N', op(A)_ik =
 *     A[i*lda + k]; for 'T', op(A)_ik = A[k*lda + i]; likewise for B.
 *   - beta == 0: C is not read (NaN/Inf in C do not propagate).
 *   - alpha == 0 or K == 0: A and B are not read; C = fl32(beta * C).
 *
 * Alongside, the oracle can return the per-element magnitude
 *   S_ij = |alpha| * sum_k |op(A)_ik * op(B)_kj| + |beta * C_ij|
 * used by the error bound |C_gpu - Cref| <= (K + 2) * 2^-24 * S_ij.
 *
 * Parallelism: OpenMP over output elements only; it does not change the
 * arithmetic of any element.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* op character -> 0 (no transpose), 1 (transpose), -1 (invalid) */
static int oracle_op(char t)
{
    if (t == 'N' || t == 'n') return 0;
    if (t == 'T' || t == 't' || t == 'C' || t == 'c') return 1;
    return -1;
}

/* Element (r, c) of op(X), X stored row-major with row stride ld. */
static double oracle_op_elem(const float *X, int64_t ld, int trans, int64_t r, int64_t c)
{
    return trans ? (double)X[c * ld + r] : (double)X[r * ld + c];
}

/*
 * Returns 0 on success, or -i when the i-th argument is invalid
 * (1 transA, 2 transB, 3 M, 4 N, 5 K, 8 lda, 10 ldb, 13 ldc, 15 lds).
 * C is updated in place.  S (may be NULL) receives S_ij at S[i*lds + j].
 */
int oracle_sgemm(char transA, char transB, int64_t M, int64_t N, int64_t K,
                 float alpha, const float *A, int64_t lda,
                 const float *B, int64_t ldb,
                 float beta, float *C, int64_t ldc,
                 double *S, int64_t lds)
{
    const int ta = oracle_op(transA);
    const int tb = oracle_op(transB);
    if (ta < 0) return -1;
    if (tb < 0) return -2;
    if (M < 0) return -3;
    if (N < 0) return -4;
    if (K < 0) return -5;
    /* stored A is M x K ('N') or K x M ('T'); stored B is K x N or N x K */
    if (lda < (ta ? (M > 1 ? M : 1) : (K > 1 ? K : 1))) return -8;
    if (ldb < (tb ? (K > 1 ? K : 1) : (N > 1 ? N : 1))) return -10;
    if (ldc < (N > 1 ? N : 1)) return -13;
    if (S && lds < (N > 1 ? N : 1)) return -15;

    const int read_ab = (alpha != 0.0f) && (K > 0);
    const int read_c = (beta != 0.0f);
    const int64_t total = M * N;

#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < total; ++e) {
        const int64_t i = e / N;
        const int64_t j = e % N;
        double sum = 0.0;
        double sum_abs = 0.0;
        if (read_ab) {
            for (int64_t k = 0; k < K; ++k) {
                const double p = oracle_op_elem(A, lda, ta, i, k) *
                                 oracle_op_elem(B, ldb, tb, k, j);
                sum += p;
                sum_abs += fabs(p);
            }
        }
        const double c_old = read_c ? (double)C[i * ldc + j] : 0.0;
        const double bc = (double)beta * c_old;
        const double r = (double)alpha * sum + bc;
        C[i * ldc + j] = (float)r;
        if (S) S[i * lds + j] = fabs((double)alpha) * sum_abs + fabs(bc);
    }
    return 0;
}

/*
 * Strided batch (the use of SGEMM for many fully connected layers at once,
 * itan.pw page, 概要): product b = 0 .. batch-1 is the SGEMM above on the
 * matrices that start at A + b*strideA, B + b*strideB and C + b*strideC
 * (strides in elements; 0 shares one matrix).  S, when given, receives
 * product b's magnitudes at S + b*strideS.  Products are computed one after
 * another in ascending b.  Returns 0, -100 for a negative stride or batch, or
 * the first product's own error status.
 */
int oracle_sgemm_strided_batched(char transA, char transB, int64_t M, int64_t N, int64_t K,
                                 float alpha, const float *A, int64_t lda, int64_t strideA,
                                 const float *B, int64_t ldb, int64_t strideB,
                                 float beta, float *C, int64_t ldc, int64_t strideC,
                                 int64_t batch, double *S, int64_t lds, int64_t strideS)
{
    if (strideA < 0 || strideB < 0 || strideC < 0 || strideS < 0 || batch < 0) return -100;
    for (int64_t b = 0; b < batch; ++b) {
        const float *Ab = A ? A + b * strideA : A;
        const float *Bb = B ? B + b * strideB : B;
        float *Cb = C ? C + b * strideC : C;
        double *Sb = S ? S + b * strideS : S;
        const int st = oracle_sgemm(transA, transB, M, N, K, alpha, Ab, lda, Bb, ldb, beta, Cb, ldc, Sb, lds);
        if (st != 0) return st;
    }
    return 0;
}

/*
 * TF32 rounding (the tensor-core format for FP32 data, youngju.dev "CUDA
 * architecture visualized", テンソルコア): 1 sign bit, the 8 exponent bits of
 * float32 and 10 fraction bits.  Its values are the floats whose 13 lowest
 * fraction bits are zero, so the spacing (quantum) of values near |x| is
 * 2^(floor(log2|x|) - 10) for normal x and 2^-136 below 2^-126.  y = x
 * rounded to the nearest such value, ties away from zero; a rounding that
 * carries past FLT_MAX gives +-Inf; +-0, +-Inf and NaN are kept.  Computed in
 * double, where every step is exact.
 */
static float oracle_tf32(float x)
{
    if (x != x || isinf(x) || x == 0.0f) return x;
    const double a = fabs((double)x);
    int e;
    frexp(a, &e);                       /* a = m * 2^e, 0.5 <= m < 1: floor(log2 a) = e - 1 */
    int qexp = (e - 1) - 10;
    if (qexp < -136) qexp = -136;       /* subnormal range: fixed quantum */
    const double q = ldexp(1.0, qexp);
    const double r = floor(a / q + 0.5) * q;   /* nearest multiple, ties away from zero */
    const double y = x < 0.0f ? -r : r;
    return (float)y;                    /* exact, or +-Inf past FLT_MAX */
}

void oracle_round_tf32(const float *x, float *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_tf32(x[i]);
}

/*
 * BF16 rounding (the other tensor-core input format for FP32-range data the
 * page names, youngju.dev "CUDA architecture visualized", テンソルコア): 1 sign
 * bit, float32's 8 exponent bits and 7 fraction bits, so the quantum near |x|
 * is 2^(floor(log2|x|) - 7) for normal x and 2^-133 below 2^-126.  y = x
 * rounded to the nearest such value, ties to the one whose last kept bit is
 * 0 (IEEE round to nearest even; the pages give no rule, so the IEEE default);
 * past the largest BF16 value (2 - 2^-7) 2^127 to +-Inf; +-0, +-Inf and NaN
 * kept.  Computed in double, where every step is exact.
 */
static float oracle_bf16(float x)
{
    if (x != x || isinf(x) || x == 0.0f) return x;
    const double a = fabs((double)x);
    int e;
    frexp(a, &e);                       /* floor(log2 a) = e - 1 */
    int qexp = (e - 1) - 7;
    if (qexp < -133) qexp = -133;       /* subnormal range: fixed quantum */
    const double q = ldexp(1.0, qexp);
    const double n = a / q;             /* exact: a has at most 24 significant bits */
    double m = floor(n);
    const double frac = n - m;
    if (frac > 0.5 || (frac == 0.5 && fmod(m, 2.0) != 0.0)) m += 1.0;   /* nearest, ties to even */
    const double r = m * q;
    const double y = (x < 0.0f) ? -r : r;
    return (float)y;                    /* exact, or +-Inf past the largest BF16 value */
}

void oracle_round_bf16(const float *x, float *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_bf16(x[i]);
}

/* Sets the number of OpenMP threads later oracle calls use (n >= 1). */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Number of OpenMP threads a parallel region of the oracle uses. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
