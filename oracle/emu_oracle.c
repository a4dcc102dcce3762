/*
 * emu_oracle.c -- plain, slow CPU oracle for the emulated-FP32 GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this file:
 * only the tests, the smoke check and the CPU-baseline leg of the benchmark
 * load it.  It shares no code, header or table with the CUDA library.
 *
 * What it computes (sources are the web pages about the method):
 *
 *  - "Unlocking Tensor Core Performance for Machine Learning Interatomic
 *    Potentials" (NVIDIA technical blog, Chinese edition), Figure 1 caption:
 *    each FP32 operand is split into three scaled BF16 components, giving nine
 *    pairwise products that are accumulated in FP32 over five anti-diagonal
 *    bands.  Same page, Figure 2 and the equation under it: TF32x3 keeps a
 *    leading TF32 part and a residual TF32 part, no scale factors, and drops
 *    the residual*residual product.
 *  - "NVIDIA, 재학습 없이 MLIP 분자 동역학을 최대 1.7배 가속한 Tensor Core FP32
 *    기법 실측 기법 공개" (discuss.pytorch.kr), section "Blackwell의 BF16x9":
 *    x = x0 + 2^-8 x1 + 2^-16 x2, eight significant bits per piece, the 3x3
 *    products grouped into five bands by scale and added to the FP32
 *    accumulator smallest band first.  Section "Ampere의 TF32x3": the same
 *    three-product TF32 identity.
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes of the repository):
 *  R1  every rounding to BF16 / TF32 is round-to-nearest, ties to even, and the
 *      residuals are signed (x - x0 may be negative);
 *  R2  a finite value whose nearest BF16 (TF32) would be infinite is truncated
 *      toward zero instead, so the residual stays finite;
 *  R3  +-inf splits into (x, +0, +0); NaN splits into canonical quiet NaNs;
 *  R4  inside a band the products are added in k order, and for one k in
 *      ascending i (i + j = band); TF32x3 adds the two residual products of
 *      every k first, then the leading products (smallest band first, as for
 *      BF16x9);
 *  R15 (Ootomo-Yokota variant) the residual is scaled by 2^11 before its
 *      TF32 rounding and the residual band is scaled back by 2^-11;
 *  R5  C = alpha*acc + beta*C0 in FP32: the product alpha*acc, the product
 *      beta*C0 and their sum are each rounded; C0 is not read when beta == 0
 *      and A, B are not read when alpha == 0 (BLAS convention).
 *
 * Matrices are row major.  op(X)[r][c] is X[r*ld + c] when trans == 0 and
 * X[c*ld + r] when trans == 1.  Build with -ffp-contract=off: the emulation
 * relies on every FP32 product and sum being rounded separately.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

static float op_at(const float* X, int64_t ld, int trans, int64_t r, int64_t c) {
    return trans ? X[c * ld + r] : X[r * ld + c];
}

/* ------------------------------------------------------------------------ */
/* Rounding of an FP32 value to BF16 and TF32 (readings R1-R3).              */
/* ------------------------------------------------------------------------ */

/* BF16 keeps the top 16 bits of the FP32 pattern.  Adding 0x7FFF plus the
 * lowest kept bit and truncating is round-to-nearest, ties to even, on the
 * magnitude (the carry may ripple into the exponent, which is correct). */
uint16_t oracle_bf16_rne(float x) {
    uint32_t u = f2u(x);
    if ((u & 0x7F800000u) == 0x7F800000u) {
        if (u & 0x007FFFFFu) return 0x7FC0u;          /* NaN (R3) */
        return (uint16_t)(u >> 16);                   /* +-inf */
    }
    uint32_t r = u + 0x7FFFu + ((u >> 16) & 1u);
    if ((r & 0x7F800000u) == 0x7F800000u)             /* would round to inf: R2 */
        return (uint16_t)(u >> 16);
    return (uint16_t)(r >> 16);
}

float oracle_bf16_to_f32(uint16_t h) { return u2f((uint32_t)h << 16); }

/* TF32 keeps sign, 8 exponent bits and 10 explicit mantissa bits: the low 13
 * bits of the FP32 pattern are zero. */
uint32_t oracle_tf32_rne_bits(float x) {
    uint32_t u = f2u(x);
    if ((u & 0x7F800000u) == 0x7F800000u) {
        if (u & 0x007FFFFFu) return 0x7FC00000u;      /* NaN (R3) */
        return u;                                     /* +-inf */
    }
    uint32_t r = (u + 0x0FFFu + ((u >> 13) & 1u)) & 0xFFFFE000u;
    if ((r & 0x7F800000u) == 0x7F800000u)             /* R2 */
        return u & 0xFFFFE000u;
    return r;
}

/* ------------------------------------------------------------------------ */
/* The splits.                                                               */
/* ------------------------------------------------------------------------ */

/* x = x0 + 2^-8 x1 + 2^-16 x2, each x_i BF16, x1 and x2 stored scaled. */
static void split3_one(float x, uint16_t* h0, uint16_t* h1, uint16_t* h2) {
    uint32_t u = f2u(x);
    if ((u & 0x7F800000u) == 0x7F800000u) {           /* R3 */
        if (u & 0x007FFFFFu) { *h0 = *h1 = *h2 = 0x7FC0u; return; }
        *h0 = (uint16_t)(u >> 16); *h1 = 0; *h2 = 0;
        return;
    }
    uint16_t p0 = oracle_bf16_rne(x);
    float r1 = x - oracle_bf16_to_f32(p0);            /* exact */
    float s1 = r1 * 256.0f;                           /* exact: power of two */
    uint16_t p1 = oracle_bf16_rne(s1);
    float r2 = s1 - oracle_bf16_to_f32(p1);           /* exact */
    float s2 = r2 * 256.0f;                           /* exact */
    uint16_t p2 = oracle_bf16_rne(s2);                /* s2 has <= 8 bits */
    *h0 = p0; *h1 = p1; *h2 = p2;
}

/* x = hi + lo, both TF32, no scaling. */
static void split2_one(float x, float* hi, float* lo) {
    uint32_t u = f2u(x);
    if ((u & 0x7F800000u) == 0x7F800000u) {
        if (u & 0x007FFFFFu) { *hi = *lo = u2f(0x7FC00000u); return; }
        *hi = x; *lo = 0.0f;
        return;
    }
    float h = u2f(oracle_tf32_rne_bits(x));
    float r = x - h;                                  /* exact */
    *hi = h;
    *lo = u2f(oracle_tf32_rne_bits(r));
}

/* The scaled residual of the Ootomo-Yokota correction (discuss.pytorch.kr
 * page, section "Ampere의 TF32x3": the paper it links adds scaling and
 * accumulates outside the tensor core).  Reading R15: hi as above, and the
 * residual multiplied by 2^11 before it is rounded to TF32, so that it keeps
 * its 11 bits where the unscaled residual would fall among FP32 subnormals.
 * x - hi is exact and the power-of-two scaling is exact. */
static void split2s_one(float x, float* hi, float* lo) {
    uint32_t u = f2u(x);
    if ((u & 0x7F800000u) == 0x7F800000u) {
        if (u & 0x007FFFFFu) { *hi = *lo = u2f(0x7FC00000u); return; }
        *hi = x; *lo = 0.0f;
        return;
    }
    float h = u2f(oracle_tf32_rne_bits(x));
    float r = ldexpf(x - h, 11);
    *hi = h;
    *lo = u2f(oracle_tf32_rne_bits(r));
}

/* Planes of op(X), rows x cols, written densely (row r at r*cols). */
void oracle_split_bf16x3(const float* X, int64_t rows, int64_t cols, int64_t ld,
                         int trans, uint16_t* P0, uint16_t* P1, uint16_t* P2) {
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            split3_one(op_at(X, ld, trans, r, c),
                       &P0[r * cols + c], &P1[r * cols + c], &P2[r * cols + c]);
}

void oracle_split_tf32x2(const float* X, int64_t rows, int64_t cols, int64_t ld,
                         int trans, float* HI, float* LO) {
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            split2_one(op_at(X, ld, trans, r, c), &HI[r * cols + c], &LO[r * cols + c]);
}

void oracle_split_tf32x2s(const float* X, int64_t rows, int64_t cols, int64_t ld,
                          int trans, float* HI, float* LO) {
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            split2s_one(op_at(X, ld, trans, r, c), &HI[r * cols + c], &LO[r * cols + c]);
}

/* Single-threaded vector form, for callers that parallelise themselves. */
void oracle_split_bf16x3_vec(const float* x, int64_t n,
                             uint16_t* P0, uint16_t* P1, uint16_t* P2) {
    for (int64_t i = 0; i < n; ++i) split3_one(x[i], &P0[i], &P1[i], &P2[i]);
}

void oracle_split_tf32x2_vec(const float* x, int64_t n, float* HI, float* LO) {
    for (int64_t i = 0; i < n; ++i) split2_one(x[i], &HI[i], &LO[i]);
}

/* ------------------------------------------------------------------------ */
/* Reference result in FP64.                                                 */
/* ------------------------------------------------------------------------ */

/* For each requested output (m = mi[p], n = ni[p]):
 *   Cref[p] = alpha * sum_k op(A)[m][k] op(B)[k][n] + beta * C0[m*ldc0 + n]
 *   Sabs[p] = sum_k |op(A)[m][k]| |op(B)[k][n]|
 * in FP64; an FP32 x FP32 product is exact in FP64. */
void oracle_gemm_f64(int transA, int transB, int64_t M, int64_t N, int64_t K,
                     float alpha, const float* A, int64_t lda,
                     const float* B, int64_t ldb,
                     float beta, const float* C0, int64_t ldc0,
                     const int64_t* mi, const int64_t* ni, int64_t npairs,
                     double* Cref, double* Sabs) {
    (void)M; (void)N;
    #pragma omp parallel for schedule(dynamic, 64)
    for (int64_t p = 0; p < npairs; ++p) {
        int64_t m = mi[p], n = ni[p];
        double s = 0.0, sa = 0.0;
        if (alpha != 0.0f) {
            for (int64_t k = 0; k < K; ++k) {
                double a = op_at(A, lda, transA, m, k);
                double b = op_at(B, ldb, transB, k, n);
                s += a * b;
                sa += fabs(a) * fabs(b);
            }
        }
        double c = (double)alpha * s;
        if (beta != 0.0f) c += (double)beta * (double)C0[m * ldc0 + n];
        Cref[p] = c;
        if (Sabs) Sabs[p] = sa;
    }
}

/* FP32 epilogue, reading R5. */
static float epilogue(float alpha, float acc, float beta, const float* C0,
                      int64_t ldc0, int64_t m, int64_t n) {
    float r = (alpha != 0.0f) ? alpha * acc : 0.0f;
    if (beta != 0.0f) {
        float t = beta * C0[m * ldc0 + n];
        r = r + t;
    }
    return r;
}

/* ------------------------------------------------------------------------ */
/* CPU BF16x9 emulation.                                                     */
/* ------------------------------------------------------------------------ */

/* For each requested output: split row m of op(A) and column n of op(B),
 * then, for band b = 4, 3, 2, 1, 0 (smallest scale first), for k, for i
 * ascending with j = b - i in 0..2:
 *      acc += 2^(-8b) * (a_i[k] * b_j[k])          (FP32, R4)
 * The BF16 x BF16 product is exact in FP32 and the power-of-two scale is exact
 * unless the result is subnormal.  When band_sums is not NULL the same terms
 * are also summed per band in FP64 (band_sums[5p + b] = sum of a_i b_j with
 * i + j = b, unscaled), so the set of terms can be checked on its own. */
void oracle_gemm_bf16x9(int transA, int transB, int64_t M, int64_t N, int64_t K,
                        float alpha, const float* A, int64_t lda,
                        const float* B, int64_t ldb,
                        float beta, const float* C0, int64_t ldc0,
                        const int64_t* mi, const int64_t* ni, int64_t npairs,
                        float* C, double* band_sums) {
    (void)M; (void)N;
    #pragma omp parallel
    {
        int64_t kk = K > 0 ? K : 1;
        uint16_t* ap = (uint16_t*)malloc(sizeof(uint16_t) * 3 * kk);
        uint16_t* bp = (uint16_t*)malloc(sizeof(uint16_t) * 3 * kk);
        #pragma omp for schedule(dynamic, 16)
        for (int64_t p = 0; p < npairs; ++p) {
            int64_t m = mi[p], n = ni[p];
            float acc = 0.0f;
            double bs[5] = {0, 0, 0, 0, 0};
            if (alpha != 0.0f) {
                for (int64_t k = 0; k < K; ++k) {
                    split3_one(op_at(A, lda, transA, m, k), &ap[k], &ap[kk + k], &ap[2 * kk + k]);
                    split3_one(op_at(B, ldb, transB, k, n), &bp[k], &bp[kk + k], &bp[2 * kk + k]);
                }
                for (int b = 4; b >= 0; --b) {
                    int ilo = b > 2 ? b - 2 : 0;
                    int ihi = b < 2 ? b : 2;
                    for (int64_t k = 0; k < K; ++k) {
                        for (int i = ilo; i <= ihi; ++i) {
                            int j = b - i;
                            float ai = oracle_bf16_to_f32(ap[i * kk + k]);
                            float bj = oracle_bf16_to_f32(bp[j * kk + k]);
                            float prod = ai * bj;
                            acc += ldexpf(prod, -8 * b);
                            bs[b] += (double)ai * (double)bj;
                        }
                    }
                }
            }
            C[p] = epilogue(alpha, acc, beta, C0, ldc0, m, n);
            if (band_sums)
                for (int b = 0; b < 5; ++b) band_sums[5 * p + b] = bs[b];
        }
        free(ap);
        free(bp);
    }
}

/* ------------------------------------------------------------------------ */
/* CPU TF32x3 emulation.                                                     */
/* ------------------------------------------------------------------------ */

/* acc accumulates, for every k, a_hi b_lo then a_lo b_hi (the residual band),
 * then, for every k, a_hi b_hi; the a_lo b_lo product is not formed.  A TF32
 * x TF32 product (11 x 11 significant bits) is exact in FP32.  band_sums, if
 * not NULL, receives per output [sum a_hi b_hi, sum (a_hi b_lo + a_lo b_hi)]
 * in FP64. */
void oracle_gemm_tf32x3(int transA, int transB, int64_t M, int64_t N, int64_t K,
                        float alpha, const float* A, int64_t lda,
                        const float* B, int64_t ldb,
                        float beta, const float* C0, int64_t ldc0,
                        const int64_t* mi, const int64_t* ni, int64_t npairs,
                        float* C, double* band_sums) {
    (void)M; (void)N;
    #pragma omp parallel
    {
        int64_t kk = K > 0 ? K : 1;
        float* ah = (float*)malloc(sizeof(float) * kk);
        float* al = (float*)malloc(sizeof(float) * kk);
        float* bh = (float*)malloc(sizeof(float) * kk);
        float* bl = (float*)malloc(sizeof(float) * kk);
        #pragma omp for schedule(dynamic, 16)
        for (int64_t p = 0; p < npairs; ++p) {
            int64_t m = mi[p], n = ni[p];
            float acc = 0.0f;
            double s0 = 0.0, s1 = 0.0;
            if (alpha != 0.0f) {
                for (int64_t k = 0; k < K; ++k) {
                    split2_one(op_at(A, lda, transA, m, k), &ah[k], &al[k]);
                    split2_one(op_at(B, ldb, transB, k, n), &bh[k], &bl[k]);
                }
                for (int64_t k = 0; k < K; ++k) {
                    float t1 = ah[k] * bl[k];
                    acc += t1;
                    float t2 = al[k] * bh[k];
                    acc += t2;
                    s1 += (double)ah[k] * (double)bl[k] + (double)al[k] * (double)bh[k];
                }
                for (int64_t k = 0; k < K; ++k) {
                    float t0 = ah[k] * bh[k];
                    acc += t0;
                    s0 += (double)ah[k] * (double)bh[k];
                }
            }
            C[p] = epilogue(alpha, acc, beta, C0, ldc0, m, n);
            if (band_sums) { band_sums[2 * p] = s0; band_sums[2 * p + 1] = s1; }
        }
        free(ah); free(al); free(bh); free(bl);
    }
}

/* ------------------------------------------------------------------------ */
/* The cheaper rungs the pages set BF16x9 and TF32x3 against.                */
/* ------------------------------------------------------------------------ */

/* "FP32 as the sum of two BF16" (the discuss.pytorch.kr page, on PyTorch's
 * "high" matmul precision): the first two pieces of the three-way split,
 * x ~ x0 + 2^-8 x1, and the three products a0 b0, a0 b1, a1 b0 -- band 1
 * (a0 b1 then a1 b0 for each k) before band 0, each product scaled by its
 * band weight; a1 b1 and the third pieces are dropped. */
void oracle_gemm_bf16x3(int transA, int transB, int64_t M, int64_t N, int64_t K,
                        float alpha, const float* A, int64_t lda,
                        const float* B, int64_t ldb,
                        float beta, const float* C0, int64_t ldc0,
                        const int64_t* mi, const int64_t* ni, int64_t npairs, float* C) {
    (void)M; (void)N;
    #pragma omp parallel
    {
        int64_t kk = K > 0 ? K : 1;
        uint16_t* ap = (uint16_t*)malloc(sizeof(uint16_t) * 3 * kk);
        uint16_t* bp = (uint16_t*)malloc(sizeof(uint16_t) * 3 * kk);
        #pragma omp for schedule(dynamic, 16)
        for (int64_t p = 0; p < npairs; ++p) {
            int64_t m = mi[p], n = ni[p];
            float acc = 0.0f;
            if (alpha != 0.0f) {
                for (int64_t k = 0; k < K; ++k) {
                    split3_one(op_at(A, lda, transA, m, k), &ap[k], &ap[kk + k], &ap[2 * kk + k]);
                    split3_one(op_at(B, ldb, transB, k, n), &bp[k], &bp[kk + k], &bp[2 * kk + k]);
                }
                for (int64_t k = 0; k < K; ++k) {
                    float t1 = oracle_bf16_to_f32(ap[k]) * oracle_bf16_to_f32(bp[kk + k]);
                    acc += ldexpf(t1, -8);
                    float t2 = oracle_bf16_to_f32(ap[kk + k]) * oracle_bf16_to_f32(bp[k]);
                    acc += ldexpf(t2, -8);
                }
                for (int64_t k = 0; k < K; ++k)
                    acc += oracle_bf16_to_f32(ap[k]) * oracle_bf16_to_f32(bp[k]);
            }
            C[p] = epilogue(alpha, acc, beta, C0, ldc0, m, n);
        }
        free(ap);
        free(bp);
    }
}

/* Ootomo-Yokota style TF32x3 (R15): the residual band with scaled
 * residuals, a_hi b_lo' then a_lo' b_hi for every k, each exact product
 * scaled back by 2^-11 and added to the FP32 accumulator, then a_hi b_hi for
 * every k; all additions are FP32 round-to-nearest (the accumulation happens
 * outside the tensor core). */
void oracle_gemm_tf32x3_oy(int transA, int transB, int64_t M, int64_t N, int64_t K,
                           float alpha, const float* A, int64_t lda,
                           const float* B, int64_t ldb,
                           float beta, const float* C0, int64_t ldc0,
                           const int64_t* mi, const int64_t* ni, int64_t npairs, float* C) {
    (void)M; (void)N;
    #pragma omp parallel
    {
        int64_t kk = K > 0 ? K : 1;
        float* ah = (float*)malloc(sizeof(float) * kk);
        float* al = (float*)malloc(sizeof(float) * kk);
        float* bh = (float*)malloc(sizeof(float) * kk);
        float* bl = (float*)malloc(sizeof(float) * kk);
        #pragma omp for schedule(dynamic, 16)
        for (int64_t p = 0; p < npairs; ++p) {
            int64_t m = mi[p], n = ni[p];
            float acc = 0.0f;
            if (alpha != 0.0f) {
                for (int64_t k = 0; k < K; ++k) {
                    split2s_one(op_at(A, lda, transA, m, k), &ah[k], &al[k]);
                    split2s_one(op_at(B, ldb, transB, k, n), &bh[k], &bl[k]);
                }
                for (int64_t k = 0; k < K; ++k) {
                    acc += ldexpf(ah[k] * bl[k], -11);
                    acc += ldexpf(al[k] * bh[k], -11);
                }
                for (int64_t k = 0; k < K; ++k)
                    acc += ah[k] * bh[k];
            }
            C[p] = epilogue(alpha, acc, beta, C0, ldc0, m, n);
        }
        free(ah); free(al); free(bh); free(bl);
    }
}

/* Single-pass TF32 ([NV] Figures 5-8, "one-pass TF32"): hi_a * hi_b only. */
void oracle_gemm_tf32(int transA, int transB, int64_t M, int64_t N, int64_t K,
                      float alpha, const float* A, int64_t lda,
                      const float* B, int64_t ldb,
                      float beta, const float* C0, int64_t ldc0,
                      const int64_t* mi, const int64_t* ni, int64_t npairs, float* C) {
    (void)M; (void)N;
    #pragma omp parallel for schedule(dynamic, 16)
    for (int64_t p = 0; p < npairs; ++p) {
        int64_t m = mi[p], n = ni[p];
        float acc = 0.0f;
        if (alpha != 0.0f) {
            for (int64_t k = 0; k < K; ++k) {
                float ah, al, bh, bl;
                split2_one(op_at(A, lda, transA, m, k), &ah, &al);
                split2_one(op_at(B, ldb, transB, k, n), &bh, &bl);
                acc += ah * bh;
            }
        }
        C[p] = epilogue(alpha, acc, beta, C0, ldc0, m, n);
    }
}

/* ------------------------------------------------------------------------ */
/* Plain FP32 GEMM (the "native FP32" the pages compare against).            */
/* ------------------------------------------------------------------------ */

/* acc = acc + fl(a*b) for k = 0..K-1: every product and every sum rounded
 * to FP32 separately. */
void oracle_gemm_fp32(int transA, int transB, int64_t M, int64_t N, int64_t K,
                      float alpha, const float* A, int64_t lda,
                      const float* B, int64_t ldb,
                      float beta, const float* C0, int64_t ldc0,
                      const int64_t* mi, const int64_t* ni, int64_t npairs,
                      float* C) {
    (void)M; (void)N;
    #pragma omp parallel for schedule(dynamic, 16)
    for (int64_t p = 0; p < npairs; ++p) {
        int64_t m = mi[p], n = ni[p];
        float acc = 0.0f;
        if (alpha != 0.0f) {
            for (int64_t k = 0; k < K; ++k) {
                float prod = op_at(A, lda, transA, m, k) * op_at(B, ldb, transB, k, n);
                acc = acc + prod;
            }
        }
        C[p] = epilogue(alpha, acc, beta, C0, ldc0, m, n);
    }
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
