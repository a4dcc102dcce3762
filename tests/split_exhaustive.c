/*
 * Exhaustive check of a three-way BF16 split and a two-way TF32 split over
 * all 2^32 FP32 bit patterns.  Test code: it is handed the split under test as
 * a function pointer and checks it against properties written down here,
 * without sharing any arithmetic with it.
 *
 * BF16 split (x = x0 + 2^-8 x1 + 2^-16 x2, "Blackwell의 BF16x9" section of
 * the discuss.pytorch.kr page on the method; rounding reading: nearest, ties
 * to even, signed residuals), for every finite x:
 *   - x0 is the BF16 value nearest to x (ties: even last kept bit), except
 *     that a value whose nearest BF16 is infinite takes the BF16 just below it
 *     in magnitude;
 *   - v1 = 2^8 (x - x0) is an FP32 value and x1 is the BF16 nearest to it;
 *   - v2 = 2^8 (v1 - x1) is exactly representable in BF16 and x2 == v2;
 *   - x0 + 2^-8 x1 + 2^-16 x2 == x exactly (in double).
 * +-inf must give (x, +0, +0) and NaN three canonical quiet NaNs (0x7FC0).
 *
 * TF32 split (x = hi + lo, no scaling, Figure 2 of the NVIDIA blog post):
 *   - hi is the TF32 value (10 explicit mantissa bits) nearest to x, ties
 *     even, with the same overflow rule; lo is the TF32 value nearest to
 *     x - hi; both have their low 13 bits zero.
 *
 * "Nearest" is found by brute force: the two candidates on either side of x
 * are built from the bit pattern and their distances to x compared in
 * double, which is exact for these operands.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef void (*split3_vec_fn)(const float*, int64_t, uint16_t*, uint16_t*, uint16_t*);
typedef void (*split2_vec_fn)(const float*, int64_t, float*, float*);

static float bits_f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* Nearest value with `drop` low bits cleared, on a finite FP32 pattern.
 * Returns the pattern of the chosen candidate. */
static uint32_t nearest_pattern(uint32_t u, int drop) {
    uint32_t mask = ~((1u << drop) - 1u);
    uint32_t lo = u & mask;                 /* toward zero */
    uint32_t hi = lo + (1u << drop);        /* away from zero (next in magnitude) */
    double x = (double)bits_f(u);
    double vlo = (double)bits_f(lo);
    int hi_inf = ((hi & 0x7F800000u) == 0x7F800000u);
    double vhi = hi_inf ? ldexp(x < 0 ? -1.0 : 1.0, 128) : (double)bits_f(hi);
    double dlo = fabs(x - vlo), dhi = fabs(vhi - x);
    uint32_t pick;
    if (dlo < dhi) pick = lo;
    else if (dhi < dlo) pick = hi;
    else pick = ((lo >> drop) & 1u) ? hi : lo;        /* tie: even */
    if (pick == hi && hi_inf) pick = lo;               /* overflow reading */
    return pick;
}

static double bf16_val(uint16_t h) { return (double)bits_f((uint32_t)h << 16); }

/* Returns the number of failing patterns; *first receives the first one. */
int64_t check_bf16x3_exhaustive(split3_vec_fn split, uint32_t* first) {
    int64_t fails = 0;
    uint32_t first_bad = 0xFFFFFFFFu;
    #pragma omp parallel
    {
        float* xs = (float*)malloc(sizeof(float) * 65536);
        uint16_t* p0 = (uint16_t*)malloc(2 * 65536);
        uint16_t* p1 = (uint16_t*)malloc(2 * 65536);
        uint16_t* p2 = (uint16_t*)malloc(2 * 65536);
        int64_t my_fails = 0;
        uint32_t my_first = 0xFFFFFFFFu;
        #pragma omp for schedule(dynamic, 64)
        for (int64_t top = 0; top < 65536; ++top) {
            for (uint32_t lo16 = 0; lo16 < 65536; ++lo16)
                xs[lo16] = bits_f(((uint32_t)top << 16) | lo16);
            split(xs, 65536, p0, p1, p2);
            for (uint32_t i = 0; i < 65536; ++i) {
                uint32_t u = ((uint32_t)top << 16) | i;
                int ok = 1;
                if ((u & 0x7F800000u) == 0x7F800000u) {
                    if (u & 0x007FFFFFu)
                        ok = p0[i] == 0x7FC0 && p1[i] == 0x7FC0 && p2[i] == 0x7FC0;
                    else
                        ok = p0[i] == (uint16_t)(u >> 16) && p1[i] == 0 && p2[i] == 0;
                } else {
                    double x = (double)xs[i];
                    uint32_t e0 = nearest_pattern(u, 16);
                    ok &= (p0[i] == (uint16_t)(e0 >> 16));
                    double v1 = (x - bf16_val(p0[i])) * 256.0;          /* exact in double */
                    float v1f = (float)v1;
                    ok &= ((double)v1f == v1);
                    uint32_t e1 = nearest_pattern(f_bits(v1f), 16);
                    ok &= (p1[i] == (uint16_t)(e1 >> 16));
                    double v2 = (v1 - bf16_val(p1[i])) * 256.0;
                    ok &= (bf16_val(p2[i]) == v2);
                    double rec = bf16_val(p0[i]) + ldexp(bf16_val(p1[i]), -8)
                               + ldexp(bf16_val(p2[i]), -16);
                    ok &= (rec == x);
                    /* +-0 splits into (+-0, +0, +0) */
                    if (x == 0.0) ok &= (p0[i] == (uint16_t)(u >> 16)) && p1[i] == 0 && p2[i] == 0;
                }
                if (!ok) { ++my_fails; if (u < my_first) my_first = u; }
            }
        }
        #pragma omp critical
        {
            fails += my_fails;
            if (my_first < first_bad) first_bad = my_first;
        }
        free(xs); free(p0); free(p1); free(p2);
    }
    *first = first_bad;
    return fails;
}

int64_t check_tf32x2_exhaustive(split2_vec_fn split, uint32_t* first) {
    int64_t fails = 0;
    uint32_t first_bad = 0xFFFFFFFFu;
    #pragma omp parallel
    {
        float* xs = (float*)malloc(sizeof(float) * 65536);
        float* hi = (float*)malloc(sizeof(float) * 65536);
        float* lo = (float*)malloc(sizeof(float) * 65536);
        int64_t my_fails = 0;
        uint32_t my_first = 0xFFFFFFFFu;
        #pragma omp for schedule(dynamic, 64)
        for (int64_t top = 0; top < 65536; ++top) {
            for (uint32_t lo16 = 0; lo16 < 65536; ++lo16)
                xs[lo16] = bits_f(((uint32_t)top << 16) | lo16);
            split(xs, 65536, hi, lo);
            for (uint32_t i = 0; i < 65536; ++i) {
                uint32_t u = ((uint32_t)top << 16) | i;
                uint32_t h = f_bits(hi[i]), l = f_bits(lo[i]);
                int ok = 1;
                if ((u & 0x7F800000u) == 0x7F800000u) {
                    if (u & 0x007FFFFFu) ok = (h == 0x7FC00000u && l == 0x7FC00000u);
                    else ok = (h == u && l == 0);
                } else {
                    ok &= ((h & 0x1FFFu) == 0) && ((l & 0x1FFFu) == 0);
                    ok &= (h == nearest_pattern(u, 13));
                    double r = (double)xs[i] - (double)hi[i];
                    float rf = (float)r;
                    ok &= ((double)rf == r);
                    ok &= (l == nearest_pattern(f_bits(rf), 13));
                    /* |x - hi - lo| <= 2^-22 |x| + 2^-137 (the residual of a
                     * value near the subnormal range keeps fewer bits: TF32
                     * spacing there is 2^-136) */
                    double e = fabs((double)xs[i] - (double)hi[i] - (double)lo[i]);
                    ok &= (e <= ldexp(fabs((double)xs[i]), -22) + ldexp(1.0, -137));
                }
                if (!ok) { ++my_fails; if (u < my_first) my_first = u; }
            }
        }
        #pragma omp critical
        {
            fails += my_fails;
            if (my_first < first_bad) first_bad = my_first;
        }
        free(xs); free(hi); free(lo);
    }
    *first = first_bad;
    return fails;
}
