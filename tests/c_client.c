/*
 * c_client.c -- a plain C caller of libemusgemm, with no CUDA headers and no
 * Python: it includes only include/emu_sgemm.h, runs emu_sgemm_host on host
 * buffers (the library copies them to the GPU and back) in BF16X9 mode, and
 * checks every element against a double-precision triple loop with the
 * library's documented bound
 *     |C - C_exact| <= (2K + 2) 2^-24 |alpha| sum_k |a_mk||b_kn| + 2^-23 |beta C0|.
 * Prints "ok <max err/bound>" and exits 0, or prints the failure and exits 1.
 *
 *   gcc -std=c11 -O2 -I include tests/c_client.c -L<libdir> -lemusgemm -lm
 */
#include <math.h>
#include <stdio.h>
#include <stdlib.h>

#include "emu_sgemm.h"

/* a small deterministic generator (xorshift32), values in [-1, 1) */
static unsigned rng_state = 2463534242u;
static float next_value(void) {
    rng_state ^= rng_state << 13;
    rng_state ^= rng_state >> 17;
    rng_state ^= rng_state << 5;
    return (float)((double)(rng_state >> 8) / 8388608.0 - 1.0);
}

int main(void) {
    const int64_t M = 300, N = 257, K = 520;
    const float alpha = 1.25f, beta = -0.5f;
    float* A = malloc(sizeof(float) * M * K);
    float* B = malloc(sizeof(float) * K * N);
    float* C = malloc(sizeof(float) * M * N);
    float* C0 = malloc(sizeof(float) * M * N);
    if (!A || !B || !C || !C0) return 1;
    for (int64_t i = 0; i < M * K; ++i) A[i] = next_value();
    for (int64_t i = 0; i < K * N; ++i) B[i] = next_value();
    for (int64_t i = 0; i < M * N; ++i) C[i] = C0[i] = next_value();

    emu_status_t st = emu_sgemm_host(0, 0, M, N, K, alpha, A, K, B, N, beta, C, N,
                                     EMU_MODE_BF16X9, NULL);
    if (st != EMU_OK) {
        printf("emu_sgemm_host: %s (%d)\n", emu_status_string(st), (int)st);
        return 1;
    }
    double worst = 0.0;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0, sabs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double p = (double)A[m * K + k] * (double)B[k * N + n];
                s += p;
                sabs += fabs(p);
            }
            const double exact = (double)alpha * s + (double)beta * (double)C0[m * N + n];
            const double bound = (2.0 * K + 2.0) * ldexp(1.0, -24) * fabs((double)alpha) * sabs +
                                 ldexp(1.0, -23) * fabs((double)beta * (double)C0[m * N + n]) +
                                 (9.0 * K + 4.0) * ldexp(1.0, -149);
            const double r = fabs((double)C[m * N + n] - exact) / bound;
            if (!(r <= 1.0)) {
                printf("element (%lld, %lld): %.9g vs %.17g, bound %.3g\n", (long long)m,
                       (long long)n, (double)C[m * N + n], exact, bound);
                return 1;
            }
            if (r > worst) worst = r;
        }
    }
    emu_shutdown();
    printf("ok %.6f\n", worst);
    free(A); free(B); free(C); free(C0);
    return 0;
}
