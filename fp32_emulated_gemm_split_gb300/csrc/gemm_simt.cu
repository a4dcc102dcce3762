// gemm_simt.cu -- plain FP32 GEMM on the CUDA cores (FFMA), the library's
// own "native FP32" baseline that the pages measure their speedups against
// ("Unlocking Tensor Core Performance for Machine Learning Interatomic
// Potentials", Figure 3: BF16x9 against native FP32 SGEMM).  Also the small
// helper kernels: C = beta*C for the degenerate cases and the bounded-wait
// self-test.
//
// 128 x 128 tile per 256-thread block, K in steps of 16 through a
// double-buffered shared-memory tile; each thread accumulates an 8 x 8 block
// (rows ty*4..+3 and 64+ty*4..+3, columns tx*4..+3 and 64+tx*4..+3) with
// sequential FMAs over K.
#include "emu_device.cuh"

namespace emu {
namespace {

constexpr int SBM = 128, SBN = 128, SBK = 16;

__global__ void __launch_bounds__(256)
gemm_simt_kernel(int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha,
                 const float* __restrict__ A, int64_t lda, const float* __restrict__ B, int64_t ldb,
                 float beta, float* __restrict__ C, int64_t ldc) {
    __shared__ __align__(16) float As[2][SBK][SBM];
    __shared__ __align__(16) float Bs[2][SBK][SBN];
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const int64_t m0 = (int64_t)blockIdx.y * SBM, n0 = (int64_t)blockIdx.x * SBN;

    // each thread loads 8 elements of the A tile and 8 of the B tile per K step
    auto load_tiles = [&](int buf, int64_t k0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = tid + 256 * i;           // 0 .. 2047
            int mm, kk;
            if (transA) { mm = e % SBM; kk = e / SBM; }   // contiguous along m in memory
            else        { kk = e % SBK; mm = e / SBK; }   // contiguous along k
            const int64_t gm = m0 + mm, gk = k0 + kk;
            float v = 0.0f;
            if (gm < M && gk < K) v = transA ? A[gk * lda + gm] : A[gm * lda + gk];
            As[buf][kk][mm] = v;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = tid + 256 * i;
            int nn, kk;
            if (transB) { kk = e % SBK; nn = e / SBK; }   // contiguous along k
            else        { nn = e % SBN; kk = e / SBN; }   // contiguous along n
            const int64_t gn = n0 + nn, gk = k0 + kk;
            float v = 0.0f;
            if (gn < N && gk < K) v = transB ? B[gn * ldb + gk] : B[gk * ldb + gn];
            Bs[buf][kk][nn] = v;
        }
    };

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

    const int64_t ksteps = (K + SBK - 1) / SBK;
    load_tiles(0, 0);
    __syncthreads();
    for (int64_t s = 0; s < ksteps; ++s) {
        const int buf = s & 1;
        if (s + 1 < ksteps) load_tiles(buf ^ 1, (s + 1) * SBK);
#pragma unroll
        for (int kk = 0; kk < SBK; ++kk) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][64 + ty * 4]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][64 + tx * 4]);
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t gm = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
        if (gm >= M) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int64_t gn = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
            if (gn >= N) continue;
            float v = alpha * acc[i][j];
            if (beta != 0.0f) v = fmaf(beta, C[gm * ldc + gn], v);
            C[gm * ldc + gn] = v;
        }
    }
}

__global__ void scale_kernel(int64_t M, int64_t N, float beta, float* __restrict__ C, int64_t ldc) {
    const int64_t total = M * N;
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = t / N, c = t - r * N;
        float* p = C + r * ldc + c;
        *p = (beta == 0.0f) ? 0.0f : beta * *p;
    }
}

// Waits on an mbarrier that nothing will ever arrive on; the bounded wait
// gives up after limit_ns and records the timeout code.
__global__ void timeout_probe_kernel(int* err, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
        mbar_wait(smem_u32(&bar), 0, err, kDevErrTimeout, limit_ns);
    }
}

}  // namespace

cudaError_t launch_gemm_simt(int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha,
                             const float* A, int64_t lda, const float* B, int64_t ldb, float beta,
                             float* C, int64_t ldc, cudaStream_t stream) {
    if (M == 0 || N == 0) return cudaSuccess;
    dim3 grid((unsigned)((N + SBN - 1) / SBN), (unsigned)((M + SBM - 1) / SBM));
    gemm_simt_kernel<<<grid, 256, 0, stream>>>(transA, transB, M, N, K, alpha, A, lda, B, ldb,
                                               beta, C, ldc);
    return cudaGetLastError();
}

cudaError_t launch_scale(int64_t M, int64_t N, float beta, float* C, int64_t ldc,
                         cudaStream_t stream) {
    if (M == 0 || N == 0) return cudaSuccess;
    const int64_t blocks = (M * N + 255) / 256;
    scale_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(M, N, beta, C, ldc);
    return cudaGetLastError();
}

cudaError_t launch_timeout_probe(int* err, uint64_t limit_ns, cudaStream_t stream) {
    timeout_probe_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace emu
