// gemm_tc.cu -- the tensor-core GEMM of the two-pass path.
//
// Inputs are the pieces written by split.cu: for BF16x9 three BF16 planes
// per operand, for TF32x3 two TF32 planes, each K-major (op(A) as M x K,
// op(B)^T as N x K) with a row stride that is a multiple of 16 bytes.
//
// Method ("Unlocking Tensor Core Performance for Machine Learning Interatomic
// Potentials", Figure 1 caption; discuss.pytorch.kr summary, section
// "Blackwell의 BF16x9"): the nine products a_i b_j fall into five bands
// b = i + j with weight 2^-8b, and the bands are added to one FP32
// accumulator smallest band first.  Here the accumulator lives in tensor
// memory and the bands are processed one after the other over the whole K
// range: band 4 (a2 b2), band 3 (a1 b2, a2 b1), band 2, band 1, band 0.  The
// first MMA of each later band is issued with scale-input-d = 8, i.e.
// D = A*B + 2^-8 D, so the finished bands are shifted down by one band
// weight before the next band is added on top of them:
//     acc = S0 + 2^-8 (S1 + 2^-8 (S2 + 2^-8 (S3 + 2^-8 S4))).
// TF32x3 (Figure 2 and its equation) runs the residual band (hi*lo, lo*hi)
// first and then hi*hi into the same accumulator, without scaling.
//
// Structure (one CTA per 128 x 256 tile of C, one CTA per SM):
//   warp 4, one thread   TMA producer: streams (A piece, B piece) K-blocks
//                        through a 4-stage shared-memory ring;
//   warp 5, one thread   MMA issuer: 4 tcgen05.mma (kind::f16 K=16 or
//                        kind::tf32 K=8) per stage, commit frees the stage;
//   warps 0-3            epilogue: TMEM -> registers (tcgen05.ld), then
//                        C = alpha*acc + beta*C in FP32.
// Each stage is one 128-byte-wide K block of a piece: the pipeline sees the
// same operand traffic per MMA as a plain BF16 GEMM whose K is 9x longer.
#include "emu_device.cuh"

namespace emu {
namespace {

constexpr int BM = kTcBM, BN = kTcBN, S = kTcStages;
constexpr int kStageA = BM * kTcBKBytes;            // 16 KB
constexpr int kStageB = BN * kTcBKBytes;            // 32 KB
constexpr int kStageBytes = kStageA + kStageB;      // 48 KB
constexpr int kSmemBytes = S * kStageBytes + 1024 /*barriers*/ + 1024 /*alignment*/;
constexpr uint32_t kTmemCols = 256;

// Pairs (i, j) of pieces in processing order, grouped by band, packed four
// bits per pair (i in bits 2-3, j in bits 0-1) so that no thread needs an
// indexed local array; band lengths packed four bits per band.
struct Schedule {
    uint64_t pairs;
    uint32_t band_len;
    int nbands;
    int scale8;            // 1: shift the accumulator by 2^-8 between bands
    __device__ __forceinline__ int pi(int t) const { return int((pairs >> (4 * t + 2)) & 3u); }
    __device__ __forceinline__ int pj(int t) const { return int((pairs >> (4 * t)) & 3u); }
    __device__ __forceinline__ int len(int b) const { return int((band_len >> (4 * b)) & 15u); }
};

constexpr uint64_t pack_pairs(const int (&ij)[9][2], int n) {
    uint64_t v = 0;
    for (int t = 0; t < n; ++t) v |= uint64_t((ij[t][0] << 2) | ij[t][1]) << (4 * t);
    return v;
}

// BF16x9: band 4: (2,2) | band 3: (1,2) (2,1) | band 2: (0,2) (1,1) (2,0) |
//         band 1: (0,1) (1,0) | band 0: (0,0)
constexpr int kBf16Pairs[9][2] = {{2, 2}, {1, 2}, {2, 1}, {0, 2}, {1, 1}, {2, 0}, {0, 1}, {1, 0}, {0, 0}};
// TF32x3 (piece 0 = hi, 1 = lo): residual band (hi,lo) (lo,hi) | leading band (hi,hi)
constexpr int kTf32Pairs[9][2] = {{0, 1}, {1, 0}, {0, 0}};
constexpr uint64_t kBf16Packed = pack_pairs(kBf16Pairs, 9);
constexpr uint64_t kTf32Packed = pack_pairs(kTf32Pairs, 3);

__device__ __forceinline__ Schedule schedule_for(int tf32) {
    Schedule s;
    if (!tf32) {
        s.pairs = kBf16Packed;
        s.band_len = 1u | (2u << 4) | (3u << 8) | (2u << 12) | (1u << 16);
        s.nbands = 5;
        s.scale8 = 1;
    } else {
        s.pairs = kTf32Packed;
        s.band_len = 2u | (1u << 4);
        s.nbands = 2;
        s.scale8 = 0;
    }
    return s;
}

template <int TF32>
__global__ void __launch_bounds__(kTcThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
               const TcGemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * kStageBytes);
    // bars[0..S): full, bars[S..2S): empty, bars[2S]: accumulator ready
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Tile coordinates, grouped so that CTAs running together share rows of A.
    constexpr int kGroupM = 8;
    const int pid = blockIdx.x;
    const int per_group = kGroupM * p.tiles_n;
    const int group = pid / per_group;
    const int first_m = group * kGroupM;
    const int gm = min(p.tiles_m - first_m, kGroupM);
    const int tile_m = first_m + (pid % per_group) % gm;
    const int tile_n = (pid % per_group) / gm;
    const int m0 = tile_m * BM, n0 = tile_n * BN;

    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S), accum = smem_u32(bars + 2 * S);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        mbar_init(accum, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&mapA);
        tma_prefetch_desc(&mapB);
    }
    if (warp == 0) tmem_alloc_cta1(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const Schedule sc = schedule_for(TF32);

    if (warp == 4 && lane == 0) {
        // ---------------------------------------------------- TMA producer
        constexpr int kElems = TF32 ? kTcBKBytes / 4 : kTcBKBytes / 2;
        int stage = 0;
        uint32_t phase = 0;
        int t0 = 0;
        bool ok = true;
        for (int b = 0; b < sc.nbands && ok; ++b) {
            for (int kb = 0; kb < p.num_kb && ok; ++kb) {
                for (int t = t0; t < t0 + sc.len(b); ++t) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, p.err, kDevErrTimeout) || *abort_flag) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full0 + 8 * stage;
                    mbar_arrive_expect_tx(fb, kStageBytes);
                    const uint32_t sa = smem_u32(smem + stage * kStageBytes);
                    tma_load_3d(sa, &mapA, fb, kb * kElems, m0, sc.pi(t));
                    tma_load_3d(sa + kStageA, &mapB, fb, kb * kElems, n0, sc.pj(t));
                    if (++stage == S) { stage = 0; phase ^= 1; }
                }
            }
            t0 += sc.len(b);
        }
        if (!ok) {
            *abort_flag = 1;
            // let loads already in flight land before the CTA can exit
            for (int s = 0; s < S; ++s) mbar_wait(full0 + 8 * s, 0, p.err, kDevErrTimeout, 20000000ull);
        }
    } else if (warp == 5 && lane == 0) {
        // ------------------------------------------------------ MMA issuer
        const uint32_t idesc = make_idesc(TF32 ? 2u : 1u, BM, BN);
        int stage = 0;
        uint32_t phase = 0;
        int t0 = 0;
        bool ok = true;
        bool first = true;
        for (int b = 0; b < sc.nbands && ok; ++b) {
            for (int kb = 0; kb < p.num_kb && ok; ++kb) {
                for (int t = t0; t < t0 + sc.len(b); ++t) {
                    if (!mbar_wait(full0 + 8 * stage, phase, p.err, kDevErrTimeout) || *abort_flag) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * kStageBytes);
                    const uint64_t adesc = make_sw128_kmajor_desc(sa);
                    const uint64_t bdesc = make_sw128_kmajor_desc(sa + kStageA);
                    const bool band_start = (kb == 0 && t == t0);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        // advance 32 bytes along K inside the 128-byte swizzled row
                        const uint64_t koff = static_cast<uint64_t>((k * 32) >> 4);
                        if (k == 0 && band_start && sc.scale8 && !first) {
                            mma_cta1_scaled8<TF32>(tmem, adesc + koff, bdesc + koff, idesc);
                        } else {
                            mma_cta1<TF32>(tmem, adesc + koff, bdesc + koff, idesc,
                                           (first && k == 0) ? 0u : 1u);
                        }
                    }
                    first = false;
                    tc_commit_cta1(empty0 + 8 * stage);
                    if (++stage == S) { stage = 0; phase ^= 1; }
                }
            }
            t0 += sc.len(b);
        }
        if (!ok) *abort_flag = 1;
        // accumulator ready (or, after an abort, all issued MMAs finished)
        tc_commit_cta1(accum);
    } else if (warp < 4) {
        // -------------------------------------------------------- epilogue
        const bool ready = mbar_wait(accum, 0, p.err, kDevErrTimeout);
        tc_fence_after();
        if (ready && !*abort_flag) {
            const int row = m0 + warp * 32 + lane;
            const bool row_ok = row < p.M;
            float* crow = p.C + (int64_t)row * p.ldc;
            const bool vec = ((p.ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(p.C) & 15) == 0);
            for (int c = 0; c < BN; c += 32) {
                if (n0 + c >= p.N) break;          // warp-uniform
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c, r);
                tmem_ld_wait();
                if (!row_ok) continue;
                const int col0 = n0 + c;
                if (vec && col0 + 32 <= p.N) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        float4 v;
                        v.x = p.alpha * __uint_as_float(r[4 * q + 0]);
                        v.y = p.alpha * __uint_as_float(r[4 * q + 1]);
                        v.z = p.alpha * __uint_as_float(r[4 * q + 2]);
                        v.w = p.alpha * __uint_as_float(r[4 * q + 3]);
                        float4* dst = reinterpret_cast<float4*>(crow + col0 + 4 * q);
                        if (p.beta != 0.0f) {
                            const float4 o = *dst;
                            v.x = fmaf(p.beta, o.x, v.x);
                            v.y = fmaf(p.beta, o.y, v.y);
                            v.z = fmaf(p.beta, o.z, v.z);
                            v.w = fmaf(p.beta, o.w, v.w);
                        }
                        *dst = v;
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        if (col0 + q < p.N) {
                            float v = p.alpha * __uint_as_float(r[q]);
                            if (p.beta != 0.0f) v = fmaf(p.beta, crow[col0 + q], v);
                            crow[col0 + q] = v;
                        }
                    }
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc_cta1(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_gemm_tc(int tf32, const CUtensorMap& mapA, const CUtensorMap& mapB,
                           const TcGemmParams& p, cudaStream_t stream) {
    const int tiles = p.tiles_m * p.tiles_n;
    if (tiles == 0) return cudaSuccess;
    if (tf32) {
        static bool attr = false;
        if (!attr) {
            cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<1>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 kSmemBytes);
            if (e != cudaSuccess) return e;
            attr = true;
        }
        gemm_tc_kernel<1><<<tiles, kTcThreads, kSmemBytes, stream>>>(mapA, mapB, p);
    } else {
        static bool attr = false;
        if (!attr) {
            cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<0>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 kSmemBytes);
            if (e != cudaSuccess) return e;
            attr = true;
        }
        gemm_tc_kernel<0><<<tiles, kTcThreads, kSmemBytes, stream>>>(mapA, mapB, p);
    }
    return cudaGetLastError();
}

}  // namespace emu
