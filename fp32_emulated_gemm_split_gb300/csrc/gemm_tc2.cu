// gemm_tc2.cu -- the tensor-core GEMM of the two-pass path on CTA pairs.
//
// Same method and band schedule as gemm_tc.cu (bands of the nine BF16
// products b = i + j processed one after the other, 4 down to 0, into one FP32
// accumulator that the first MMA of each later band scales by 2^-8 through
// the scale-input-d operand; TF32x3 runs its residual band, then hi*hi).
// Source: "Unlocking Tensor Core Performance for Machine Learning Interatomic
// Potentials", Figure 1 caption; discuss.pytorch.kr summary, section
// "Blackwell의 BF16x9".
//
// Layout on the GPU:
//   * a cluster of two CTAs (one per SM of an SM pair) owns a 256 x 256 tile
//     of C; each CTA stages 128 rows of the A piece and 128 rows of the B^T
//     piece per K block, and one tcgen05.mma.cta_group::2 (M = 256, N = 256)
//     reads both CTAs' shared memory, so each SM streams half of B instead
//     of all of it;
//   * the kernel is persistent: one cluster per SM pair walks the tiles;
//   * tensor memory holds two 256-column accumulators, so the epilogue of
//     one tile overlaps the main loop of the next.
// Warp roles in each CTA (256 threads):
//   warp 0   TMA producer (both CTAs; completion counted on the leader CTA's
//            barrier through the .cta_group::2 form of the tensor copy)
//   warp 1   MMA issuer (leader CTA only)
//   warp 2   tensor-memory allocation (both CTAs, collectively)
//   warps 4-7  epilogue: TMEM lanes 32(w-4) .. +31 -> C = alpha*acc + beta*C
#include "emu_device.cuh"

namespace emu {
namespace {

constexpr int kPairBM = 256, kPairBN = 256, kHalf = 128;
constexpr int kStageA = kHalf * kTcBKBytes;          // 16 KB
constexpr int kStageB = kHalf * kTcBKBytes;          // 16 KB
constexpr int kStage = kStageA + kStageB;            // 32 KB per CTA
constexpr int kThreads2 = 256;
constexpr uint32_t kAccCols = 256;                   // one accumulator
constexpr uint32_t kTmemCols2 = 512;                 // two accumulators

template <int S>
constexpr int smem_bytes2() { return S * kStage + 1024 + 1024; }

// ------------------------------------------------------------ schedule --

// Pieces (i, j) in processing order, four bits per pair; band lengths four
// bits per band (see gemm_tc.cu for the order and its reason).
struct Sched2 {
    uint64_t pairs;
    uint32_t lens;
    int nbands, scale8;
    __device__ __forceinline__ int pi(int t) const { return int((pairs >> (4 * t + 2)) & 3u); }
    __device__ __forceinline__ int pj(int t) const { return int((pairs >> (4 * t)) & 3u); }
    __device__ __forceinline__ int len(int b) const { return int((lens >> (4 * b)) & 15u); }
};

// (2,2) | (1,2) (2,1) | (0,2) (1,1) (2,0) | (0,1) (1,0) | (0,0)
constexpr uint64_t kPairsBf16 =
    (uint64_t(0xA) << 0) | (uint64_t(0x6) << 4) | (uint64_t(0x9) << 8) | (uint64_t(0x2) << 12) |
    (uint64_t(0x5) << 16) | (uint64_t(0x8) << 20) | (uint64_t(0x1) << 24) | (uint64_t(0x4) << 28) |
    (uint64_t(0x0) << 32);
// (hi,lo) (lo,hi) | (hi,hi)
constexpr uint64_t kPairsTf32 = (uint64_t(0x1) << 0) | (uint64_t(0x4) << 4) | (uint64_t(0x0) << 8);

template <int TF32>
__device__ __forceinline__ Sched2 sched2() {
    Sched2 s;
    if constexpr (TF32) {
        s.pairs = kPairsTf32; s.lens = 2u | (1u << 4); s.nbands = 2; s.scale8 = 0;
    } else {
        s.pairs = kPairsBf16; s.lens = 1u | (2u << 4) | (3u << 8) | (2u << 12) | (1u << 16);
        s.nbands = 5; s.scale8 = 1;
    }
    return s;
}

__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int& tm, int& tn) {
    constexpr int G = 8;                       // tiles of M walked together (L2 reuse of B)
    const int per_group = G * tiles_n;
    const int group = tile / per_group;
    const int first_m = group * G;
    const int gm = min(tiles_m - first_m, G);
    const int r = tile - group * per_group;
    tm = first_m + r % gm;
    tn = r / gm;
}

template <int TF32, int S>
__global__ void __launch_bounds__(kThreads2, 1)
gemm_tc2_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                const TcGemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * kStage);
    // [0,S) full (leader) | [S,2S) empty | 2S,2S+1 tmem full | 2S+2,2S+3 tmem empty (leader)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int cluster_id = blockIdx.x >> 1, num_clusters = gridDim.x >> 1;
    const int total = p.tiles_m * p.tiles_n;

    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S);
    const uint32_t tfull0 = smem_u32(bars + 2 * S), tempty0 = smem_u32(bars + 2 * S + 2);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        mbar_init(tfull0, 1);
        mbar_init(tfull0 + 8, 1);
        mbar_init(tempty0, 8);          // 4 epilogue warps in each of the 2 CTAs
        mbar_init(tempty0 + 8, 8);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&mapA);
        tma_prefetch_desc(&mapB);
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(tmem_slot)), "r"(kTmemCols2) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Sched2 sc = sched2<TF32>();
    constexpr int kElems = TF32 ? kTcBKBytes / 4 : kTcBKBytes / 2;

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------- TMA producer
        const uint32_t full_leader0 = map_to_rank(full0, 0);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int tile = cluster_id; tile < total && ok; tile += num_clusters) {
            int tm, tn;
            tile_coords(tile, p.tiles_m, p.tiles_n, tm, tn);
            const int arow = tm * kPairBM + int(rank) * kHalf;
            const int brow = tn * kPairBN + int(rank) * kHalf;
            int t0 = 0;
            for (int b = 0; b < sc.nbands && ok; ++b) {
                for (int kb = 0; kb < p.num_kb && ok; ++kb) {
                    for (int t = t0; t < t0 + sc.len(b); ++t) {
                        if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, p.err, kDevErrTimeout) ||
                            *abort_flag) {
                            ok = false;
                            break;
                        }
                        if (leader) mbar_arrive_expect_tx(full0 + 8 * stage, 2 * kStage);
                        const uint32_t fb = full_leader0 + 8 * stage;
                        const uint32_t sa = smem_u32(smem + stage * kStage);
                        tma_load_3d_pair(sa, &mapA, fb, kb * kElems, arow, sc.pi(t));
                        tma_load_3d_pair(sa + kStageA, &mapB, fb, kb * kElems, brow, sc.pj(t));
                        if (++stage == S) { stage = 0; phase ^= 1; }
                    }
                }
                t0 += sc.len(b);
            }
        }
        if (!ok) *abort_flag = 1;
    } else if (warp == 1 && lane == 0 && leader) {
        // ------------------------------------------------------ MMA issuer
        const uint32_t idesc = make_idesc(TF32 ? 2u : 1u, kPairBM, kPairBN);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        int i = 0;
        for (int tile = cluster_id; tile < total && ok; tile += num_clusters, ++i) {
            const int buf = i & 1;
            const uint32_t aph = (i >> 1) & 1;
            if (!mbar_wait(tempty0 + 8 * buf, aph ^ 1, p.err, kDevErrTimeout)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d = tmem + buf * kAccCols;
            bool first = true;
            int t0 = 0;
            for (int b = 0; b < sc.nbands && ok; ++b) {
                for (int kb = 0; kb < p.num_kb && ok; ++kb) {
                    for (int t = t0; t < t0 + sc.len(b); ++t) {
                        if (!mbar_wait(full0 + 8 * stage, phase, p.err, kDevErrTimeout) ||
                            *abort_flag) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sa = smem_u32(smem + stage * kStage);
                        const uint64_t adesc = make_sw128_kmajor_desc(sa);
                        const uint64_t bdesc = make_sw128_kmajor_desc(sa + kStageA);
                        const bool band_start = (kb == 0 && t == t0);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint64_t koff = static_cast<uint64_t>((k * 32) >> 4);
                            if (k == 0 && band_start && sc.scale8 && !first)
                                mma_cta2_scaled8<TF32>(d, adesc + koff, bdesc + koff, idesc);
                            else
                                mma_cta2<TF32>(d, adesc + koff, bdesc + koff, idesc,
                                               (first && k == 0) ? 0u : 1u);
                        }
                        first = false;
                        tc_commit_pair(empty0 + 8 * stage);
                        if (++stage == S) { stage = 0; phase ^= 1; }
                    }
                }
                t0 += sc.len(b);
            }
            tc_commit_pair(tfull0 + 8 * buf);
        }
        if (!ok) *abort_flag = 1;
    } else if (warp >= 4) {
        // -------------------------------------------------------- epilogue
        const int q = warp - 4;                 // TMEM lane quadrant of this warp
        const uint32_t tempty_leader0 = map_to_rank(tempty0, 0);
        const bool vec = ((p.ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(p.C) & 15) == 0);
        int i = 0;
        for (int tile = cluster_id; tile < total; tile += num_clusters, ++i) {
            const int buf = i & 1;
            const uint32_t aph = (i >> 1) & 1;
            if (!mbar_wait(tfull0 + 8 * buf, aph, p.err, kDevErrTimeout)) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            int tm, tn;
            tile_coords(tile, p.tiles_m, p.tiles_n, tm, tn);
            const int row = tm * kPairBM + int(rank) * kHalf + q * 32 + lane;
            const int n0 = tn * kPairBN;
            const bool row_ok = row < p.M && !*abort_flag;
            float* crow = p.C + (int64_t)row * p.ldc;
            for (int c = 0; c < kPairBN; c += 32) {
                if (n0 + c >= p.N) break;                       // warp-uniform
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem + buf * kAccCols + c + (static_cast<uint32_t>(q * 32) << 16), r);
                tmem_ld_wait();
                if (!row_ok) continue;
                const int col0 = n0 + c;
                if (vec && col0 + 32 <= p.N) {
#pragma unroll
                    for (int v4 = 0; v4 < 8; ++v4) {
                        float4 v;
                        v.x = p.alpha * __uint_as_float(r[4 * v4 + 0]);
                        v.y = p.alpha * __uint_as_float(r[4 * v4 + 1]);
                        v.z = p.alpha * __uint_as_float(r[4 * v4 + 2]);
                        v.w = p.alpha * __uint_as_float(r[4 * v4 + 3]);
                        float4* dst = reinterpret_cast<float4*>(crow + col0 + 4 * v4);
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
                    for (int v1 = 0; v1 < 32; ++v1) {
                        if (col0 + v1 < p.N) {
                            float v = p.alpha * __uint_as_float(r[v1]);
                            if (p.beta != 0.0f) v = fmaf(p.beta, crow[col0 + v1], v);
                            crow[col0 + v1] = v;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(tempty_leader0 + 8 * buf);
        }
    }

    __syncwarp();
    tc_fence_before();
    cluster_sync();
    if (warp == 2) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;"
                     :: "r"(tmem), "r"(kTmemCols2) : "memory");
    }
}

template <int TF32, int S>
cudaError_t launch2(const CUtensorMap& mapA, const CUtensorMap& mapB, const TcGemmParams& p,
                    int num_clusters, cudaStream_t stream) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(gemm_tc2_kernel<TF32, S>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             smem_bytes2<S>());
        if (e != cudaSuccess) return e;
        attr = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * num_clusters);
    cfg.blockDim = dim3(kThreads2);
    cfg.dynamicSmemBytes = smem_bytes2<S>();
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_tc2_kernel<TF32, S>, mapA, mapB, p);
}

constexpr int kPairStages = 6;

}  // namespace

int tc2_max_clusters(int sms) {
    // one cluster per SM pair; the kernel needs a whole SM (shared memory, TMEM)
    return sms / 2;
}

cudaError_t launch_gemm_tc2(int tf32, const CUtensorMap& mapA, const CUtensorMap& mapB,
                            const TcGemmParams& p, int sms, cudaStream_t stream) {
    const int tiles = p.tiles_m * p.tiles_n;
    if (tiles == 0) return cudaSuccess;
    const int clusters = tiles < tc2_max_clusters(sms) ? tiles : tc2_max_clusters(sms);
    cudaError_t e = tf32 ? launch2<1, kPairStages>(mapA, mapB, p, clusters, stream)
                         : launch2<0, kPairStages>(mapA, mapB, p, clusters, stream);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace emu
