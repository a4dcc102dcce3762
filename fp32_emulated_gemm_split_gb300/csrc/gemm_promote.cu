// gemm_promote.cu -- the tensor-core GEMM of the two-pass path with FP32
// accumulation of the bands on the CUDA cores.
//
// Method ("Unlocking Tensor Core Performance for Machine Learning Interatomic
// Potentials", Figure 1 caption; discuss.pytorch.kr summary, section
// "Blackwell의 BF16x9"): the nine products a_i b_j of the three BF16 pieces
// fall into five bands b = i + j of weight 2^-8b, and the bands are added to
// an FP32 accumulator smallest band first.  TF32x3 (Figure 2 and its
// equation): the residual band hi*lo + lo*hi first, then hi*hi.
//
// Why the accumulation leaves the tensor core: an MMA adds its products to
// the TMEM accumulator with a truncating alignment, so a long chain of MMAs
// into one accumulator loses about half an ulp per MMA, always toward zero;
// over K = 8192 (512 BF16 MMAs) that bias reaches ~1e-5 relative, worse than
// plain FP32.  Here the tensor core only sums short chunks (kChunk stages =
// 16 MMAs) into a TMEM buffer; eight "accumulator" warps read each finished
// chunk (tcgen05.ld) and add it, times its band weight (exact), to FP32
// registers with round-to-nearest adds, band 4 first, band 0 last.  Two TMEM
// chunk buffers let the tensor core fill one while the other is drained.
//
// Layout: a cluster of two CTAs (an SM pair) owns a 256 x 256 tile of C; each
// CTA stages 128 rows of the A piece and 128 rows of the B^T piece per K
// block and one tcgen05.mma.cta_group::2 (M = N = 256) reads both CTAs'
// shared memory.  Persistent: one cluster per SM pair walks the tiles.
// Warps (576 threads per CTA):
//   warp 0      TMA producer (both CTAs; completion counted on the leader's
//               barrier) and tensor-memory allocation
//   warp 1      MMA issuer (leader CTA only)
//   warps 2-17  accumulators: warp w owns TMEM lanes 32(w%4)..+31 and the
//               column quarter (w-2)/4 of the tile: 64 FP32 registers per
//               thread; they also write C = alpha*acc + beta*C.
// (Each SM sub-partition has its own 16K-register file, so per-thread
// registers are capped by the warps that share a sub-partition; 64 columns
// per thread keeps the accumulators in registers without spilling.)
#include "emu_device.cuh"

namespace emu {
namespace {

constexpr int kBM = 256, kBN = 256, kHalfRows = 128;
constexpr int kStA = kHalfRows * kTcBKBytes;         // 16 KB
constexpr int kStB = kHalfRows * kTcBKBytes;         // 16 KB
constexpr int kSt = kStA + kStB;                     // 32 KB per CTA per stage
constexpr int kStages = 6;
constexpr int kChunk = 4;                            // stages per TMEM chunk (16 MMAs)
constexpr int kAccWarps = 16;                        // 4 lane quadrants x 4 column quarters
constexpr int kAccCols = kBN / 4;                    // 64 columns per accumulator thread
constexpr int kThreadsP = (2 + kAccWarps) * 32;
constexpr uint32_t kBufCols = 256;
constexpr uint32_t kTmemColsP = 512;
constexpr int kSmemP = kStages * kSt + 1024 + 1024;

// Pieces (i, j) in processing order, four bits each (i << 2 | j); band
// lengths four bits each.  BF16x9: (2,2) | (1,2) (2,1) | (0,2) (1,1) (2,0) |
// (0,1) (1,0) | (0,0).  TF32x3 (0 = hi, 1 = lo): (hi,lo) (lo,hi) | (hi,hi).
constexpr uint64_t kOrderBf16 = 0xA | (0x6ull << 4) | (0x9ull << 8) | (0x2ull << 12) |
                                (0x5ull << 16) | (0x8ull << 20) | (0x1ull << 24) | (0x4ull << 28);
constexpr uint32_t kLensBf16 = 1u | (2u << 4) | (3u << 8) | (2u << 12) | (1u << 16);
constexpr uint64_t kOrderTf32 = 0x1 | (0x4ull << 4);
constexpr uint32_t kLensTf32 = 2u | (1u << 4);

template <int TF32>
struct Order {
    static constexpr uint64_t pairs = TF32 ? kOrderTf32 : kOrderBf16;
    static constexpr uint32_t lens = TF32 ? kLensTf32 : kLensBf16;
    static constexpr int nbands = TF32 ? 2 : 5;
    __device__ __forceinline__ static int pi(int t) { return int((pairs >> (4 * t + 2)) & 3u); }
    __device__ __forceinline__ static int pj(int t) { return int((pairs >> (4 * t)) & 3u); }
    __device__ __forceinline__ static int len(int b) { return int((lens >> (4 * b)) & 15u); }
    // weight of the b-th band processed: 2^-8(4-b) for BF16x9, 1 for TF32x3
    __device__ __forceinline__ static float weight(int b) {
        return TF32 ? 1.0f : __uint_as_float(uint32_t(127 - 8 * (4 - b)) << 23);
    }
};

__device__ __forceinline__ void tile_of(int tile, int tiles_m, int tiles_n, int& tm, int& tn) {
    constexpr int G = 8;                  // tiles of M walked together: B tiles stay in L2
    const int per_group = G * tiles_n;
    const int group = tile / per_group;
    const int first_m = group * G;
    const int gm = min(tiles_m - first_m, G);
    const int r = tile - group * per_group;
    tm = first_m + r % gm;
    tn = r / gm;
}

template <int TF32>
__global__ void __launch_bounds__(kThreadsP, 1)
gemm_promote_kernel(const __grid_constant__ CUtensorMap mapA,
                    const __grid_constant__ CUtensorMap mapB, const TcGemmParams p) {
    using O = Order<TF32>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kSt);
    // [0,S) stage full (leader) | [S,2S) stage empty | 2S..2S+1 chunk full |
    // 2S+2..2S+3 chunk empty (leader)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int cluster_id = blockIdx.x >> 1, num_clusters = gridDim.x >> 1;
    const int total = p.tiles_m * p.tiles_n;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kStages);
    const uint32_t cfull0 = smem_u32(bars + 2 * kStages), cempty0 = smem_u32(bars + 2 * kStages + 2);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        mbar_init(cfull0, 1);
        mbar_init(cfull0 + 8, 1);
        mbar_init(cempty0, 2 * kAccWarps);   // accumulator warps of both CTAs of the pair
        mbar_init(cempty0 + 8, 2 * kAccWarps);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&mapA);
            tma_prefetch_desc(&mapB);
        }
        __syncwarp();
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(tmem_slot)), "r"(kTmemColsP) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    constexpr int kElems = TF32 ? kTcBKBytes / 4 : kTcBKBytes / 2;

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------- TMA producer
        const uint32_t full_leader0 = map_to_rank(full0, 0);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int tile = cluster_id; tile < total && ok; tile += num_clusters) {
            int tm, tn;
            tile_of(tile, p.tiles_m, p.tiles_n, tm, tn);
            const int arow = tm * kBM + int(rank) * kHalfRows;
            const int brow = tn * kBN + int(rank) * kHalfRows;
            int t0 = 0;
            for (int b = 0; b < O::nbands && ok; ++b) {
                const int L = O::len(b);
                for (int kb = 0; kb < p.num_kb && ok; ++kb) {
                    for (int t = t0; t < t0 + L; ++t) {
                        if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, p.err, kDevErrTimeout) ||
                            *abort_flag) {
                            ok = false;
                            break;
                        }
                        if (leader) mbar_arrive_expect_tx(full0 + 8 * stage, 2 * kSt);
                        const uint32_t fb = full_leader0 + 8 * stage;
                        const uint32_t sa = smem_u32(smem + stage * kSt);
                        tma_load_3d_pair(sa, &mapA, fb, kb * kElems, arow, O::pi(t));
                        tma_load_3d_pair(sa + kStA, &mapB, fb, kb * kElems, brow, O::pj(t));
                        if (++stage == kStages) { stage = 0; phase ^= 1; }
                    }
                }
                t0 += L;
            }
        }
        if (!ok) *abort_flag = 1;
    } else if (warp == 1 && lane == 0 && leader) {
        // ------------------------------------------------------ MMA issuer
        const uint32_t idesc = make_idesc(TF32 ? 2u : 1u, kBM, kBN);
        int stage = 0;
        uint32_t phase = 0;
        uint32_t chunk = 0;                      // chunks issued so far (all tiles)
        bool ok = true;
        for (int tile = cluster_id; tile < total && ok; tile += num_clusters) {
            int t0 = 0;
            for (int b = 0; b < O::nbands && ok; ++b) {
                const int L = O::len(b);
                const int nst = L * p.num_kb;    // stages of this band, kb-major
                for (int s0 = 0; s0 < nst && ok; s0 += kChunk, ++chunk) {
                    const uint32_t buf = chunk & 1, cph = (chunk >> 1) & 1;
                    if (!mbar_wait(cempty0 + 8 * buf, cph ^ 1, p.err, kDevErrTimeout)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + buf * kBufCols;
                    const int s1 = min(s0 + kChunk, nst);
                    for (int st = s0; st < s1; ++st) {
                        if (!mbar_wait(full0 + 8 * stage, phase, p.err, kDevErrTimeout) ||
                            *abort_flag) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sa = smem_u32(smem + stage * kSt);
                        const uint64_t adesc = make_sw128_kmajor_desc(sa);
                        const uint64_t bdesc = make_sw128_kmajor_desc(sa + kStA);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint64_t koff = static_cast<uint64_t>((k * 32) >> 4);
                            mma_cta2<TF32>(d, adesc + koff, bdesc + koff, idesc,
                                           (st == s0 && k == 0) ? 0u : 1u);
                        }
                        tc_commit_pair(empty0 + 8 * stage);
                        if (++stage == kStages) { stage = 0; phase ^= 1; }
                    }
                    tc_commit_pair(cfull0 + 8 * buf);
                }
                t0 += L;
            }
        }
        if (!ok) *abort_flag = 1;
    } else if (warp >= 2) {
        // ------------------------------------------------ accumulator warps
        const int q = warp & 3;                        // TMEM lane quadrant
        const int h = (warp - 2) >> 2;                 // column quarter of the tile
        const uint32_t cempty_leader0 = map_to_rank(cempty0, 0);
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const bool vec = ((p.ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(p.C) & 15) == 0);
        uint32_t chunk = 0;
        bool ok = true;
        for (int tile = cluster_id; tile < total && ok; tile += num_clusters) {
            float acc[kAccCols];
#pragma unroll
            for (int j = 0; j < kAccCols; ++j) acc[j] = 0.0f;
            for (int b = 0; b < O::nbands && ok; ++b) {
                const float w = O::weight(b);
                const int nst = O::len(b) * p.num_kb;
                for (int s0 = 0; s0 < nst; s0 += kChunk, ++chunk) {
                    const uint32_t buf = chunk & 1, cph = (chunk >> 1) & 1;
                    if (!mbar_wait(cfull0 + 8 * buf, cph, p.err, kDevErrTimeout)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t col0 = tmem + buf * kBufCols + h * kAccCols + lane_off;
#pragma unroll
                    for (int g = 0; g < kAccCols / 8; ++g) {
                        uint32_t r[8];
                        tmem_ld_32x32b_x8(col0 + 8 * g, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            acc[8 * g + j] = fmaf(w, __uint_as_float(r[j]), acc[8 * g + j]);
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_remote(cempty_leader0 + 8 * buf);
                }
            }
            if (!ok || *abort_flag) break;
            // ---- epilogue: C = alpha * acc + beta * C
            int tm, tn;
            tile_of(tile, p.tiles_m, p.tiles_n, tm, tn);
            const int row = tm * kBM + int(rank) * kHalfRows + q * 32 + lane;
            const int col_base = tn * kBN + h * kAccCols;
            if (row < p.M && col_base < p.N) {
                float* crow = p.C + (int64_t)row * p.ldc + col_base;
                if (vec && col_base + kAccCols <= p.N) {
#pragma unroll
                    for (int v4 = 0; v4 < kAccCols / 4; ++v4) {
                        float4 v;
                        v.x = p.alpha * acc[4 * v4 + 0];
                        v.y = p.alpha * acc[4 * v4 + 1];
                        v.z = p.alpha * acc[4 * v4 + 2];
                        v.w = p.alpha * acc[4 * v4 + 3];
                        float4* dst = reinterpret_cast<float4*>(crow + 4 * v4);
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
                    for (int j = 0; j < kAccCols; ++j) {
                        if (col_base + j < p.N) {
                            float v = p.alpha * acc[j];
                            if (p.beta != 0.0f) v = fmaf(p.beta, crow[j], v);
                            crow[j] = v;
                        }
                    }
                }
            }
        }
        if (!ok) *abort_flag = 1;
    }

    __syncwarp();
    tc_fence_before();
    cluster_sync();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;"
                     :: "r"(tmem), "r"(kTmemColsP) : "memory");
    }
}

template <int TF32>
cudaError_t launch_promote(const CUtensorMap& mapA, const CUtensorMap& mapB, const TcGemmParams& p,
                           int clusters, cudaStream_t stream) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(gemm_promote_kernel<TF32>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemP);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(kThreadsP);
    cfg.dynamicSmemBytes = kSmemP;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_promote_kernel<TF32>, mapA, mapB, p);
}

}  // namespace

cudaError_t launch_gemm_promote(int tf32, const CUtensorMap& mapA, const CUtensorMap& mapB,
                                const TcGemmParams& p, int sms, cudaStream_t stream) {
    const int tiles = p.tiles_m * p.tiles_n;
    if (tiles == 0) return cudaSuccess;
    const int clusters = tiles < sms / 2 ? tiles : sms / 2;
    cudaError_t e = tf32 ? launch_promote<1>(mapA, mapB, p, clusters, stream)
                         : launch_promote<0>(mapA, mapB, p, clusters, stream);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace emu
