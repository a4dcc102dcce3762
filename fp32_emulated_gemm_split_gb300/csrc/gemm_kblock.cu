// gemm_kblock.cu -- the tensor-core GEMM of the two-pass path: one K block
// at a time, all bands of the block in the tensor core, the blocks summed in
// FP32 registers.
//
// Method ("Unlocking Tensor Core Performance for Machine Learning Interatomic
// Potentials", Figure 1 caption; discuss.pytorch.kr summary, section
// "Blackwell의 BF16x9"): three BF16 pieces per operand, nine products a_i b_j
// in five bands b = i + j of weight 2^-8b, accumulated in FP32 smallest band
// first.  TF32x3 (Figure 2 and its equation): residual band hi*lo + lo*hi,
// then hi*hi, no scaling.
//
// Schedule.  For each 64-element K block (32 for TF32x3) the three A pieces
// and three B pieces are staged once, and the tensor core runs the bands of
// that block smallest first into a fresh TMEM accumulator: band 4 (a2 b2),
// then band 3 with its first MMA issued with scale-input-d = 8
// (D = A*B + 2^-8 D), band 2, band 1, band 0 the same way.  The block's
// partial sum -- sum_b 2^-8b S_b over the block, shifted by the tensor core's
// own scaling -- is then added to FP32 registers with a round-to-nearest add.
// Only the four band-0 MMAs of a block run at full magnitude, so the
// tensor core's truncating accumulation costs a few 2^-24 per block, and the
// register sum over blocks rounds to nearest.  Each staged piece tile feeds 3
// MMA groups on average (6 tile loads per 9 groups), a third of the operand
// traffic of running every band over the whole K.
//
// Layout: a cluster of two CTAs (an SM pair) owns a 256 x 256 tile of C; per
// K block each CTA stages 128 rows of the three A pieces and of the three B^T
// pieces (6 x 16 KB, 128-byte swizzled rows); one tcgen05.mma.cta_group::2
// (M = N = 256) reads both CTAs' shared memory.  Two stages (K blocks) are in
// flight; each stage has one "full" barrier per piece index so the band-4
// MMAs start when pieces 2 land.  Persistent: one cluster per SM pair walks
// the tiles; two TMEM partial buffers let the tensor core fill one block's
// partial while the other is added to the registers.
// Warps (576 threads per CTA):
//   warp 0      TMA producer (both CTAs; completion counted on the leader's
//               barriers) and tensor-memory allocation
//   warp 1      MMA issuer (leader CTA only)
//   warps 2-17  accumulators: warp w owns TMEM lanes 32(w%4)..+31 and the
//               column quarter (w-2)/4 of the tile (64 FP32 registers per
//               thread) and writes C = alpha*acc + beta*C.
#include "emu_device.cuh"

namespace emu {
namespace {

constexpr int kBM = 256, kBN = 256, kHalfRows = 128;
constexpr int kPieceTile = kHalfRows * kTcBKBytes;   // 16 KB: 128 rows x 128 bytes
constexpr int kAccWarps = 16;
constexpr int kAccCols = kBN / 4;                    // 64 columns per accumulator thread
constexpr int kThreadsK = (2 + kAccWarps) * 32;
constexpr uint32_t kBufCols = 256;
constexpr uint32_t kTmemColsK = 512;

template <int TF32>
struct KCfg {
    static constexpr int pieces = TF32 ? 2 : 3;
    static constexpr int stage_bytes = 2 * pieces * kPieceTile;   // A pieces then B pieces
    static constexpr int stages = TF32 ? 3 : 2;
    static constexpr int elems = TF32 ? kTcBKBytes / 4 : kTcBKBytes / 2;
    static constexpr int smem = stages * stage_bytes + 1024 + 1024;
};

__device__ __forceinline__ void tile_pos(int tile, int tiles_m, int tiles_n, int& tm, int& tn) {
    constexpr int G = 8;                  // tiles of M walked together: B tiles stay in L2
    const int per_group = G * tiles_n;
    const int group = tile / per_group;
    const int first_m = group * G;
    const int gm = min(tiles_m - first_m, G);
    const int r = tile - group * per_group;
    tm = first_m + r % gm;
    tn = r / gm;
}

// The MMAs of one piece pair (i, j) for one K block: four K=16 (BF16) or
// K=8 (TF32) steps inside the 128-byte swizzled rows.  `first` marks the
// first MMA of a fresh accumulator; `shift` asks the first step to scale the
// accumulator by 2^-8 (start of a new, larger band).
template <int TF32>
__device__ __forceinline__ void mma_pair(uint32_t d, uint32_t a_tile, uint32_t b_tile,
                                         uint32_t idesc, bool first, bool shift) {
    const uint64_t adesc = make_sw128_kmajor_desc(a_tile);
    const uint64_t bdesc = make_sw128_kmajor_desc(b_tile);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint64_t koff = static_cast<uint64_t>((k * 32) >> 4);
        if (k == 0 && shift)
            mma_cta2_scaled8<TF32>(d, adesc + koff, bdesc + koff, idesc);
        else
            mma_cta2<TF32>(d, adesc + koff, bdesc + koff, idesc, (k == 0 && first) ? 0u : 1u);
    }
}

template <int TF32>
__global__ void __launch_bounds__(kThreadsK, 1)
gemm_kblock_kernel(const __grid_constant__ CUtensorMap mapA,
                   const __grid_constant__ CUtensorMap mapB, const TcGemmParams p) {
    using Cfg = KCfg<TF32>;
    constexpr int S = Cfg::stages, P = Cfg::pieces;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * Cfg::stage_bytes);
    // [0, S*P) piece full (leader), index s*P + piece | [S*P, S*P+S) stage empty |
    // then 2 partial full, 2 partial empty (leader)
    const int nb_full = S * P;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + nb_full + S + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int cluster_id = blockIdx.x >> 1, num_clusters = gridDim.x >> 1;
    const int total = p.tiles_m * p.tiles_n;
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + nb_full);
    const uint32_t cfull0 = smem_u32(bars + nb_full + S);
    const uint32_t cempty0 = smem_u32(bars + nb_full + S + 2);

    if (threadIdx.x == 0) {
        for (int i = 0; i < nb_full; ++i) mbar_init(full0 + 8 * i, 1);
        for (int s = 0; s < S; ++s) mbar_init(empty0 + 8 * s, 1);
        mbar_init(cfull0, 1);
        mbar_init(cfull0 + 8, 1);
        mbar_init(cempty0, 2 * kAccWarps);   // accumulator warps of both CTAs
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
                     :: "r"(smem_u32(tmem_slot)), "r"(kTmemColsK) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------- TMA producer
        const uint32_t full_leader0 = map_to_rank(full0, 0);
        uint32_t kbg = 0;                         // K blocks staged so far (all tiles)
        bool ok = true;
        for (int tile = cluster_id; tile < total && ok; tile += num_clusters) {
            int tm, tn;
            tile_pos(tile, p.tiles_m, p.tiles_n, tm, tn);
            const int arow = tm * kBM + int(rank) * kHalfRows;
            const int brow = tn * kBN + int(rank) * kHalfRows;
            for (int kb = 0; kb < p.num_kb; ++kb, ++kbg) {
                const uint32_t s = kbg % S, ph = (kbg / S) & 1;
                if (!mbar_wait(empty0 + 8 * s, ph ^ 1, p.err, kDevErrTimeout) || *abort_flag) {
                    ok = false;
                    break;
                }
                const uint32_t st = smem_u32(smem + s * Cfg::stage_bytes);
                // largest piece index first: the first band needs it first
                for (int pc = P - 1; pc >= 0; --pc) {
                    const uint32_t fb = full0 + 8 * (s * P + pc);
                    if (leader) mbar_arrive_expect_tx(fb, 4 * kPieceTile);
                    const uint32_t fbl = full_leader0 + 8 * (s * P + pc);
                    tma_load_3d_pair(st + pc * kPieceTile, &mapA, fbl, kb * Cfg::elems, arow, pc);
                    tma_load_3d_pair(st + (P + pc) * kPieceTile, &mapB, fbl, kb * Cfg::elems,
                                     brow, pc);
                }
            }
        }
        if (!ok) *abort_flag = 1;
    } else if (warp == 1 && lane == 0 && leader) {
        // ------------------------------------------------------ MMA issuer
        const uint32_t idesc = make_idesc(TF32 ? 2u : 1u, kBM, kBN);
        uint32_t kbg = 0;
        bool ok = true;
        for (int tile = cluster_id; tile < total && ok; tile += num_clusters) {
            for (int kb = 0; kb < p.num_kb; ++kb, ++kbg) {
                const uint32_t s = kbg % S, ph = (kbg / S) & 1;
                const uint32_t buf = kbg & 1, cph = (kbg >> 1) & 1;
                if (!mbar_wait(cempty0 + 8 * buf, cph ^ 1, p.err, kDevErrTimeout)) {
                    ok = false;
                    break;
                }
                const uint32_t d = tmem + buf * kBufCols;
                const uint32_t st = smem_u32(smem + s * Cfg::stage_bytes);
                auto A = [&](int i) { return st + i * kPieceTile; };
                auto B = [&](int j) { return st + (P + j) * kPieceTile; };
                auto ready = [&](int pc) {
                    const bool r = mbar_wait(full0 + 8 * (s * P + pc), ph, p.err, kDevErrTimeout) &&
                                   !*abort_flag;
                    tc_fence_after();
                    return r;
                };
                if constexpr (!TF32) {
                    if (!ready(2)) { ok = false; break; }
                    mma_pair<0>(d, A(2), B(2), idesc, true, false);           // band 4
                    if (!ready(1)) { ok = false; break; }
                    mma_pair<0>(d, A(1), B(2), idesc, false, true);           // band 3
                    mma_pair<0>(d, A(2), B(1), idesc, false, false);
                    if (!ready(0)) { ok = false; break; }
                    mma_pair<0>(d, A(0), B(2), idesc, false, true);           // band 2
                    mma_pair<0>(d, A(1), B(1), idesc, false, false);
                    mma_pair<0>(d, A(2), B(0), idesc, false, false);
                    mma_pair<0>(d, A(0), B(1), idesc, false, true);           // band 1
                    mma_pair<0>(d, A(1), B(0), idesc, false, false);
                    mma_pair<0>(d, A(0), B(0), idesc, false, true);           // band 0
                } else {
                    if (!ready(1) || !ready(0)) { ok = false; break; }
                    mma_pair<1>(d, A(0), B(1), idesc, true, false);           // hi*lo
                    mma_pair<1>(d, A(1), B(0), idesc, false, false);          // lo*hi
                    mma_pair<1>(d, A(0), B(0), idesc, false, false);          // hi*hi
                }
                tc_commit_pair(empty0 + 8 * s);
                tc_commit_pair(cfull0 + 8 * buf);
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
        uint32_t kbg = 0;
        bool ok = true;
        for (int tile = cluster_id; tile < total && ok; tile += num_clusters) {
            float acc[kAccCols];
#pragma unroll
            for (int j = 0; j < kAccCols; ++j) acc[j] = 0.0f;
            for (int kb = 0; kb < p.num_kb; ++kb, ++kbg) {
                const uint32_t buf = kbg & 1, cph = (kbg >> 1) & 1;
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
                    for (int j = 0; j < 8; ++j) acc[8 * g + j] += __uint_as_float(r[j]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(cempty_leader0 + 8 * buf);
            }
            if (!ok || *abort_flag) break;
            // ---- epilogue: C = alpha * acc + beta * C
            int tm, tn;
            tile_pos(tile, p.tiles_m, p.tiles_n, tm, tn);
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
                     :: "r"(tmem), "r"(kTmemColsK) : "memory");
    }
}

template <int TF32>
cudaError_t launch_kblock_t(const CUtensorMap& mapA, const CUtensorMap& mapB,
                            const TcGemmParams& p, int clusters, cudaStream_t stream) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(gemm_kblock_kernel<TF32>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             KCfg<TF32>::smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(kThreadsK);
    cfg.dynamicSmemBytes = KCfg<TF32>::smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_kblock_kernel<TF32>, mapA, mapB, p);
}

}  // namespace

cudaError_t launch_gemm_kblock(int tf32, const CUtensorMap& mapA, const CUtensorMap& mapB,
                               const TcGemmParams& p, int sms, cudaStream_t stream) {
    const int tiles = p.tiles_m * p.tiles_n;
    if (tiles == 0) return cudaSuccess;
    const int clusters = tiles < sms / 2 ? tiles : sms / 2;
    cudaError_t e = tf32 ? launch_kblock_t<1>(mapA, mapB, p, clusters, stream)
                         : launch_kblock_t<0>(mapA, mapB, p, clusters, stream);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace emu
