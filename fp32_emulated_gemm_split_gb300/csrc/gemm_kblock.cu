// gemm_kblock.cu -- the tensor-core GEMM: one K block at a time, all bands of
// the block in the tensor core, the blocks summed in FP32 registers.  Used by
// the two-pass path (pieces of A and B read from the workspace) and by the
// fused path (A read as FP32 and split on chip into tensor memory; B's
// pieces from the workspace).
//
// Method ("Unlocking Tensor Core Performance for Machine Learning Interatomic
// Potentials", Figure 1 caption; discuss.pytorch.kr summary, section
// "Blackwell의 BF16x9"): three BF16 pieces per operand, nine products a_i b_j
// in five bands b = i + j of weight 2^-8b, accumulated in FP32 smallest band
// first.  TF32x3 (Figure 2 and its equation): residual band hi*lo + lo*hi,
// then hi*hi, no scaling.  The two cheaper rungs the pages compare against
// run on the same pipeline: two BF16 pieces (band 1 = a0 b1 + a1 b0, then
// band 0 = a0 b0 after a 2^-8 shift; the discuss.pytorch.kr page's "FP32 as
// the sum of two BF16") and single-pass TF32 (one product, the blog post's
// one-pass TF32 of Figures 5-8).  The Ootomo-Yokota variant of TF32x3
// (linked from the discuss.pytorch.kr page's TF32x3 section: scaling, and
// accumulation outside the tensor core) stores the residual times 2^11 and
// runs the residual band, then hi*hi with scale-input-d = 11.
//
// Schedule.  For each 64-element K block (32 for TF32x3) the pieces of A and
// B are staged once, and the tensor core runs the bands of that block
// smallest first into a fresh TMEM accumulator: band 4 (a2 b2), then band 3
// with its first MMA issued with scale-input-d = 8 (D = A*B + 2^-8 D), band
// 2, band 1, band 0 the same way.  The block's partial -- sum_b 2^-8b S_b over
// the block, shifted by the tensor core's own scaling -- is then added to
// FP32 registers with a round-to-nearest add.  Only the four band-0 MMAs of a
// block run at full magnitude, so the tensor core's truncating accumulation
// costs a few 2^-24 per block, and the sum over blocks rounds to nearest.
// Each staged piece tile feeds three MMA groups on average.
//
// Layout: a cluster of two CTAs (an SM pair) owns a 256 x BN tile of C
// (BN = 256 or 128); per K block each CTA stages 128 rows of each A piece and
// BN/2 rows of each B^T piece (128-byte swizzled rows); one
// tcgen05.mma.cta_group::2 (M = 256, N = BN) reads both CTAs' shared memory.
// Two-pass BF16 pieces may instead be M- or N-major (K rows of M or N
// elements, from a row-wise split of A stored K x M or B stored K x N): the
// CTA's 128 rows or BN/2 columns then arrive as 64-element chunks of 64 K
// rows, 8 KB apart, and the MMA reads them through an MN-major descriptor and
// the transpose bit of its instruction descriptor (TcGemmParams::a_mn, b_mn).
// Each stage has one "full" barrier per piece index so the band-4 MMAs start
// when pieces 2 land.  Persistent: one cluster per SM pair walks the tiles;
// tensor memory holds 512/BN partial buffers, so the tensor core fills the
// next partials (of this tile or the next) while earlier ones are added to
// the registers and the epilogue stores C.  The last, partial round of tiles
// runs stream-K (schedule.h): its K blocks are shared evenly by all
// clusters in consecutive ranges; a range that starts inside a tile leaves
// that part's FP32 sums and a flag in global memory, and the part holding the
// tile's first K block adds them in K order and writes C.
//
// Fused A in shared memory (BF16x9, FUSED = 3, BN = 256 or 128): the
// two-pass layout, but the producer loads only B's pieces; eight split warps
// read each K block of FP32 A from global memory (prefetched into L2 two
// blocks ahead, across tile boundaries, and loaded before the stage-free
// wait), split it and store the
// three pieces into the stage's A half in the same 128-byte swizzled layout
// the TMA would have written, fence, meet at a named barrier, and one
// thread signals the leader CTA, whose MMA waits for both CTAs' halves.
//
// Fused A in tensor memory (BF16x9, FUSED = 1, BN = 128): the producer
// loads the FP32 A block (128 rows x 64, two 128-byte-swizzled boxes) into
// one of two staging buffers; sixteen split warps turn it (16 elements per
// thread) into the three BF16 pieces and store them into tensor memory
// (tcgen05.st; two 96-column A stages beside two 128-column accumulator
// buffers), fence, meet at a named barrier, and one thread signals the
// leader CTA; the MMA reads A from tensor memory and only B's pieces from
// shared memory.
//
// Warps (576 threads per CTA; 832 on either fused path):
//   warp 0      TMA producer (both CTAs; completion counted on the leader's
//               barriers) and tensor-memory allocation
//   warp 1      MMA issuer (leader CTA only)
//   warps 2..   accumulators (16, or 8 in tensor-memory fused): warp w owns
//               TMEM lanes 32(w%4)..+31 and column group (w-2)/4 of the tile
//               (BN/4, or BN/2 in tensor-memory fused, FP32 registers per
//               thread) and writes C = alpha*acc + beta*C
//   then        split warps: 8 (shared-memory fused) or 16 (tensor-memory
//               fused).
#include <mutex>

#include "emu_device.cuh"
#include "schedule.h"

namespace emu {
namespace {

constexpr int kBM = 256, kHalfRows = 128;
constexpr int kATile = kHalfRows * kTcBKBytes;       // 16 KB: 128 rows x 128 bytes
// FUSED selects how A's pieces reach the tensor core: 0 (two-pass) TMA
// loads from the workspace the split kernel wrote; 1 (tensor-memory fused)
// split warps store them into tensor memory; 3 (shared-memory fused) split
// warps store them into the A half of each shared-memory stage, where the
// two-pass path's TMA would have put them.
// Warp roles: warp 0 is the TMA producer (and allocates tensor memory),
// warp 1 the MMA issuer, then come the accumulator warps -- 16 (a column
// quarter each), or 8 (a column half each) on the tensor-memory path, which
// also runs 16 split warps and must stay within 1024 threads -- and the split
// warps: 8 of 16 rows each on the shared-memory path (their loads in flight
// must cover the latency of reading A: fewer warps starve them).
template <int FUSED>
struct Roles {
    static constexpr int acc = FUSED == 1 ? 8 : 16;
    static constexpr int split = FUSED == 1 ? 16 : FUSED == 3 ? 8 : 0;
    static constexpr int producer = 0, mma = 1, acc0 = 2, split0 = 2 + acc;
    static constexpr int warps = 2 + acc + split;
};
template <int FUSED>
constexpr int acc_warps() { return Roles<FUSED>::acc; }
constexpr int kSplitWarps = 16;                       // tensor-memory path
constexpr int kSmemSplitWarps = 8;                    // shared-memory path
constexpr int kSmemSplitRows = 128 / kSmemSplitWarps;
template <int FUSED>
constexpr int threads_k() { return Roles<FUSED>::warps * 32; }
constexpr int kSmemMax = 232448;                      // dynamic shared memory per CTA
constexpr int kA32Box = 128 * 128;                    // FP32 box: 128 rows x 32 floats
constexpr int kA32Buf = 2 * kA32Box;                  // one 64-wide K block of FP32 A
constexpr int kA32Bufs = 2;

template <int MODE, int BN, int FUSED>
struct KCfg {
    static constexpr bool TM = FUSED == 1, SMS = FUSED == 3;
    static constexpr bool tf32 = mode_is_tf32(MODE);
    static constexpr int pieces = mode_pieces(MODE);
    static constexpr int b_rows = BN / 2;                        // B^T rows per CTA
    static constexpr int b_tile = b_rows * kTcBKBytes;
    // fused: only B's pieces are staged in shared memory; A's go to tensor
    // memory (a_tm_stages rings of 96 columns after the accumulators)
    static constexpr int stage_bytes = pieces * ((TM ? 0 : kATile) + b_tile);
    static constexpr int a32_bytes = TM ? kA32Bufs * kA32Buf : 0;
    // epilogue staging for bulk tensor stores: 32 rows x 16 FP32 per
    // accumulator warp (2 KB)
    // (two per warp on the fused path, which has the shared memory to spare:
    // one is filled while the other's store is still reading it)
    static constexpr int c_bufs = TM ? 2 : 1;
    static constexpr int c_bytes = ::emu::acc_warps<FUSED>() * 2048 * c_bufs;
    static constexpr int avail = kSmemMax - 2048 - a32_bytes - c_bytes;
    static constexpr int max_stages = pieces == 1 ? 6 : 4;
    static constexpr int stages = avail / stage_bytes > max_stages ? max_stages : avail / stage_bytes;
    static constexpr int elems = tf32 ? kTcBKBytes / 4 : kTcBKBytes / 2;
    // K blocks summed in one TMEM partial before it is added to the registers.
    // TF32x3 has no band shift, so two short blocks (12 MMAs each) share a
    // partial, and single-pass TF32 eight blocks (32 MMAs; its 2^-11 piece
    // error dwarfs the tensor core's truncation).  A BF16x9 partial holds one
    // block, because the 2^-8 shift at a band change would also shift a
    // previous block's finished sum.  The two-band modes (BF16x3 and the
    // Ootomo-Yokota TF32x3) run two blocks band-major instead: band 1 of
    // both, then band 0 of both, the shift at the first band-0 MMA, so both
    // stages stay held until band 0 (band_major below).
    static constexpr bool band_major = MODE == kModeBf16x3 || MODE == kModeTf32x3Oy;
    static constexpr int band_shift = MODE == kModeTf32x3Oy ? 11 : 8;
    static constexpr int kb_per_partial =
        MODE == kModeTf32x3 || band_major ? 2 : MODE == kModeTf32 ? 8 : 1;
    // TMEM partial buffers of BN columns each (all 512 columns): 2 at BN = 256,
    // 4 at BN = 128, so the tensor core can run further ahead of the epilogue.
    static constexpr int nbuf = TM ? 2 : 512 / BN;
    static constexpr int a_tm_stages = TM ? 2 : 0;
    static constexpr int a_tm_ring = a_tm_stages > 0 ? a_tm_stages : 1;   // modulus (no zero)
    static constexpr int a_tm_cols = 3 * (kTcBKBytes / 4);            // 3 pieces x 32 columns
    static constexpr int a_tm_base = nbuf * BN;
    static_assert(a_tm_base + a_tm_stages * a_tm_cols <= 512, "tensor memory overflow");
    static constexpr int acc_warps = ::emu::acc_warps<FUSED>();
    static constexpr int acc_cols = BN / (acc_warps / 4);         // columns per accumulator thread
    static constexpr uint32_t tmem_cols = 512;
    static constexpr int smem = stages * stage_bytes + a32_bytes + c_bytes + 2048;
    // bytes a piece barrier waits for (both CTAs)
    static constexpr uint32_t piece_tx = TM || SMS ? 2 * b_tile : 2 * (kATile + b_tile);
    static_assert(stages >= 2, "shared memory too small for two stages");
    static_assert(!(FUSED == 1 && MODE != kModeBf16x9) &&
                      !(FUSED == 3 && MODE != kModeBf16x9 && MODE != kModeTf32x3),
                  "the fused paths split BF16x9 pieces (and, in shared memory, TF32x3 ones)");
    // 128-byte lines in one row of one K block of FP32 A (64 BF16-mode
    // elements: 2; 32 TF32-mode elements: 1)
    static constexpr int a32_lines = elems * 4 / 128;
};

__device__ __forceinline__ void st_release_gpu(unsigned* a, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_acq_rel_gpu() {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* a) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}

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

// An M- or N-major piece tile in shared memory: chunks of 64 elements of M
// or N by one K block (64 rows of 128 bytes), this far apart.
constexpr uint32_t kMnBox = 64 * kTcBKBytes;          // 8 KB

// The MMAs of one piece pair (i, j) for one K block: four K=16 (BF16) or
// K=8 (TF32) steps.  A K-major tile advances 32 bytes along its swizzled
// rows per step; an M- or N-major one (bit 0 of `mn` for A, bit 1 for B;
// BF16 only) 16 K rows, 2048 bytes.  `first` marks the first MMA of a fresh
// accumulator; `shift` asks the first step to scale the accumulator by
// 2^-SHIFT (start of a new, larger band).
template <int TF32, int SHIFT = 8>
__device__ __forceinline__ void mma_pair(uint32_t d, uint32_t a_tile, uint32_t b_tile,
                                         uint32_t idesc, bool first, bool shift, int mn = 0) {
    const uint64_t adesc = (mn & 1) ? make_sw128_mn_desc(a_tile, kMnBox) : make_sw128_kmajor_desc(a_tile);
    const uint64_t bdesc = (mn & 2) ? make_sw128_mn_desc(b_tile, kMnBox) : make_sw128_kmajor_desc(b_tile);
    const uint64_t astep = (mn & 1) ? (2048 >> 4) : (32 >> 4);
    const uint64_t bstep = (mn & 2) ? (2048 >> 4) : (32 >> 4);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint64_t ak = adesc + k * astep, bk = bdesc + k * bstep;
        if (k == 0 && shift)
            mma_cta2_scaled<TF32, SHIFT>(d, ak, bk, idesc);
        else
            mma_cta2<TF32>(d, ak, bk, idesc, (k == 0 && first) ? 0u : 1u);
    }
}

// The same with A in tensor memory (fused path): `a_tm` is the first column
// of the piece's 64-element K block (32 columns, K=16 step = 8 columns).
__device__ __forceinline__ void mma_pair_ta(uint32_t d, uint32_t a_tm, uint32_t b_tile,
                                            uint32_t idesc, bool first, bool shift) {
    const uint64_t bdesc = make_sw128_kmajor_desc(b_tile);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint64_t koff = static_cast<uint64_t>((k * 32) >> 4);
        if (k == 0 && shift)
            mma_cta2_ta_scaled<8>(d, a_tm + 8 * k, bdesc + koff, idesc);
        else
            mma_cta2_ta(d, a_tm + 8 * k, bdesc + koff, idesc, (k == 0 && first) ? 0u : 1u);
    }
}

// Split this thread's share of a 128 x 64 FP32 A block (two swizzled 128 x
// 32 boxes at `a32`) into the three BF16 pieces and store them to tensor
// memory at column `col` (piece i at col + 32 i; BF16 pairs, two elements
// per 32-bit column, rows = lanes).  A warp reaches only its own 32 lanes
// (warp % 4), so row r = 32 (warp % 4) + lane, and the four split warps of a
// lane quadrant take elements 16 kpart .. +15.  The 32 lanes read the same
// logical 16-byte chunk of 32 consecutive rows, which the 128-byte swizzle
// spreads over 8 distinct bank groups per 8 rows: conflict-free.
__device__ __forceinline__ void split_block_tm(const uint8_t* a32, uint32_t col, int r, int kpart) {
    const uint8_t* row = a32 + (kpart >> 1) * kA32Box + r * 128;
    uint32_t w0[8], w1[8], w2[8];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int c4 = (kpart & 1) * 4 + c;
        const float4 x = *reinterpret_cast<const float4*>(row + ((c4 ^ (r & 7)) << 4));
        split_bf16x3_pair(x.x, x.y, w0[2 * c], w1[2 * c], w2[2 * c]);
        split_bf16x3_pair(x.z, x.w, w0[2 * c + 1], w1[2 * c + 1], w2[2 * c + 1]);
    }
    tmem_st_32x32b_x8(col, w0);
    tmem_st_32x32b_x8(col + 32, w1);
    tmem_st_32x32b_x8(col + 64, w2);
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint4& v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                 :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// Named barrier `id` over `nthreads` threads that also ANDs a predicate: every
// participating warp reaches it once per use, whatever its predicate, so a
// warp whose wait gave up still meets the others and all leave together.
__device__ __forceinline__ bool bar_and(int id, int nthreads, bool v) {
    uint32_t r;
    asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n"
                 " bar.red.and.pred p, %2, %3, q;\n selp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(r) : "r"(uint32_t(v)), "r"(id), "r"(nthreads) : "memory");
    return r != 0;
}
constexpr int kSplitBarrier = 1;                      // named barrier of the split warps

template <int MODE, int BN, int FUSED>
__global__ void __launch_bounds__(threads_k<FUSED>(), 1)
gemm_kblock_kernel(const __grid_constant__ CUtensorMap mapA,
                   const __grid_constant__ CUtensorMap mapB,
                   const __grid_constant__ CUtensorMap mapC, const TcGemmParams p) {
    using Cfg = KCfg<MODE, BN, FUSED>;
    using R = Roles<FUSED>;
    constexpr int S = Cfg::stages, P = Cfg::pieces, kAccCols = Cfg::acc_cols;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* a32 = smem + S * Cfg::stage_bytes;           // FP32 A staging (fused only)
    uint8_t* cstage = a32 + Cfg::a32_bytes;               // epilogue staging for C
    uint64_t* bars = reinterpret_cast<uint64_t*>(cstage + Cfg::c_bytes);
    // [0, S*P) piece full (leader), index s*P + piece | S stage empty |
    // 2 partial full | 2 partial empty (leader) | fused: S A-pieces ready
    // (leader), 2 FP32 full, 2 FP32 free
    const int nb_full = S * P;
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = full0 + 8 * nb_full;
    constexpr int NB = Cfg::nbuf;
    const uint32_t cfull0 = empty0 + 8 * S;
    const uint32_t cempty0 = cfull0 + 8 * NB;
    const uint32_t aready0 = cempty0 + 8 * NB;
    const uint32_t afull0 = aready0 + 8 * S;
    const uint32_t afree0 = afull0 + 8 * kA32Bufs;
    // fused: 2 tensor-memory A stages free (each CTA, arrived by the MMA commit)
    const uint32_t atfree0 = afree0 + 8 * kA32Bufs;
    uint32_t* tmem_slot =
        reinterpret_cast<uint32_t*>(bars + nb_full + 2 * S + 2 * NB + 2 * kA32Bufs + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int cluster_id = blockIdx.x >> 1, num_clusters = gridDim.x >> 1;
    const TileSchedule sch = {p.tiles_m * p.tiles_n, p.num_kb, p.tail_tiles, p.tail_clusters,
                              num_clusters};
    const int nunits = sched_units(sch, cluster_id);

    if constexpr (Cfg::SMS) {
        // split warps: start the first two K blocks of their rows of A on
        // their way to L2 while the prologue runs (a hint; see griddep_wait
        // below for the reads)
        if (warp >= R::split0 && warp < R::split0 + R::split && nunits > 0) {
            const Unit u0 = sched_unit(sch, cluster_id, 0);
            int tm0, tn0;
            tile_pos(u0.tile, p.tiles_m, p.tiles_n, tm0, tn0);
            const int row0 = tm0 * kBM + int(rank) * kHalfRows +
                             kSmemSplitRows * (warp - R::split0);
            constexpr int L = Cfg::a32_lines;
            for (int d = 0; d < 2 && u0.kb0 + d < u0.kb1; ++d) {
                for (int t = lane; t < L * kSmemSplitRows; t += 32) {
                    const int prow = row0 + t / L;
                    const int pk = (u0.kb0 + d) * Cfg::elems + 32 * (t % L);
                    if (prow < p.M && pk < p.K)
                        asm volatile("prefetch.global.L2 [%0];"
                                     :: "l"(p.A32 + (int64_t)prow * p.lda + pk));
                }
            }
        }
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < nb_full; ++i) mbar_init(full0 + 8 * i, 1);
        for (int s = 0; s < S; ++s) mbar_init(empty0 + 8 * s, 1);
        for (int b = 0; b < NB; ++b) {
            mbar_init(cfull0 + 8 * b, 1);
            mbar_init(cempty0 + 8 * b, 2 * Cfg::acc_warps);   // accumulator warps of both CTAs
        }
        if (Cfg::SMS) {
            // A half of stage s written (leader; one arrive per CTA)
            for (int s = 0; s < S; ++s) mbar_init(aready0 + 8 * s, 2);
        }
        if (Cfg::TM) {
            // A pieces of tensor-memory stage t written (leader; one per CTA)
            for (int t = 0; t < Cfg::a_tm_stages; ++t) mbar_init(aready0 + 8 * t, 2);
            for (int t = 0; t < Cfg::a_tm_stages; ++t) mbar_init(atfree0 + 8 * t, 1);
            for (int f = 0; f < kA32Bufs; ++f) {
                mbar_init(afull0 + 8 * f, 1);
                mbar_init(afree0 + 8 * f, 1);
            }
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == R::producer) {
        if (lane == 0) {
            tma_prefetch_desc(&mapA);
            tma_prefetch_desc(&mapB);
        }
        __syncwarp();
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(tmem_slot)), "r"(Cfg::tmem_cols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // operand layouts of the pieces (bit 0: A M-major, bit 1: B N-major):
    // two-pass BF16 modes only
    const int mn = (Cfg::TM || Cfg::SMS || Cfg::tf32) ? 0 : ((p.a_mn ? 1 : 0) | (p.b_mn ? 2 : 0));
    // A kernel launched behind this one as a programmatic dependent (the next
    // GEMM of a run of calls on already-split weights) may start now on SMs
    // this grid leaves free: every one of its reads and writes of global
    // memory waits for this grid's completion (griddep_wait), and its CTAs
    // cannot share an SM with this grid's (each takes most of the shared
    // memory), so the overlap covers only its launch and prologue.
    griddep_launch_dependents();
    if (warp == R::producer) {
        if (lane == 0) {
            // ---------------------------------------------------- TMA producer
            griddep_wait();                           // the split ahead has written the pieces
            const uint32_t full_leader0 = map_to_rank(full0, 0);
            uint32_t kbg = 0;                         // K blocks staged so far (all units)
            bool ok = true;
            for (int i = 0; i < nunits && ok; ++i) {
                const Unit w = sched_unit(sch, cluster_id, i);
                int tm, tn;
                tile_pos(w.tile, p.tiles_m, p.tiles_n, tm, tn);
                const int arow = tm * kBM + int(rank) * kHalfRows;
                const int brow = tn * BN + int(rank) * Cfg::b_rows;
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++kbg) {
                    const uint32_t s = kbg % S, ph = (kbg / S) & 1;
                    if (Cfg::TM) {
                        const uint32_t f = kbg % kA32Bufs, fph = (kbg / kA32Bufs) & 1;
                        if (!mbar_wait(afree0 + 8 * f, fph ^ 1, p.err, kDevErrTimeout) || *abort_flag) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(afull0 + 8 * f, kA32Buf);
                        const uint32_t dst = smem_u32(a32 + f * kA32Buf);
                        // FP32 A map is (K, M, 1): the two 32-wide boxes of this K block
                        tma_load_3d(dst, &mapA, afull0 + 8 * f, kb * 64, arow, 0);
                        tma_load_3d(dst + kA32Box, &mapA, afull0 + 8 * f, kb * 64 + 32, arow, 0);
                    }
                    if (!mbar_wait(empty0 + 8 * s, ph ^ 1, p.err, kDevErrTimeout) || *abort_flag) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = smem_u32(smem + s * Cfg::stage_bytes);
                    // largest piece index first: the first band needs it first
                    for (int pc = P - 1; pc >= 0; --pc) {
                        if (leader) mbar_arrive_expect_tx(full0 + 8 * (s * P + pc), Cfg::piece_tx);
                        const uint32_t fbl = full_leader0 + 8 * (s * P + pc);
                        // K-major maps are (K, rows, piece); M- or N-major
                        // ones (K rows of M or N elements: two-pass BF16
                        // only) are (element, K, 64-element chunk, piece),
                        // the CTA's chunks one box, kMnBox apart
                        if (!Cfg::TM && !Cfg::SMS) {
                            const uint32_t adst = st + pc * kATile;
                            if (mn & 1)
                                tma_load_4d_pair(adst, &mapA, fbl, 0, kb * Cfg::elems, arow / 64, pc);
                            else
                                tma_load_3d_pair(adst, &mapA, fbl, kb * Cfg::elems, arow, pc);
                        }
                        const uint32_t bdst = st + P * (Cfg::TM ? 0 : kATile) + pc * Cfg::b_tile;
                        if (mn & 2)
                            tma_load_4d_pair(bdst, &mapB, fbl, 0, kb * Cfg::elems, brow / 64, pc);
                        else
                            tma_load_3d_pair(bdst, &mapB, fbl, kb * Cfg::elems, brow, pc);
                    }
                }
            }
            if (!ok) *abort_flag = 1;
        }
    } else if (warp == R::mma) {
        if (lane == 0 && leader) {
            // ------------------------------------------------------ MMA issuer
            const uint32_t idesc = make_idesc(Cfg::tf32 ? 2u : 1u, kBM, BN) |
                                   ((mn & 1) ? kIdescAMn : 0u) | ((mn & 2) ? kIdescBMn : 0u);
            constexpr int KBP = Cfg::kb_per_partial;
            uint32_t kbg = 0, part = 0;              // K blocks and TMEM partials so far
            uint32_t prev_s = 0;                     // band-major: stage of the pair's first block
            bool ok = true;
            for (int i = 0; i < nunits && ok; ++i) {
                const Unit w = sched_unit(sch, cluster_id, i);
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++kbg) {
                    const uint32_t s = kbg % S, ph = (kbg / S) & 1;
                    const uint32_t buf = part % NB, cph = (part / NB) & 1;
                    const bool fresh = ((kb - w.kb0) % KBP) == 0;   // first block of a partial
                    const bool close = ((kb - w.kb0) % KBP) == KBP - 1 || kb == w.kb1 - 1;
                    if (fresh && !mbar_wait(cempty0 + 8 * buf, cph ^ 1, p.err, kDevErrTimeout)) {
                        ok = false;
                        break;
                    }
                    // fused: A's pieces of this block in tensor-memory stage t
                    const uint32_t t = Cfg::TM ? kbg % Cfg::a_tm_ring : 0;
                    const uint32_t tph = Cfg::TM ? (kbg / Cfg::a_tm_ring) & 1 : 0;
                    if (Cfg::TM) {
                        if (!mbar_wait(aready0 + 8 * t, tph, p.err, kDevErrTimeout)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    if (Cfg::SMS) {
                        // both CTAs' split warps have written A's pieces into stage s
                        if (!mbar_wait(aready0 + 8 * s, ph, p.err, kDevErrTimeout)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    const uint32_t d = tmem + buf * BN;
                    const uint32_t st = smem_u32(smem + s * Cfg::stage_bytes);
                    constexpr int a_smem = Cfg::TM ? 0 : kATile;
                    auto A = [&](int i) { return st + i * a_smem; };
                    auto B = [&](int j) { return st + P * a_smem + j * Cfg::b_tile; };
                    const uint32_t a_tm0 = tmem + Cfg::a_tm_base + t * Cfg::a_tm_cols;
                    auto ready = [&](int pc) {
                        const bool r = mbar_wait(full0 + 8 * (s * P + pc), ph, p.err, kDevErrTimeout) &&
                                       !*abort_flag;
                        tc_fence_after();
                        return r;
                    };
                    if constexpr (Cfg::TM) {
                        // A pieces from tensor memory, 32 columns apart
                        auto pr = [&](int i, int j, bool first, bool shift) {
                            mma_pair_ta(d, a_tm0 + 32 * i, B(j), idesc, first, shift);
                        };
                        if (!ready(2)) { ok = false; break; }
                        pr(2, 2, true, false);                                    // band 4
                        if (!ready(1)) { ok = false; break; }
                        pr(1, 2, false, true);                                    // band 3
                        pr(2, 1, false, false);
                        if (!ready(0)) { ok = false; break; }
                        pr(0, 2, false, true);                                    // band 2
                        pr(1, 1, false, false);
                        pr(2, 0, false, false);
                        pr(0, 1, false, true);                                    // band 1
                        pr(1, 0, false, false);
                        pr(0, 0, false, true);                                    // band 0
                    } else if constexpr (MODE == kModeBf16x9) {
                        if (!ready(2)) { ok = false; break; }
                        mma_pair<0>(d, A(2), B(2), idesc, true, false, mn);       // band 4
                        if (!ready(1)) { ok = false; break; }
                        mma_pair<0>(d, A(1), B(2), idesc, false, true, mn);       // band 3
                        mma_pair<0>(d, A(2), B(1), idesc, false, false, mn);
                        if (!ready(0)) { ok = false; break; }
                        mma_pair<0>(d, A(0), B(2), idesc, false, true, mn);       // band 2
                        mma_pair<0>(d, A(1), B(1), idesc, false, false, mn);
                        mma_pair<0>(d, A(2), B(0), idesc, false, false, mn);
                        mma_pair<0>(d, A(0), B(1), idesc, false, true, mn);       // band 1
                        mma_pair<0>(d, A(1), B(0), idesc, false, false, mn);
                        mma_pair<0>(d, A(0), B(0), idesc, false, true, mn);       // band 0
                    } else if constexpr (MODE == kModeTf32x3) {
                        if (!ready(1) || !ready(0)) { ok = false; break; }
                        mma_pair<1>(d, A(0), B(1), idesc, fresh, false);          // hi*lo
                        mma_pair<1>(d, A(1), B(0), idesc, false, false);          // lo*hi
                        mma_pair<1>(d, A(0), B(0), idesc, false, false);          // hi*hi
                    } else if constexpr (Cfg::band_major) {
                        // BF16x3: band 1 = a0 b1 + a1 b0, band 0 = a0 b0, shift 2^-8.
                        // Ootomo-Yokota: hi lo' + lo' hi, then hi hi, shift 2^-11.
                        constexpr int T = Cfg::tf32 ? 1 : 0, SH = Cfg::band_shift;
                        if (!ready(1) || !ready(0)) { ok = false; break; }
                        mma_pair<T>(d, A(0), B(1), idesc, fresh, false, mn);      // band 1
                        mma_pair<T>(d, A(1), B(0), idesc, false, false, mn);
                        if (!close) {
                            prev_s = s;                  // band 0 after the next block's band 1
                            continue;                    // stage held: no empty commit yet
                        }
                        if (!fresh) {
                            // band 0 of the pair's first block (shift), free its stage
                            const uint32_t pst = smem_u32(smem + prev_s * Cfg::stage_bytes);
                            mma_pair<T, SH>(d, pst, pst + P * kATile, idesc, false, true, mn);
                            tc_commit_pair(empty0 + 8 * prev_s);
                            mma_pair<T>(d, A(0), B(0), idesc, false, false, mn);
                        } else {
                            mma_pair<T, SH>(d, A(0), B(0), idesc, false, true, mn);
                        }
                    } else {
                        if (!ready(0)) { ok = false; break; }
                        mma_pair<1>(d, A(0), B(0), idesc, fresh, false);          // hi*hi
                    }
                    tc_commit_pair(empty0 + 8 * s);
                    if (Cfg::TM) tc_commit_pair(atfree0 + 8 * t);    // tensor-memory A stage free
                    if (close) {
                        tc_commit_pair(cfull0 + 8 * buf);
                        ++part;
                    }
                }
            }
            if (!ok) *abort_flag = 1;
        }
    } else if (Cfg::SMS && warp >= R::split0 && warp < R::split0 + R::split) {
        // ------------------------------------- split warps (shared memory)
        // For every K block of this cluster's units, in the producer's order:
        // prefetch this warp's rows of the block two ahead into L2 (across
        // tile boundaries); load this block's rows, then, once the MMA has
        // consumed the block that last used stage s, split this CTA's 128
        // rows of FP32 A (warp w: rows 16 w .. +15, four rows per step, eight
        // lanes per row, each lane one 16-byte chunk of the 128-byte rows of
        // the pieces: 8 elements for BF16x9, whose K block is 64 wide, 4 for
        // TF32x3, whose block is 32 wide) and store the pieces into the
        // stage's A half in the 128-byte swizzled K-major layout the MMA
        // reads (chunk j of row r at chunk j ^ (r % 8): the eight lanes of a
        // row hit eight bank groups; zeros past M and K); fence for the
        // tensor core, meet the other split warps, and one thread counts this
        // CTA in on the leader's barrier.
        constexpr bool TF = Cfg::tf32;
        constexpr int EL = TF ? 4 : 8;            // FP32 elements per lane and row
        constexpr int L = Cfg::a32_lines;
        const int sw = warp - R::split0;
        const int rsub = lane >> 3, chunk = lane & 7;
        const uint32_t aready_leader0 = map_to_rank(aready0, 0);
        constexpr int RW = kSmemSplitRows, IT = RW / 4;   // rows per warp, 4-row steps
        // L2 prefetch of this warp's rows of one block (L 128-byte lines per
        // row); a hint only, so it may run ahead of the grid dependency below
        auto prefetch_block = [&](int arow_, int kb_) {
#pragma unroll
            for (int t = lane; t < L * RW; t += 32) {
                const int prow = arow_ + RW * sw + t / L;
                const int pk = kb_ * Cfg::elems + 32 * (t % L);
                if (prow < p.M && pk < p.K)
                    asm volatile("prefetch.global.L2 [%0];"
                                 :: "l"(p.A32 + (int64_t)prow * p.lda + pk));
            }
        };
        auto unit_arow = [&](const Unit& u) {
            int tm_, tn_;
            tile_pos(u.tile, p.tiles_m, p.tiles_n, tm_, tn_);
            return tm_ * kBM + int(rank) * kHalfRows;
        };
        constexpr int kAhead = 2;                 // blocks prefetched ahead
        Unit wnext = {};
        int arow_next = 0;
        if (nunits > 0) {                         // (its first blocks: prefetched at entry)
            wnext = sched_unit(sch, cluster_id, 0);
            arow_next = unit_arow(wnext);
        }
        // A may be the output of the kernel ahead in the stream (a
        // programmatic dependent launch starts before it ends)
        griddep_wait();
        uint32_t g = 0;
        bool ok = true;
        for (int i = 0; i < nunits && ok; ++i) {
            const Unit w = wnext;
            const int arow = arow_next;
            if (i + 1 < nunits) {
                wnext = sched_unit(sch, cluster_id, i + 1);
                arow_next = unit_arow(wnext);
            }
            for (int kb = w.kb0; kb < w.kb1; ++kb, ++g) {
                const uint32_t s = g % S, ph = (g / S) & 1;
                // the block kAhead ahead in this cluster's sequence, which
                // may lie in the next unit (the next tile's rows)
                if (kb + kAhead < w.kb1)
                    prefetch_block(arow, kb + kAhead);
                else if (i + 1 < nunits && wnext.kb0 + (kb + kAhead - w.kb1) < wnext.kb1)
                    prefetch_block(arow_next, wnext.kb0 + (kb + kAhead - w.kb1));
                // this block's FP32 rows first: their latency overlaps the wait
                const int k = kb * Cfg::elems + chunk * EL;
                float4 x[IT][EL / 4];
#pragma unroll
                for (int it = 0; it < IT; ++it) {
                    const int row = arow + RW * sw + 4 * it + rsub;
#pragma unroll
                    for (int v = 0; v < EL / 4; ++v) x[it][v] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (row < p.M && k < p.K) {
                        const float* src = p.A32 + (int64_t)row * p.lda + k;
                        if (k + EL - 1 < p.K) {
#pragma unroll
                            for (int v = 0; v < EL / 4; ++v)
                                x[it][v] = __ldg(reinterpret_cast<const float4*>(src + 4 * v));
                        } else {
                            float t[EL];
#pragma unroll
                            for (int j = 0; j < EL; ++j) t[j] = 0.f;
                            for (int j = 0; j < EL && k + j < p.K; ++j) t[j] = src[j];
#pragma unroll
                            for (int v = 0; v < EL / 4; ++v)
                                x[it][v] = make_float4(t[4 * v], t[4 * v + 1], t[4 * v + 2],
                                                       t[4 * v + 3]);
                        }
                    }
                }
                const bool good = mbar_wait(empty0 + 8 * s, ph ^ 1, p.err, kDevErrTimeout) &&
                                  !*abort_flag;
                if (good) {
                    const uint32_t st = smem_u32(smem + s * Cfg::stage_bytes);
#pragma unroll
                    for (int it = 0; it < IT; ++it) {
                        const int r = RW * sw + 4 * it + rsub;
                        const uint32_t off = r * 128 + ((chunk ^ (r & 7)) << 4);
                        if constexpr (TF) {
                            // TF32x3: hi and lo, FP32 containers (no scaling)
                            float4 hi, lo;
                            split_tf32x2(x[it][0].x, hi.x, lo.x);
                            split_tf32x2(x[it][0].y, hi.y, lo.y);
                            split_tf32x2(x[it][0].z, hi.z, lo.z);
                            split_tf32x2(x[it][0].w, hi.w, lo.w);
                            st_shared_v4(st + off, make_uint4(__float_as_uint(hi.x),
                                                              __float_as_uint(hi.y),
                                                              __float_as_uint(hi.z),
                                                              __float_as_uint(hi.w)));
                            st_shared_v4(st + kATile + off,
                                         make_uint4(__float_as_uint(lo.x), __float_as_uint(lo.y),
                                                    __float_as_uint(lo.z), __float_as_uint(lo.w)));
                        } else {
                            uint4 q0, q1, q2;
                            split_bf16x3_pair(x[it][0].x, x[it][0].y, q0.x, q1.x, q2.x);
                            split_bf16x3_pair(x[it][0].z, x[it][0].w, q0.y, q1.y, q2.y);
                            split_bf16x3_pair(x[it][EL / 8].x, x[it][EL / 8].y, q0.z, q1.z, q2.z);
                            split_bf16x3_pair(x[it][EL / 8].z, x[it][EL / 8].w, q0.w, q1.w, q2.w);
                            st_shared_v4(st + off, q0);
                            st_shared_v4(st + kATile + off, q1);
                            st_shared_v4(st + 2 * kATile + off, q2);
                        }
                    }
                    fence_proxy_async_smem();        // generic writes -> the tensor core
                }
                if (!bar_and(kSplitBarrier, kSmemSplitWarps * 32, good)) {
                    ok = false;
                    break;
                }
                if (sw == 0 && lane == 0) mbar_arrive_remote(aready_leader0 + 8 * s);
            }
        }
    } else if (Cfg::TM && warp >= R::split0 && warp < R::split0 + R::split) {
        // ------------------------------------------------------ split warps
        // Split every K block of this cluster's tiles, as soon as its FP32
        // block has landed and its tensor-memory A stage is free, ahead of
        // the tensor core.
        const int w = warp - R::split0;
        const int kpart = w >> 2;                      // 16-element part of the 64
        const int r = 32 * (warp & 3) + lane;          // row: this warp's TMEM lanes
        const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        const uint32_t aready_leader0 = map_to_rank(aready0, 0);
        uint32_t my_blocks = 0;
        for (int i = 0; i < nunits; ++i) {
            const Unit w = sched_unit(sch, cluster_id, i);
            my_blocks += uint32_t(w.kb1 - w.kb0);
        }
        for (uint32_t g = 0; g < my_blocks; ++g) {
            const uint32_t f = g % kA32Bufs, fph = (g / kA32Bufs) & 1;
            const uint32_t t = g % Cfg::a_tm_ring, tph = (g / Cfg::a_tm_ring) & 1;
            const bool ok = mbar_wait(afull0 + 8 * f, fph, p.err, kDevErrTimeout) &&
                            mbar_wait(atfree0 + 8 * t, tph ^ 1, p.err, kDevErrTimeout) &&
                            !*abort_flag;
            if (ok) {
                tc_fence_after();
                split_block_tm(a32 + f * kA32Buf,
                               (tmem + Cfg::a_tm_base + t * Cfg::a_tm_cols + 8 * kpart) | lane_off,
                               r, kpart);
                tmem_st_wait();
                tc_fence_before();           // tensor-memory stores -> the MMA
            }
            // all 16 split warps done with this block; one thread signals, so
            // one cluster-scope release per block instead of sixteen
            if (!bar_and(kSplitBarrier, kSplitWarps * 32, ok)) {
                *abort_flag = 1;
                break;
            }
            if (w == 0 && lane == 0) {
                mbar_arrive(afree0 + 8 * f);
                mbar_arrive_remote(aready_leader0 + 8 * t);
            }
        }
    } else if (warp >= R::acc0 && warp < R::acc0 + R::acc) {
        // ------------------------------------------------ accumulator warps
        const int q = warp & 3;                        // TMEM lane quadrant
        const int h = (warp - R::acc0) >> 2;           // column group of the tile
        const uint32_t cempty_leader0 = map_to_rank(cempty0, 0);
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const bool vec = ((p.ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(p.C) & 15) == 0);
        bool ok = true;
        constexpr int KBP = Cfg::kb_per_partial;
        uint32_t part = 0;
        for (int i = 0; i < nunits && ok; ++i) {
            const Unit w = sched_unit(sch, cluster_id, i);
            const int nparts = (w.kb1 - w.kb0 + KBP - 1) / KBP;   // TMEM partials of this unit
            const int tile = w.tile;
            if (p.beta != 0.0f && w.publish < 0) {
                // the epilogue will read this thread's row of C: start it on
                // its way to L2 now, while the tensor core works
                int tm_, tn_;
                tile_pos(tile, p.tiles_m, p.tiles_n, tm_, tn_);
                const int prow = tm_ * kBM + int(rank) * kHalfRows + q * 32 + lane;
                const int pcol = tn_ * BN + h * kAccCols;
                if (prow < p.M) {
#pragma unroll
                    for (int c = 0; c < kAccCols; c += 32)
                        if (pcol + c < p.N)
                            asm volatile("prefetch.global.L2 [%0];"
                                         :: "l"(p.C + (int64_t)prow * p.ldc + pcol + c));
                }
            }
            float acc[kAccCols];
#pragma unroll
            for (int j = 0; j < kAccCols; ++j) acc[j] = 0.0f;
            for (int pi = 0; pi < nparts; ++pi, ++part) {
                const uint32_t buf = part % NB, cph = (part / NB) & 1;
                if (!mbar_wait(cfull0 + 8 * buf, cph, p.err, kDevErrTimeout)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t col0 = tmem + buf * BN + h * kAccCols + lane_off;
                if constexpr (FUSED == 0) {
                    // 16 columns per load and wait (the fused kernels, at 72
                    // registers a thread, load 8)
#pragma unroll
                    for (int g = 0; g < kAccCols / 16; ++g) {
                        uint32_t r[16];
                        tmem_ld_32x32b_x16(col0 + 16 * g, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j) acc[16 * g + j] += __uint_as_float(r[j]);
                    }
                } else {
#pragma unroll
                    for (int g = 0; g < kAccCols / 8; ++g) {
                        uint32_t r[8];
                        tmem_ld_32x32b_x8(col0 + 8 * g, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc[8 * g + j] += __uint_as_float(r[j]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(cempty_leader0 + 8 * buf);
            }
            if (!ok || *abort_flag) break;
            // stream-K tail: one FP32 slot per (cluster, CTA rank, accumulator
            // warp); this thread's sums as 16-byte groups, lane-contiguous per
            // group, so that a warp writes and reads 512 contiguous bytes at a
            // time
            const int aw = warp - R::acc0;
            auto slot = [&](int c) { return (c * 2 + int(rank)) * Cfg::acc_warps + aw; };
            if (w.publish >= 0) {
                // a later part of a split tile: leave the sums for the owner
                float4* dst = reinterpret_cast<float4*>(p.part_ws) +
                              (size_t)slot(w.publish) * (kAccCols / 4 * 32) + lane;
#pragma unroll
                for (int j = 0; j < kAccCols / 4; ++j)
                    __stcg(dst + j * 32, make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2],
                                                     acc[4 * j + 3]));
                fence_acq_rel_gpu();                   // each lane's stores before the flag
                __syncwarp();
                if (lane == 0) st_release_gpu(p.flags + slot(w.publish), p.epoch);
                continue;                              // the owner writes C
            }
            // owner of a split tile: add the later parts' sums in K order
            // (bounded waits; those clusters publish before they wait on anything)
            for (int o = 1; o <= w.others && ok; ++o) {
                const unsigned* f = p.flags + slot(cluster_id + o);
                const uint64_t t0 = global_timer_ns();
                while (ld_acquire_gpu(f) != p.epoch) {
                    __nanosleep(64);
                    if (global_timer_ns() - t0 > EMU_WAIT_LIMIT_NS) {
                        record_error(p.err, kDevErrTimeout);
                        ok = false;
                        break;
                    }
                }
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                const float4* src = reinterpret_cast<const float4*>(p.part_ws) +
                                    (size_t)slot(cluster_id + o) * (kAccCols / 4 * 32) + lane;
                constexpr int kBatch = kAccCols / 4 < 8 ? kAccCols / 4 : 8;   // loads in flight
#pragma unroll
                for (int j0 = 0; j0 < kAccCols / 4; j0 += kBatch) {
                    float4 v[kBatch];
#pragma unroll
                    for (int b = 0; b < kBatch; ++b) v[b] = __ldcg(src + (j0 + b) * 32);
#pragma unroll
                    for (int b = 0; b < kBatch; ++b) {
                        acc[4 * (j0 + b)] += v[b].x;
                        acc[4 * (j0 + b) + 1] += v[b].y;
                        acc[4 * (j0 + b) + 2] += v[b].z;
                        acc[4 * (j0 + b) + 3] += v[b].w;
                    }
                }
                // consumed: clear the flag, so that a replay of the same
                // launch (a CUDA graph bakes the epoch in) waits afresh
                __syncwarp();
                if (lane == 0) *const_cast<volatile unsigned*>(f) = 0u;
            }
            if (!ok) { *abort_flag = 1; break; }
            // ---- epilogue: C = alpha * acc + beta * C
            int tm, tn;
            tile_pos(tile, p.tiles_m, p.tiles_n, tm, tn);
            const int row0 = tm * kBM + int(rank) * kHalfRows + q * 32;
            const int row = row0 + lane;
            const int col_base = tn * BN + h * kAccCols;
            if (p.tma_store) {
                // Stage 32 rows x 16 columns at a time in this warp's 2 KB
                // buffer (64-byte swizzle: conflict-free writes) and let one
                // bulk tensor store write them, coalesced and clipped at the
                // edge of the C map, which ends at column N & ~3 (a bulk store
                // clips in whole 16-byte units); each lane stores its row's
                // last N % 4 columns itself.  With beta != 0 each lane first
                // reads its own row's 16 values of C (16-byte loads where
                // they fit).
                constexpr int CB = Cfg::c_bufs;
                const int n4 = p.N & ~3;                    // the C map's width
                const uint32_t cst0 = smem_u32(cstage + (warp - R::acc0) * 2048 * CB);
                // The cluster's last unit: all its MMAs have completed (this
                // warp has drained the last partial), so no stage is read or
                // written any more and each warp stages all its chunks in
                // stage memory at once -- no wait for a buffer to be read out.
                constexpr int kChunks = kAccCols / 16;
                static_assert(Cfg::acc_warps * kChunks * 2048 <= S * Cfg::stage_bytes,
                              "stage memory holds the last unit's C");
                const bool last = i == nunits - 1;
                const uint32_t lst0 = smem_u32(smem) + (warp - R::acc0) * kChunks * 2048;
                // alpha * acc (+ beta * C) of 16 columns into a 2 KB staging
                // buffer: lane = row, 64-byte swizzle
                auto stage_chunk = [&](int ch, uint32_t cst) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int j = 16 * ch + 4 * c;
                        float4 v = make_float4(p.alpha * acc[j], p.alpha * acc[j + 1],
                                               p.alpha * acc[j + 2], p.alpha * acc[j + 3]);
                        const int gc = col_base + j;
                        if (p.beta != 0.0f && row < p.M && gc < p.N) {
                            const float* src = p.C + (int64_t)row * p.ldc + gc;
                            if (gc + 3 < p.N) {
                                const float4 o = *reinterpret_cast<const float4*>(src);
                                v.x = fmaf(p.beta, o.x, v.x);
                                v.y = fmaf(p.beta, o.y, v.y);
                                v.z = fmaf(p.beta, o.z, v.z);
                                v.w = fmaf(p.beta, o.w, v.w);
                            } else {
                                v.x = fmaf(p.beta, src[0], v.x);
                                if (gc + 1 < p.N) v.y = fmaf(p.beta, src[1], v.y);
                                if (gc + 2 < p.N) v.z = fmaf(p.beta, src[2], v.z);
                            }
                        }
                        const uint32_t a = cst + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4);
                        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};"
                                     :: "r"(a), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                                     : "memory");
                        // gc is a multiple of 4: a group at or past N & ~3
                        // holds the (at most 3) columns the map leaves out
                        if (gc >= n4 && gc < p.N && row < p.M) {
                            float* dst = p.C + (int64_t)row * p.ldc + gc;
                            dst[0] = v.x;
                            if (gc + 1 < p.N) dst[1] = v.y;
                            if (gc + 2 < p.N) dst[2] = v.z;
                        }
                    }
                };
                if (row0 < p.M && last) {
                    // every chunk staged, one proxy fence, then all the stores
                    int nch = 0;
#pragma unroll
                    for (int ch = 0; ch < kChunks; ++ch) {
                        if (col_base + 16 * ch >= p.N) break;          // warp-uniform
                        stage_chunk(ch, lst0 + ch * 2048);
                        ++nch;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        for (int ch = 0; ch < nch; ++ch)
                            if (col_base + 16 * ch < n4)
                                tma_store_2d(&mapC, col_base + 16 * ch, row0, lst0 + ch * 2048);
                        bulk_commit();
                    }
                } else if (row0 < p.M) {
#pragma unroll
                    for (int ch = 0; ch < kChunks; ++ch) {
                        if (col_base + 16 * ch >= p.N) break;          // warp-uniform
                        const uint32_t cst = cst0 + (ch % CB) * 2048;
                        if (lane == 0) bulk_wait_read_n<CB - 1>();      // this buffer free again
                        __syncwarp();
                        stage_chunk(ch, cst);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            if (col_base + 16 * ch < n4) tma_store_2d(&mapC, col_base + 16 * ch, row0, cst);
                            bulk_commit();
                        }
                    }
                }
            } else if (row < p.M && col_base < p.N) {
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
        if (p.tma_store && lane == 0) bulk_wait_all();        // C written before exit
    }

    __syncwarp();
    tc_fence_before();
    cluster_sync();
    if (warp == R::producer) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;"
                     :: "r"(tmem), "r"(Cfg::tmem_cols) : "memory");
    }
}

// Host-side state of one kernel variant, per device: whether its dynamic
// shared-memory limit has been raised there, and how many of its clusters
// can be resident.  emu_sgemm and emu_sgemm_noalloc take different locks, so
// this state has a lock of its own: their first calls may come from two
// host threads at once.
constexpr int kMaxDevices = 64;
struct VariantState {
    std::mutex mu;
    bool attr[kMaxDevices] = {};
    int clusters[kMaxDevices] = {};
};

template <int MODE, int BN, int FUSED>
VariantState& variant_state() {
    static VariantState st;
    return st;
}

int current_device_index() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

template <int MODE, int BN, int FUSED>
cudaError_t set_smem_attr_locked(VariantState& st, int dev) {
    using Cfg = KCfg<MODE, BN, FUSED>;
    if (dev >= 0 && st.attr[dev]) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(gemm_kblock_kernel<MODE, BN, FUSED>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::smem);
    if (e == cudaSuccess && dev >= 0) st.attr[dev] = true;
    return e;
}

template <int MODE, int BN, int FUSED>
cudaError_t set_smem_attr() {
    VariantState& st = variant_state<MODE, BN, FUSED>();
    std::lock_guard<std::mutex> lock(st.mu);
    return set_smem_attr_locked<MODE, BN, FUSED>(st, current_device_index());
}

// Clusters of this kernel that can be resident at once (at most sms / 2).
// The persistent grid never exceeds it, so every cluster runs concurrently:
// the owner of a stream-K tail tile waits for the clusters that hold the
// tile's later K ranges, which must not be queued behind it.
template <int MODE, int BN, int FUSED>
int max_clusters_t(int sms) {
    using Cfg = KCfg<MODE, BN, FUSED>;
    VariantState& st = variant_state<MODE, BN, FUSED>();
    std::lock_guard<std::mutex> lock(st.mu);
    const int dev = current_device_index();
    int n = dev >= 0 ? st.clusters[dev] : 0;
    if (n <= 0) {
        n = sms / 2;
        if (set_smem_attr_locked<MODE, BN, FUSED>(st, dev) == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2 * (sms / 2));
            cfg.blockDim = dim3(threads_k<FUSED>());
            cfg.dynamicSmemBytes = Cfg::smem;
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = 2;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            int m = 0;
            if (cudaOccupancyMaxActiveClusters(&m, gemm_kblock_kernel<MODE, BN, FUSED>, &cfg) ==
                    cudaSuccess && m > 0)
                n = m;
            else
                cudaGetLastError();
        }
        if (dev >= 0) st.clusters[dev] = n;
    }
    return n < sms / 2 ? n : sms / 2;
}

template <int MODE, int BN, int FUSED>
cudaError_t launch_kblock_t(const CUtensorMap& mapA, const CUtensorMap& mapB,
                            const CUtensorMap& mapC, const TcGemmParams& p, int clusters,
                            cudaStream_t stream, bool pdl) {
    using Cfg = KCfg<MODE, BN, FUSED>;
    cudaError_t e = set_smem_attr<MODE, BN, FUSED>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(threads_k<FUSED>());
    cfg.dynamicSmemBytes = Cfg::smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, gemm_kblock_kernel<MODE, BN, FUSED>, mapA, mapB, mapC, p);
}

}  // namespace

int gemm_kblock_clusters(int mode, int bn, int fused, int sms) {
    if (fused == 3 && mode == kModeTf32x3)
        return bn == 128 ? max_clusters_t<kModeTf32x3, 128, 3>(sms)
                         : max_clusters_t<kModeTf32x3, 256, 3>(sms);
    if (fused == 3)
        return bn == 128 ? max_clusters_t<kModeBf16x9, 128, 3>(sms)
                         : max_clusters_t<kModeBf16x9, 256, 3>(sms);
    if (fused) return max_clusters_t<kModeBf16x9, 128, 1>(sms);
    switch (mode) {
        case kModeTf32x3:
            return bn == 128 ? max_clusters_t<kModeTf32x3, 128, 0>(sms)
                             : max_clusters_t<kModeTf32x3, 256, 0>(sms);
        case kModeBf16x9:
            return bn == 128 ? max_clusters_t<kModeBf16x9, 128, 0>(sms)
                             : max_clusters_t<kModeBf16x9, 256, 0>(sms);
        case kModeBf16x3: return max_clusters_t<kModeBf16x3, 256, 0>(sms);
        case kModeTf32: return max_clusters_t<kModeTf32, 256, 0>(sms);
        case kModeTf32x3Oy: return max_clusters_t<kModeTf32x3Oy, 256, 0>(sms);
        default: return sms / 2;
    }
}

cudaError_t launch_gemm_kblock(int mode, int bn, int fused, const CUtensorMap& mapA,
                               const CUtensorMap& mapB, const CUtensorMap& mapC,
                               const TcGemmParams& p, int sms, cudaStream_t stream, bool pdl) {
    const int tiles = p.tiles_m * p.tiles_n;
    if (tiles == 0) return cudaSuccess;
    TcGemmParams q = p;
    const int resident = gemm_kblock_clusters(mode, bn, fused, sms);
    // A stream-K tail is used only as planned for this many resident
    // clusters: whole tiles fill complete rounds of all of them and every
    // cluster sharing the tail runs at once (an owner waits for the others).
    const int first = tiles - q.tail_tiles;
    const bool split_ok = q.tail_tiles > 0 && q.tail_tiles <= tiles && q.part_ws && q.flags &&
                          q.tail_clusters >= 1 && q.tail_clusters <= resident &&
                          q.num_kb >= 2 && first % resident == 0;
    if (!split_ok) {                         // whole tiles only
        q.tail_tiles = 0;
        q.tail_clusters = 0;
    }
    const int clusters = sched_grid_clusters(tiles, q.tail_tiles, q.tail_clusters, resident);
    cudaError_t e;
    if (fused == 3) {
        if ((mode != kModeBf16x9 && mode != kModeTf32x3) || !q.A32) return cudaErrorInvalidValue;
        if (mode == kModeTf32x3)
            e = bn == 128 ? launch_kblock_t<kModeTf32x3, 128, 3>(mapA, mapB, mapC, q, clusters, stream, pdl)
                          : launch_kblock_t<kModeTf32x3, 256, 3>(mapA, mapB, mapC, q, clusters, stream, pdl);
        else
            e = bn == 128 ? launch_kblock_t<kModeBf16x9, 128, 3>(mapA, mapB, mapC, q, clusters, stream, pdl)
                          : launch_kblock_t<kModeBf16x9, 256, 3>(mapA, mapB, mapC, q, clusters, stream, pdl);
    } else if (fused) {
        if (mode != kModeBf16x9 || bn != 128) return cudaErrorInvalidValue;
        e = launch_kblock_t<kModeBf16x9, 128, 1>(mapA, mapB, mapC, q, clusters, stream, pdl);
    } else if (mode == kModeTf32x3) {
        e = bn == 128 ? launch_kblock_t<kModeTf32x3, 128, 0>(mapA, mapB, mapC, q, clusters, stream, pdl)
                      : launch_kblock_t<kModeTf32x3, 256, 0>(mapA, mapB, mapC, q, clusters, stream, pdl);
    } else if (mode == kModeBf16x9) {
        e = bn == 128 ? launch_kblock_t<kModeBf16x9, 128, 0>(mapA, mapB, mapC, q, clusters, stream, pdl)
                      : launch_kblock_t<kModeBf16x9, 256, 0>(mapA, mapB, mapC, q, clusters, stream, pdl);
    } else if (mode == kModeBf16x3 && bn == 256) {
        e = launch_kblock_t<kModeBf16x3, 256, 0>(mapA, mapB, mapC, q, clusters, stream, pdl);
    } else if (mode == kModeTf32 && bn == 256) {
        e = launch_kblock_t<kModeTf32, 256, 0>(mapA, mapB, mapC, q, clusters, stream, pdl);
    } else if (mode == kModeTf32x3Oy && bn == 256) {
        e = launch_kblock_t<kModeTf32x3Oy, 256, 0>(mapA, mapB, mapC, q, clusters, stream, pdl);
    } else {
        return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace emu
