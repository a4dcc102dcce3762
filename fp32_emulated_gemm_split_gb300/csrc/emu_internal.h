// emu_internal.h -- declarations shared by the translation units of
// libemusgemm (host launchers and kernel parameters).  Not installed.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "schedule.h"

namespace emu {

// Device error codes recorded in the sticky error word (same values as the
// public emu_status_t).
enum : int {
    kDevErrTimeout = -5,
};

// Tensor-core GEMM variants (the values of the public emu_mode_t):
// pieces per operand and the products each K block runs.
enum : int {
    kModeBf16x9 = 0,     // 3 BF16 pieces, 9 products in 5 bands
    kModeTf32x3 = 1,     // 2 TF32 pieces, 3 products
    kModeFp32Simt = 2,   // no pieces: the CUDA-core FP32 kernel
    kModeBf16x3 = 3,     // 2 BF16 pieces, 3 products in 2 bands
    kModeTf32 = 4,       // 1 TF32 piece, 1 product
    kModeTf32x3Oy = 5,   // 2 TF32 pieces (residual scaled by 2^11), 3 products
};
constexpr bool valid_mode(int m) { return m >= kModeBf16x9 && m <= kModeTf32x3Oy; }
constexpr bool mode_is_tf32(int m) { return m == kModeTf32x3 || m == kModeTf32 || m == kModeTf32x3Oy; }
constexpr int mode_pieces(int m) { return m == kModeBf16x9 ? 3 : m == kModeTf32 ? 1 : 2; }

// K extent of one staged piece tile in bytes: one 128-byte swizzled row
// (64 BF16 or 32 TF32 elements).
constexpr int kTcBKBytes = 128;

// Row stride, in elements, of the split pieces in the workspace: a multiple
// of 8 so that every row starts on a 16-byte boundary (a TMA requirement).
inline int64_t plane_ld(int64_t K) { return (K + 7) / 8 * 8; }

struct TcGemmParams {
    int* err;            // the device's sticky error word
    int M, N, K;
    int num_kb;          // number of K stages: ceil(K / elements per stage)
    int tiles_m, tiles_n;
    float alpha, beta;
    float* C;
    int64_t ldc;
    int tma_store;       // 1: the C tensor map is valid (bulk tensor stores of C)
    // Stream-K tail (schedule.h): the K blocks of the last tail_tiles tiles
    // are shared by tail_clusters clusters in consecutive ranges; a cluster
    // whose range starts inside a tile leaves that part's FP32 sums in its
    // slot of part_ws and raises its flag (value epoch); the tile's owner
    // adds them and writes C.  tail_tiles = 0: whole tiles only.
    int tail_tiles, tail_clusters;
    // shared-memory fused path only: FP32 A (row-major, 16-byte aligned,
    // lda % 4 == 0), read by the kernel's split warps
    const float* A32;
    int64_t lda;
    float* part_ws;
    unsigned* flags;
    unsigned epoch;
    // Two-pass BF16 modes: the layout of each operand's pieces.  0: K-major
    // (planes of op(A)'s rows, or op(B)^T's, along K: what the split writes
    // from a matrix stored with K contiguous).  1: M-major (A) or N-major
    // (B): planes of K rows of M or N elements, what a plain row-wise split
    // writes from A stored K x M (transA) or B stored K x N; the tensor core
    // reads them through the transpose bits of its instruction descriptor,
    // so no transposed split is needed.
    int a_mn, b_mn;
};

// Launchers (return the launch status; nothing is synchronised).
cudaError_t launch_split_bf16x3(const float* X, int64_t rows, int64_t cols, int64_t ld, int trans,
                                uint16_t* P0, uint16_t* P1, uint16_t* P2, int64_t ldp,
                                cudaStream_t stream, bool pdl = false);
// lo_scale: 1 (TF32x3) or 2^11 (the residual scaled before its rounding)
cudaError_t launch_split_tf32x2(const float* X, int64_t rows, int64_t cols, int64_t ld, int trans,
                                float* HI, float* LO, int64_t ldp, cudaStream_t stream,
                                float lo_scale = 1.0f, bool pdl = false);
// The pieces a tensor-core mode reads, as planes of rows x ldp elements
// (BF16 bits or TF32-valued FP32) starting at `planes`, plane_rows rows of
// ldp apart (0: rows, consecutive planes; more: the rows of a panel of a
// larger set of planes).
// pdl: launch as a programmatic dependent of the kernel ahead in the stream
// (only where the two are independent); the split still completes after it.
cudaError_t launch_split_pieces(int mode, const float* X, int64_t rows, int64_t cols, int64_t ld,
                                int trans, void* planes, int64_t ldp, cudaStream_t stream,
                                bool pdl = false, int64_t plane_rows = 0);
// Bytes of one piece element of a mode.
constexpr int mode_piece_bytes(int m) { return mode_is_tf32(m) ? 4 : 2; }
// mode: one of the kMode* variants; bn: tile width 128 or 256 (the two
// cheaper modes: 256 only); fused: mapA is an FP32 map over op(A) (box
// 32 x 128) split in shared memory (BF16x9, bn 128 only)
// pdl: the GEMM may start (prologue: barriers, tensor memory, descriptor
// prefetch) while the split ahead of it runs; its producer waits for that
// split before the first piece load.
cudaError_t launch_gemm_kblock(int mode, int bn, int fused, const CUtensorMap& mapA,
                               const CUtensorMap& mapB, const CUtensorMap& mapC,
                               const TcGemmParams& p, int sms, cudaStream_t stream,
                               bool pdl = false);
// Clusters of the GEMM variant that can be resident at once on a GPU with
// `sms` SMs (at most sms / 2); the persistent grid uses this many.
int gemm_kblock_clusters(int mode, int bn, int fused, int sms);
cudaError_t launch_gemm_simt(int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha,
                             const float* A, int64_t lda, const float* B, int64_t ldb, float beta,
                             float* C, int64_t ldc, cudaStream_t stream);
cudaError_t launch_scale(int64_t M, int64_t N, float beta, float* C, int64_t ldc,
                         cudaStream_t stream);
cudaError_t launch_timeout_probe(int* err, uint64_t limit_ns, cudaStream_t stream);

// PERFORMANT strategy (chooser.cu): the mode that runs for a requested mode
// (the FP32 SIMT kernel where it is predicted faster), and the two time
// estimates in microseconds; sms is the device's SM count.
// What handing one part's sums to the tile's owner costs, in half K blocks
// of the mode (the split tail's planner, schedule.h, and the time model of
// the PERFORMANT strategy use it): writing and reading a slot takes about 4
// us for 256-wide tiles (2 us for 128-wide ones, whose K blocks also take half
// as long), against measured K blocks of 2.7 us (BF16x9), 1.1 us (TF32x3, its
// Ootomo-Yokota variant and BF16x3) and 0.53 us (single-pass TF32).
inline int handover_half_blocks(int mode) {
    switch (mode) {
        case kModeBf16x9: return 3;
        case kModeTf32x3:
        case kModeTf32x3Oy: return 8;
        case kModeBf16x3: return 7;
        default: return 15;
    }
}
int choose_mode(int64_t M, int64_t N, int64_t K, int mode, int performant, int sms);
double predict_tc_us(int64_t M, int64_t N, int64_t K, int mode, int sms);
double predict_simt_us(int64_t M, int64_t N, int64_t K, int sms);

// Device address of the sticky error word of the current device.
int* device_error_word();

}  // namespace emu
