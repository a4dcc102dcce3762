// emu_sgemm.cu -- host side of libemusgemm: the C ABI declared in
// include/emu_sgemm.h.  Argument checks, the per-device workspace, TMA tensor
// maps, dispatch between the two-pass, fused and SIMT paths, kernel timing
// and the host-buffer entry point.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "emu_device.cuh"
#include "emu_sgemm.h"

namespace emu {

__device__ int g_emu_error = 0;

static_assert(kModeBf16x9 == int(EMU_MODE_BF16X9) && kModeTf32x3 == int(EMU_MODE_TF32X3) &&
                  kModeFp32Simt == int(EMU_MODE_FP32_SIMT) && kModeBf16x3 == int(EMU_MODE_BF16X3) &&
                  kModeTf32 == int(EMU_MODE_TF32) && kModeTf32x3Oy == int(EMU_MODE_TF32X3_OY),
              "kernel variants follow emu_mode_t");

namespace {

constexpr int kMaxDevices = 64;
constexpr int kHostChunksMax = 8;        // row chunks of emu_sgemm_host's copy/compute pipeline

struct DeviceState {
    int checked = 0;           // 0 unknown, 1 supported, -1 unsupported
    int sms = 0;
    int* err = nullptr;        // device address of g_emu_error
    void* ws = nullptr;        // workspace for the split pieces
    size_t ws_bytes = 0;
    void* stage = nullptr;     // device staging for emu_sgemm_host
    size_t stage_bytes = 0;
    // emu_sgemm_host's pipeline: host->device and device->host copy streams
    // and per-chunk events (created on first use, kept until exit)
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t ev_in[kHostChunksMax] = {}, ev_done[kHostChunksMax] = {};
    cudaEvent_t ev_panel = nullptr;      // each column panel of op(B) landed
    // the GEMM's stream-K tail: one slot of partial sums per cluster (grown on
    // demand), flags (zeroed once) and the epoch that marks this call's flags
    void* part = nullptr;
    size_t part_bytes = 0;
    unsigned* flags = nullptr;
    unsigned epoch = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
int g_path = -1;               // -1: not yet read from the environment
int g_strategy = -1;           // same

// ------------------------------------------------------------ profiling --
struct ProfRecord { int kind; cudaEvent_t start, stop; };
bool g_prof_on = false;
std::vector<ProfRecord> g_prof_pending;
std::vector<cudaEvent_t> g_event_pool;
int64_t g_prof_launches[5] = {0, 0, 0, 0, 0};
double g_prof_ms[5] = {0, 0, 0, 0, 0};

cudaEvent_t pool_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

struct ProfScope {
    int kind;
    cudaStream_t stream;
    cudaEvent_t start = nullptr;
    ProfScope(int k, cudaStream_t s) : kind(k), stream(s) {
        if (g_prof_on) {
            start = pool_event();
            cudaEventRecord(start, stream);
        }
    }
    ~ProfScope() {
        if (start) {
            cudaEvent_t stop = pool_event();
            cudaEventRecord(stop, stream);
            g_prof_pending.push_back({kind, start, stop});
        }
    }
};

// ----------------------------------------------------------- helpers --

cudaError_t g_last_cuda_error = cudaSuccess;

emu_status_t from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return EMU_OK;
    g_last_cuda_error = e;
    if (e == cudaErrorMemoryAllocation) return EMU_ERR_ALLOC;
    if (e == cudaErrorLaunchFailure || e == cudaErrorInvalidConfiguration ||
        e == cudaErrorLaunchOutOfResources || e == cudaErrorInvalidDeviceFunction ||
        e == cudaErrorNoKernelImageForDevice)
        return EMU_ERR_LAUNCH;
    return EMU_ERR_CUDA;
}

// Tile width of the K-block kernel on the two-pass path: 128 when N <= 128
// (a 256-wide tile would compute at least half zeros), else 256.
int kblock_bn(int64_t N) { return N <= 128 ? 128 : 256; }

int read_strategy_env() {
    const char* s = std::getenv("EMU_SGEMM_STRATEGY");
    if (s && !std::strcmp(s, "performant")) return EMU_STRATEGY_PERFORMANT;
    return EMU_STRATEGY_EAGER;
}

int read_path_env() {
    const char* s = std::getenv("EMU_SGEMM_PATH");
    if (!s) return EMU_PATH_AUTO;
    if (!std::strcmp(s, "twopass")) return EMU_PATH_TWOPASS;
    if (!std::strcmp(s, "fused")) return EMU_PATH_FUSED;
    if (!std::strcmp(s, "fused_tmem")) return EMU_PATH_FUSED_TMEM;
    return EMU_PATH_AUTO;
}

// Current device state, checking the architecture once.
emu_status_t current_device(DeviceState** out, int* dev_out = nullptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return EMU_ERR_CUDA;
    DeviceState& d = g_dev[dev];
    if (d.checked == 0) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        d.checked = (major == 10 && minor == 3) ? 1 : -1;
        if (d.checked > 0 &&
            cudaGetSymbolAddress(reinterpret_cast<void**>(&d.err), g_emu_error) != cudaSuccess) {
            cudaGetLastError();
            d.checked = 0;
            return EMU_ERR_CUDA;
        }
    }
    if (d.checked < 0) return EMU_ERR_ARCH;
    *out = &d;
    if (dev_out) *dev_out = dev;
    return EMU_OK;
}

emu_status_t ensure_buffer(void** buf, size_t* have, size_t need) {
    if (need <= *have) return EMU_OK;
    if (*buf) {
        cudaFree(*buf);   // synchronises the device: no kernel still reads the old buffer
        *buf = nullptr;
        *have = 0;
    }
    size_t bytes = need + need / 8;   // some headroom against repeated growth
    if (cudaMalloc(buf, bytes) != cudaSuccess) {
        cudaGetLastError();
        *buf = nullptr;
        return EMU_ERR_ALLOC;
    }
    *have = bytes;
    return EMU_OK;
}

// cuTensorMapEncodeTiled, fetched from the driver through the runtime so the
// library needs no link-time dependency on libcuda.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// Tensor map over `planes` row-major planes of rows x cols elements (row
// stride ld elements, plane stride plane_rows*ld, plane_rows 0 meaning
// rows), box of box_cols x box_rows, 128-byte swizzle, zero fill outside the
// matrix.
emu_status_t make_plane_map(CUtensorMap* map, const void* base, bool fp32, int64_t rows,
                            int64_t cols, int64_t ld, int planes, int box_cols, int box_rows,
                            int64_t plane_rows = 0) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return EMU_ERR_CUDA;
    const int esize = fp32 ? 4 : 2;
    const int64_t prow = plane_rows > 0 ? plane_rows : rows;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)planes};
    cuuint64_t strides[2] = {(cuuint64_t)(ld * esize), (cuuint64_t)(prow * ld * esize)};
    cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
    cuuint32_t elem_strides[3] = {1, 1, 1};
    CUresult r = enc(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     3, const_cast<void*>(base), dims, strides, box, elem_strides,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? EMU_OK : EMU_ERR_CUDA;
}

// 4-D map over M- or N-major pieces: `planes` planes of K rows x ld
// elements (ld a multiple of 64; planes plane_rows rows apart, 0: K), each
// row seen as ceil(cols / 64) chunks of 64 elements: dimensions (element,
// K row, chunk, piece).  A box of 64 elements x box_k rows x `chunks`
// chunks lands in shared memory as the chunks one after another, each K
// row 128 bytes (128-byte swizzle): the M- or N-major layout the tensor
// core reads.  K rows past K and chunks past the last are zero-filled; the
// elements of the last chunk past `cols` are read from the row's padding
// and reach only outputs that are never stored.
emu_status_t make_plane_map_mn(CUtensorMap* map, const void* base, int64_t cols, int64_t K,
                               int64_t ld, int planes, int box_k, int chunks,
                               int64_t plane_rows = 0) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return EMU_ERR_CUDA;
    if (ld % 64 != 0) return EMU_ERR_INVALID_VALUE;
    const int64_t prow = plane_rows > 0 ? plane_rows : K;
    cuuint64_t dims[4] = {64, (cuuint64_t)K, (cuuint64_t)((cols + 63) / 64), (cuuint64_t)planes};
    cuuint64_t strides[3] = {(cuuint64_t)(ld * 2), 128, (cuuint64_t)(prow * ld * 2)};
    cuuint32_t box[4] = {64, (cuuint32_t)box_k, (cuuint32_t)chunks, 1};
    cuuint32_t elem_strides[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                     strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? EMU_OK : EMU_ERR_CUDA;
}

// 2-D map over C for the bulk tensor stores of the GEMM epilogue (any beta;
// with beta != 0 the epilogue reads C itself first): box of 16 columns x 32
// rows, 64-byte swizzle.  The map covers the first N & ~3 columns only: a
// bulk store clips a box at the edge of the map in whole 16-byte units
// (measured on GB300: with N = 4k + 1..3 it wrote zeros up to column 4k + 3,
// past C), so the epilogue stores the last N % 4 columns of each row itself.
// Returns false (and the kernel stores C directly) when C's rows are not
// 16-byte aligned or C is narrower than 4 columns.
bool make_c_map(CUtensorMap* map, float* C, int64_t M, int64_t N, int64_t ldc) {
    if ((ldc % 4) != 0 || (reinterpret_cast<uintptr_t>(C) & 15) != 0 || N < 4) return false;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)(N & ~int64_t(3)), (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)(ldc * 4)};
    cuuint32_t box[2] = {16, 32};
    cuuint32_t elem_strides[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, C, dims, strides, box, elem_strides,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Plan the tail of the persistent GEMM (schedule.h) for the clusters of
// this GEMM variant that can be resident at once, and give it its
// workspace: one slot of bm x bn FP32 sums and 2 x 16 flags per cluster
// sharing the tail.  Sets p.tail_*, p.part_ws, p.flags and p.epoch.
constexpr int kFlagsBytes = 64 << 10;

emu_status_t plan_tail(TcGemmParams& p, int mode, int bm, int bn, int fused, DeviceState* d) {
    const int tiles = p.tiles_m * p.tiles_n;
    const int clusters = gemm_kblock_clusters(mode, bn, fused, d->sms);
    p.tail_tiles = 0;
    p.tail_clusters = 0;
    p.part_ws = nullptr;
    p.flags = nullptr;
    p.epoch = 0;
    int tail_tiles = 0, tail_clusters = 0;
    sched_plan_tail(tiles, p.num_kb, clusters, handover_half_blocks(mode), &tail_tiles,
                    &tail_clusters);
    if (tail_tiles == 0) return EMU_OK;
    if ((size_t)tail_clusters * 2 * 16 * sizeof(unsigned) > (size_t)kFlagsBytes) return EMU_OK;
    const size_t need = (size_t)tail_clusters * bm * bn * sizeof(float);
    emu_status_t st = ensure_buffer(&d->part, &d->part_bytes, need);
    if (st != EMU_OK) return st;
    if (!d->flags) {
        if (cudaMalloc(&d->flags, kFlagsBytes) != cudaSuccess) {
            cudaGetLastError();
            d->flags = nullptr;
            return EMU_ERR_ALLOC;
        }
        if (cudaMemset(d->flags, 0, kFlagsBytes) != cudaSuccess) return from_cuda(cudaGetLastError());
    }
    p.tail_tiles = tail_tiles;
    p.tail_clusters = tail_clusters;
    p.part_ws = static_cast<float*>(d->part);
    p.flags = d->flags;
    p.epoch = ++d->epoch == 0 ? ++d->epoch : d->epoch;   // never 0 (the flags' initial value)
    return EMU_OK;
}

// a * b + c, or false when it does not fit in 62 bits (no allocation that
// large can succeed; the check keeps every later size product from wrapping).
bool fits_mul_add(uint64_t a, uint64_t b, uint64_t c, size_t* out) {
    uint64_t p = 0;
    if (__builtin_mul_overflow(a, b, &p) || __builtin_add_overflow(p, c, &p) ||
        p > (uint64_t(1) << 62))
        return false;
    *out = (size_t)p;
    return true;
}

// The largest workspace any mode needs for this shape: 3 pieces x 4 bytes x
// ldp per row of op(A) and op(B)^T, plus the 1 KB alignment of A's region.
// Beyond 2^62 bytes the call returns EMU_ERR_ALLOC before any size product
// is formed (M, N, K up to INT32_MAX would otherwise wrap a 64-bit size).
bool workspace_fits(int64_t M, int64_t N, int64_t K) {
    size_t bytes = 0;
    // K-major pieces, and M- or N-major ones (K rows of M and N rounded up to 64)
    return fits_mul_add((uint64_t)M + (uint64_t)N, 12 * (uint64_t)plane_ld(K), 2048, &bytes) &&
           fits_mul_add((uint64_t)M + (uint64_t)N + 128, 12 * (uint64_t)K, 2048, &bytes);
}

emu_status_t check_gemm_args(int transA, int transB, int64_t M, int64_t N, int64_t K,
                             const float* A, int64_t lda, const float* B, int64_t ldb,
                             float beta, float* C, int64_t ldc, int mode) {
    if ((transA != 0 && transA != 1) || (transB != 0 && transB != 1)) return EMU_ERR_INVALID_VALUE;
    if (!valid_mode(mode)) return EMU_ERR_INVALID_VALUE;
    if (M < 0 || N < 0 || K < 0) return EMU_ERR_INVALID_VALUE;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return EMU_ERR_INVALID_VALUE;
    const int64_t a_cols = transA ? M : K, b_cols = transB ? K : N;
    if (lda < 1 || lda < a_cols || ldb < 1 || ldb < b_cols || ldc < 1 || ldc < N)
        return EMU_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return EMU_OK;
    if (C == nullptr) return EMU_ERR_INVALID_VALUE;
    if (K > 0 && (A == nullptr || B == nullptr)) return EMU_ERR_INVALID_VALUE;
    (void)beta;
    return EMU_OK;
}

// Workspace layout: op(B)^T's pieces first (at offset 0, so that they stay
// where they are for any M), then op(A)'s at a 1 KB boundary.  b_ready: B's
// pieces for this B, mode and K are already there (an earlier row chunk of
// the same emu_sgemm_host call put them) and are not split again.
// B's pieces supplied by the caller (emu_sgemm_bsplit): the pieces of
// op(B)^T as consecutive planes of N rows x ldbp elements.
struct BPieces {
    const void* p = nullptr;
    int64_t ld = 0;
};

// Where one operand's pieces are: planes starting at p, ld elements per
// row, plane_rows rows apart (0: the planes' own row count).  mn = 0:
// K-major, a row per row of op(A) (or of op(B)^T), K elements long.  mn = 1
// (two-pass BF16 modes): M- or N-major, a row per K index, M (or N) elements
// long, ld a multiple of 64 (mn_ld) -- what a row-wise split writes from A
// stored K x M or B stored K x N.
struct PieceSet {
    const void* p;
    int64_t ld;
    int64_t plane_rows;
    int mn;
};

// Whether a two-pass call keeps an operand's pieces M- or N-major: an
// operand stored with K as its row index (A with transA, B without transB),
// whose split is then a row-wise one instead of a transposed one (about
// 20 us less per 8192^2 operand on GB300).  BF16x9 always: measured on GB300
// with launches of the two layouts alternating on one box (40-60 pairs,
// median of the pair differences), the GEMM takes the same time on N-major
// as on K-major pieces at 8192^3, 4096^3, 12288 x 1024 x 256 and 1.1M x 1024
// x 256 (within 0.1 %), and less for deep K (1024^2 x 32768 7 %, the weight
// gradients 256 x 256, 256 x 1024 and 1024^2 x 1,105,920 6-10 %: a tile's K
// rows of 512 bytes follow each other in memory, where K-major rows millions
// of elements long do not).  BF16x3 only when K is at least 4 times the
// operand's M (or N): at 8192^3 N-major pieces cost it 4-5 % with the same
// L2 and DRAM traffic and less tensor-pipe activity (75.9 against 72.5 % at
// 4096^3), which an L2 prefetch of the next K block did not change.  TF32
// pieces stay K-major.  The rule depends
// on K and the operand's own extent only, so a row chunk of op(A) never
// changes B's layout.
inline bool mn_pieces(int mode, bool k_is_row, int64_t K, int64_t extent) {
    if (!k_is_row) return false;
    return mode == kModeBf16x9 || (mode == kModeBf16x3 && K >= 4 * extent);
}

// Row length of M- or N-major pieces: whole 64-element chunks (the tensor
// copies read them a chunk at a time).
inline int64_t mn_ld(int64_t cols) { return (cols + 63) / 64 * 64; }

// Bytes of one operand's pieces: `rows` rows of op(A) (or of op(B)^T) over K.
inline size_t piece_bytes(int mode, bool mn, int64_t rows, int64_t K) {
    const size_t per = (size_t)mode_pieces(mode) * mode_piece_bytes(mode);
    return mn ? per * (size_t)K * mn_ld(rows) : per * (size_t)rows * plane_ld(K);
}

// The tensor-core GEMM on pieces already in device memory (op(A)'s and
// op(B)^T's, as PieceSet says).  Launched as a programmatic dependent of the
// split ahead of it in the stream.
emu_status_t gemm_on_pieces(int mode, const PieceSet& a, const PieceSet& b, int64_t M, int64_t N,
                            int64_t K, float alpha, float beta, float* C, int64_t ldc,
                            DeviceState* d, cudaStream_t stream) {
    const int tf32 = mode_is_tf32(mode);
    const int planes = mode_pieces(mode);
    const int box_cols = tf32 ? kTcBKBytes / 4 : kTcBKBytes / 2;
    // the two cheaper modes are built for 256-wide tiles only
    const int bn = (mode == kModeBf16x9 || mode == kModeTf32x3) ? kblock_bn(N) : 256;
    if ((a.mn || b.mn) && tf32) return EMU_ERR_INVALID_VALUE;     // caller's bug
    // K-major planes: a (K, rows, piece) map read in boxes of one K block x
    // the CTA's rows; M- or N-major: boxes of one K block x the CTA's
    // 64-element chunks
    CUtensorMap mapA, mapB;
    emu_status_t st = a.mn ? make_plane_map_mn(&mapA, a.p, M, K, a.ld, planes, box_cols, 128 / 64,
                                               a.plane_rows)
                           : make_plane_map(&mapA, a.p, tf32, M, K, a.ld, planes, box_cols, 128,
                                            a.plane_rows);
    if (st != EMU_OK) return st;
    st = b.mn ? make_plane_map_mn(&mapB, b.p, N, K, b.ld, planes, box_cols, bn / 2 / 64,
                                  b.plane_rows)
              : make_plane_map(&mapB, b.p, tf32, N, K, b.ld, planes, box_cols, bn / 2, b.plane_rows);
    if (st != EMU_OK) return st;

    TcGemmParams p = {};
    p.err = d->err;
    p.M = (int)M; p.N = (int)N; p.K = (int)K;
    p.num_kb = (int)((K + box_cols - 1) / box_cols);
    p.tiles_m = (int)((M + 255) / 256);
    p.tiles_n = (int)((N + bn - 1) / bn);
    p.alpha = alpha; p.beta = beta; p.C = C; p.ldc = ldc;
    p.a_mn = a.mn; p.b_mn = b.mn;
    CUtensorMap mapC = mapB;                 // placeholder when C is stored directly
    p.tma_store = make_c_map(&mapC, C, M, N, ldc) ? 1 : 0;
    st = plan_tail(p, mode, 256, bn, 0, d);
    if (st != EMU_OK) return st;
    ProfScope ps(1, stream);
    return from_cuda(launch_gemm_kblock(mode, bn, 0, mapA, mapB, mapC, p, d->sms, stream, true));
}

emu_status_t run_two_pass(int mode, int transA, int transB, int64_t M, int64_t N, int64_t K,
                          float alpha, const float* A, int64_t lda, const float* B, int64_t ldb,
                          float beta, float* C, int64_t ldc, DeviceState* d, cudaStream_t stream,
                          bool b_ready = false, BPieces bext = {}) {
    const int64_t ldp = plane_ld(K);
    const bool a_mn = mn_pieces(mode, transA, K, M);
    const bool b_mn = mn_pieces(mode, !transB, K, N) && !bext.p;
    const size_t a_bytes = piece_bytes(mode, a_mn, M, K);
    const size_t b_bytes = bext.p ? 0 : piece_bytes(mode, b_mn, N, K);
    const size_t b_region = (b_bytes + 1023) / 1024 * 1024;
    if (b_ready && d->ws_bytes < b_region + a_bytes) return EMU_ERR_INVALID_VALUE;  // caller's bug
    emu_status_t st = ensure_buffer(&d->ws, &d->ws_bytes, b_region + a_bytes);
    if (st != EMU_OK) return st;
    uint8_t* wb = static_cast<uint8_t*>(d->ws);
    uint8_t* wa = wb + b_region;

    const PieceSet as{wa, a_mn ? mn_ld(M) : ldp, 0, a_mn ? 1 : 0};
    const PieceSet bs = bext.p ? PieceSet{bext.p, bext.ld, 0, 0}
                               : PieceSet{wb, b_mn ? mn_ld(N) : ldp, 0, b_mn ? 1 : 0};
    cudaError_t e;
    {
        // op(A) is M x K: A itself when transA == 0; A stored K x M split
        // row-wise into M-major pieces (BF16) or transposed (TF32)
        ProfScope ps(0, stream);
        e = a_mn ? launch_split_pieces(mode, A, K, M, lda, 0, wa, as.ld, stream)
                 : launch_split_pieces(mode, A, M, K, lda, transA, wa, ldp, stream);
    }
    if (e != cudaSuccess) return from_cuda(e);
    if (!b_ready && !bext.p) {
        // op(B)^T is N x K: B itself when transB == 1; B stored K x N split
        // row-wise into N-major pieces (BF16) or transposed (TF32)
        ProfScope ps(0, stream);
        // independent of A's split: may run beside it (programmatic launch)
        e = b_mn ? launch_split_pieces(mode, B, K, N, ldb, 0, wb, bs.ld, stream, true)
                 : launch_split_pieces(mode, B, N, K, ldb, !transB, wb, ldp, stream, true);
    }
    if (e != cudaSuccess) return from_cuda(e);
    return gemm_on_pieces(mode, as, bs, M, N, K, alpha, beta, C, ldc, d, stream);
}

// Whether op(A) can be read directly by the fused kernel: K-major rows that
// start on 16-byte boundaries (a TMA requirement).
bool fused_ok(int mode, int transA, const float* A, int64_t lda) {
    return (mode == EMU_MODE_BF16X9 || mode == EMU_MODE_TF32X3) && transA == 0 &&
           (lda % 4) == 0 && (reinterpret_cast<uintptr_t>(A) & 15) == 0;
}

// Tensor-memory fused path: B's three pieces go to the workspace (one split
// kernel); A is read as FP32 by the GEMM kernel (TMA into shared memory) and
// split by its split warps into tensor memory, where the MMA reads it
// (128-wide tiles).
emu_status_t run_fused_tmem(int transB, int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                       int64_t lda, const float* B, int64_t ldb, float beta, float* C,
                       int64_t ldc, DeviceState* d, cudaStream_t stream, bool b_ready = false,
                       BPieces bext = {}) {
    int64_t ldp = plane_ld(K);
    uint16_t* pb = nullptr;
    emu_status_t st;
    if (bext.p) {
        pb = const_cast<uint16_t*>(static_cast<const uint16_t*>(bext.p));
        ldp = bext.ld;
    } else {
        if (b_ready && d->ws_bytes < (size_t)3 * N * ldp * 2) return EMU_ERR_INVALID_VALUE;
        st = ensure_buffer(&d->ws, &d->ws_bytes, (size_t)3 * N * ldp * 2);
        if (st != EMU_OK) return st;
        pb = static_cast<uint16_t*>(d->ws);
    }
    cudaError_t e = cudaSuccess;
    if (!b_ready && !bext.p) {
        ProfScope ps(0, stream);
        e = launch_split_bf16x3(B, N, K, ldb, !transB, pb, pb + N * ldp, pb + 2 * N * ldp, ldp,
                                stream);
    }
    if (e != cudaSuccess) return from_cuda(e);
    constexpr int bn = 128;
    CUtensorMap mapA, mapB;
    st = make_plane_map(&mapA, A, true, M, K, lda, 1, 32, 128);   // FP32 A: (K, M, 1)
    if (st != EMU_OK) return st;
    st = make_plane_map(&mapB, pb, false, N, K, ldp, 3, 64, bn / 2);
    if (st != EMU_OK) return st;
    TcGemmParams p = {};
    p.err = d->err;
    p.M = (int)M; p.N = (int)N; p.K = (int)K;
    p.num_kb = (int)((K + 63) / 64);
    p.tiles_m = (int)((M + 255) / 256);
    p.tiles_n = (int)((N + bn - 1) / bn);
    p.alpha = alpha; p.beta = beta; p.C = C; p.ldc = ldc;
    CUtensorMap mapC = mapB;
    p.tma_store = make_c_map(&mapC, C, M, N, ldc) ? 1 : 0;
    st = plan_tail(p, kModeBf16x9, 256, bn, 1, d);
    if (st != EMU_OK) return st;
    {
        ProfScope ps(2, stream);
        e = launch_gemm_kblock(0, bn, 1, mapA, mapB, mapC, p, d->sms, stream, true);
    }
    return from_cuda(e);
}

// Shared-memory fused path (BF16x9): B's pieces go to the workspace (one
// split kernel); the GEMM kernel's split warps read FP32 A and store its
// pieces straight into the A half of each shared-memory stage, where the
// two-pass path's TMA would have put them: 256-wide tiles, A read from HBM
// once as FP32, its pieces never written out.
emu_status_t run_fused_smem(int mode, int transB, int64_t M, int64_t N, int64_t K, float alpha,
                            const float* A, int64_t lda, const float* B, int64_t ldb, float beta,
                            float* C, int64_t ldc, DeviceState* d, cudaStream_t stream,
                            bool b_ready = false, BPieces bext = {}) {
    // BF16x9: three BF16 pieces per K block of 64; TF32x3: hi and lo (FP32
    // containers) per K block of 32
    const bool tf32 = mode == kModeTf32x3;
    const int pieces = mode_pieces(mode), es = mode_piece_bytes(mode);
    const int box_k = tf32 ? kTcBKBytes / 4 : kTcBKBytes / 2;
    int64_t ldp = plane_ld(K);
    uint8_t* pb = nullptr;
    emu_status_t st;
    if (bext.p) {
        pb = const_cast<uint8_t*>(static_cast<const uint8_t*>(bext.p));
        ldp = bext.ld;
    } else {
        const size_t need = (size_t)pieces * N * ldp * es;
        if (b_ready && d->ws_bytes < need) return EMU_ERR_INVALID_VALUE;
        st = ensure_buffer(&d->ws, &d->ws_bytes, need);
        if (st != EMU_OK) return st;
        pb = static_cast<uint8_t*>(d->ws);
    }
    cudaError_t e = cudaSuccess;
    if (!b_ready && !bext.p) {
        ProfScope ps(0, stream);
        e = launch_split_pieces(mode, B, N, K, ldb, !transB, pb, ldp, stream);
    }
    if (e != cudaSuccess) return from_cuda(e);
    const int bn = kblock_bn(N);
    CUtensorMap mapB;
    st = make_plane_map(&mapB, pb, tf32, N, K, ldp, pieces, box_k, bn / 2);
    if (st != EMU_OK) return st;
    const CUtensorMap mapA = mapB;           // not read: the split warps fill A's stages
    TcGemmParams p = {};
    p.err = d->err;
    p.M = (int)M; p.N = (int)N; p.K = (int)K;
    p.num_kb = (int)((K + box_k - 1) / box_k);
    p.tiles_m = (int)((M + 255) / 256);
    p.tiles_n = (int)((N + bn - 1) / bn);
    p.alpha = alpha; p.beta = beta; p.C = C; p.ldc = ldc;
    p.A32 = A; p.lda = lda;
    CUtensorMap mapC = mapB;
    p.tma_store = make_c_map(&mapC, C, M, N, ldc) ? 1 : 0;
    st = plan_tail(p, mode, 256, bn, 3, d);
    if (st != EMU_OK) return st;
    {
        ProfScope ps(2, stream);
        e = launch_gemm_kblock(mode, bn, 3, mapA, mapB, mapC, p, d->sms, stream, true);
    }
    return from_cuda(e);
}

// What one call runs: the kernel mode after the strategy's choice, and
// which path takes it (0 two-pass, 1 tensor-memory fused, 3 shared-memory
// fused).
struct Plan {
    int mode;
    int fused;
};

Plan plan_call(int transA, int64_t M, int64_t N, int64_t K, const float* A, int64_t lda, int mode,
               const DeviceState* d, bool keep_mode = false) {
    if (g_strategy < 0) g_strategy = read_strategy_env();
    if (g_path < 0) g_path = read_path_env();
    Plan pl;
    // PERFORMANT: the plain FP32 kernel where it is predicted faster (not
    // when B comes already split: the pieces are what the caller gives)
    pl.mode = keep_mode ? mode
                        : choose_mode(M, N, K, mode, g_strategy == EMU_STRATEGY_PERFORMANT, d->sms);
    // AUTO, for BF16x9 with M >= 4096 and N <= 256 (the MLIP layers), where
    // splitting A in the GEMM kernel saves more than the split kernel's HBM
    // round trip costs (measured on GB300, graph replays, shared-memory fused
    // / tensor-memory fused / two-pass): for 128 < N <= 256 the shared-memory
    // path (131072 x 256 x 1024 387 / 476 / 532 us; 131072 x 256 x 256 123 /
    // 142 / 150 us; 12288 x 256 x 1024 55.2 / 60.6 / 63.3 us; 12288 x 256 x
    // 256 24.3 / 26.8 / 26.8 us), for N <= 128 the tensor-memory path, whose
    // 128-wide tiles then waste nothing (131072 x 128 x 256 95 / 79 / 114 us);
    // two-pass elsewhere (N = 1024: 394 us two-pass against 447, as A's
    // pieces are then reused by four column tiles).
    const bool small_n = g_path == EMU_PATH_AUTO && N <= 256 && M >= 4096;
    const bool on_chip = pl.mode != EMU_MODE_FP32_SIMT && fused_ok(pl.mode, transA, A, lda);
    // the tensor-memory kernel splits BF16x9 pieces only; TF32x3 has the
    // shared-memory one, which AUTO does not take: measured on GB300 against
    // two-pass (20 calls back to back) it is no faster on the MLIP layers
    // (1.1M x 256 x 256 1212 / 1216 us, 1.1M x 256 x 1024 4477 / 4385 us,
    // 12288 x 256 x 256 33.9 / 25.8 us): a TF32 K block is a third of a BF16x9
    // one's MMA time, so the per-tile epilogue and hand-offs dominate either way
    const bool tm = pl.mode == EMU_MODE_BF16X9;
    pl.fused = !on_chip ? 0
             : g_path == EMU_PATH_FUSED_TMEM ? (tm ? 1 : 0)
             : g_path == EMU_PATH_FUSED ? 3
             : !small_n ? 0
             : pl.mode == EMU_MODE_TF32X3 ? 0
             : (N > 128 ? 3 : 1);
    return pl;
}

emu_status_t run_planned(const Plan& pl, int transA, int transB, int64_t M, int64_t N, int64_t K,
                         float alpha, const float* A, int64_t lda, const float* B, int64_t ldb,
                         float beta, float* C, int64_t ldc, DeviceState* d, cudaStream_t stream,
                         bool b_ready, BPieces bext = {}) {
    if (pl.mode == EMU_MODE_FP32_SIMT) {
        ProfScope ps(3, stream);
        return from_cuda(launch_gemm_simt(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C,
                                          ldc, stream));
    }
    if (pl.fused == 3)
        return run_fused_smem(pl.mode, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, d,
                              stream, b_ready, bext);
    if (pl.fused == 1)
        return run_fused_tmem(transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, d, stream,
                              b_ready, bext);
    return run_two_pass(pl.mode, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, d,
                        stream, b_ready, bext);
}

emu_status_t sgemm_device(int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha,
                          const float* A, int64_t lda, const float* B, int64_t ldb, float beta,
                          float* C, int64_t ldc, int mode, cudaStream_t stream) {
    emu_status_t st = check_gemm_args(transA, transB, M, N, K, A, lda, B, ldb, beta, C, ldc, mode);
    if (st != EMU_OK) return st;
    if (M == 0 || N == 0) return EMU_OK;
    if (!workspace_fits(M, N, K)) return EMU_ERR_ALLOC;
    DeviceState* d = nullptr;
    st = current_device(&d);
    if (st != EMU_OK) return st;
    if (K == 0 || alpha == 0.0f) {
        ProfScope ps(4, stream);
        return from_cuda(launch_scale(M, N, beta, C, ldc, stream));
    }
    const Plan pl = plan_call(transA, M, N, K, A, lda, mode, d);
    return run_planned(pl, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, d, stream,
                       false);
}

emu_status_t check_split_args(const void* X, int64_t rows, int64_t cols, int64_t ld, int trans,
                              const void* P0, const void* P1, const void* P2, int64_t ldp) {
    if (trans != 0 && trans != 1) return EMU_ERR_INVALID_VALUE;
    if (rows < 0 || cols < 0) return EMU_ERR_INVALID_VALUE;
    if (ld < 1 || ld < (trans ? rows : cols) || ldp < 1 || ldp < cols) return EMU_ERR_INVALID_VALUE;
    if (rows == 0 || cols == 0) return EMU_OK;
    if (!X || !P0 || !P1 || !P2) return EMU_ERR_INVALID_VALUE;
    return EMU_OK;
}

}  // namespace

// Device address of the sticky error word on the current device (nullptr if
// it cannot be resolved).  Used by entry points defined in other files.
int* device_error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    DeviceState* d = nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (current_device(&d) != EMU_OK) return nullptr;
    return d->err;
}

}  // namespace emu

using namespace emu;

extern "C" {

emu_status_t emu_sgemm(int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha,
                       const float* A, int64_t lda, const float* B, int64_t ldb, float beta,
                       float* C, int64_t ldc, int mode, emu_stream_t stream) {
    std::lock_guard<std::mutex> lock(g_mu);
    return sgemm_device(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, mode,
                        reinterpret_cast<cudaStream_t>(stream));
}

// emu_sgemm_host for large problems.  Host->device copies go on a copy
// stream in the order the GEMMs need them; each GEMM runs on the caller's
// stream as soon as its operands have landed, and each row chunk of C goes
// back on a second copy stream while the next chunk computes.  When op(B) is
// wide (the two-pass kernels, N >= 2 panels), the first row chunk of op(A)
// crosses first and is split once, then op(B) crosses in column panels, each
// split into its rows of B's pieces and multiplied by that first chunk as it
// lands, so that the tensor cores start after one panel rather than after
// all of B (on GB300 the link moves about 210 GB/s to the device: 8192^2
// FP32 take 1.3 ms).  The remaining row chunks then run full width with B's
// pieces split once, in chunks of about 48 MB, then 96 MB, then 48 MB again
// and a last one of 256 rows: the first lands soon after B, the middle ones
// make fewer and fuller launches, and the last one's copy back is the tail
// that nothing overlaps (measured at 8192^3: 1.8-2.3 % faster than equal
// chunks; the 256-row last chunk 1.6 % more, 5.68 against 5.77 ms a call
// on one box, a first chunk of 2560 rows 4.6 % slower).  Otherwise B
// crosses first, whole, and the first chunk splits it.  Row chunks of C are
// independent, so the result is what one call computes (up to the last
// wave's K split, which follows the tile count of each launch).
constexpr int64_t kHostPanelCols = 1024;    // op(B) columns per panel
constexpr int64_t kHostPanelRows = 2048;    // rows of the first chunk with panels
constexpr int64_t kHostChunkBytes = int64_t(48) << 20;   // op(A) and C bytes per later chunk

emu_status_t host_pipelined(int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha,
                            const float* A, int64_t lda, const float* B, int64_t ldb, float beta,
                            float* C, int64_t ldc, int mode, DeviceState* d, float* dA, float* dB,
                            float* dC, size_t b_bytes, cudaStream_t stream) {
    cudaError_t e = cudaSuccess;
    if (!d->s_in) {
        e = cudaStreamCreateWithFlags(&d->s_in, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&d->s_out, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d->ev_panel, cudaEventDisableTiming);
        for (int i = 0; i < kHostChunksMax && e == cudaSuccess; ++i) {
            e = cudaEventCreateWithFlags(&d->ev_in[i], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d->ev_done[i], cudaEventDisableTiming);
        }
        if (e != cudaSuccess) return from_cuda(e);
    }
    const Plan pl = plan_call(transA, M, N, K, dA, lda, mode, d);
    const bool panels = pl.mode != EMU_MODE_FP32_SIMT && pl.fused == 0 &&
                        N >= 2 * kHostPanelCols && b_bytes >= (size_t(16) << 20);
    // at most 64 panels: wider ones for very wide B (multiples of 256 columns)
    int64_t pw = kHostPanelCols;
    if (panels && (N + pw - 1) / pw > 64) pw = ((N + 63) / 64 + 255) / 256 * 256;

    // row chunks of whole 256-row tiles (at most kHostChunksMax): with panels
    // the first is kHostPanelRows rows; the rest about kHostChunkBytes of
    // op(A) and C each, or growing then shrinking after panels
    const int64_t row_bytes = (transA ? 1 : lda) * 4 * (transA ? K : 1) + N * 4;
    int64_t bounds[kHostChunksMax + 1];
    int nch = 0;
    bounds[0] = 0;
    int64_t m0 = 0;
    if (panels) {
        m0 = M < kHostPanelRows ? M : kHostPanelRows;
        bounds[++nch] = m0;
    }
    if (m0 < M) {
        const int64_t rest = M - m0;
        const int64_t cap = kHostChunksMax - nch;
        // rows of one kHostChunkBytes chunk, in whole tiles
        int64_t u = (kHostChunkBytes / row_bytes) / 256 * 256;
        u = u < 256 ? 256 : u;
        // after the panels, a last chunk of one tile row when the short
        // chunks are longer: its copy back is the tail that nothing overlaps
        const int64_t t = u > 256 ? 256 : 0;
        const int64_t mid = rest - 2 * u - t;
        const int64_t nmid = mid > 0 ? (mid + 2 * u - 1) / (2 * u) : 0;
        if (panels && mid > 0 && 2 + nmid + (t > 0 ? 1 : 0) <= cap) {
            // after the panels: a short chunk (it lands soon after B), double
            // chunks (fewer, fuller launches), a short one and the tile row
            const int64_t mc = ((mid + nmid - 1) / nmid + 255) / 256 * 256;
            bounds[++nch] = m0 + u;
            for (int64_t r = m0 + u; r < M - u - t; r += mc)
                bounds[++nch] = (M - u - t - r < mc) ? M - u - t : r + mc;
            if (t > 0) bounds[++nch] = M - t;
            bounds[++nch] = M;
        } else {
            int64_t n = (rest * row_bytes) / kHostChunkBytes;
            n = n < 2 ? 2 : n;
            n = n > cap ? cap : n;
            const int64_t mc = (((rest + n - 1) / n) + 255) / 256 * 256;
            for (int64_t r = m0; r < M; r += mc) bounds[++nch] = (M - r < mc) ? M : r + mc;
        }
    }

    // size the workspace for the largest chunk now: no reallocation (and no
    // loss of B's pieces) inside the loop; the layouts are run_two_pass's
    const int64_t ldp = plane_ld(K);
    const bool simt = pl.mode == EMU_MODE_FP32_SIMT;
    auto a_mn_rows = [&](int64_t rows) {
        return !simt && !pl.fused && mn_pieces(pl.mode, transA, K, rows);
    };
    const bool b_mn = !simt && !pl.fused && mn_pieces(pl.mode, !transB, K, N);
    const size_t b_region = simt ? 0 : (piece_bytes(pl.mode, b_mn, N, K) + 1023) / 1024 * 1024;
    if (!simt) {
        size_t a_max = 0;                    // the largest chunk's A pieces, in its layout
        for (int i = 0; i < nch; ++i) {
            const int64_t rows = bounds[i + 1] - bounds[i];
            const size_t a = piece_bytes(pl.mode, a_mn_rows(rows), rows, K);
            a_max = a > a_max ? a : a_max;
        }
        const size_t need = pl.fused ? piece_bytes(pl.mode, false, N, K) : b_region + a_max;
        emu_status_t st = ensure_buffer(&d->ws, &d->ws_bytes, need);
        if (st != EMU_OK) return st;
    }
    uint8_t* wb = static_cast<uint8_t*>(d->ws);
    uint8_t* wa = wb + b_region;
    // bytes from one row (K-major) or column (N-major) of B's pieces to the next
    const size_t es = simt ? 0 : mode_piece_bytes(pl.mode);
    const size_t prow = es * ldp;
    const int64_t ldbn = mn_ld(N);

    // the copy streams start after the caller's earlier work on its stream
    e = cudaEventRecord(d->ev_done[0], stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(d->s_in, d->ev_done[0], 0);
    if (e == cudaSuccess && b_bytes && !panels)
        e = cudaMemcpyAsync(dB, B, b_bytes, cudaMemcpyHostToDevice, d->s_in);
    emu_status_t st = EMU_OK;
    for (int i = 0; i < nch && e == cudaSuccess && st == EMU_OK; ++i) {
        const int64_t r0 = bounds[i], rows = bounds[i + 1] - bounds[i];
        if (transA == 0) {
            e = cudaMemcpyAsync(dA + r0 * lda, A + r0 * lda, size_t((rows - 1) * lda + K) * 4,
                                cudaMemcpyHostToDevice, d->s_in);
        } else {   // op(A)'s rows r0.. are columns of the stored K x M matrix
            e = cudaMemcpy2DAsync(dA + r0, size_t(lda) * 4, A + r0, size_t(lda) * 4,
                                  size_t(rows) * 4, size_t(K), cudaMemcpyHostToDevice, d->s_in);
        }
        const size_t c_chunk = size_t((rows - 1) * ldc + N) * 4;
        if (e == cudaSuccess && beta != 0.0f)
            e = cudaMemcpyAsync(dC + r0 * ldc, C + r0 * ldc, c_chunk, cudaMemcpyHostToDevice,
                                d->s_in);
        if (e == cudaSuccess) e = cudaEventRecord(d->ev_in[i], d->s_in);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, d->ev_in[i], 0);
        if (e != cudaSuccess) break;
        const float* Ai = transA ? dA + r0 : dA + r0 * lda;
        if (panels && i == 0) {
            const bool a_mn = a_mn_rows(rows);
            const PieceSet as{wa, a_mn ? mn_ld(rows) : ldp, 0, a_mn ? 1 : 0};
            {
                ProfScope ps(0, stream);
                e = a_mn ? launch_split_pieces(pl.mode, Ai, K, rows, lda, 0, wa, as.ld, stream)
                         : launch_split_pieces(pl.mode, Ai, rows, K, lda, transA, wa, ldp, stream);
            }
            for (int64_t j0 = 0; j0 < N && e == cudaSuccess && st == EMU_OK; j0 += pw) {
                const int64_t w = N - j0 < pw ? N - j0 : pw;
                // op(B)'s columns j0..j0+w: rows of B (transB) or a column block
                if (transB)
                    e = cudaMemcpyAsync(dB + j0 * ldb, B + j0 * ldb, size_t((w - 1) * ldb + K) * 4,
                                        cudaMemcpyHostToDevice, d->s_in);
                else
                    e = cudaMemcpy2DAsync(dB + j0, size_t(ldb) * 4, B + j0, size_t(ldb) * 4,
                                          size_t(w) * 4, size_t(K), cudaMemcpyHostToDevice,
                                          d->s_in);
                if (e == cudaSuccess) e = cudaEventRecord(d->ev_panel, d->s_in);
                if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, d->ev_panel, 0);
                if (e != cudaSuccess) break;
                {
                    // into rows j0.. of B's K-major pieces (planes N rows
                    // apart), or row-wise into columns j0.. of its N-major
                    // ones (planes K rows apart)
                    ProfScope ps(0, stream);
                    e = b_mn ? launch_split_pieces(pl.mode, dB + j0, K, w, ldb, 0, wb + j0 * es,
                                                   ldbn, stream, false, K)
                             : launch_split_pieces(pl.mode, transB ? dB + j0 * ldb : dB + j0, w, K,
                                                   ldb, !transB, wb + j0 * prow, ldp, stream,
                                                   false, N);
                }
                const PieceSet bs = b_mn ? PieceSet{wb + j0 * es, ldbn, K, 1}
                                         : PieceSet{wb + j0 * prow, ldp, N, 0};
                if (e == cudaSuccess)
                    st = gemm_on_pieces(pl.mode, as, bs, rows, w, K, alpha, beta, dC + j0, ldc, d,
                                        stream);
            }
        } else {
            st = run_planned(pl, transA, transB, rows, N, K, alpha, Ai, lda, dB, ldb, beta,
                             dC + r0 * ldc, ldc, d, stream, i > 0);
        }
        if (st != EMU_OK || e != cudaSuccess) break;
        e = cudaEventRecord(d->ev_done[i], stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(d->s_out, d->ev_done[i], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(C + r0 * ldc, dC + r0 * ldc, c_chunk, cudaMemcpyDeviceToHost,
                                d->s_out);
    }
    // wait for everything issued, whatever failed
    const cudaError_t e1 = cudaStreamSynchronize(d->s_in);
    const cudaError_t e2 = cudaStreamSynchronize(stream);
    const cudaError_t e3 = cudaStreamSynchronize(d->s_out);
    if (st != EMU_OK) return st;
    if (e == cudaSuccess) e = e1 != cudaSuccess ? e1 : (e2 != cudaSuccess ? e2 : e3);
    return from_cuda(e);
}

emu_status_t emu_sgemm_host(int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha,
                            const float* A, int64_t lda, const float* B, int64_t ldb, float beta,
                            float* C, int64_t ldc, int mode, emu_stream_t stream_) {
    std::lock_guard<std::mutex> lock(g_mu);
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    emu_status_t st = check_gemm_args(transA, transB, M, N, K, A, lda, B, ldb, beta, C, ldc, mode);
    if (st != EMU_OK) return st;
    if (M == 0 || N == 0) return EMU_OK;
    DeviceState* d = nullptr;
    st = current_device(&d);
    if (st != EMU_OK) return st;
    if (!workspace_fits(M, N, K)) return EMU_ERR_ALLOC;
    // stored extents: A is (transA ? K : M) rows of lda, B is (transB ? N : K)
    // rows of ldb; sizes that do not fit in 62 bits cannot be staged
    const int64_t a_rows = transA ? K : M, b_rows = transB ? N : K;
    size_t a_el = 0, b_el = 0, c_el = 0;
    if (K > 0 && (!fits_mul_add((uint64_t)(a_rows - 1), (uint64_t)lda, (uint64_t)(transA ? M : K), &a_el) ||
                  !fits_mul_add((uint64_t)(b_rows - 1), (uint64_t)ldb, (uint64_t)(transB ? K : N), &b_el)))
        return EMU_ERR_ALLOC;
    if (!fits_mul_add((uint64_t)(M - 1), (uint64_t)ldc, (uint64_t)N, &c_el) ||
        (a_el + b_el + c_el) > (size_t(1) << 60))
        return EMU_ERR_ALLOC;
    const size_t a_bytes = a_el * 4, b_bytes = b_el * 4, c_bytes = c_el * 4;
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    st = ensure_buffer(&d->stage, &d->stage_bytes, up(a_bytes) + up(b_bytes) + up(c_bytes));
    if (st != EMU_OK) return st;
    uint8_t* base = static_cast<uint8_t*>(d->stage);
    float* dA = reinterpret_cast<float*>(base);
    float* dB = reinterpret_cast<float*>(base + up(a_bytes));
    float* dC = reinterpret_cast<float*>(base + up(a_bytes) + up(b_bytes));
    const size_t moved = a_bytes + b_bytes + c_bytes * (beta != 0.0f ? 2 : 1);
    if (K > 0 && alpha != 0.0f && M >= 512 && moved >= (size_t(64) << 20))
        return host_pipelined(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, mode,
                              d, dA, dB, dC, b_bytes, stream);
    cudaError_t e = cudaSuccess;
    if (a_bytes) e = cudaMemcpyAsync(dA, A, a_bytes, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess && b_bytes) e = cudaMemcpyAsync(dB, B, b_bytes, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess && beta != 0.0f)
        e = cudaMemcpyAsync(dC, C, c_bytes, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return from_cuda(e);
    st = sgemm_device(transA, transB, M, N, K, alpha, K > 0 ? dA : nullptr, lda,
                      K > 0 ? dB : nullptr, ldb, beta, dC, ldc, mode, stream);
    if (st != EMU_OK) return st;
    e = cudaMemcpyAsync(C, dC, c_bytes, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    return from_cuda(e);
}

emu_status_t emu_sgemm_bsplit(int transA, int64_t M, int64_t N, int64_t K, float alpha,
                              const float* A, int64_t lda, const void* Bp, int64_t ldbp,
                              float beta, float* C, int64_t ldc, int mode,
                              emu_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (transA != 0 && transA != 1) return EMU_ERR_INVALID_VALUE;
    if (!valid_mode(mode) || mode == EMU_MODE_FP32_SIMT) return EMU_ERR_INVALID_VALUE;
    if (M < 0 || N < 0 || K < 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
        return EMU_ERR_INVALID_VALUE;
    if (lda < 1 || lda < (transA ? M : K) || ldc < 1 || ldc < N) return EMU_ERR_INVALID_VALUE;
    // the pieces are read by TMA: 16-byte aligned base and rows
    if (ldbp < K || ldbp < 1 || (ldbp % 8) != 0 || ldbp > INT32_MAX) return EMU_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return EMU_OK;
    if (C == nullptr) return EMU_ERR_INVALID_VALUE;
    if (K > 0 && (A == nullptr || Bp == nullptr || (reinterpret_cast<uintptr_t>(Bp) & 15) != 0))
        return EMU_ERR_INVALID_VALUE;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!workspace_fits(M, N, K)) return EMU_ERR_ALLOC;
    DeviceState* d = nullptr;
    emu_status_t st = current_device(&d);
    if (st != EMU_OK) return st;
    if (K == 0 || alpha == 0.0f) {
        ProfScope ps(4, stream);
        return from_cuda(launch_scale(M, N, beta, C, ldc, stream));
    }
    const Plan pl = plan_call(transA, M, N, K, A, lda, mode, d, true);
    BPieces bext;
    bext.p = Bp;
    bext.ld = ldbp;
    // transB and B are not used: op(B)^T's pieces are given
    return run_planned(pl, transA, 0, M, N, K, alpha, A, lda, nullptr, 0, beta, C, ldc, d, stream,
                       false, bext);
}

emu_status_t emu_split_bf16x3(const float* X, int64_t rows, int64_t cols, int64_t ld, int trans,
                              uint16_t* P0, uint16_t* P1, uint16_t* P2, int64_t ldp,
                              emu_stream_t stream) {
    emu_status_t st = check_split_args(X, rows, cols, ld, trans, P0, P1, P2, ldp);
    if (st != EMU_OK || rows == 0 || cols == 0) return st;
    DeviceState* d = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        st = current_device(&d);
    }
    if (st != EMU_OK) return st;
    return from_cuda(launch_split_bf16x3(X, rows, cols, ld, trans, P0, P1, P2, ldp,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

emu_status_t emu_split_tf32x2(const float* X, int64_t rows, int64_t cols, int64_t ld, int trans,
                              float* HI, float* LO, int64_t ldp, emu_stream_t stream) {
    emu_status_t st = check_split_args(X, rows, cols, ld, trans, HI, LO, LO, ldp);
    if (st != EMU_OK || rows == 0 || cols == 0) return st;
    DeviceState* d = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        st = current_device(&d);
    }
    if (st != EMU_OK) return st;
    return from_cuda(launch_split_tf32x2(X, rows, cols, ld, trans, HI, LO, ldp,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

emu_status_t emu_split_tf32x2_scaled(const float* X, int64_t rows, int64_t cols, int64_t ld,
                                     int trans, float* HI, float* LO, int64_t ldp,
                                     emu_stream_t stream) {
    emu_status_t st = check_split_args(X, rows, cols, ld, trans, HI, LO, LO, ldp);
    if (st != EMU_OK || rows == 0 || cols == 0) return st;
    DeviceState* d = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        st = current_device(&d);
    }
    if (st != EMU_OK) return st;
    return from_cuda(launch_split_tf32x2(X, rows, cols, ld, trans, HI, LO, ldp,
                                         reinterpret_cast<cudaStream_t>(stream), 2048.0f));
}

emu_status_t emu_set_path(int path) {
    if (path != EMU_PATH_AUTO && path != EMU_PATH_TWOPASS && path != EMU_PATH_FUSED &&
        path != EMU_PATH_FUSED_TMEM)
        return EMU_ERR_INVALID_VALUE;
    std::lock_guard<std::mutex> lock(g_mu);
    g_path = path;
    return EMU_OK;
}

int emu_get_path(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_path < 0) g_path = read_path_env();
    return g_path;
}

emu_status_t emu_set_strategy(int strategy) {
    if (strategy != EMU_STRATEGY_EAGER && strategy != EMU_STRATEGY_PERFORMANT)
        return EMU_ERR_INVALID_VALUE;
    std::lock_guard<std::mutex> lock(g_mu);
    g_strategy = strategy;
    return EMU_OK;
}

int emu_get_strategy(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_strategy < 0) g_strategy = read_strategy_env();
    return g_strategy;
}

int emu_choose_mode(int64_t M, int64_t N, int64_t K, int mode, int strategy, int sms) {
    if (!valid_mode(mode) || M < 0 || N < 0 || K < 0) return -1;
    if (strategy < 0) strategy = emu_get_strategy();
    if (strategy != EMU_STRATEGY_EAGER && strategy != EMU_STRATEGY_PERFORMANT) return -1;
    if (sms <= 0) {
        DeviceState* d = nullptr;
        std::lock_guard<std::mutex> lock(g_mu);
        if (current_device(&d) != EMU_OK) return -1;
        sms = d->sms;
    }
    return choose_mode(M, N, K, mode, strategy == EMU_STRATEGY_PERFORMANT, sms);
}

double emu_predict_us(int64_t M, int64_t N, int64_t K, int mode, int sms) {
    if (!valid_mode(mode) || M < 0 || N < 0 || K < 0 || sms <= 0) return -1.0;
    return mode == EMU_MODE_FP32_SIMT ? predict_simt_us(M, N, K, sms)
                                      : predict_tc_us(M, N, K, mode, sms);
}

size_t emu_workspace_size(int64_t M, int64_t N, int64_t K, int mode) {
    if (M <= 0 || N <= 0 || K <= 0 || mode == EMU_MODE_FP32_SIMT) return 0;
    if (!valid_mode(mode) || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return 0;
    if (!workspace_fits(M, N, K)) return SIZE_MAX;
    // B's pieces, then A's at a 1 KB boundary (run_two_pass), each in the
    // larger of its layouts: the transposes decide which one a call takes
    auto most = [&](int64_t rows) {
        const size_t k_major = piece_bytes(mode, false, rows, K);
        const size_t mn = mn_pieces(mode, true, K, rows) ? piece_bytes(mode, true, rows, K) : 0;
        return k_major > mn ? k_major : mn;
    };
    return (most(N) + 1023) / 1024 * 1024 + most(M);
}

emu_status_t emu_get_last_device_error(void) {
    int v = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return from_cuda(e);
    e = cudaMemcpyFromSymbol(&v, g_emu_error, sizeof(int));
    if (e != cudaSuccess) return from_cuda(e);
    return static_cast<emu_status_t>(v);
}

emu_status_t emu_clear_device_error(void) {
    const int zero = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_emu_error, &zero, sizeof(int));
    return from_cuda(e);
}

emu_status_t emu_selftest_timeout(int limit_us, emu_stream_t stream) {
    if (limit_us < 1 || limit_us > 1000000) return EMU_ERR_INVALID_VALUE;
    DeviceState* d = nullptr;
    emu_status_t st;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        st = current_device(&d);
    }
    if (st != EMU_OK) return st;
    cudaError_t e = launch_timeout_probe(d->err, (uint64_t)limit_us * 1000ull,
                                         reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return from_cuda(e);
    return emu_get_last_device_error();
}

emu_status_t emu_profile_enable(int on) {
    std::lock_guard<std::mutex> lock(g_mu);
    for (auto& r : g_prof_pending) {
        g_event_pool.push_back(r.start);
        g_event_pool.push_back(r.stop);
    }
    g_prof_pending.clear();
    for (int i = 0; i < 5; ++i) { g_prof_launches[i] = 0; g_prof_ms[i] = 0.0; }
    g_prof_on = on != 0;
    return EMU_OK;
}

emu_status_t emu_profile_read(int kind, int64_t* launches, double* total_ms) {
    if (kind < 0 || kind >= 5 || !launches || !total_ms) return EMU_ERR_INVALID_VALUE;
    std::lock_guard<std::mutex> lock(g_mu);
    for (auto& r : g_prof_pending) {
        cudaError_t e = cudaEventSynchronize(r.stop);
        if (e != cudaSuccess) return from_cuda(e);
        float ms = 0.0f;
        cudaEventElapsedTime(&ms, r.start, r.stop);
        g_prof_launches[r.kind] += 1;
        g_prof_ms[r.kind] += ms;
        g_event_pool.push_back(r.start);
        g_event_pool.push_back(r.stop);
    }
    g_prof_pending.clear();
    *launches = g_prof_launches[kind];
    *total_ms = g_prof_ms[kind];
    return EMU_OK;
}

const char* emu_last_cuda_error(void) { return cudaGetErrorName(g_last_cuda_error); }

const char* emu_status_string(emu_status_t s) {
    switch (s) {
        case EMU_OK: return "EMU_OK";
        case EMU_ERR_INVALID_VALUE: return "EMU_ERR_INVALID_VALUE";
        case EMU_ERR_ARCH: return "EMU_ERR_ARCH";
        case EMU_ERR_ALLOC: return "EMU_ERR_ALLOC";
        case EMU_ERR_LAUNCH: return "EMU_ERR_LAUNCH";
        case EMU_ERR_TIMEOUT: return "EMU_ERR_TIMEOUT";
        case EMU_ERR_CUDA: return "EMU_ERR_CUDA";
    }
    return "EMU_ERR_UNKNOWN";
}

emu_status_t emu_shutdown(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    for (int i = 0; i < kMaxDevices; ++i) {
        DeviceState& d = g_dev[i];
        if (!d.ws && !d.stage && !d.s_in && !d.part && !d.flags) continue;
        cudaSetDevice(i);
        if (d.ws) cudaFree(d.ws);
        if (d.stage) cudaFree(d.stage);
        d.ws = d.stage = nullptr;
        d.ws_bytes = d.stage_bytes = 0;
        if (d.part) cudaFree(d.part);
        if (d.flags) cudaFree(d.flags);
        d.part = nullptr;
        d.part_bytes = 0;
        d.flags = nullptr;
        if (d.s_in) {
            cudaStreamDestroy(d.s_in);
            cudaStreamDestroy(d.s_out);
            for (int j = 0; j < kHostChunksMax; ++j) {
                if (d.ev_in[j]) cudaEventDestroy(d.ev_in[j]);
                if (d.ev_done[j]) cudaEventDestroy(d.ev_done[j]);
                d.ev_in[j] = d.ev_done[j] = nullptr;
            }
            if (d.ev_panel) cudaEventDestroy(d.ev_panel);
            d.ev_panel = nullptr;
            d.s_in = d.s_out = nullptr;
        }
    }
    cudaSetDevice(cur);
    return EMU_OK;
}

int emu_version(void) { return 100; }

}  // extern "C"
