// noalloc.cu -- emu_sgemm_noalloc: the two-pass emulated GEMM for callers
// that cannot allocate device memory.
//
// emu_sgemm keeps the split pieces of A and B in a workspace it allocates
// (and grows) with cudaMalloc.  Some callers cannot let a library do that:
// code whose device memory is owned entirely by another allocator or a fixed
// memory budget (a framework's caching allocator, a service that reserves
// its memory up front), where an extra cudaMalloc can fail or break the
// owner's accounting; and code that cannot afford the device-wide
// synchronisation that cudaMalloc / cudaFree impose in the middle of its
// stream work.  For them this file holds the pieces in a fixed array in
// device memory instead, reserved when the library's device code is loaded
// on a GPU and kept until the process exits, so a call allocates nothing.
//
// The array is shared by every call on a device: calls whose work overlaps
// on the GPU (different streams, or host threads without ordering) race on
// it and must be serialised by the caller.  Nothing in it needs to start at
// zero: each call's split kernels write every element its GEMM kernel reads
// (the tensor maps stop at K and at the matrix rows, and read zeros beyond
// them), so the contents left by the previous call do not matter.
#include <cstring>
#include <mutex>

#include "emu_device.cuh"
#include "emu_sgemm.h"

namespace emu {
namespace {

constexpr size_t kNoAllocBytes = size_t(64) << 20;      // 64 MiB
constexpr int kMaxDev = 64;

// The fixed scratch: split pieces of op(A) (M x ldp per piece), then of
// op(B)^T (N x ldp per piece) at the next 1 KB boundary.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocBytes];

struct Slot {
    void* scratch = nullptr;   // device address of g_noalloc_scratch on this device
    int* err = nullptr;        // device address of the library's error word
    int sms = 0;
    bool ready = false;
};

std::mutex g_noalloc_mu;
Slot g_slot[kMaxDev];

// Once per device, with that device current: check the architecture and
// resolve the array's device address.  (In host code the array's name is
// only a host-side stand-in for the symbol, never a device pointer.)
emu_status_t setup_current_device(Slot** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return EMU_ERR_CUDA;
    Slot& s = g_slot[dev];
    if (!s.ready) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (!(major == 10 && minor == 3)) return EMU_ERR_ARCH;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return EMU_ERR_CUDA;
        }
        int* err = device_error_word();
        if (err == nullptr) return EMU_ERR_CUDA;
        cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, dev);
        s.scratch = p;
        s.err = err;
        s.ready = true;
    }
    *out = &s;
    return EMU_OK;
}

typedef CUresult (*EncodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    }
    return fn;
}

// 3-D map (K, rows, piece) over pieces stored row-major with row stride ld.
bool piece_map(CUtensorMap* map, void* base, bool fp32, int64_t rows, int64_t K, int64_t ld,
               int pieces, int box_k, int box_rows) {
    EncodeTiled enc = encoder();
    if (!enc) return false;
    const int es = fp32 ? 4 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)rows, (cuuint64_t)pieces};
    cuuint64_t strides[2] = {(cuuint64_t)(ld * es), (cuuint64_t)(rows * ld * es)};
    cuuint32_t box[3] = {(cuuint32_t)box_k, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
               base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

emu_status_t status_of(cudaError_t e) {
    if (e == cudaSuccess) return EMU_OK;
    if (e == cudaErrorLaunchOutOfResources || e == cudaErrorInvalidConfiguration ||
        e == cudaErrorLaunchFailure || e == cudaErrorNoKernelImageForDevice)
        return EMU_ERR_LAUNCH;
    return EMU_ERR_CUDA;
}

}  // namespace
}  // namespace emu

using namespace emu;

extern "C" emu_status_t emu_sgemm_noalloc(int transA, int transB, int64_t M, int64_t N,
                                          int64_t K, float alpha, const float* A, int64_t lda,
                                          const float* B, int64_t ldb, float beta, float* C,
                                          int64_t ldc, int mode, emu_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    // the same argument rules as emu_sgemm
    if ((transA != 0 && transA != 1) || (transB != 0 && transB != 1)) return EMU_ERR_INVALID_VALUE;
    if (!valid_mode(mode)) return EMU_ERR_INVALID_VALUE;
    if (M < 0 || N < 0 || K < 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
        return EMU_ERR_INVALID_VALUE;
    if (lda < 1 || lda < (transA ? M : K) || ldb < 1 || ldb < (transB ? K : N) || ldc < 1 ||
        ldc < N)
        return EMU_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return EMU_OK;
    if (C == nullptr || (K > 0 && (A == nullptr || B == nullptr))) return EMU_ERR_INVALID_VALUE;

    const bool tf32 = mode_is_tf32(mode);
    const int pieces = mode_pieces(mode), es = mode_piece_bytes(mode);
    const int64_t ldp = plane_ld(K);
    const bool uses_scratch = mode != EMU_MODE_FP32_SIMT && K > 0 && alpha != 0.0f;
    // Bytes of one row of pieces (at most 3 * 4 * (2^31 + 7), no overflow).
    // M + N rows must fit before any product of sizes is formed: with M, N
    // and K near INT32_MAX, (M + N) * row_bytes would wrap past 2^64.
    const size_t row_bytes = (size_t)pieces * es * (size_t)ldp;
    size_t a_region = 0;
    if (uses_scratch) {
        if ((size_t)M + (size_t)N > kNoAllocBytes / row_bytes) return EMU_ERR_INVALID_VALUE;
        a_region = ((size_t)M * row_bytes + 1023) / 1024 * 1024;
        if (a_region + (size_t)N * row_bytes > kNoAllocBytes) return EMU_ERR_INVALID_VALUE;
    }

    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    Slot* s = nullptr;
    emu_status_t st = setup_current_device(&s);
    if (st != EMU_OK) return st;
    if (K == 0 || alpha == 0.0f) return status_of(launch_scale(M, N, beta, C, ldc, stream));
    if (mode == EMU_MODE_FP32_SIMT)
        return status_of(launch_gemm_simt(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C,
                                          ldc, stream));

    uint8_t* wa = static_cast<uint8_t*>(s->scratch);
    uint8_t* wb = wa + a_region;
    cudaError_t e = launch_split_pieces(mode, A, M, K, lda, transA, wa, ldp, stream);
    if (e == cudaSuccess) e = launch_split_pieces(mode, B, N, K, ldb, !transB, wb, ldp, stream);
    if (e != cudaSuccess) return status_of(e);

    const int box_k = tf32 ? kTcBKBytes / 4 : kTcBKBytes / 2;
    CUtensorMap mapA, mapB;
    if (!piece_map(&mapA, wa, tf32, M, K, ldp, pieces, box_k, 128) ||
        !piece_map(&mapB, wb, tf32, N, K, ldp, pieces, box_k, 128))
        return EMU_ERR_CUDA;
    TcGemmParams p = {};
    p.err = s->err;
    p.M = (int)M; p.N = (int)N; p.K = (int)K;
    p.num_kb = (int)((K + box_k - 1) / box_k);
    p.tiles_m = (int)((M + 255) / 256);
    p.tiles_n = (int)((N + 255) / 256);
    p.alpha = alpha; p.beta = beta; p.C = C; p.ldc = ldc;
    p.tma_store = 0;                         // C stored directly by the epilogue warps
    return status_of(launch_gemm_kblock(mode, 256, 0, mapA, mapB, mapB, p, s->sms, stream));
}
