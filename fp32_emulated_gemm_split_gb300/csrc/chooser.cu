// chooser.cu -- the PERFORMANT strategy: run an emulated mode only where it
// is predicted to be faster than the plain FP32 kernel.
//
// The discuss.pytorch.kr page (section "PyTorch에서 직접 써 보려면") and the
// NVIDIA blog post (MD-step results) describe two strategies for cuBLAS's
// BF16x9: "performant" uses the emulation only where a speedup is expected,
// "eager" whenever the operation supports it.  This library's choice is a
// small time model of its own kernels, one estimate per path, with constants
// fitted to a shape sweep on GB300 (device time per call, CUDA-graph replay,
// so host overhead is left out):
//   tensor-core path:  two split launches + the split's HBM bytes
//                      + one GEMM launch + waves x (tile cost + K blocks x block cost)
//   FP32 SIMT kernel:  one launch + waves x (tile cost + K x per-K cost)
// where a wave is one round of output tiles over the GPU (256 x 256 tiles on
// SM pairs for the tensor core, 128 x 128 tiles for SIMT).
#include "emu_internal.h"

namespace emu {

namespace {

// Fitted on GB300 (152 SMs) -- microseconds.
constexpr double kLaunchUs = 2.5;          // one kernel launch and its gap, in a graph
constexpr double kHbmBytesPerUs = 5.5e6;   // split kernels' effective bandwidth
constexpr double kTcTileUs = 3.0;          // pipeline fill and epilogue of one tile
constexpr double kSimtTileUs = 1.0;
constexpr double kSimtKUs = 0.25;          // one K step of a 128 x 128 SIMT tile
constexpr int kSimtCtasPerSm = 2;

// Tensor-core time of one K block (64 BF16 / 32 TF32 elements) of a
// 256 x 256 tile on an SM pair, from the 8192^3 runs of each mode.
double block_us(int mode) {
    switch (mode) {
        case kModeBf16x9: return 2.63;
        case kModeTf32x3: return 0.93;
        case kModeTf32x3Oy: return 0.95;
        case kModeBf16x3: return 1.46;
        case kModeTf32: return 0.41;
        default: return 0.0;
    }
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

double predict_tc_us(int64_t M, int64_t N, int64_t K, int mode, int sms) {
    const int pieces = mode_pieces(mode), esz = mode_piece_bytes(mode);
    const double split_bytes = double(M + N) * double(K) * (4.0 + pieces * esz);
    const int64_t tiles = cdiv(M, 256) * cdiv(N, 256);
    const int64_t waves = cdiv(tiles, sms / 2 > 0 ? sms / 2 : 1);
    const int64_t kb = cdiv(K, mode_is_tf32(mode) ? 32 : 64);
    return 3 * kLaunchUs + split_bytes / kHbmBytesPerUs +
           double(waves) * (kTcTileUs + double(kb) * block_us(mode));
}

double predict_simt_us(int64_t M, int64_t N, int64_t K, int sms) {
    const int64_t tiles = cdiv(M, 128) * cdiv(N, 128);
    const int64_t waves = cdiv(tiles, int64_t(sms) * kSimtCtasPerSm);
    return kLaunchUs + double(waves) * (kSimtTileUs + double(K) * kSimtKUs);
}

int choose_mode(int64_t M, int64_t N, int64_t K, int mode, int performant, int sms) {
    if (!performant || mode == kModeFp32Simt) return mode;
    if (M <= 0 || N <= 0 || K <= 0) return mode;     // nothing to multiply
    return predict_simt_us(M, N, K, sms) < predict_tc_us(M, N, K, mode, sms) ? kModeFp32Simt
                                                                               : mode;
}

}  // namespace emu
