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
//   tensor-core path:  fixed (three launches) + the split's bytes
//                      + waves x (wave cost + K blocks x block cost)
//   FP32 SIMT kernel:  waves x (wave cost + K x per-K cost)
// where a wave is one round of output tiles over the GPU (256 x 256 tiles on
// SM pairs for the tensor core, 128 x 128 tiles for SIMT).
#include "emu_internal.h"

namespace emu {

namespace {

// Fitted on GB300 (152 SMs), microseconds, by least squares on relative error
// over 86 shapes (M, N in 64..4096, K in 16..4096, and the MLIP layer
// shapes), CUDA-graph replay of 20 calls each, with the second split and the
// GEMM launched as programmatic dependents.  Median model error 5 % (BF16x9,
// TF32x3), 3 % (SIMT); the choice named the faster kernel in all 86 shapes.
struct TcFit {
    double fixed_us;      // three launches (two splits, the GEMM), partly overlapped
    double us_per_mb;     // split traffic, per MB read and written
    double wave_us;       // per wave of tiles: pipeline fill and epilogue
    double block_us;      // per K block (64 BF16 / 32 TF32 elements) per wave
};

TcFit tc_fit(int mode) {
    // BF16x9 and TF32x3 fitted; the other modes scale the K-block cost by
    // their measured 8192^3 GEMM time relative to the fitted mode's
    // (BF16x3 1.849 / 4.708 ms, TF32 1.457 / 3.348, Ootomo-Yokota 3.426 / 3.348).
    switch (mode) {
        case kModeBf16x9: return {6.76, 0.141, 2.72, 2.27};
        case kModeBf16x3: return {6.76, 0.141, 2.72, 0.89};
        case kModeTf32x3: return {6.19, 0.262, 3.61, 0.89};
        case kModeTf32x3Oy: return {6.19, 0.262, 3.61, 0.91};
        case kModeTf32: return {6.19, 0.262, 3.61, 0.39};
        default: return {0, 0, 0, 0};
    }
}

// FP32 SIMT kernel: 128 x 128 tiles, two resident per SM.  A K step costs
// less when the tiles fit on the SMs one each.
constexpr double kSimtWaveUs = 3.25;
constexpr double kSimtKUsAlone = 0.145;
constexpr double kSimtKUsShared = 0.260;
constexpr int kSimtCtasPerSm = 2;

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

double predict_tc_us(int64_t M, int64_t N, int64_t K, int mode, int sms) {
    const TcFit f = tc_fit(mode);
    const int pieces = mode_pieces(mode), esz = mode_piece_bytes(mode);
    const double split_mb = double(M + N) * double(K) * (4.0 + pieces * esz) * 1e-6;
    // N <= 128 runs 128-wide tiles (BF16x9, TF32x3): half the MMA work each
    const bool narrow = N <= 128 && (mode == kModeBf16x9 || mode == kModeTf32x3);
    const int64_t bn = narrow ? 128 : 256;
    const int64_t tiles = cdiv(M, 256) * cdiv(N, bn);
    const int64_t waves = cdiv(tiles, sms / 2 > 0 ? sms / 2 : 1);
    const int64_t kb = cdiv(K, mode_is_tf32(mode) ? 32 : 64);
    const double block = f.block_us * (narrow ? 0.5 : 1.0);
    return f.fixed_us + split_mb * f.us_per_mb + double(waves) * (f.wave_us + double(kb) * block);
}

double predict_simt_us(int64_t M, int64_t N, int64_t K, int sms) {
    const int64_t tiles = cdiv(M, 128) * cdiv(N, 128);
    const int64_t waves = cdiv(tiles, int64_t(sms) * kSimtCtasPerSm);
    const double k_us = tiles <= sms ? kSimtKUsAlone : kSimtKUsShared;
    return double(waves) * (kSimtWaveUs + double(K) * k_us);
}

int choose_mode(int64_t M, int64_t N, int64_t K, int mode, int performant, int sms) {
    if (!performant || mode == kModeFp32Simt) return mode;
    if (M <= 0 || N <= 0 || K <= 0) return mode;     // nothing to multiply
    return predict_simt_us(M, N, K, sms) < predict_tc_us(M, N, K, mode, sms) ? kModeFp32Simt
                                                                               : mode;
}

}  // namespace emu
