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
//                      + rounds x round cost + K blocks x block cost
//                      + hand-overs x hand-over cost
//   FP32 SIMT kernel:  waves x (wave cost + K x per-K cost)
// where a round is one set of 256-wide output tiles over the SM pairs; the
// rounds, the K blocks of the longest cluster and its hand-overs follow the
// GEMM's own tail plan (schedule.h), so that a few deep tiles spread over
// every cluster are estimated as they run.  The SIMT kernel's waves are 128 x
// 128 tiles, two per SM.
#include "emu_internal.h"
#include "schedule.h"

namespace emu {

namespace {

// Fitted on GB300 (152 SMs), microseconds, by least squares on relative error
// over 96 shapes (M, N in 64..4096, K in 16..4096, the MLIP layer shapes, and
// ten deep-K shapes up to 256 x 256 x 262144), CUDA-graph replay of 20 calls
// each.  Median model error 6.7 % (BF16x9), 7.6 % (TF32x3), 2.6 % (SIMT);
// the choice named the faster kernel in 94 of the 96 shapes (the two misses
// within 1 % of a tie).
struct TcFit {
    double fixed_us;      // three launches (two splits, the GEMM), partly overlapped
    double us_per_mb;     // split traffic, per MB read and written
    double round_us;      // per round of tiles: pipeline fill and epilogue
    double block_us;      // per K block (64 BF16 / 32 TF32 elements) of the longest cluster
    double handover_us;   // per hand-over of a split tile's part to its owner
};

TcFit tc_fit(int mode) {
    // BF16x9 and TF32x3 fitted; the other modes scale the K-block cost by
    // their measured 8192^3 GEMM time relative to the fitted mode's
    // (BF16x3 1.849 / 4.708 ms, TF32 1.457 / 3.348, Ootomo-Yokota 3.426 / 3.348).
    switch (mode) {
        case kModeBf16x9: return {7.07, 0.1345, 2.51, 2.586, 7.52};
        case kModeBf16x3: return {7.07, 0.1345, 2.51, 2.586 * 1.849 / 4.708, 7.52};
        case kModeTf32x3: return {6.50, 0.1799, 3.31, 1.038, 8.73};
        case kModeTf32x3Oy: return {6.50, 0.1799, 3.31, 1.038 * 3.426 / 3.348, 8.73};
        case kModeTf32: return {6.50, 0.1799, 3.31, 1.038 * 1.457 / 3.348, 8.73};
        default: return {0, 0, 0, 0, 0};
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
    const double half = narrow ? 0.5 : 1.0;
    const int64_t bn = narrow ? 128 : 256;
    const int64_t tiles = cdiv(M, 256) * cdiv(N, bn);
    const int64_t res = sms / 2 > 0 ? sms / 2 : 1;
    const int64_t kb = cdiv(K, mode_is_tf32(mode) ? 32 : 64);
    // the tail plan of the GEMM (schedule.h): rounds, the longest cluster's
    // K blocks and its hand-overs
    const int fix2 = handover_half_blocks(mode);
    int tt = 0, tc = 0;
    if (tiles <= INT32_MAX && kb <= INT32_MAX)
        sched_plan_tail(static_cast<int>(tiles), static_cast<int>(kb), static_cast<int>(res), fix2,
                        &tt, &tc);
    double rounds, blocks, hands = 0.0;
    if (tt == 0) {
        rounds = double(cdiv(tiles, res));
        blocks = rounds * double(kb);
    } else {
        const int64_t whole = (tiles - tt) / res;
        const int64_t smax = res / tt < kb / 2 ? res / tt : kb / 2;
        const double rd = double((fix2 + 2) / 3) / double(fix2 > 0 ? fix2 : 1);
        rounds = double(whole + 1);
        if (tc % tt == 0 && tc / tt <= smax) {                  // aligned parts
            const int64_t s = tc / tt;
            blocks = double(whole * kb + cdiv(kb, s));
            hands = 1.0 + double(s > 8 ? s - 8 : 0) * rd;
        } else {                                                // stream-K ranges
            const int64_t parts = cdiv(tc, tt);
            blocks = double(whole * kb + cdiv(int64_t(tt) * kb, tc));
            hands = 2.0 + double(parts > 8 ? parts - 8 : 0) * rd;
        }
    }
    return f.fixed_us + split_mb * f.us_per_mb + rounds * f.round_us +
           blocks * f.block_us * half + hands * f.handover_us * half;
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
