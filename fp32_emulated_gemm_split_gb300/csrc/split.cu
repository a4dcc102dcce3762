// split.cu -- the split/pack step of the two-pass path: FP32 op(X) -> BF16
// pieces (BF16x9) or TF32 pieces (TF32x3), written row-major with a padded
// row stride so that the GEMM can stage them with TMA.
//
// The split itself is x = x0 + 2^-8 x1 + 2^-16 x2 ("Blackwell의 BF16x9"
// section of the discuss.pytorch.kr page on the method; Figure 1 of the
// NVIDIA blog post "Unlocking Tensor Core Performance for Machine Learning
// Interatomic Potentials") and x = hi + lo (Figure 2 of that post).  These
// kernels are bound by HBM bandwidth: BF16x9 reads 4 bytes and writes 6 bytes
// per element, TF32x3 reads 4 and writes 8.  A null last plane (P2, LO) skips
// its writes: the two-piece BF16 and single-pass TF32 modes do not read it.
// The Ootomo-Yokota variant scales the TF32 residual by 2^11 (lo_scale)
// before rounding it.
#include <atomic>

#include "emu_device.cuh"

namespace emu {
namespace {

// ------------------------------------------------------ row-wise (no transpose)

// Each thread splits 8 consecutive elements of one row: two 16-byte loads,
// one 16-byte store per piece.  Requires 16-byte aligned rows in and out.
// U groups per thread per step, all loaded before any is split: with U = 1
// each thread keeps one 32-byte read in flight, too few to cover HBM's
// latency.  Measured on GB300 (an L2 flush before each launch): 8192^2 115.3
// / 111.3 / 109.2 us for U = 1 / 2 / 4 (U = 4: 6.15 TB/s, the speed of a
// plain stream with the same 4-byte-read, 6-byte-write mix); 1.1M x 256
// 480 / 451 / 442 us; 12288 x 256 10.9 us with U = 1, 12.9 with U = 4 (too
// few groups to go round), so the launcher keeps U = 1 for small splits.
template <int U>
__global__ void __launch_bounds__(256) split3_rows_vec8(const float* __restrict__ X, int64_t rows,
                                                        int64_t cols, int64_t ld,
                                                        uint16_t* __restrict__ P0,
                                                        uint16_t* __restrict__ P1,
                                                        uint16_t* __restrict__ P2, int64_t ldp) {
    griddep_launch_dependents();
    const int64_t groups = cols / 8;
    const int64_t total = rows * groups;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t t0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t0 < total; t0 += U * stride) {
        float4 a[U], b[U];
        int64_t o[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t t = t0 + u * stride;
            if (t < total) {
                const int64_t r = t / groups;
                const int64_t c = (t - r * groups) * 8;
                const float4* src = reinterpret_cast<const float4*>(X + r * ld + c);
                a[u] = __ldcs(src);
                b[u] = __ldcs(src + 1);
                o[u] = r * ldp + c;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (t0 + u * stride < total) {
                uint4 o0, o1, o2;
                split_bf16x3_pair(a[u].x, a[u].y, o0.x, o1.x, o2.x);
                split_bf16x3_pair(a[u].z, a[u].w, o0.y, o1.y, o2.y);
                split_bf16x3_pair(b[u].x, b[u].y, o0.z, o1.z, o2.z);
                split_bf16x3_pair(b[u].z, b[u].w, o0.w, o1.w, o2.w);
                *reinterpret_cast<uint4*>(P0 + o[u]) = o0;
                *reinterpret_cast<uint4*>(P1 + o[u]) = o1;
                if (P2) *reinterpret_cast<uint4*>(P2 + o[u]) = o2;
            }
        }
    }
    griddep_wait();          // see launch_pdl: complete only after the kernel ahead
}

// Any shape and alignment: one element per thread.
__global__ void __launch_bounds__(256) split3_rows_scalar(const float* __restrict__ X, int64_t rows,
                                                          int64_t cols, int64_t ld,
                                                          uint16_t* __restrict__ P0,
                                                          uint16_t* __restrict__ P1,
                                                          uint16_t* __restrict__ P2, int64_t ldp) {
    griddep_launch_dependents();
    const int64_t total = rows * cols;
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = t / cols;
        const int64_t c = t - r * cols;
        uint16_t h0, h1, h2;
        split_bf16x3(X[r * ld + c], h0, h1, h2);
        const int64_t o = r * ldp + c;
        P0[o] = h0; P1[o] = h1;
        if (P2) P2[o] = h2;
    }
    griddep_wait();          // see launch_pdl: complete only after the kernel ahead
}

// TF32 pieces, 4 consecutive elements per group, U groups per thread per
// step as above (8192^2: 158 / 150 / 140 us for U = 1 / 2 / 4; 1.1M x 256:
// 644 / 609 / 578 us).
template <int U>
__global__ void __launch_bounds__(256) split2_rows_vec4(const float* __restrict__ X, int64_t rows,
                                                        int64_t cols, int64_t ld,
                                                        float* __restrict__ HI,
                                                        float* __restrict__ LO, int64_t ldp, float lo_scale) {
    griddep_launch_dependents();
    const int64_t groups = cols / 4;
    const int64_t total = rows * groups;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t t0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t0 < total; t0 += U * stride) {
        float4 a[U];
        int64_t o[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t t = t0 + u * stride;
            if (t < total) {
                const int64_t r = t / groups;
                const int64_t c = (t - r * groups) * 4;
                a[u] = __ldcs(reinterpret_cast<const float4*>(X + r * ld + c));
                o[u] = r * ldp + c;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (t0 + u * stride < total) {
                float4 h, l;
                split_tf32x2(a[u].x, h.x, l.x, lo_scale);
                split_tf32x2(a[u].y, h.y, l.y, lo_scale);
                split_tf32x2(a[u].z, h.z, l.z, lo_scale);
                split_tf32x2(a[u].w, h.w, l.w, lo_scale);
                *reinterpret_cast<float4*>(HI + o[u]) = h;
                if (LO) *reinterpret_cast<float4*>(LO + o[u]) = l;
            }
        }
    }
    griddep_wait();          // see launch_pdl: complete only after the kernel ahead
}

__global__ void __launch_bounds__(256) split2_rows_scalar(const float* __restrict__ X, int64_t rows,
                                                          int64_t cols, int64_t ld,
                                                          float* __restrict__ HI,
                                                          float* __restrict__ LO, int64_t ldp, float lo_scale) {
    griddep_launch_dependents();
    const int64_t total = rows * cols;
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = t / cols;
        const int64_t c = t - r * cols;
        float h, l;
        split_tf32x2(X[r * ld + c], h, l, lo_scale);
        HI[r * ldp + c] = h;
        if (LO) LO[r * ldp + c] = l;
    }
    griddep_wait();          // see launch_pdl: complete only after the kernel ahead
}

// ------------------------------------------------------------- transposed
//
// op(X) = X^T: op(X)[r][c] = X[c * ld + r].  A 64 x 64 tile goes through
// shared memory so that both the FP32 reads (along stored rows) and the
// piece writes (along op rows, two BF16 per 4-byte store) are coalesced.
// Grid: x walks the tiles along op columns (stored rows), y the tiles along
// op rows, looping where there are more than gridDim.y of them.  Consecutive
// blocks thus write neighbouring 128-byte segments of the same op rows:
// measured on GB300 at 8192^2 (B's split for the square benchmark), 124.2 us
// against 130.9 us with x along op rows; grouping the tiles in squares of
// 2-16 or streaming stores gained nothing more.
constexpr int kT = 64;

__global__ void __launch_bounds__(256) split3_transposed(const float* __restrict__ X, int64_t rows,
                                                         int64_t cols, int64_t ld,
                                                         uint16_t* __restrict__ P0,
                                                         uint16_t* __restrict__ P1,
                                                         uint16_t* __restrict__ P2, int64_t ldp) {
    griddep_launch_dependents();
    __shared__ float tile[kT][kT + 1];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8
    const int64_t c0 = (int64_t)blockIdx.x * kT;              // op cols  = stored rows
    for (int64_t rt = blockIdx.y; rt * kT < rows; rt += gridDim.y) {
        const int64_t r0 = rt * kT;                           // op rows  = stored columns
        // load: stored row (c0 + i), stored columns r0 + tx, r0 + tx + 32
        for (int i = ty; i < kT; i += 8) {
            const int64_t sr = c0 + i;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t sc = r0 + tx + 32 * h;
                tile[i][tx + 32 * h] = (sr < cols && sc < rows) ? __ldcs(X + sr * ld + sc) : 0.0f;
            }
        }
        __syncthreads();
        // store: op row (r0 + j), op columns c0 + 2*tx, c0 + 2*tx + 1
        for (int j = ty; j < kT; j += 8) {
            const int64_t r = r0 + j;
            if (r >= rows) break;
            const int64_t c = c0 + 2 * tx;
            uint16_t a0, a1, a2, b0, b1, b2;
            split_bf16x3(tile[2 * tx][j], a0, a1, a2);
            split_bf16x3(tile[2 * tx + 1][j], b0, b1, b2);
            const int64_t o = r * ldp + c;
            if (c + 1 < cols && (o & 1) == 0) {
                *reinterpret_cast<uint32_t*>(P0 + o) = a0 | (uint32_t(b0) << 16);
                *reinterpret_cast<uint32_t*>(P1 + o) = a1 | (uint32_t(b1) << 16);
                if (P2) *reinterpret_cast<uint32_t*>(P2 + o) = a2 | (uint32_t(b2) << 16);
            } else {
                if (c < cols) { P0[o] = a0; P1[o] = a1; if (P2) P2[o] = a2; }
                if (c + 1 < cols) { P0[o + 1] = b0; P1[o + 1] = b1; if (P2) P2[o + 1] = b2; }
            }
        }
        __syncthreads();         // the tile is refilled by the next op-row tile
    }
    griddep_wait();          // see launch_pdl: complete only after the kernel ahead
}

// Vectorised form for full 64 x 64 tiles with 16-byte aligned rows on both
// sides: each thread loads four float4 along stored rows; then for each half
// of an op row, lanes 4i..4i+3 of a warp write its pieces as 16-byte stores
// of consecutive 8-element groups: 64 contiguous bytes per piece and store,
// and the four lanes' shared-memory reads fall on distinct banks.  Tiles at
// the ragged edges use the kernel above.  Measured on GB300 at 8192^2 (an L2
// flush before each launch): 127.6 us when each lane wrote a 16-element run
// as two stores 32 bytes apart.
__global__ void __launch_bounds__(256) split3_transposed_vec(const float* __restrict__ X, int64_t rows,
                                                             int64_t cols, int64_t ld,
                                                             uint16_t* __restrict__ P0,
                                                             uint16_t* __restrict__ P1,
                                                             uint16_t* __restrict__ P2, int64_t ldp) {
    griddep_launch_dependents();
    __shared__ float tile[kT][kT + 1];               // [op col (stored row)][op row]
    const int tid = threadIdx.x;
    const int64_t c0 = (int64_t)blockIdx.x * kT;     // op cols  = stored rows
    for (int64_t rt = blockIdx.y; rt * kT < rows; rt += gridDim.y) {
        const int64_t r0 = rt * kT;                  // op rows  = stored columns
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int idx = tid + 256 * i;               // 0 .. 1023
            const int k = idx >> 4, r4 = (idx & 15) * 4;
            const float4 v = __ldcs(reinterpret_cast<const float4*>(X + (c0 + k) * ld + r0 + r4));
            tile[k][r4 + 0] = v.x;
            tile[k][r4 + 1] = v.y;
            tile[k][r4 + 2] = v.z;
            tile[k][r4 + 3] = v.w;
        }
        __syncthreads();
        const int rr = tid >> 2, cp = tid & 3;           // op row in tile, 8-element group
        const int64_t o = (r0 + rr) * ldp + c0 + 8 * cp;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int j = 32 * q + 8 * cp;               // op columns c0 + j .. + 7
            uint32_t w0[4], w1[4], w2[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                split_bf16x3_pair(tile[j + 2 * i][rr], tile[j + 2 * i + 1][rr], w0[i], w1[i], w2[i]);
            *reinterpret_cast<uint4*>(P0 + o + 32 * q) = make_uint4(w0[0], w0[1], w0[2], w0[3]);
            *reinterpret_cast<uint4*>(P1 + o + 32 * q) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
            if (P2)
                *reinterpret_cast<uint4*>(P2 + o + 32 * q) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
        }
        __syncthreads();         // the tile is refilled by the next op-row tile
    }
    griddep_wait();          // see launch_pdl: complete only after the kernel ahead
}

__global__ void __launch_bounds__(256) split2_transposed(const float* __restrict__ X, int64_t rows,
                                                         int64_t cols, int64_t ld,
                                                         float* __restrict__ HI,
                                                         float* __restrict__ LO, int64_t ldp, float lo_scale) {
    griddep_launch_dependents();
    __shared__ float tile[kT][kT + 1];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int64_t c0 = (int64_t)blockIdx.x * kT;
    for (int64_t rt = blockIdx.y; rt * kT < rows; rt += gridDim.y) {
        const int64_t r0 = rt * kT;
        for (int i = ty; i < kT; i += 8) {
            const int64_t sr = c0 + i;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t sc = r0 + tx + 32 * h;
                tile[i][tx + 32 * h] = (sr < cols && sc < rows) ? __ldcs(X + sr * ld + sc) : 0.0f;
            }
        }
        __syncthreads();
        for (int j = ty; j < kT; j += 8) {
            const int64_t r = r0 + j;
            if (r >= rows) break;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t c = c0 + tx + 32 * h;
                if (c < cols) {
                    float hi, lo;
                    split_tf32x2(tile[tx + 32 * h][j], hi, lo, lo_scale);
                    HI[r * ldp + c] = hi;
                    if (LO) LO[r * ldp + c] = lo;
                }
            }
        }
        __syncthreads();         // the tile is refilled by the next op-row tile
    }
    griddep_wait();          // see launch_pdl: complete only after the kernel ahead
}

// Vectorised TF32 form for full 64 x 64 tiles with 16-byte aligned rows on
// both sides: each thread loads four float4 along stored rows; then for
// each of four 16-element parts of an op row, lanes 4i..4i+3 of a warp write
// its hi (and lo) values as 16-byte stores, 64 contiguous bytes per plane and
// store.  Tiles at the ragged edges use the kernel above.  Measured on GB300
// at 8192^2 (an L2 flush before each launch): the kernel above 158 us (5.1
// TB/s of the 12 bytes an element moves), the row-wise split 142 us.
__global__ void __launch_bounds__(256) split2_transposed_vec(const float* __restrict__ X, int64_t rows,
                                                             int64_t cols, int64_t ld,
                                                             float* __restrict__ HI,
                                                             float* __restrict__ LO, int64_t ldp,
                                                             float lo_scale) {
    griddep_launch_dependents();
    __shared__ float tile[kT][kT + 1];               // [op col (stored row)][op row]
    const int tid = threadIdx.x;
    const int64_t c0 = (int64_t)blockIdx.x * kT;     // op cols  = stored rows
    for (int64_t rt = blockIdx.y; rt * kT < rows; rt += gridDim.y) {
        const int64_t r0 = rt * kT;                  // op rows  = stored columns
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int idx = tid + 256 * i;               // 0 .. 1023
            const int k = idx >> 4, r4 = (idx & 15) * 4;
            const float4 v = __ldcs(reinterpret_cast<const float4*>(X + (c0 + k) * ld + r0 + r4));
            tile[k][r4 + 0] = v.x;
            tile[k][r4 + 1] = v.y;
            tile[k][r4 + 2] = v.z;
            tile[k][r4 + 3] = v.w;
        }
        __syncthreads();
        const int rr = tid >> 2, cp = tid & 3;           // op row in tile, 4-element group
        const int64_t o = (r0 + rr) * ldp + c0 + 4 * cp;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int j = 16 * q + 4 * cp;               // op columns c0 + j .. + 3
            float4 h, l;
            split_tf32x2(tile[j + 0][rr], h.x, l.x, lo_scale);
            split_tf32x2(tile[j + 1][rr], h.y, l.y, lo_scale);
            split_tf32x2(tile[j + 2][rr], h.z, l.z, lo_scale);
            split_tf32x2(tile[j + 3][rr], h.w, l.w, lo_scale);
            *reinterpret_cast<float4*>(HI + o + 16 * q) = h;
            if (LO) *reinterpret_cast<float4*>(LO + o + 16 * q) = l;
        }
        __syncthreads();         // the tile is refilled by the next op-row tile
    }
    griddep_wait();          // see launch_pdl: complete only after the kernel ahead
}

// Launch `kern` on `stream`; with pdl, as a programmatic dependent of the
// kernel ahead of it: it may start while that kernel runs (this library only
// asks for it where the two are independent), and because every split
// kernel calls griddep_wait() before it exits, it completes only after the
// kernel ahead -- so whatever waits for it (the GEMM's producer) also waits
// for that one.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, cudaStream_t stream, bool pdl,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The transposed kernels' grid: op-column tiles along x, op-row tiles along
// y (at most 65535; the kernels loop over the rest).
dim3 transposed_grid(int64_t rows, int64_t cols) {
    const int64_t rt = (rows + kT - 1) / kT;
    return dim3((unsigned)((cols + kT - 1) / kT), (unsigned)(rt < 65535 ? rt : 65535));
}

int grid_for(int64_t work, int threads) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (work + threads - 1) / threads;
    const int64_t cap = (int64_t)sms * 8;     // 8 resident 256-thread blocks per SM
    return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

// Blocks of 256 threads of `kern` resident at once on the device (at most
// 8 per SM), cached per kernel.
template <typename K>
int resident_blocks(K kern, std::atomic<int>& cache) {
    int v = cache.load(std::memory_order_relaxed);
    if (v > 0) return v;
    int dev = 0, sms = 148, per = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kern, 256, 0) != cudaSuccess || per < 1) {
        cudaGetLastError();
        per = 1;
    }
    v = sms * (per < 8 ? per : 8);
    cache.store(v, std::memory_order_relaxed);
    return v;
}

// Launch a row-wise split kernel over `groups` groups: four groups per
// thread per step (resident grid) when there are at least four per resident
// thread, else one (grid_for).
template <typename K4, typename K1, typename... Args>
cudaError_t launch_rows(K4 k4, K1 k1, std::atomic<int>& cache4, int64_t groups, cudaStream_t stream,
                        bool pdl, Args... args) {
    const int res = resident_blocks(k4, cache4);
    if (groups >= 4 * (int64_t)res * 256)
        return launch_pdl(k4, dim3(res), stream, pdl, args...);
    return launch_pdl(k1, dim3(grid_for(groups, 256)), stream, pdl, args...);
}
std::atomic<int> g_res_split3{0}, g_res_split2{0};

}  // namespace

cudaError_t launch_split_bf16x3(const float* X, int64_t rows, int64_t cols, int64_t ld, int trans,
                                uint16_t* P0, uint16_t* P1, uint16_t* P2, int64_t ldp,
                                cudaStream_t stream, bool pdl) {
    if (rows == 0 || cols == 0) return cudaSuccess;
    cudaError_t e;
    if (trans) {
        const dim3 grid = transposed_grid(rows, cols);
        if (rows % kT == 0 && cols % kT == 0 && ld % 4 == 0 && ldp % 8 == 0 && aligned16(X) &&
            aligned16(P0) && aligned16(P1) && aligned16(P2))
            e = launch_pdl(split3_transposed_vec, grid, stream, pdl, X, rows, cols, ld, P0, P1, P2,
                           ldp);
        else
            e = launch_pdl(split3_transposed, grid, stream, pdl, X, rows, cols, ld, P0, P1, P2, ldp);
    } else if (cols % 8 == 0 && ld % 4 == 0 && ldp % 8 == 0 && aligned16(X) && aligned16(P0) &&
               aligned16(P1) && aligned16(P2)) {
        e = launch_rows(split3_rows_vec8<4>, split3_rows_vec8<1>, g_res_split3, rows * (cols / 8),
                        stream, pdl, X, rows, cols, ld, P0, P1, P2, ldp);
    } else {
        e = launch_pdl(split3_rows_scalar, dim3(grid_for(rows * cols, 256)), stream, pdl, X, rows,
                       cols, ld, P0, P1, P2, ldp);
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_split_tf32x2(const float* X, int64_t rows, int64_t cols, int64_t ld, int trans,
                                float* HI, float* LO, int64_t ldp, cudaStream_t stream,
                                float lo_scale, bool pdl) {
    if (rows == 0 || cols == 0) return cudaSuccess;
    cudaError_t e;
    if (trans) {
        const dim3 grid = transposed_grid(rows, cols);
        if (rows % kT == 0 && cols % kT == 0 && ld % 4 == 0 && ldp % 4 == 0 && aligned16(X) &&
            aligned16(HI) && aligned16(LO))
            e = launch_pdl(split2_transposed_vec, grid, stream, pdl, X, rows, cols, ld, HI, LO, ldp,
                           lo_scale);
        else
            e = launch_pdl(split2_transposed, grid, stream, pdl, X, rows, cols, ld, HI, LO, ldp,
                           lo_scale);
    } else if (cols % 4 == 0 && ld % 4 == 0 && ldp % 4 == 0 && aligned16(X) && aligned16(HI) &&
               aligned16(LO)) {
        e = launch_rows(split2_rows_vec4<4>, split2_rows_vec4<1>, g_res_split2, rows * (cols / 4),
                        stream, pdl, X, rows, cols, ld, HI, LO, ldp, lo_scale);
    } else {
        e = launch_pdl(split2_rows_scalar, dim3(grid_for(rows * cols, 256)), stream, pdl, X, rows,
                       cols, ld, HI, LO, ldp, lo_scale);
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_split_pieces(int mode, const float* X, int64_t rows, int64_t cols, int64_t ld,
                                int trans, void* planes, int64_t ldp, cudaStream_t stream,
                                bool pdl, int64_t plane_rows) {
    const int64_t n = (plane_rows > 0 ? plane_rows : rows) * ldp;
    if (mode_is_tf32(mode)) {
        float* hi = static_cast<float*>(planes);
        return launch_split_tf32x2(X, rows, cols, ld, trans, hi,
                                   mode_pieces(mode) > 1 ? hi + n : nullptr, ldp, stream,
                                   mode == kModeTf32x3Oy ? 2048.0f : 1.0f, pdl);
    }
    uint16_t* p0 = static_cast<uint16_t*>(planes);
    return launch_split_bf16x3(X, rows, cols, ld, trans, p0, p0 + n,
                               mode_pieces(mode) > 2 ? p0 + 2 * n : nullptr, ldp, stream, pdl);
}

}  // namespace emu
