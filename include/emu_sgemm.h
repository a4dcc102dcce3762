/*
 * emu_sgemm.h -- C ABI of libemusgemm: FP32 matrix multiplication emulated
 * on the BF16 (or TF32) tensor cores of one GB300 GPU (sm_103a).
 *
 * The method is the one described on the web pages about it:
 *
 *  - "Unlocking Tensor Core Performance for Machine Learning Interatomic
 *    Potentials" (NVIDIA technical blog), Figure 1 and its caption (BF16x9:
 *    three scaled BF16 pieces per FP32 operand, nine pairwise products,
 *    accumulated in FP32 over five anti-diagonal bands), Figure 2 and the
 *    equation under it (TF32x3: a leading and a residual TF32 piece, no
 *    scaling, the residual*residual product dropped);
 *  - the discuss.pytorch.kr summary of that post, section "Blackwell의
 *    BF16x9: 세 조각, 아홉 번의 곱" (x = x0 + 2^-8 x1 + 2^-16 x2; the bands are
 *    added to the FP32 accumulator smallest band first) and section "Ampere의
 *    TF32x3: 두 조각, 세 번의 곱".
 *
 * The interface keeps what the pages require of it: FP32 in, FP32 out, the
 * caller's code unchanged apart from the call ("FP32 in and out" in the
 * CUTLASS paragraph of the blog post's TF32x3 section).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  Storage   Row major.  op(X) = X when trans == 0, X^T when trans == 1.  The
 *            leading dimension (ld*) is the distance, in elements, between
 *            consecutive rows of the matrix AS STORED.  A column-major caller
 *            computes C^T = op(B)^T op(A)^T instead.
 *  Pointers  Unless an entry point says otherwise, matrix pointers are CUDA
 *            device pointers (or managed memory) on the current device, owned
 *            by the caller; the library never frees them.
 *  Streams   `stream` is a cudaStream_t (0 = the legacy default stream).
 *            Work is enqueued asynchronously; a call returns once its kernels
 *            are launched.
 *  Errors    Arguments are checked on the host before anything is launched;
 *            a bad argument returns EMU_ERR_INVALID_VALUE and touches nothing.
 *            No entry point aborts the process, traps on the device or spins
 *            without a bound: device-side waits give up after a time limit
 *            and record EMU_ERR_TIMEOUT in a sticky per-device error word that
 *            emu_get_last_device_error() returns.
 *  Scratch   The two-pass path stores the split operands in a workspace that
 *            the library allocates per device, grows on demand and releases
 *            in emu_shutdown().  Calls on one device share it, so concurrent
 *            calls on different streams of one device must be serialised by
 *            the caller.  Growing it calls cudaMalloc / cudaFree, which must
 *            not happen during stream capture.
 */
#ifndef EMU_SGEMM_H
#define EMU_SGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, declared here without the CUDA headers. */
typedef struct CUstream_st* emu_stream_t;

typedef enum {
    /* three BF16 pieces per operand, nine products in five bands */
    EMU_MODE_BF16X9 = 0,
    /* two TF32 pieces per operand, three products (residual*residual dropped) */
    EMU_MODE_TF32X3 = 1,
    /* plain FP32 FMA on the CUDA cores (the library's own baseline) */
    EMU_MODE_FP32_SIMT = 2,
    /* cheaper, less accurate rungs: two BF16 pieces per operand, three
       products a0 b0, a0 b1, a1 b0 (about 2^-16 relative per product) */
    EMU_MODE_BF16X3 = 3,
    /* one TF32 piece per operand, one product (about 2^-10 per product) */
    EMU_MODE_TF32 = 4,
    /* TF32X3 with the Ootomo-Yokota correction: the residual is scaled by
       2^11 before its TF32 rounding and the residual band by 2^-11 */
    EMU_MODE_TF32X3_OY = 5
} emu_mode_t;

typedef enum {
    EMU_OK = 0,
    EMU_ERR_INVALID_VALUE = -1,   /* bad argument; nothing was launched */
    EMU_ERR_ARCH = -2,            /* current device is not compute capability 10.3 */
    EMU_ERR_ALLOC = -3,           /* workspace or staging allocation failed */
    EMU_ERR_LAUNCH = -4,          /* a kernel launch failed */
    EMU_ERR_TIMEOUT = -5,         /* a device-side wait ran out (see the errors note) */
    EMU_ERR_CUDA = -6             /* another CUDA runtime error */
} emu_status_t;

/* Which implementation emu_sgemm uses for the tensor-core modes. */
typedef enum {
    EMU_PATH_AUTO = 0,     /* the library chooses per call */
    EMU_PATH_TWOPASS = 1,  /* split kernels write the pieces to the workspace, then the GEMM */
    EMU_PATH_FUSED = 2,    /* one kernel reads FP32 A and splits it into shared memory
                              (BF16x9 and TF32x3) */
    EMU_PATH_FUSED_TMEM = 3 /* the same, split into tensor memory (128-wide tiles) */
} emu_path_t;

/*
 * emu_sgemm -- C = alpha * op(A) * op(B) + beta * C.
 *
 *  transA, transB  0 or 1 (see Storage above).
 *  M, N, K         op(A) is M x K, op(B) is K x N, C is M x N; each >= 0.
 *  A, lda          device FP32; lda >= (transA ? M : K), lda >= 1.
 *  B, ldb          device FP32; ldb >= (transB ? K : N), ldb >= 1.
 *  C, ldc          device FP32, read (when beta != 0) and written; ldc >= N.
 *                  C must not overlap A or B.
 *  mode            an emu_mode_t.
 *
 * BF16X9 (the method of Figure 1 of the blog post): every element of op(A)
 * and op(B) is split exactly into x = x0 + 2^-8 x1 + 2^-16 x2 (three BF16
 * pieces, rounding to nearest even, signed residuals).  The nine products
 * a_i b_j are formed on the tensor cores and grouped into bands b = i + j,
 * taken in the order 4, 3, 2, 1, 0; the result is
 *     sum_b 2^-8b S_b,  S_b = sum_{i+j=b} sum_k a_i[m,k] b_j[k,n],
 * accumulated in FP32 smallest band first: the tensor core sums short runs
 * of K (16 MMAs) and each partial is added, times 2^-8b, to an FP32
 * accumulator with round-to-nearest.  TF32X3 (Figure 2): x = hi + lo (TF32,
 * nearest even, no scaling); the band hi*lo + lo*hi is accumulated first,
 * then hi*hi; lo*lo is dropped.  BF16X3 keeps the first two BF16 pieces
 * and runs band 1 (a0 b1 + a1 b0) then band 0 (a0 b0), the way PyTorch's
 * "high" matmul precision is described on the discuss.pytorch.kr page;
 * TF32 runs hi*hi alone (one-pass TF32, Figures 5-8 of the blog post).
 * TF32X3_OY is the variant of the Ootomo-Yokota paper that the
 * discuss.pytorch.kr page's TF32x3 section links (scaling, accumulation
 * outside the tensor core): lo' = tf32(2^11 (x - hi)), the residual band
 * hi*lo' + lo'*hi first, then hi*hi with the band scaled by 2^-11, each
 * 32-element K block's partial added to FP32 registers with round to
 * nearest.  It equals TF32X3 wherever x - hi is a normal FP32 number and
 * keeps 11 residual bits below that range.
 * Neither meets FP32 accuracy; they complete the accuracy ladder the pages
 * compare BF16X9 with.  The epilogue is C = alpha*acc + beta*C in
 * FP32; C is not read when beta == 0, and A, B are not read when alpha == 0
 * or K == 0 (BLAS convention).  M == 0 or N == 0 is a no-op.
 *
 * Non-finite inputs: the split keeps +-inf as (x, +0, +0) and NaN as NaN
 * pieces, so an output that meets an infinity is usually NaN (products such
 * as inf * 0 with a zero residual piece), where an IEEE FP32 dot product
 * would give +-inf; outputs that meet no infinity or NaN are unaffected.
 *
 * Accuracy: for BF16X9 every element satisfies
 *     |C - C_exact| <= (2K + 2) 2^-24 |alpha| sum_k |a_mk||b_kn| + 2^-23 |beta C|
 * (TF32X3 and TF32X3_OY add 2^-20 |alpha| sum_k |a_mk||b_kn|, BF16X3 2^-16 and TF32
 * 2^-10 + 2^-21), where C_exact is the result in exact arithmetic.
 *
 * Returns EMU_OK once the kernels are enqueued on `stream`.
 *
 * CUDA graphs: a call can be captured on `stream` once a call of the same
 * shape and mode (or one needing at least as much workspace) has run on the
 * device outside capture -- the library sizes its buffers with cudaMalloc,
 * which a capture does not allow.  Replays reuse the captured workspace and
 * must not overlap one another or other calls on the GPU.  A later call that
 * needs more workspace than any before it reallocates it, which invalidates
 * graphs captured earlier: capture after the largest call has run (or
 * re-capture).
 */
emu_status_t emu_sgemm(int transA, int transB, int64_t M, int64_t N, int64_t K,
                       float alpha, const float* A, int64_t lda,
                       const float* B, int64_t ldb,
                       float beta, float* C, int64_t ldc,
                       int mode, emu_stream_t stream);

/*
 * emu_sgemm_host -- emu_sgemm on HOST buffers, end to end.
 *
 * A, B and C are host pointers (pageable or pinned).  The call copies op's
 * operands (and C when beta != 0) to library-owned device buffers on
 * `stream`, runs emu_sgemm there and copies C back, then synchronises the
 * stream before it returns, so C holds the result on return.  Same
 * arguments, layout and error codes as emu_sgemm; the device buffers are
 * grown on demand and released by emu_shutdown().  When more than 64 MB
 * move (and M >= 512), the copies are pipelined with the GEMM: op(A) and C
 * cross in row chunks of whole 256-row tiles on a library-owned copy
 * stream, each chunk's GEMM runs on `stream` as its rows land, and C's
 * chunks go back on a second library-owned stream.  B crosses first, whole,
 * and the first chunk splits it -- except where the two-pass kernels run
 * with N >= 2048 and B of at least 16 MiB: there op(A)'s first 2048 rows
 * cross first, then op(B) in column panels of 1024 columns (wider when there
 * would be more than 64), each split into its rows of B's pieces and
 * multiplied by those first rows as it lands, so that the tensor cores start
 * after one panel instead of all of B; the later chunks reuse B's pieces.
 * The result meets the same accuracy bound as one emu_sgemm call; it is bit
 * for bit the same unless the split of the GEMM's last wave along K (which
 * depends on the tile count of each launch) differs between the call and
 * its chunks or panels.  Host buffers in pinned memory let the copies
 * overlap; pageable ones work too.
 */
emu_status_t emu_sgemm_host(int transA, int transB, int64_t M, int64_t N, int64_t K,
                            float alpha, const float* A, int64_t lda,
                            const float* B, int64_t ldb,
                            float beta, float* C, int64_t ldc,
                            int mode, emu_stream_t stream);

/*
 * emu_sgemm_bsplit -- emu_sgemm with op(B) given already split.
 *
 * For a B that stays the same over many calls -- the weight of a linear
 * layer, applied to batch after batch of activations, as in the MLIP layers
 * the blog post measures (Figure 3) -- split it once and pass its pieces:
 * a call then runs no split of B, and in BF16X9 with A stored K-major
 * (transA == 0, lda % 4 == 0, A 16-byte aligned) and N <= 256, M >= 4096
 * it is a single kernel launch that splits A on chip (the FUSED or
 * FUSED_TMEM path of emu_set_path; EMU_PATH_TWOPASS splits A into the
 * workspace first).  Consecutive calls on one stream overlap each kernel's
 * launch and prologue with the end of the one before it (programmatic
 * dependent launch).
 *
 *  Bp, ldbp   the pieces of op(B)^T (N x K, K-major) as the mode's
 *             consecutive planes of N rows x ldbp elements, plane i at
 *             element offset i * N * ldbp:
 *               BF16X9  3 planes of BF16 bits (uint16), as emu_split_bf16x3
 *                       writes them for op(B)^T (trans = !transB);
 *               BF16X3  the first 2 of those planes;
 *               TF32X3  2 FP32 planes (HI, LO) of emu_split_tf32x2;
 *               TF32X3_OY  HI and LO of emu_split_tf32x2_scaled;
 *               TF32    1 plane, HI.
 *             Device memory owned by the caller, 16-byte aligned; ldbp >= K
 *             and a multiple of 8; columns K..ldbp-1 are not read.  The
 *             pieces must not change while a call that reads them runs.
 *  mode       any emu_mode_t but EMU_MODE_FP32_SIMT; the strategy
 *             (emu_set_strategy) does not apply: the call runs `mode`.
 * The other arguments, the layout of A and C, the results and the error
 * codes are emu_sgemm's (with B given by its pieces, the result is the one
 * emu_sgemm computes for that B).  Uses the library's workspace for A's
 * pieces only where A is split into it.
 */
emu_status_t emu_sgemm_bsplit(int transA, int64_t M, int64_t N, int64_t K, float alpha,
                              const float* A, int64_t lda, const void* Bp, int64_t ldbp,
                              float beta, float* C, int64_t ldc, int mode, emu_stream_t stream);

/*
 * emu_split_bf16x3 -- the split/pack step of BF16X9 on its own.
 *
 * Writes the three BF16 pieces (raw bit patterns) of op(X), rows x cols:
 * P_i[r * ldp + c] holds piece i of op(X)[r][c] with
 *     op(X)[r][c] = P0 + 2^-8 P1 + 2^-16 P2   exactly, for every finite value.
 * This is the same kernel the two-pass GEMM uses to fill its workspace (A is
 * split as op(A); B as op(B)^T, i.e. with trans = !transB, so that both are
 * K-major).  X: device FP32 with leading dimension ld (ld >= (trans ? rows :
 * cols)); P0, P1, P2: device, ldp >= cols; columns cols..ldp-1 are not
 * written.  Rounding to nearest even; a finite value whose nearest BF16 is
 * infinite takes the truncated BF16; +-inf -> (x, +0, +0); NaN -> 0x7FC0 in
 * all three.
 */
emu_status_t emu_split_bf16x3(const float* X, int64_t rows, int64_t cols, int64_t ld,
                              int trans, uint16_t* P0, uint16_t* P1, uint16_t* P2,
                              int64_t ldp, emu_stream_t stream);

/*
 * emu_split_tf32x2 -- the split step of TF32X3 on its own: HI and LO (FP32
 * containers with the low 13 mantissa bits zero) with op(X) ~ HI + LO, HI the
 * nearest TF32 of x (ties even), LO the nearest TF32 of x - HI.  Same layout,
 * ownership and rules as emu_split_bf16x3.
 */
emu_status_t emu_split_tf32x2(const float* X, int64_t rows, int64_t cols, int64_t ld,
                              int trans, float* HI, float* LO, int64_t ldp,
                              emu_stream_t stream);

/*
 * emu_split_tf32x2_scaled -- the split step of TF32X3_OY on its own: HI as
 * in emu_split_tf32x2, LO the nearest TF32 of 2^11 (x - HI), so that
 * op(X) ~ HI + 2^-11 LO.  Same layout, ownership and rules as
 * emu_split_tf32x2.
 */
emu_status_t emu_split_tf32x2_scaled(const float* X, int64_t rows, int64_t cols, int64_t ld,
                                     int trans, float* HI, float* LO, int64_t ldp,
                                     emu_stream_t stream);

/*
 * emu_sgemm_noalloc -- emu_sgemm that allocates no device memory.
 *
 * The pages have no counterpart: this entry point exists for callers of this
 * library that cannot let it call cudaMalloc -- code whose device memory is
 * owned by another allocator or a fixed budget (where an extra allocation
 * can fail or break that owner's accounting), or code that cannot take the
 * device-wide synchronisation of cudaMalloc / cudaFree in the middle of its
 * stream work.  Instead of the growable workspace it keeps the split pieces
 * in one fixed 64 MiB array in device memory, which every GPU that loads
 * the library holds until the process exits.
 *
 * Same arguments, layout, modes and error codes as emu_sgemm, and its
 * results meet the same accuracy bound.  It always runs the two-pass split
 * and GEMM kernels with 256-wide tiles, whole tiles only (no split of the
 * last wave along K) and C stored by the epilogue warps, so its results are
 * bit for bit emu_sgemm's only where emu_sgemm takes that same path (N > 128,
 * no split tail, the two-pass path).  One limit: the pieces must fit in the
 * array,
 *     BF16X9:  3 * 2 * (M + N) * ldp  bytes  (plus < 1 KB of alignment),
 *     TF32X3:  2 * 4 * (M + N) * ldp  bytes,   ldp = K rounded up to 8,
 *     BF16X3:  2 * 2 * (M + N) * ldp  bytes,   TF32: 1 * 4 * (M + N) * ldp,
 *     TF32X3_OY: as TF32X3,
 * at most 64 MiB; a larger request returns EMU_ERR_INVALID_VALUE and
 * launches nothing (the check is made before any size product is formed, so
 * no M, N, K can wrap it; FP32_SIMT and the K == 0 / alpha == 0 cases use no
 * scratch and have no limit).  Once the first call on a device has
 * returned, later calls change neither the device's free memory nor any
 * allocator's state.  The first call on a device, with that device
 * current, resolves the array's device address (cudaGetSymbolAddress) once;
 * make that first call before any stream capture.  All calls on a device
 * share the array: calls whose work overlaps on the GPU (other streams,
 * unordered host threads) race on it and must be serialised by the caller.
 * Nothing in the array has to start at zero -- each call writes every piece
 * its GEMM reads -- so the contents a previous call left do not matter.
 */
emu_status_t emu_sgemm_noalloc(int transA, int transB, int64_t M, int64_t N, int64_t K,
                               float alpha, const float* A, int64_t lda,
                               const float* B, int64_t ldb,
                               float beta, float* C, int64_t ldc,
                               int mode, emu_stream_t stream);

/* Select the implementation of the tensor-core modes for later calls on this
 * process (EMU_PATH_AUTO by default; the environment variable
 * EMU_SGEMM_PATH=auto|twopass|fused|fused_tmem sets the initial value).
 * FUSED applies to BF16x9 and TF32x3, FUSED_TMEM to BF16x9, each with
 * op(A) = A stored with 16-byte aligned rows (lda % 4 == 0); other calls run
 * two-pass.  AUTO takes FUSED for BF16x9 with M >= 4096 and 128 < N <= 256,
 * FUSED_TMEM for BF16x9 with M >= 4096 and N <= 128, two-pass otherwise
 * (TF32x3 split on chip was measured no faster than two-pass).  Not
 * thread-safe with respect to concurrent emu_sgemm calls. */
emu_status_t emu_set_path(int path);
int emu_get_path(void);

/* Whether an emulated mode always runs as asked.  The discuss.pytorch.kr
 * page (section "PyTorch에서 직접 써 보려면") and the blog post's MD-step
 * results contrast cuBLAS's two strategies for its BF16x9: "eager" uses the
 * emulation wherever it applies, "performant" only where it is expected to be
 * faster than native FP32.  This library's strategies: */
typedef enum {
    EMU_STRATEGY_EAGER = 0,       /* every call runs the mode it asks for (default) */
    EMU_STRATEGY_PERFORMANT = 1   /* a call in a tensor-core mode runs the FP32 SIMT
                                     kernel instead where that is predicted faster */
} emu_strategy_t;

/* Select the strategy of later emu_sgemm / emu_sgemm_host calls in this
 * process (EMU_STRATEGY_EAGER by default; EMU_SGEMM_STRATEGY=performant sets
 * the initial value).  emu_sgemm_noalloc always runs the mode it is given.
 * Under PERFORMANT a result meets the FP32 SIMT kernel's accuracy (the
 * BF16X9 bound) where the kernel is swapped.  Returns EMU_ERR_INVALID_VALUE
 * for another value.  Not thread-safe with respect to concurrent calls. */
emu_status_t emu_set_strategy(int strategy);
int emu_get_strategy(void);

/* The mode emu_sgemm would run for an M x N x K request in `mode` under
 * `strategy` (-1: the current one) on a GPU with `sms` SMs (<= 0: the
 * current device's, which needs a device).  A pure host function; -1 for
 * invalid arguments.  The choice compares two time estimates of this
 * library's kernels, fitted to measurements on GB300: */
int emu_choose_mode(int64_t M, int64_t N, int64_t K, int mode, int strategy, int sms);
/* ... the estimated device time of one call in microseconds (-1 on invalid
 * arguments; sms must be > 0). */
double emu_predict_us(int64_t M, int64_t N, int64_t K, int mode, int sms);

/* Bytes of workspace the two-pass path needs for one call of this shape,
 * whatever its transposes.  The pieces of an operand stored with K as its
 * row index (A with transA, B without transB) are M- or N-major (K rows of
 * M or N elements, rounded up to 64) in BF16x9, and in BF16x3 when K is at
 * least 4 times that operand's M (or N); all other pieces are K-major (rows
 * of K elements, rounded up to 8).  This is the larger of the two for each
 * operand, B's region rounded up to 1 KB. */
size_t emu_workspace_size(int64_t M, int64_t N, int64_t K, int mode);

/* Read the sticky device error word of the current device (synchronises the
 * device).  Returns EMU_OK when no device-side wait has given up. */
emu_status_t emu_get_last_device_error(void);
/* Clear that word (synchronises the device). */
emu_status_t emu_clear_device_error(void);

/* Exercise the bounded-wait machinery: one tiny kernel waits on an mbarrier
 * that nothing arrives on, gives up after `limit_us` microseconds (1 to
 * 1,000,000), records EMU_ERR_TIMEOUT and exits normally.  Returns the
 * device error word after the kernel (EMU_ERR_TIMEOUT when the machinery
 * works); the word is left set. */
emu_status_t emu_selftest_timeout(int limit_us, emu_stream_t stream);

/* Kernel-level timing.  While enabled, every kernel that emu_sgemm launches
 * is bracketed by CUDA events recorded on the caller's stream.
 * emu_profile_read synchronises on the recorded events and returns, for
 * kernel kind `kind` (0 = split/pack, 1 = tensor-core GEMM, 2 = fused GEMM,
 * 3 = SIMT GEMM, 4 = epilogue-only scale), the number of launches and their
 * summed duration in milliseconds since the last emu_profile_enable(1). */
emu_status_t emu_profile_enable(int on);
emu_status_t emu_profile_read(int kind, int64_t* launches, double* total_ms);

/* Name of the last CUDA runtime error that an entry point of this library
 * turned into a non-OK status (for example "cudaErrorLaunchOutOfResources"),
 * or "cudaSuccess" if none; a static string.  Process-wide, not thread-safe. */
const char* emu_last_cuda_error(void);

/* Name of a status code (static string). */
const char* emu_status_string(emu_status_t status);

/* Release the workspace and staging buffers of every device. */
emu_status_t emu_shutdown(void);

/* Library version as 10000*major + 100*minor + patch. */
int emu_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EMU_SGEMM_H */
