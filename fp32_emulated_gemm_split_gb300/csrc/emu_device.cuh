// emu_device.cuh -- device-side building blocks shared by the library's
// kernels: inline-PTX wrappers for mbarriers, TMA, tcgen05 (TMEM allocation,
// MMA, commit, loads), bounded waits and the sticky device error word.
//
// Every wait in this library is bounded: a wait that has not completed after
// EMU_WAIT_LIMIT_NS of %globaltimer records an error code in the device's
// sticky error word (its address is a kernel argument) and returns false, and
// the calling kernel winds down instead of spinning forever.  No kernel traps.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "emu_internal.h"

namespace emu {

#ifndef EMU_WAIT_LIMIT_NS
#define EMU_WAIT_LIMIT_NS 2000000000ull   // 2 s: far above any legitimate wait
#endif

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void record_error(int* err, int code) {
    atomicCAS(err, 0, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier --

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done) : "r"(bar), "r"(parity) : "memory");
    return done != 0;
}

// Wait for the phase with the given parity to complete.  Returns false (and
// records `code` in *err) if it has not completed within the limit.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* err, int code,
                                          uint64_t limit_ns = EMU_WAIT_LIMIT_NS) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0 && global_timer_ns() - t0 > limit_ns) {
            record_error(err, code);
            return false;
        }
    }
}

// --------------------------------------------------------------------- TMA --

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(map) : "memory");
}

// 3-D tiled load into this CTA's shared memory, completion signalled on `bar`
// as transaction bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t c0, int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        :: "r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar) : "memory");
}

// 2-D tiled store from this CTA's shared memory to global memory (bulk
// group completion; out-of-range parts of the box are not written).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int32_t c0, int32_t c1,
                                             uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                 :: "l"(map), "r"(c0), "r"(c1), "r"(src) : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until the shared memory of all committed bulk stores has been read.
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// ... all but the most recent N bulk stores have finished reading.
template <int N>
__device__ __forceinline__ void bulk_wait_read_n() {
    asm volatile("cp.async.bulk.wait_group.read %0;" :: "n"(N) : "memory");
}
// Wait until all committed bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05 --

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 "matrix descriptor") for a K-major
// operand tile stored with the 128-byte swizzle: rows of 128 bytes, groups of
// 8 rows 1024 bytes apart.  Fields: start address >> 4 in bits 0-13, leading
// byte offset >> 4 in bits 16-29 (unused by this swizzled K-major layout),
// stride byte offset >> 4 in bits 32-45, the fixed value 1 in bits 46-47,
// base offset 0 (tiles are 1024-byte aligned), swizzle mode 2 (128-byte) in
// bits 61-63.
__device__ __forceinline__ uint64_t make_sw128_kmajor_desc(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1u) << 16;                 // LBO: 16 bytes (ignored)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;         // SBO: 1024 bytes
    d |= static_cast<uint64_t>(1u) << 46;                 // descriptor version
    d |= static_cast<uint64_t>(2u) << 61;                 // 128-byte swizzle
    return d;
}

// The same for an M- or N-major operand (PTX ISA, tcgen05 shared memory
// descriptor; canonical MN-major layout with 128-byte swizzle): a tensor
// copy of a box of 64 elements (128 bytes, the contiguous M or N direction)
// by 64 K rows puts K row r at byte 128 r, its 16-byte chunks swizzled by
// r % 8, so the 8-row swizzle atoms of 1024 bytes follow each other along K
// (stride byte offset 1024) and the next 64 elements of M or N are `lbo`
// bytes further (leading byte offset: the next box).  One K = 16 step of a
// BF16 MMA is 16 K rows: two atoms, 2048 bytes.
__device__ __forceinline__ uint64_t make_sw128_mn_desc(uint32_t smem_addr, uint32_t lbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(lbo >> 4) << 16;           // LBO: next 64 elements of M or N
    d |= static_cast<uint64_t>(1024u >> 4) << 32;         // SBO: next 8 K rows
    d |= static_cast<uint64_t>(1u) << 46;                 // descriptor version
    d |= static_cast<uint64_t>(2u) << 61;                 // 128-byte swizzle
    return d;
}

// Instruction descriptor for a dense tcgen05.mma with FP32 accumulation and
// both operands K-major: D format F32 (bits 4-5 = 1), A and B formats in bits
// 7-9 and 10-12 (kind::f16: 1 = BF16; kind::tf32: 2 = TF32), N >> 3 in bits
// 17-22, M >> 4 in bits 24-28.  Bit 15 (A) and bit 16 (B) ask for an M- or
// N-major operand instead (kIdescAMn, kIdescBMn).
__host__ __device__ constexpr uint32_t make_idesc(uint32_t ab_format, uint32_t M, uint32_t N) {
    return (1u << 4) | (ab_format << 7) | (ab_format << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}
constexpr uint32_t kIdescAMn = 1u << 15, kIdescBMn = 1u << 16;

// 32 lanes x 8 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_32x32b_x8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr) : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr) : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------- CTA pairs (clusters of 2) --

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];"
                 :: "r"(cluster_addr) : "memory");
}

// The same over a 4-D map (M- or N-major pieces: element, K row, 64-element
// chunk, piece).
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t c0, int32_t c1,
                                                 int32_t c2, int32_t c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile"
        ".mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];"
        :: "r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar_cluster) : "memory");
}

// Tensor copy into this CTA's shared memory whose completion is counted on
// an mbarrier that may live in the peer CTA of the pair.
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t c0, int32_t c1,
                                                 int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile"
        ".mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        :: "r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar_cluster) : "memory");
}

template <int TF32>
__device__ __forceinline__ void mma_cta2(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
    if constexpr (TF32) {
        asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                     " tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n}\n"
                     :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
    } else {
        asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                     " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n"
                     :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
    }
}

// D = A*B + 2^-SHIFT D (scale-input-d = SHIFT).
template <int TF32, int SHIFT>
__device__ __forceinline__ void mma_cta2_scaled(uint32_t d, uint64_t a, uint64_t b,
                                                uint32_t idesc) {
    static_assert(SHIFT >= 1 && SHIFT <= 15, "scale-input-d takes 0..15");
    if constexpr (TF32) {
        asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, 1, 0;\n"
                     " tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p, %4;\n}\n"
                     :: "r"(d), "l"(a), "l"(b), "r"(idesc), "n"(SHIFT) : "memory");
    } else {
        asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, 1, 0;\n"
                     " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p, %4;\n}\n"
                     :: "r"(d), "l"(a), "l"(b), "r"(idesc), "n"(SHIFT) : "memory");
    }
}

// The same with the A operand in tensor memory: `a` is the TMEM address of
// the first 32-bit column of this K step's A (rows = lanes, two 16-bit
// elements per column).
__device__ __forceinline__ void mma_cta2_ta(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                 " tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
                 :: "r"(d), "r"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}

template <int SHIFT>
__device__ __forceinline__ void mma_cta2_ta_scaled(uint32_t d, uint32_t a, uint64_t b,
                                                   uint32_t idesc) {
    static_assert(SHIFT >= 1 && SHIFT <= 15, "scale-input-d takes 0..15");
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, 1, 0;\n"
                 " tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p, %4;\n}\n"
                 :: "r"(d), "r"(a), "l"(b), "r"(idesc), "n"(SHIFT) : "memory");
}

// Store 8 consecutive 32-bit columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
           "r"(r[6]), "r"(r[7]) : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Arrive on the barrier at this offset in both CTAs of the pair once the
// MMAs issued so far have completed.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster"
                 ".multicast::cluster.b64 [%0], %1;" :: "r"(bar), "h"((uint16_t)3) : "memory");
}

// ------------------------------------------------------------- the split --

// Nearest BF16 (ties to even) of a finite FP32 value; a value whose nearest
// BF16 would be infinite takes the largest finite BF16 of its sign, which is
// the truncated value (the `satfinite` form of the conversion).
__device__ __forceinline__ uint16_t bf16_rn_sat(float x) {
    uint16_t h;
    asm("cvt.rn.satfinite.bf16.f32 %0, %1;" : "=h"(h) : "f"(x));
    return h;
}

__device__ __forceinline__ float bf16_as_f32(uint16_t h) {
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// x = x0 + 2^-8 x1 + 2^-16 x2 with three BF16 pieces, x1 and x2 scaled up by
// 2^8 and 2^16 so that each piece keeps a full BF16 significand.  Rounding is
// to nearest, ties to even, with signed residuals; +-inf -> (x, +0, +0); NaN ->
// three canonical quiet NaNs.  The subtraction and the scaling are exact.
__device__ __forceinline__ void split_bf16x3(float x, uint16_t& h0, uint16_t& h1, uint16_t& h2) {
    const uint32_t u = __float_as_uint(x);
    if ((u & 0x7F800000u) == 0x7F800000u) {
        const bool nan = (u & 0x007FFFFFu) != 0;
        h0 = nan ? uint16_t(0x7FC0) : uint16_t(u >> 16);
        h1 = nan ? uint16_t(0x7FC0) : uint16_t(0);
        h2 = h1;
        return;
    }
    h0 = bf16_rn_sat(x);
    const float s1 = __fmul_rn(__fsub_rn(x, bf16_as_f32(h0)), 256.0f);
    h1 = bf16_rn_sat(s1);
    const float s2 = __fmul_rn(__fsub_rn(s1, bf16_as_f32(h1)), 256.0f);
    h2 = bf16_rn_sat(s2);
}

// Two neighbouring elements at once: the same pieces as split_bf16x3, packed
// as BF16 pairs (element a in the low half, b in the high half), with one
// cvt.rn.satfinite.bf16x2.f32 per piece instead of two conversions and a
// pack.  satfinite turns a finite value whose nearest BF16 is infinite into
// the largest finite BF16, which is its truncation (the R2 rule); pairs
// holding an infinity or a NaN take the scalar path.
__device__ __forceinline__ uint32_t cvt_bf16x2(float hi, float lo) {
    uint32_t d;
    asm("cvt.rn.satfinite.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ void split_bf16x3_pair(float a, float b, uint32_t& p0, uint32_t& p1,
                                                  uint32_t& p2) {
    const uint32_t ua = __float_as_uint(a), ub = __float_as_uint(b);
    if (((ua & 0x7F800000u) == 0x7F800000u) || ((ub & 0x7F800000u) == 0x7F800000u)) {
        uint16_t a0, a1, a2, b0, b1, b2;
        split_bf16x3(a, a0, a1, a2);
        split_bf16x3(b, b0, b1, b2);
        p0 = uint32_t(a0) | (uint32_t(b0) << 16);
        p1 = uint32_t(a1) | (uint32_t(b1) << 16);
        p2 = uint32_t(a2) | (uint32_t(b2) << 16);
        return;
    }
    p0 = cvt_bf16x2(b, a);
    const float sa1 = __fmul_rn(__fsub_rn(a, __uint_as_float(p0 << 16)), 256.0f);
    const float sb1 = __fmul_rn(__fsub_rn(b, __uint_as_float(p0 & 0xFFFF0000u)), 256.0f);
    p1 = cvt_bf16x2(sb1, sa1);
    const float sa2 = __fmul_rn(__fsub_rn(sa1, __uint_as_float(p1 << 16)), 256.0f);
    const float sb2 = __fmul_rn(__fsub_rn(sb1, __uint_as_float(p1 & 0xFFFF0000u)), 256.0f);
    p2 = cvt_bf16x2(sb2, sa2);
}

// Nearest TF32 (10 explicit mantissa bits, ties to even) kept in an FP32
// container with the low 13 bits zero; overflow to inf is replaced by the
// truncated value.  Integer rounding on the bit pattern.
__device__ __forceinline__ uint32_t tf32_rn_bits(float x) {
    const uint32_t u = __float_as_uint(x);
    const uint32_t r = (u + 0x0FFFu + ((u >> 13) & 1u)) & 0xFFFFE000u;
    return ((r & 0x7F800000u) == 0x7F800000u) ? (u & 0xFFFFE000u) : r;
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start before the kernel ahead of it in the stream has
// finished; griddep_wait() makes the calling thread wait until that kernel
// has completed and its writes are visible (it returns at once when nothing
// is pending), and griddep_launch_dependents() lets the next such kernel
// start launching now.
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// x = hi + lo / lo_scale, both TF32: lo_scale = 1 for TF32x3, 2^11 for the
// Ootomo-Yokota variant (the residual is scaled before its rounding; the
// scaling by a power of two is exact).
__device__ __forceinline__ void split_tf32x2(float x, float& hi, float& lo, float lo_scale = 1.0f) {
    const uint32_t u = __float_as_uint(x);
    if ((u & 0x7F800000u) == 0x7F800000u) {
        const bool nan = (u & 0x007FFFFFu) != 0;
        hi = nan ? __uint_as_float(0x7FC00000u) : x;
        lo = nan ? __uint_as_float(0x7FC00000u) : 0.0f;
        return;
    }
    hi = __uint_as_float(tf32_rn_bits(x));
    lo = __uint_as_float(tf32_rn_bits(__fmul_rn(__fsub_rn(x, hi), lo_scale)));
}

}  // namespace emu
