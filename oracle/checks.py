"""Acceptance criteria for an emulated-FP32 GEMM result (test infrastructure).

The pages say that BF16x9 matches or beats native FP32 accuracy against an
FP64 reference ("Unlocking Tensor Core Performance for Machine Learning
Interatomic Potentials", section "Limitations and decision criteria"); the
criteria below make that concrete:

* element-wise, with u = 2^-24 (unit roundoff of FP32):
      |C - C_ref| <= (2K + 2) u |alpha| S_abs + 2 u |beta C0|
                     + ((9K + 4) |alpha| + 2) 2^-149
  where S_abs = sum_k |a_mk||b_kn|.  2K u |alpha| S_abs is the worst case of a
  K-term FP32 accumulation (one rounding per step, each at most u times the
  running magnitude); the 2u terms cover the two roundings of the epilogue
  alpha*acc + beta*C0; the last term covers products and partial sums that
  land among FP32 subnormals (absolute spacing 2^-149): those roundings
  happen in the accumulator, which the epilogue then multiplies by alpha,
  and the epilogue's own roundings of a subnormal result add up to 2^-149.
* TF32x3 drops the residual*residual product and its residual is itself
  rounded to TF32, which costs at most 3 * 2^-22 |a||b| < 2^-20 |a||b| per
  product, so its bound adds 2^-20 |alpha| S_abs.  The cheaper rungs (two
  BF16 pieces, single-pass TF32) add their own representation error
  (MODE_EXTRA).
* below FP32's normal range the pieces of the split rungs are rounded to
  their format's subnormal quantum, an absolute error per operand
  (MODE_SUB_ABS), and the tensor core's accumulation loses some bits of
  products with an FP32-subnormal operand (TC_SUB_ABS, measured); callers
  that pass S1 = sum_k |a_mk| + |b_kn| get both added.
* relative Frobenius error ||C - C_ref||_F / ||C_ref||_F <= 2e-6 on
  normally distributed inputs.
"""
from __future__ import annotations

import numpy as np

U = 2.0 ** -24
SUB = 2.0 ** -149
FROBENIUS_TOL = 2e-6


# Representation error of the cheaper modes, per product, relative to |a||b|.
# Two BF16 pieces (8 significant bits each, unit roundoff 2^-8): |x - x0| <=
# 2^-8 |x| and |x1| <= (1 + 2^-8) |x|; the second rounding, of 2^8 (x - x0)
# (at most |x| in magnitude, so a half ulp is at most 2^-9 |x| there), leaves
# |x - x0 - 2^-8 x1| <= 2^-17 |x|.  With a^ = a0 + 2^-8 a1 and r_a = a - a^,
# ab minus the kept products a0 b0 + 2^-8 (a0 b1 + a1 b0) is 2^-16 a1 b1 +
# a^ r_b + r_a b^ + r_a r_b, at most (2^-16 (1 + 2^-8)^2 + 2 * 2^-17 (1 +
# 2^-17) + 2^-34) |a||b| < 2^-15 + 2^-22 (random pairs reach 2^-15.1).  One
# TF32 piece leaves |x - hi| <= 2^-11 |x|, so the product misses at most
# 2 * 2^-11 + 2^-22 < 2^-10 + 2^-21.
MODE_EXTRA = {"bf16x9": 0.0, "tf32x3": 2.0 ** -20, "tf32x3_oy": 2.0 ** -20,
              "bf16x3": 2.0 ** -15 + 2.0 ** -22, "tf32": 2.0 ** -10 + 2.0 ** -21}


# Below FP32's normal range (2^-126) a piece is rounded with its format's
# subnormal quantum: TF32 keeps the top 10 of FP32's 23 mantissa bits
# (quantum 2^-136), BF16 the top 7 (2^-133).  So the pieces leave an absolute
# error per operand on top of the relative one: TF32x3 and single-pass TF32 up
# to 2^-137 (the last piece's half quantum), the Ootomo-Yokota split 2^-148
# (its residual is scaled by 2^11 before rounding), two BF16 pieces 2^-142
# (the second piece is scaled by 2^-8), BF16x9 nothing (its third piece
# reaches 2^-149, FP32's own quantum).  A product a b then misses by up to
# E (|a| + |b|) more, and a sum by E S1 with S1 = sum_k |a_mk| + |b_kn|.
MODE_SUB_ABS = {"bf16x9": 0.0, "tf32x3": 2.0 ** -137, "tf32x3_oy": 2.0 ** -148,
                "bf16x3": 2.0 ** -142, "tf32": 2.0 ** -137}

# The tensor core's own loss on FP32-subnormal operands, measured on GB300
# (not a representation error: BF16x9's pieces are exact): with K = 1, a
# product a b whose |a| is below 2^-126 came out up to 64 ulps of the product
# off (2^-17 of |a b|; within 2 ulps from 2^-126 up), so by less than
# 2^-17 * 2^-126 |b| = 2^-143 |b|.  Bound: 2^-142 per unit of the other
# operand, added to every tensor-core mode's E (tests/test_gpu_gemm.py pins
# it: held, and needed).
TC_SUB_ABS = 2.0 ** -142


def operand_l1(A, B, transA=False, transB=False, pairs=None):
    """S1 = sum_k |op(A)[m, k]| + |op(B)[k, n]| (FP64), at `pairs` or for all
    outputs: the weight of MODE_SUB_ABS in the bound."""
    a = np.abs(np.asarray(A, np.float64))
    b = np.abs(np.asarray(B, np.float64))
    ra = a.sum(axis=0) if transA else a.sum(axis=1)          # per row of op(A)
    cb = b.sum(axis=1) if transB else b.sum(axis=0)          # per column of op(B)
    if pairs is None:
        return ra[:, None] + cb[None, :]
    return ra[pairs[0]] + cb[pairs[1]]


def elementwise_bound(K, alpha, beta, Sabs, C0=None, mode="bf16x9", S1=None):
    base = (2 * K + 2) * U + MODE_EXTRA[mode]
    b = base * abs(float(alpha)) * np.asarray(Sabs, np.float64)
    if beta != 0.0:
        b = b + 2 * U * abs(float(beta)) * np.abs(np.asarray(C0, np.float64))
    if S1 is not None:
        e = MODE_SUB_ABS[mode] + TC_SUB_ABS
        b = b + e * (1 + 2.0 ** -10) * abs(float(alpha)) * np.asarray(S1, np.float64)
    return b + ((9 * K + 4) * abs(float(alpha)) + 2) * SUB


def error_ratio(C, Cref, Sabs, K, alpha, beta, C0=None, mode="bf16x9", S1=None):
    """max |C - C_ref| / bound; the result passes when this is <= 1.  With
    operands that reach FP32's subnormals, pass S1 (operand_l1) so that the
    split rungs' absolute error there is allowed for."""
    err = np.abs(np.asarray(C, np.float64) - np.asarray(Cref, np.float64))
    bound = elementwise_bound(K, alpha, beta, Sabs, C0, mode, S1)
    if err.size == 0:
        return 0.0
    return float(np.max(err / bound))


def rel_frobenius(C, Cref):
    Cref = np.asarray(Cref, np.float64)
    d = np.asarray(C, np.float64) - Cref
    den = np.linalg.norm(Cref)
    return float(np.linalg.norm(d) / den) if den > 0 else float(np.linalg.norm(d))
