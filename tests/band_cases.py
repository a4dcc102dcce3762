"""Seeded GEMM inputs in which each of the nine BF16x9 products leaves its
own bit in a result that FP32 holds exactly.

Why such inputs exist.  The three-way split x = x0 + 2^-8 x1 + 2^-16 x2
("Blackwell의 BF16x9" section of the discuss.pytorch.kr page; Figure 1 caption
of the NVIDIA blog post) rounds each piece to BF16, whose subnormals stop at
2^-133 while FP32's go down to 2^-149.  So

* an FP32 subnormal of magnitude at most 2^-142 rounds to zero at the first
  two steps: the whole value is its third piece, x = 2^-16 x2;
* one of magnitude at most 2^-134 that is a multiple of 2^-141 is its second
  piece alone, x = 2^-8 x1;
* 2^E (1 + 2^-9 + 2^-17), 2^E (1 + 2^-8 - 2^-17) and 2^E (1.5 + 2^-9 + 2^-17)
  have three nonzero power-of-two pieces (2^E, 2^(E-1), 2^(E-1)), (2^E, 2^E,
  -2^(E-1)) and (1.5 2^E, 2^(E-1), 2^(E-1)).

A product of a one-piece operand with a three-piece one is then three
products a_i b_j in three consecutive bands, each contributing a single
distinct bit pattern, and nothing else: with a1-only A the products are a1 b0,
a1 b1, a1 b2 (bands 1-3); with a2-only A, a2 b0, a2 b1, a2 b2 (bands 2-4);
the mirrored kinds put the one-piece values in B.  Keeping at most four such
terms per output and exponents within a factor four makes every partial sum,
in any order, exact in FP32 (at most 22 significant bits), so the exact
product is the only correct answer and a kernel that skips any one of the
products it touches returns different bits.

The three-piece values are also exact sums of two TF32 pieces, hi + lo with
lo = +-2^(E-17) (TF32x3 of Figure 2 of the blog post), so with a first-piece
operand (kinds "a0" and "b0") the cheaper rungs are pinned the same way: each
of them returns, bit for bit, the sum of the products it keeps.

This module only draws inputs (numpy PCG64); it computes nothing of the
method.
"""
from __future__ import annotations

import numpy as np

# kind -> (which operand holds the one-piece values, their magnitudes)
#   "a0": A = +-1, +-1/2 (first piece only): products a0 b0, a0 b1, a0 b2
#   "a1": A = +-2^-135, +-2^-136 (second piece only): a1 b0, a1 b1, a1 b2
#   "a2": A = +-2^-143, +-2^-144 (third piece only): a2 b0, a2 b1, a2 b2
#   "b0", "b1", "b2": the same one-piece values in B, three-piece values in A
KINDS = ("a0", "a1", "a2", "b0", "b1", "b2")
ONE_PIECE = {
    "0": (1.0, 0.5),
    "1": (2.0 ** -135, 2.0 ** -136),
    "2": (2.0 ** -143, 2.0 ** -144),
}
# Products each kind makes (i indexes A's pieces, j B's).
TOUCHES = {
    "a0": [(0, 0), (0, 1), (0, 2)],
    "a1": [(1, 0), (1, 1), (1, 2)],
    "a2": [(2, 0), (2, 1), (2, 2)],
    "b0": [(0, 0), (1, 0), (2, 0)],
    "b1": [(0, 1), (1, 1), (2, 1)],
    "b2": [(0, 2), (1, 2), (2, 2)],
}
THREE_PIECE = (1 + 2.0 ** -9 + 2.0 ** -17, 1 + 2.0 ** -8 - 2.0 ** -17, 1.5 + 2.0 ** -9 + 2.0 ** -17)
MAX_TERMS = 4


def _three_piece(r, shape, E):
    v = np.array(THREE_PIECE)[r.integers(0, len(THREE_PIECE), shape)]
    s = np.where(r.random(shape) < 0.5, -1.0, 1.0)
    e = E - r.integers(0, 2, shape)
    return (s * np.ldexp(v, e)).astype(np.float32)


def _sparse_one_piece(r, rows, K, mags):
    """rows x K: each row holds 0..MAX_TERMS nonzeros at random positions."""
    X = np.zeros((rows, K), np.float32)
    if K == 0:
        return X
    n = r.integers(0, MAX_TERMS + 1, rows)
    n = np.minimum(n, K)
    for i in range(rows):
        cols = r.choice(K, size=int(n[i]), replace=False)
        s = np.where(r.random(cols.size) < 0.5, -1.0, 1.0)
        m = np.array(mags)[r.integers(0, len(mags), cols.size)]
        X[i, cols] = (s * m).astype(np.float32)
    return X


def make(kind: str, M: int, N: int, K: int, transA=False, transB=False, seed=0):
    """(A, B) in their stored layouts for C = op(A) op(B).  The one-piece
    operand is sparse (at most MAX_TERMS nonzeros per row of op(A), or per
    column of op(B)); the other is dense with three-piece values of exponent
    20 or 19 (so every product is a normal FP32 number)."""
    if kind not in KINDS:
        raise ValueError(kind)
    r = np.random.Generator(np.random.PCG64(seed))
    mags = ONE_PIECE[kind[1]]
    if kind[0] == "a":
        opA = _sparse_one_piece(r, M, K, mags)
        opB = _three_piece(r, (K, N), 20)
    else:
        opA = _three_piece(r, (M, K), 20)
        opB = _sparse_one_piece(r, N, K, mags).T
    A = np.ascontiguousarray(opA.T if transA else opA)
    B = np.ascontiguousarray(opB.T if transB else opB)
    return A, B


def exact(A, B, transA=False, transB=False):
    """The exact product in float64 (every sum here is exact in float64)."""
    a = (A.T if transA else A).astype(np.float64)
    b = (B.T if transB else B).astype(np.float64)
    return a @ b
