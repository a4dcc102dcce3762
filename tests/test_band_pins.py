"""CPU pins for the nine-product band test inputs (tests/band_cases.py).

Each input kind makes a known set of the nine BF16x9 products a_i b_j
("Blackwell의 BF16x9" section of the discuss.pytorch.kr page; Figure 1 caption
of the NVIDIA blog post) and keeps every partial sum exact in FP32.  These
tests show, without a GPU, that
  * the pieces of the constructed values are the ones the construction states
    (checked against the split's definition: the three pieces sum back to x
    and each is a BF16 value);
  * the exact product is an FP32 number, and the oracle's BF16x9 emulation
    returns it bit for bit;
  * an emulation that leaves out any one of the nine products -- or keeps
    only bands 0-2 (six products) or 0-3 (eight) -- returns different bits
    on a large share of the outputs, so the GPU tests built on these inputs
    cannot be passed by a kernel that skips a product;
  * the same holds for the cheaper rungs and TF32x3 (Figure 2): with a
    first-piece operand their exact result is the sum of the products they
    keep, and dropping one of them changes it.
"""
import os
import re
import tempfile

import numpy as np
import pytest

import oracle
import band_cases as BC

SHAPES = [(37, 29, 150, 0, 0), (40, 33, 200, 1, 1), (24, 64, 129, 0, 1)]


def _f(P):
    return oracle.bf16_bits_to_f32(P).astype(np.float64)


def _pieces(A, B, transA, transB):
    """float64 pieces of op(A) (M x K) and op(B)^T (N x K)."""
    pa = [_f(p) for p in oracle.split_bf16x3(A, transA)]
    pb = [_f(p) for p in oracle.split_bf16x3(B, not transB)]
    return pa, pb


def _emulate(pa, pb, keep):
    """sum over the kept (i, j) of 2^-8(i+j) a_i b_j, in float64 (exact here)."""
    C = 0.0
    for (i, j) in keep:
        C = C + np.ldexp(pa[i] @ pb[j].T, -8 * (i + j))
    return C


ALL9 = [(i, j) for i in range(3) for j in range(3)]


@pytest.mark.parametrize("x,pieces", [
    (2.0 ** -135, (0.0, 2.0 ** -127, 0.0)),
    (2.0 ** -136, (0.0, 2.0 ** -128, 0.0)),
    (2.0 ** -143, (0.0, 0.0, 2.0 ** -127)),
    (-2.0 ** -144, (0.0, 0.0, -2.0 ** -128)),
    (1 + 2.0 ** -9 + 2.0 ** -17, (1.0, 0.5, 0.5)),
    (1 + 2.0 ** -8 - 2.0 ** -17, (1.0, 1.0, -0.5)),
    (1.5 + 2.0 ** -9 + 2.0 ** -17, (1.5, 0.5, 0.5)),
])
def test_constructed_values_have_the_stated_pieces(x, pieces):
    X = np.array([[x]], np.float32)
    assert float(X[0, 0]) == x                       # representable in FP32
    got = tuple(float(oracle.bf16_bits_to_f32(p)[0, 0]) for p in oracle.split_bf16x3(X))
    assert got == pieces
    assert pieces[0] + 2.0 ** -8 * pieces[1] + 2.0 ** -16 * pieces[2] == x


def test_three_piece_values_are_two_tf32_pieces():
    for v in BC.THREE_PIECE:
        X = np.array([[v * 2.0 ** 20, -v * 2.0 ** 19]], np.float32)
        hi, lo = oracle.split_tf32x2(X)
        assert np.array_equal(hi.astype(np.float64) + lo, X.astype(np.float64))
        assert np.all(np.abs(lo) == np.array([[2.0 ** 3, 2.0 ** 2]]))


@pytest.mark.parametrize("kind", BC.KINDS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_exact_result_is_fp32_and_the_oracle_returns_it(kind, shape):
    M, N, K, tA, tB = shape
    A, B = BC.make(kind, M, N, K, tA, tB, seed=M + N + K)
    E = BC.exact(A, B, tA, tB)
    assert np.array_equal(E.astype(np.float32).astype(np.float64), E)
    assert np.count_nonzero(E) > 0.5 * E.size
    C = oracle.gemm_bf16x9(A, B, tA, tB)
    assert np.array_equal(C.astype(np.float64), E)
    Cref, _ = oracle.gemm_ref(A, B, tA, tB)
    assert np.array_equal(Cref, E)
    # the nine products of the oracle's own pieces re-sum to the same value
    pa, pb = _pieces(A, B, tA, tB)
    assert np.array_equal(_emulate(pa, pb, ALL9), E)


def test_power_of_two_alpha_keeps_the_result_exact():
    A, B = BC.make("a2", 31, 17, 90, seed=4)
    C = oracle.gemm_bf16x9(A, B, alpha=2.0 ** 64)
    assert np.array_equal(C.astype(np.float64), np.ldexp(BC.exact(A, B), 64))


@pytest.mark.parametrize("ij", ALL9, ids=lambda t: f"a{t[0]}b{t[1]}")
def test_dropping_any_one_product_changes_the_result(ij):
    """For every product a_i b_j, the kinds that make it detect its absence
    on most of their nonzero outputs."""
    kinds = [k for k in BC.KINDS if ij in BC.TOUCHES[k]]
    assert kinds
    for kind in kinds:
        for (M, N, K, tA, tB) in SHAPES:
            A, B = BC.make(kind, M, N, K, tA, tB, seed=M + N + K)
            E = BC.exact(A, B, tA, tB)
            pa, pb = _pieces(A, B, tA, tB)
            D = _emulate(pa, pb, [p for p in ALL9 if p != ij]).astype(np.float32)
            nz = E != 0
            assert np.mean(D[nz] != E[nz]) > 0.9, (kind, ij)


@pytest.mark.parametrize("kind", ["a1", "a2", "b1", "b2"])
def test_six_and_eight_product_kernels_fail(kind):
    """Keeping bands 0-2 only (six products), or bands 0-3 (eight: a2 b2
    dropped), changes the result wherever the kind reaches those bands."""
    M, N, K, tA, tB = SHAPES[0]
    A, B = BC.make(kind, M, N, K, tA, tB, seed=7)
    E = BC.exact(A, B, tA, tB)
    pa, pb = _pieces(A, B, tA, tB)
    nz = E != 0
    six = _emulate(pa, pb, [p for p in ALL9 if sum(p) <= 2]).astype(np.float32)
    assert np.mean(six[nz] != E[nz]) > 0.9
    if kind in ("a2", "b2"):
        eight = _emulate(pa, pb, [p for p in ALL9 if p != (2, 2)]).astype(np.float32)
        assert np.mean(eight[nz] != E[nz]) > 0.9


def test_mutant_oracle_without_band4_fails_the_pin():
    src = open(oracle._SRC).read()
    mutated, n = re.subn(r"acc \+= ldexpf\(prod, -8 \* b\);",
                         "if (b != 4) acc += ldexpf(prod, -8 * b);", src)
    assert n == 1
    d = tempfile.mkdtemp(prefix="oracle_mutant_")
    c = os.path.join(d, "mutant.c")
    with open(c, "w") as f:
        f.write(mutated)
    L = oracle.load(oracle.compile_c(c, os.path.join(d, "mutant.so")))
    A, B = BC.make("b2", 40, 24, 100, seed=9)
    E = BC.exact(A, B)
    assert not np.array_equal(oracle.gemm_bf16x9(A, B, L=L).astype(np.float64), E)
    assert np.array_equal(oracle.gemm_bf16x9(A, B).astype(np.float64), E)


# ---------------------------------------------------- the other modes --
# With a first-piece operand (kind a0: A = +-1, +-1/2; b0: the same in B) the
# other operand's three-piece values are hi + lo exactly in TF32, so TF32x3
# and its Ootomo-Yokota variant must return the exact product; the two
# cheaper rungs must return the exact sum of the products they keep.

def _tf32_pieces(X, trans):
    hi, lo = oracle.split_tf32x2(X, trans)
    return hi.astype(np.float64), lo.astype(np.float64)


@pytest.mark.parametrize("kind", ["a0", "b0"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_ladder_modes_return_the_sum_of_their_products(kind, shape):
    M, N, K, tA, tB = shape
    A, B = BC.make(kind, M, N, K, tA, tB, seed=M * N + K)
    E = BC.exact(A, B, tA, tB)
    nz = E != 0
    # TF32x3 and the Ootomo-Yokota variant: the exact product
    ah, al = _tf32_pieces(A, tA)
    bh, bl = _tf32_pieces(B, not tB)
    for fn in (oracle.gemm_tf32x3, oracle.gemm_tf32x3_oy):
        assert np.array_equal(fn(A, B, tA, tB).astype(np.float64), E)
    no_hl = (ah @ bh.T + al @ bh.T).astype(np.float32)     # hi*lo dropped
    no_lh = (ah @ bh.T + ah @ bl.T).astype(np.float32)     # lo*hi dropped
    dropped = no_hl if kind == "a0" else no_lh             # the one that is nonzero
    assert np.mean(dropped[nz] != E[nz]) > 0.9
    # single-pass TF32: hi * hi
    T = (ah @ bh.T)
    assert np.array_equal(T.astype(np.float32).astype(np.float64), T)
    assert np.array_equal(oracle.gemm_tf32(A, B, tA, tB).astype(np.float64), T)
    # two BF16 pieces: a0 b0 + 2^-8 (a0 b1 + a1 b0)
    pa, pb = _pieces(A, B, tA, tB)
    X3 = _emulate(pa, pb, [(0, 0), (0, 1), (1, 0)])
    assert np.array_equal(oracle.gemm_bf16x3(A, B, tA, tB).astype(np.float64), X3)
    assert np.mean(X3[nz] != E[nz]) > 0.9                  # the third pieces are gone
    one = _emulate(pa, pb, [(0, 0)]).astype(np.float32)
    assert np.mean(one[nz] != X3[nz]) > 0.9                # band 1 is there
