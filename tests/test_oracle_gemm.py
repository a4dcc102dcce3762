"""Pins for the oracle's GEMMs: the FP64 reference and the CPU BF16x9 / TF32x3
emulations.

What fixes the expected values (none is the oracle itself):
  * numpy's float64 matmul for the FP64 reference (a library routine);
  * closed forms: identity and diagonal power-of-two operands, all-ones, and
    integer inputs whose every partial sum is exact in FP32 -- the emulation
    must then return the exact product;
  * the exactness of the three-way split ("Blackwell의 BF16x9" section of the
    discuss.pytorch.kr page): the nine products, scaled by 2^-8(i+j) and
    summed, must equal sum_k a_k b_k up to double rounding, which pins the set
    of terms in the five bands;
  * the TF32x3 identity a*b ~ a_hi b_hi + a_hi b_lo + a_lo b_hi (equation
    under Figure 2 of the NVIDIA blog post);
  * the accuracy claim of the pages (BF16x9 matches or beats native FP32
    against an FP64 reference) and the element-wise and Frobenius criteria.
Mutation tests at the end compile broken copies of the C oracle and check that
these pins reject them.
"""
import os
import re
import tempfile
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import checks
from fp32_emulated_gemm_split_gb300 import workloads as W

R = lambda seed: np.random.Generator(np.random.PCG64(seed))  # noqa: E731


def _op(X, t):
    return X.T if t else X


# --------------------------------------------------------------------------
# FP64 reference
# --------------------------------------------------------------------------

@pytest.mark.parametrize("transA,transB", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_f64_reference_matches_numpy(transA, transB):
    r = R(21 + 2 * transA + transB)
    M, N, K = 37, 29, 53
    A = r.standard_normal((K, M) if transA else (M, K)).astype(np.float32)
    B = r.standard_normal((N, K) if transB else (K, N)).astype(np.float32)
    C0 = r.uniform(-1, 1, (M, N)).astype(np.float32)
    Cref, Sabs = oracle.gemm_ref(A, B, transA, transB, alpha=1.5, beta=-0.25, C0=C0)
    a = _op(A, transA).astype(np.float64)
    b = _op(B, transB).astype(np.float64)
    expect = 1.5 * (a @ b) - 0.25 * C0.astype(np.float64)
    sabs = np.abs(a) @ np.abs(b)
    assert np.allclose(Sabs, sabs, rtol=1e-13, atol=0)
    assert np.all(np.abs(Cref - expect) <= 1e-13 * (1.5 * sabs + 0.25 * np.abs(C0)))


def test_f64_reference_strided_views_and_pairs():
    r = R(5)
    big = r.standard_normal((40, 70)).astype(np.float32)
    A = big[:, 3:35]          # 40 x 32, row stride 70
    B = r.standard_normal((32, 24)).astype(np.float32)
    Cref, _ = oracle.gemm_ref(A, B)
    assert np.allclose(Cref, A.astype(np.float64) @ B.astype(np.float64), rtol=1e-12, atol=1e-12)
    mi = np.array([0, 39, 17], np.int64)
    ni = np.array([23, 0, 5], np.int64)
    Cp, _ = oracle.gemm_ref(A, B, pairs=(mi, ni))
    assert np.array_equal(Cp, Cref[mi, ni])


# --------------------------------------------------------------------------
# Closed forms: the emulation must be exact
# --------------------------------------------------------------------------

EMUS = [("bf16x9", oracle.gemm_bf16x9), ("tf32x3", oracle.gemm_tf32x3)]


@pytest.mark.parametrize("name,emu", EMUS)
def test_identity_reproduces_other_operand_bitwise(name, emu):
    r = R(31)
    X = r.standard_normal((8, 8)).astype(np.float32)
    I = np.eye(8, dtype=np.float32)
    if name == "bf16x9":
        # the three pieces of every element re-add exactly
        assert np.array_equal(emu(I, X), X)
        assert np.array_equal(emu(X, I), X)
        big = W.normal(R(32), (256, 256))
        assert np.array_equal(emu(np.eye(256, dtype=np.float32), big), big)
    else:
        # TF32x3 keeps hi + lo of each element, 22 of the 24 bits
        hi, lo = oracle.split_tf32x2(X)
        assert np.array_equal(emu(I, X), lo + hi)


def test_bf16x9_diagonal_power_of_two_scaling():
    r = R(33)
    X = r.standard_normal((8, 8)).astype(np.float32)
    e = np.arange(-4, 4)
    D = np.diag(np.ldexp(1.0, e)).astype(np.float32)
    expect = (np.ldexp(1.0, e)[:, None] * X.astype(np.float64)).astype(np.float32)
    assert np.array_equal(oracle.gemm_bf16x9(D, X), expect)


@pytest.mark.parametrize("name,emu", EMUS)
def test_ones_gives_K(name, emu):
    K = 256
    A = np.ones((4, K), np.float32)
    B = np.ones((K, 3), np.float32)
    assert np.all(emu(A, B) == K)


def _bruteforce_cases():
    r = R(41)
    cases = []
    z = np.zeros((8, 8), np.float32)
    cases.append(("zeros", z, r.standard_normal((8, 8)).astype(np.float32)))
    sgn = lambda s: np.where(r.random(s) < 0.5, -1.0, 1.0)  # noqa: E731
    p2a = (sgn((8, 8)) * np.ldexp(1.0, r.integers(-5, 6, (8, 8)))).astype(np.float32)
    p2b = (sgn((8, 8)) * np.ldexp(1.0, r.integers(-5, 6, (8, 8)))).astype(np.float32)
    cases.append(("pow2", p2a, p2b))
    # 21-bit integers (all three BF16 pieces nonzero) times {-1, 0, 1}:
    # every partial sum is an integer below 2^24, so exact in FP32.
    big = r.integers(-(1 << 20), 1 << 20, (8, 8)).astype(np.float32)
    tern = r.integers(-1, 2, (8, 8)).astype(np.float32)
    cases.append(("int21_x_ternary", big, tern))
    cases.append(("ternary_x_int21", tern, big))
    # 13-bit integers times 8-bit integers: products < 2^21, sums < 2^24
    i13 = r.integers(-(1 << 12), 1 << 12, (8, 8)).astype(np.float32)
    i8 = r.integers(-(1 << 7), 1 << 7, (8, 8)).astype(np.float32)
    cases.append(("int13_x_int8", i13, i8))
    return cases


@pytest.mark.parametrize("case", _bruteforce_cases(), ids=lambda c: c[0])
def test_bf16x9_bruteforce_8x8x8_exact(case):
    _, A, B = case
    exact = A.astype(np.float64) @ B.astype(np.float64)     # exact: small integers / powers of two
    assert np.all(np.abs(exact) < 2 ** 24)
    assert np.array_equal(oracle.gemm_bf16x9(A, B), exact.astype(np.float32))
    for ta, tb in [(1, 0), (0, 1), (1, 1)]:
        C = oracle.gemm_bf16x9(np.ascontiguousarray(_op(A, ta)), np.ascontiguousarray(_op(B, tb)),
                               transA=ta, transB=tb)
        assert np.array_equal(C, exact.astype(np.float32))


def test_bruteforce_golden_fixture():
    """Cases stored under tests/golden (closed-form expected values)."""
    path = os.path.join(os.path.dirname(__file__), "golden", "bruteforce_8x8x8.txt")
    cases = _read_golden(path)
    assert len(cases) >= 4
    for name, A, B, alpha, beta, C0, expect in cases:
        C = oracle.gemm_bf16x9(A, B, alpha=alpha, beta=beta, C0=C0)
        assert np.array_equal(C, expect), name


def _read_golden(path):
    cases = []
    with open(path) as f:
        lines = [l.strip() for l in f if l.strip() and not l.startswith("#")]
    i = 0
    while i < len(lines):
        head = lines[i].split()
        assert head[0] == "case"
        name, alpha, beta = head[1], float.fromhex(head[2]), float.fromhex(head[3])
        mats = {}
        i += 1
        for key in ("A", "B", "C0", "C"):
            assert lines[i] == key
            vals = [float.fromhex(v) for row in lines[i + 1:i + 9] for v in row.split()]
            mats[key] = np.array(vals, np.float32).reshape(8, 8)
            i += 9
        cases.append((name, mats["A"], mats["B"], alpha, beta, mats["C0"], mats["C"]))
    return cases


# --------------------------------------------------------------------------
# The set of terms: exactness of the nine-product decomposition
# --------------------------------------------------------------------------

def test_bf16x9_band_sums_recompose_the_exact_dot_product():
    r = R(51)
    M, N, K = 4, 5, 16
    A = (r.standard_normal((M, K)) * np.exp2(r.integers(-6, 6, (M, K)))).astype(np.float32)
    B = (r.standard_normal((K, N)) * np.exp2(r.integers(-6, 6, (K, N)))).astype(np.float32)
    _, bands = oracle.gemm_bf16x9(A, B, with_bands=True)
    _, Sabs = oracle.gemm_ref(A, B)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(float(A[m, k])) * Fraction(float(B[k, n])) for k in range(K))
            got = sum(Fraction(float(bands[m, n, b])) * Fraction(2) ** (-8 * b) for b in range(5))
            assert abs(float(got - exact)) <= 2.0 ** -50 * Sabs[m, n]
            # every band carries its own share: drop one and the identity breaks
            for b in range(5):
                if bands[m, n, b] != 0:
                    part = Fraction(float(bands[m, n, b])) * Fraction(2) ** (-8 * b)
                    assert abs(float(got - part - exact)) > 2.0 ** -50 * Sabs[m, n]


def test_tf32x3_band_sums_are_the_three_products():
    r = R(52)
    M, N, K = 3, 4, 16
    A = r.standard_normal((M, K)).astype(np.float32)
    B = r.standard_normal((K, N)).astype(np.float32)
    _, bands = oracle.gemm_tf32x3(A, B, with_bands=True)
    ah, al = oracle.split_tf32x2(A)
    bh, bl = oracle.split_tf32x2(B)
    F = lambda v: Fraction(float(v))  # noqa: E731
    for m in range(M):
        for n in range(N):
            hh = sum(F(ah[m, k]) * F(bh[k, n]) for k in range(K))
            mixed = sum(F(ah[m, k]) * F(bl[k, n]) + F(al[m, k]) * F(bh[k, n]) for k in range(K))
            assert abs(float(F(bands[m, n, 0]) - hh)) <= 2.0 ** -52 * abs(float(hh))
            assert abs(float(F(bands[m, n, 1]) - mixed)) <= 2.0 ** -52 * float(abs(mixed)) + 1e-300


# --------------------------------------------------------------------------
# Accuracy: the spec criteria and the pages' claim
# --------------------------------------------------------------------------

def _accuracy_case(g: W.Gemm, mode):
    A, B, C0 = W.generate(g)
    emu = oracle.gemm_bf16x9 if mode == "bf16x9" else oracle.gemm_tf32x3
    C = emu(A, B, g.transA, g.transB, g.alpha, g.beta, C0)
    Cref, Sabs = oracle.gemm_ref(A, B, g.transA, g.transB, g.alpha, g.beta, C0)
    return C, Cref, Sabs, C0


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
def test_square256_within_bounds(mode):
    g = W.WORKLOADS["square256_uniform"]
    C, Cref, Sabs, _ = _accuracy_case(g, mode)
    assert checks.error_ratio(C, Cref, Sabs, g.K, g.alpha, g.beta, mode=mode) <= 1.0
    assert checks.rel_frobenius(C, Cref) <= checks.FROBENIUS_TOL


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
def test_mlip_layer_shape_within_bounds(mode):
    g = W.Gemm("mlip_small", 512, 256, 1024, transB=True, dist="mlip", seed=9)
    C, Cref, Sabs, _ = _accuracy_case(g, mode)
    assert checks.error_ratio(C, Cref, Sabs, g.K, 1.0, 0.0, mode=mode) <= 1.0
    assert checks.rel_frobenius(C, Cref) <= checks.FROBENIUS_TOL


def test_stress_distribution_with_alpha_beta_within_bounds():
    g = W.Gemm("stress_small", 48, 40, 4096, alpha=1.5, beta=0.5, dist="stress", seed=4)
    C, Cref, Sabs, C0 = _accuracy_case(g, "bf16x9")
    assert checks.error_ratio(C, Cref, Sabs, g.K, g.alpha, g.beta, C0) <= 1.0


def test_bf16x9_at_least_as_accurate_as_plain_fp32():
    """The pages: against an FP64 reference BF16x9 matches or beats native FP32."""
    r = R(61)
    A = W.normal(r, (256, 256))
    B = W.normal(r, (256, 256))
    Cref, _ = oracle.gemm_ref(A, B)
    e9 = checks.rel_frobenius(oracle.gemm_bf16x9(A, B), Cref)
    e32 = checks.rel_frobenius(oracle.gemm_fp32(A, B), Cref)
    assert e9 <= e32


def test_k_zero_alpha_zero_and_beta_semantics():
    r = R(71)
    A = np.zeros((4, 0), np.float32)
    B = np.zeros((0, 3), np.float32)
    C0 = r.uniform(-1, 1, (4, 3)).astype(np.float32)
    for emu in (oracle.gemm_bf16x9, oracle.gemm_tf32x3, oracle.gemm_fp32):
        assert np.array_equal(emu(A, B, beta=0.5, C0=C0), (np.float32(0.5) * C0))
    A = np.full((4, 5), np.nan, np.float32)
    B = np.ones((5, 3), np.float32)
    # alpha == 0: A and B are not read; beta == 0: C0 is not read
    assert np.array_equal(oracle.gemm_bf16x9(A, B, alpha=0.0, beta=2.0, C0=C0), 2 * C0)
    C0n = np.full((4, 3), np.nan, np.float32)
    assert np.all(oracle.gemm_bf16x9(np.ones((4, 5), np.float32), B, beta=0.0, C0=C0n) == 5)


# --------------------------------------------------------------------------
# Mutation tests: broken copies of the oracle must fail the pins above
# --------------------------------------------------------------------------

def _mutant(pattern, repl):
    src = open(oracle._SRC).read()
    mutated, n = re.subn(pattern, repl, src)
    assert n >= 1, pattern
    d = tempfile.mkdtemp(prefix="oracle_mutant_")
    c = os.path.join(d, "mutant.c")
    with open(c, "w") as f:
        f.write(mutated)
    return oracle.load(oracle.compile_c(c, os.path.join(d, "mutant.so")))


def test_mutant_dropping_band4_fails_band_identity():
    L = _mutant(r"acc \+= ldexpf\(prod, -8 \* b\);\n(\s*)bs\[b\] \+= \(double\)ai \* \(double\)bj;",
                r"if (b != 4) { acc += ldexpf(prod, -8 * b); bs[b] += (double)ai * (double)bj; }")
    r = R(51)
    A = r.standard_normal((2, 16)).astype(np.float32)
    B = r.standard_normal((16, 2)).astype(np.float32)
    _, bands = oracle.gemm_bf16x9(A, B, with_bands=True, L=L)
    _, Sabs = oracle.gemm_ref(A, B)
    exact = sum(Fraction(float(A[0, k])) * Fraction(float(B[k, 0])) for k in range(16))
    got = sum(Fraction(float(bands[0, 0, b])) * Fraction(2) ** (-8 * b) for b in range(5))
    assert abs(float(got - exact)) > 2.0 ** -50 * Sabs[0, 0]


def test_mutant_wrong_band_scale_fails_identity():
    L = _mutant(r"ldexpf\(prod, -8 \* b\)", "ldexpf(prod, -7 * b)")
    X = W.normal(R(31), (8, 8))
    I = np.eye(8, dtype=np.float32)
    assert not np.array_equal(oracle.gemm_bf16x9(I, X, L=L), X)


def test_mutant_truncating_split_fails_rint_pin():
    L = _mutant(r"uint32_t r = u \+ 0x7FFFu \+ \(\(u >> 16\) & 1u\);", "uint32_t r = u;")
    x = W.normal(R(12), (1, 4096))
    p0, _, _ = oracle.split_bf16x3(x, L=L)
    ref, _, _ = oracle.split_bf16x3(x)
    # the torch/rint pins compare against nearest-even values; truncation differs
    import torch
    t = torch.from_numpy(x.ravel().copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ref.ravel(), t) and not np.array_equal(p0.ravel(), t)


def test_mutant_transposed_operand_fails_reference_pin():
    L = _mutant(r"return trans \? X\[c \* ld \+ r\] : X\[r \* ld \+ c\];",
                "return trans ? X[r * ld + c] : X[r * ld + c];")
    r = R(22)
    A = r.standard_normal((6, 6)).astype(np.float32)
    B = r.standard_normal((6, 6)).astype(np.float32)
    Cref, _ = oracle.gemm_ref(A, B, transA=1, L=L)
    assert not np.allclose(Cref, A.T.astype(np.float64) @ B.astype(np.float64))


def test_mutant_dropping_tf32_mixed_term_fails_band_pin():
    L = _mutant(r"float t2 = al\[k\] \* bh\[k\];\n(\s*)acc \+= t2;", "float t2 = 0.0f;")
    r = R(52)
    A = r.standard_normal((3, 16)).astype(np.float32)
    B = r.standard_normal((16, 4)).astype(np.float32)
    Cm = oracle.gemm_tf32x3(A, B, L=L)
    Cref, Sabs = oracle.gemm_ref(A, B)
    assert checks.error_ratio(Cm, Cref, Sabs, 16, 1.0, 0.0, mode="tf32x3") > 1.0


# --------------------------------------------------------------------------
# The cheaper rungs: two BF16 pieces (three products) and single-pass TF32
# --------------------------------------------------------------------------

def test_bf16x3_identity_keeps_the_first_two_pieces():
    X = W.normal(R(81), (64, 64))
    I = np.eye(64, dtype=np.float32)
    p0, p1, _ = oracle.split_bf16x3(X)
    f = oracle.bf16_bits_to_f32
    expect = (f(p0).astype(np.float64) + np.ldexp(f(p1), -8)).astype(np.float32)
    assert np.array_equal(oracle.gemm_bf16x3(I, X), expect)
    assert np.array_equal(oracle.gemm_bf16x3(X, I), expect)


def test_tf32_identity_keeps_the_leading_piece():
    X = W.normal(R(82), (64, 64))
    I = np.eye(64, dtype=np.float32)
    hi, _ = oracle.split_tf32x2(X)
    assert np.array_equal(oracle.gemm_tf32(I, X), hi)
    assert np.array_equal(oracle.gemm_tf32(X, I), hi)


@pytest.mark.parametrize("mode,fn", [("bf16x3", oracle.gemm_bf16x3), ("tf32", oracle.gemm_tf32)])
def test_cheaper_rungs_within_their_bounds_and_ordered(mode, fn):
    r = R(83)
    A = W.normal(r, (128, 512))
    B = W.normal(r, (512, 96))
    Cref, Sabs = oracle.gemm_ref(A, B)
    C = fn(A, B)
    assert checks.error_ratio(C, Cref, Sabs, 512, 1.0, 0.0, mode=mode) <= 1.0
    # the ladder the pages describe: the cheaper rung is less accurate
    e = checks.rel_frobenius(C, Cref)
    e9 = checks.rel_frobenius(oracle.gemm_bf16x9(A, B), Cref)
    e3 = checks.rel_frobenius(oracle.gemm_tf32x3(A, B), Cref)
    assert e > 5 * max(e9, e3)
    assert e > checks.FROBENIUS_TOL       # misses the criterion BF16x9 and TF32x3 meet


def test_bf16x3_piece_error_matches_its_bound():
    """The two-piece representation error, measured on the oracle's own
    split over 2^20 normal values: |x - x0 - 2^-8 x1| reaches 2^-17 |x| (not
    less: 2^-18 would be too small) and never exceeds it; the kept products
    of random pairs miss by more than 2^-16 |a||b| and never by more than
    the rung's allowance, 2^-15 + 2^-22."""
    r = R(85)
    x = W.normal(r, (1, 1 << 20))
    p0, p1, _ = oracle.split_bf16x3(x)
    f = lambda p: (p.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    x0, x1 = f(p0)[0], f(p1)[0]
    xd = x[0].astype(np.float64)
    rel = np.abs(xd - x0 - 2.0 ** -8 * x1) / np.abs(xd)
    assert 2.0 ** -18 < rel.max() <= 2.0 ** -17
    h = xd.size // 2
    a, b = xd[:h], xd[h:]
    kept = x0[:h] * x0[h:] + 2.0 ** -8 * (x0[:h] * x1[h:] + x1[:h] * x0[h:])
    err = np.abs(a * b - kept) / np.abs(a * b)
    assert 2.0 ** -16 < err.max() <= checks.MODE_EXTRA["bf16x3"]


def _subnormals_and_edge(r, n):
    """FP32 subnormals (random mantissa, both signs) and normals just above
    2^-126, whose residuals after the first piece are subnormal."""
    sub = (r.integers(1, 1 << 23, n, dtype=np.uint32) |
           (r.integers(0, 2, n, dtype=np.uint32) << 31)).view(np.float32)
    edge = (np.ldexp(r.uniform(1.0, 2.0, n), r.integers(-126, -118, n)) *
            np.where(r.random(n) < 0.5, -1.0, 1.0)).astype(np.float32)
    return np.concatenate([sub, edge]).reshape(1, -1)


def test_split_errors_below_the_normal_range_match_their_bounds():
    """MODE_SUB_ABS, pinned on the oracle's own splits: over 2^17 FP32
    subnormals and small normals the absolute representation error reaches
    within a factor two of each rung's constant and never exceeds it; BF16x9
    represents every one exactly (its third piece reaches 2^-149)."""
    x = _subnormals_and_edge(R(86), 1 << 16)
    xd = x[0].astype(np.float64)
    f = lambda p: (p.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    p0, p1, p2 = oracle.split_bf16x3(x)
    b0, b1, b2 = f(p0)[0], f(p1)[0], f(p2)[0]
    hi, lo = oracle.split_tf32x2(x)
    hs, ls = oracle.split_tf32x2s(x)
    err = {
        "bf16x9": np.abs(xd - b0 - 2.0 ** -8 * b1 - 2.0 ** -16 * b2),
        "bf16x3": np.abs(xd - b0 - 2.0 ** -8 * b1),
        "tf32x3": np.abs(xd - hi[0] - lo[0].astype(np.float64)),
        "tf32": np.abs(xd - hi[0]),
        "tf32x3_oy": np.abs(xd - hs[0] - 2.0 ** -11 * ls[0].astype(np.float64)),
    }
    assert err["bf16x9"].max() == 0.0
    for mode in ("bf16x3", "tf32x3", "tf32", "tf32x3_oy"):
        e = checks.MODE_SUB_ABS[mode]
        # the relative part is allowed too: |x - x^| <= rho |x| + E
        rho = {"bf16x3": 2.0 ** -17, "tf32x3": 2.0 ** -22, "tf32": 2.0 ** -11,
               "tf32x3_oy": 2.0 ** -22}[mode]
        assert np.all(err[mode] <= rho * np.abs(xd) + e), mode
        assert err[mode][: 1 << 16].max() > e / 2, mode          # attained on subnormals


def test_subnormal_partial_sums_are_scaled_by_alpha():
    """A product among FP32 subnormals keeps only a few bits in the FP32
    accumulator (spacing 2^-149), and the epilogue multiplies that error by
    alpha.  K = 1, a = 1.2345 * 2^-72, b = 1.4567 * 2^-72 (normal; a b about
    57.5 * 2^-149), alpha = 2^17: the oracle's BF16x9 misses the FP64 result
    by about 0.46 * 2^-132, over ten times the subnormal term taken in the
    result's units, and within it taken in the accumulator's (times
    |alpha|)."""
    a = np.array([[1.2345 * 2.0 ** -72]], np.float32)
    b = np.array([[1.4567 * 2.0 ** -72]], np.float32)
    alpha = 2.0 ** 17
    Cref, Sabs = oracle.gemm_ref(a, b, alpha=alpha)
    C = oracle.gemm_bf16x9(a, b, alpha=alpha)
    err = abs(float(C[0, 0]) - float(Cref[0, 0]))
    unscaled = 4 * 2.0 ** -24 * alpha * float(Sabs[0, 0]) + 13 * 2.0 ** -149
    assert err > 10 * unscaled
    assert checks.error_ratio(C, Cref, Sabs, 1, alpha, 0.0) <= 1.0


def test_subnormal_operands_need_the_absolute_term():
    """K = 1, a a subnormal that TF32 cannot hold to the last bit, b = 1.5 *
    2^30: the oracle's TF32x3 product misses by about 2^-137 * 2^30, far
    above the relative terms, and within them once the absolute term
    (operand_l1) is added."""
    a = np.array([[np.float32(np.uint32(0x00000FFF).view(np.float32))]])   # 4095 * 2^-149
    b = np.array([[np.float32(1.5 * 2.0 ** 30)]], np.float32)
    Cref, Sabs = oracle.gemm_ref(a, b)
    C = oracle.gemm_tf32x3(a, b)
    assert checks.error_ratio(C, Cref, Sabs, 1, 1.0, 0.0, mode="tf32x3") > 100
    S1 = checks.operand_l1(a, b)
    assert checks.error_ratio(C, Cref, Sabs, 1, 1.0, 0.0, mode="tf32x3", S1=S1) <= 1.0


def test_bf16x3_exact_on_16_bit_integers():
    r = R(84)
    A = r.integers(-(1 << 15), 1 << 15, (8, 8)).astype(np.float32)   # 16 significant bits
    B = r.integers(-1, 2, (8, 8)).astype(np.float32)
    exact = A.astype(np.float64) @ B.astype(np.float64)
    assert np.array_equal(oracle.gemm_bf16x3(A, B), exact.astype(np.float32))


def test_cheaper_rungs_drop_exactly_the_stated_terms():
    """1x1x1 closed forms: which pieces and products each rung keeps."""
    def one(fn, a, b):
        return float(fn(np.array([[a]], np.float32), np.array([[b]], np.float32))[0, 0])
    x = 1 + 2.0 ** -8                   # pieces (1, 1, 0)
    y = 1 + 2.0 ** -9 + 2.0 ** -18      # pieces (1, 2^-1, 2^-2)
    # two pieces: a0 b0 + 2^-8 (a0 b1 + a1 b0); a1 b1 = 2^-16 is dropped
    assert one(oracle.gemm_bf16x3, x, x) == 1 + 2.0 ** -7
    assert one(oracle.gemm_bf16x9, x, x) == 1 + 2.0 ** -7 + 2.0 ** -16
    # the third piece never enters
    assert one(oracle.gemm_bf16x3, y, y) == 1 + 2.0 ** -8
    assert one(oracle.gemm_bf16x3, x, y) == 1 + 2.0 ** -8 + 2.0 ** -9
    # single-pass TF32: 10 explicit mantissa bits kept, the rest rounded away
    z = 1 + 2.0 ** -10
    assert one(oracle.gemm_tf32, z, z) == 1 + 2.0 ** -9 + 2.0 ** -20
    assert one(oracle.gemm_tf32, 1 + 2.0 ** -11, 3.0) == 3.0           # tie to even
    assert one(oracle.gemm_tf32, 1 + 3 * 2.0 ** -12, 1.0) == 1 + 2.0 ** -10
    # TF32x3 keeps hi*lo and lo*hi
    assert one(oracle.gemm_tf32x3, 1 + 2.0 ** -11, 1 + 2.0 ** -11) == 1 + 2.0 ** -10


def test_mutant_keeping_a1b1_in_bf16x3_fails_closed_form():
    L = _mutant(r"acc \+= ldexpf\(t2, -8\);",
                "acc += ldexpf(t2, -8); acc += ldexpf(oracle_bf16_to_f32(ap[kk + k]) * "
                "oracle_bf16_to_f32(bp[kk + k]), -16);")
    x = np.array([[1 + 2.0 ** -8]], np.float32)
    assert float(oracle.gemm_bf16x3(x, x, L=L)[0, 0]) != 1 + 2.0 ** -7


# --------------------------------------------------------------------------
# The Ootomo-Yokota variant: residual scaled by 2^11 before its TF32 rounding
# --------------------------------------------------------------------------

def test_scaled_split_is_the_unscaled_split_times_2_11_in_the_normal_range():
    x = W.normal(R(91), (64, 512))
    hi, lo = oracle.split_tf32x2(x)
    hs, ls = oracle.split_tf32x2s(x)
    assert np.array_equal(hs, hi)
    assert np.array_equal(ls, np.ldexp(lo, 11).astype(np.float32))


def test_scaled_split_keeps_residual_bits_below_the_normal_range():
    x = np.float32(2.0 ** -120 * (1 + 2.0 ** -12 + 2.0 ** -21 + 2.0 ** -23))
    X = np.array([[x]], np.float32)
    hs, ls = oracle.split_tf32x2s(X)
    assert hs[0, 0] == np.float32(2.0 ** -120)
    assert ls[0, 0] == np.float32(2.0 ** -121 * (1 + 2.0 ** -9))        # tie to even at 2^-11
    hi, lo = oracle.split_tf32x2(X)
    assert lo[0, 0] == np.float32(2.0 ** -132)                          # subnormal: bits lost
    I = np.ones((1, 1), np.float32)
    assert oracle.gemm_tf32x3_oy(I, X)[0, 0] == np.float32(2.0 ** -120 * (1 + 2.0 ** -12 + 2.0 ** -21))
    assert oracle.gemm_tf32x3(I, X)[0, 0] == np.float32(2.0 ** -120 * (1 + 2.0 ** -12))


def test_oy_equals_tf32x3_bitwise_on_normal_range_data():
    # the scaling is exact there, so every product and sum is the same
    r = R(92)
    A = W.normal(r, (64, 300))
    B = W.normal(r, (300, 48))
    C0 = W.uniform(r, (64, 48))
    assert np.array_equal(oracle.gemm_tf32x3_oy(A, B, alpha=1.5, beta=-0.5, C0=C0),
                          oracle.gemm_tf32x3(A, B, alpha=1.5, beta=-0.5, C0=C0))


def test_oy_within_bound_on_wide_exponent_data():
    r = R(93)
    A = W.stress(r, (96, 512))
    B = W.stress(r, (512, 80))
    Cref, Sabs = oracle.gemm_ref(A, B)
    C = oracle.gemm_tf32x3_oy(A, B)
    assert checks.error_ratio(C, Cref, Sabs, 512, 1.0, 0.0, mode="tf32x3_oy") <= 1.0


def test_mutant_unscaled_residual_fails_oy_equality():
    L = _mutant(r"float r = ldexpf\(x - h, 11\);", "float r = ldexpf(x - h, 10);")
    r = R(94)
    A = W.normal(r, (16, 64))
    B = W.normal(r, (64, 16))
    assert not np.array_equal(oracle.gemm_tf32x3_oy(A, B, L=L), oracle.gemm_tf32x3(A, B))
