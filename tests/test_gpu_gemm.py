"""GPU parity of the emulated GEMM (BF16x9, TF32x3) and the SIMT baseline
against the CPU oracle.

Criterion (element-wise, from the method's accuracy claim): |C - C_ref| <=
(2K + 2) 2^-24 |alpha| S_abs + 2^-23 |beta C0| (+2^-20 |alpha| S_abs for
TF32x3), and a relative Frobenius error <= 2e-6 on normally distributed
inputs.  Small cases are compared on every element; the full-size workloads
on 4096 sampled outputs plus the corners, which the oracle computes one by
one.  Closed-form cases (identity, 8x8x8 integers) must match exactly."""
import os

import numpy as np
import pytest

import oracle
from oracle import checks
from fp32_emulated_gemm_split_gb300 import workloads as W
from gpu_util import emu_module, to_dev

pytestmark = pytest.mark.gpu

MODES = ["bf16x9", "tf32x3", "fp32_simt"]


@pytest.fixture(scope="module")
def emu():
    return emu_module()


def _run(emu, A, B, transA=False, transB=False, alpha=1.0, beta=0.0, C0=None, mode="bf16x9"):
    import torch
    M = A.shape[1] if transA else A.shape[0]
    N = B.shape[0] if transB else B.shape[1]
    dC = to_dev(C0) if C0 is not None else torch.full((M, N), float("nan"), device="cuda")
    emu.emu_sgemm(to_dev(A), to_dev(B), dC, transA=transA, transB=transB, alpha=alpha,
                  beta=beta, mode=mode)
    torch.cuda.synchronize()
    return dC.cpu().numpy()


def _bound_mode(mode):
    return "tf32x3" if mode == "tf32x3" else "bf16x9"


# ------------------------------------------------------------ closed forms --

@pytest.mark.parametrize("mode", ["bf16x9", "fp32_simt"])
def test_identity_gives_the_other_operand_bitwise(emu, mode):
    X = W.normal(W.rng(31), (256, 256))
    I = np.eye(256, dtype=np.float32)
    assert np.array_equal(_run(emu, I, X, mode=mode), X)
    assert np.array_equal(_run(emu, X, I, mode=mode), X)


def test_golden_bruteforce_cases_exact(emu):
    from test_oracle_gemm import _read_golden
    path = os.path.join(os.path.dirname(__file__), "golden", "bruteforce_8x8x8.txt")
    for name, A, B, alpha, beta, C0, expect in _read_golden(path):
        for mode in ("bf16x9", "fp32_simt"):
            C = _run(emu, A, B, alpha=alpha, beta=beta, C0=C0, mode=mode)
            assert np.array_equal(C, expect), (name, mode)


def test_ones_gives_K(emu):
    for mode in MODES:
        C = _run(emu, np.ones((130, 1000), np.float32), np.ones((1000, 260), np.float32), mode=mode)
        assert np.all(C == 1000), mode


# ------------------------------------------------------- small, every element --

SHAPES = [(1, 1, 1), (7, 13, 5), (128, 256, 64), (129, 257, 65), (200, 300, 136),
          (300, 513, 1000), (64, 40, 2048)]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("transA,transB", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_ragged_shapes_every_element(emu, mode, shape, transA, transB):
    M, N, K = shape
    r = W.rng(M * 7 + N * 3 + K + 2 * transA + transB)
    A = W.uniform(r, (K, M) if transA else (M, K))
    B = W.uniform(r, (N, K) if transB else (K, N))
    C0 = W.uniform(r, (M, N))
    C = _run(emu, A, B, transA, transB, 1.5, -0.75, C0, mode)
    Cref, Sabs = oracle.gemm_ref(A, B, transA, transB, 1.5, -0.75, C0)
    ratio = checks.error_ratio(C, Cref, Sabs, K, 1.5, -0.75, C0, mode=_bound_mode(mode))
    assert ratio <= 1.0, ratio


# (M, N, K): BF16x9 keeps an operand stored with K as its row index M- or
# N-major; BF16x3 only when K >= 4 times its M (or N), which holds for both
# operands here ...
LAYOUT_SHAPES = [(256, 300, 1300), (129, 257, 1100), (1, 9, 40), (64, 1000, 4100),
                 (1536, 512, 7000), (256, 256, 100000),
                 # ... only B ...
                 (200, 1, 64), (1000, 60, 2000),
                 # ... neither (K-major pieces, split transposed)
                 (300, 513, 1000), (4096, 4096, 512)]


@pytest.mark.parametrize("shape", LAYOUT_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("mode", ["bf16x9", "bf16x3", "tf32x3"])
def test_operand_layout_does_not_change_a_bit(emu, mode, shape):
    """op(A) and op(B) fixed, stored four ways (A as M x K or K x M, B as
    K x N or N x K).  BF16x9 (and BF16x3 where K is at least 4 times M or
    N) splits an operand stored with K as its row index row-wise into M- or
    N-major pieces, which the tensor core reads through the transpose bits
    of its instruction descriptor; otherwise, and always for TF32x3 (the
    control), into K-major pieces.  The products and their order are the
    same either way, so the four results are the same bits, on the two-pass
    path (1536 x 512 x 7000, 256 x 256 x 100000 and 4096^2 x 512 with
    stream-K tails)."""
    M, N, K = shape
    r = W.rng(M + 3 * N + 7 * K)
    opA = W.normal(r, (M, K))
    opB = W.normal(r, (K, N), std=K ** -0.5)
    C0 = W.uniform(r, (M, N))
    old = emu.emu_get_path()
    emu.emu_set_path("twopass")
    try:
        outs = {}
        for tA in (0, 1):
            for tB in (0, 1):
                A = np.ascontiguousarray(opA.T) if tA else opA
                B = np.ascontiguousarray(opB.T) if tB else opB
                outs[(tA, tB)] = _run(emu, A, B, tA, tB, alpha=1.5, beta=-0.5, C0=C0, mode=mode)
    finally:
        emu.emu_set_path(old)
    ref = outs[(0, 1)]                  # K-major pieces of both operands
    for k, C in outs.items():
        assert np.array_equal(C.view(np.uint32), ref.view(np.uint32)), k
    mi, ni = W.sample_pairs(M, N, 1024, seed=M)
    Cref, Sabs = oracle.gemm_ref(opA, opB, 0, 0, 1.5, -0.5, C0, pairs=(mi, ni))
    assert checks.error_ratio(ref[mi, ni], Cref, Sabs, K, 1.5, -0.5, C0[mi, ni], mode=mode) <= 1.0


def test_strided_operands_and_output(emu):
    import torch
    r = W.rng(5)
    Abig = W.normal(r, (300, 520))
    Bbig = W.normal(r, (260, 400))
    Cbig = W.normal(r, (300, 700))
    A, B = Abig[:, 8:264], Bbig[:256, 16:392]          # rows 16-byte aligned, ld > cols
    dA, dB, dC = to_dev(Abig)[:, 8:264], to_dev(Bbig)[:256, 16:392], to_dev(Cbig)
    Cv = dC[:, 100:476]
    emu.emu_sgemm(dA, dB, Cv, alpha=1.0, beta=0.5)
    torch.cuda.synchronize()
    C0 = Cbig[:, 100:476]
    Cref, Sabs = oracle.gemm_ref(A, B, alpha=1.0, beta=0.5, C0=C0)
    out = dC.cpu().numpy()
    assert checks.error_ratio(out[:, 100:476], Cref, Sabs, 256, 1.0, 0.5, C0) <= 1.0
    untouched = np.ones(700, bool)
    untouched[100:476] = False
    assert np.array_equal(out[:, untouched], Cbig[:, untouched])


def test_transposed_views_are_handled(emu):
    import torch
    r = W.rng(8)
    A = W.normal(r, (96, 160))
    B = W.normal(r, (200, 160))                        # used as B^T
    dC = emu.emu_sgemm(to_dev(A), to_dev(B).t())       # a column-major view of B
    torch.cuda.synchronize()
    Cref, Sabs = oracle.gemm_ref(A, B, transB=True)
    assert checks.error_ratio(dC.cpu().numpy(), Cref, Sabs, 160, 1.0, 0.0) <= 1.0


# ------------------------------------------------------------- workloads --

def _sampled_check(emu, g, mode, n=4096):
    import torch
    A, B, C0 = W.generate(g)
    dA, dB = to_dev(A), to_dev(B)
    dC = to_dev(C0) if C0 is not None else torch.empty((g.M, g.N), device="cuda")
    emu.emu_sgemm(dA, dB, dC, transA=g.transA, transB=g.transB, alpha=g.alpha, beta=g.beta,
                  mode=mode)
    torch.cuda.synchronize()
    mi, ni = W.sample_pairs(g.M, g.N, n)
    # whole first and last rows as well
    mi = np.concatenate([mi, np.zeros(g.N, np.int64), np.full(g.N, g.M - 1, np.int64)])
    ni = np.concatenate([ni, np.arange(g.N), np.arange(g.N)])
    got = dC[torch.from_numpy(mi).cuda(), torch.from_numpy(ni).cuda()].cpu().numpy()
    Cref, Sabs = oracle.gemm_ref(A, B, g.transA, g.transB, g.alpha, g.beta, C0, pairs=(mi, ni))
    C0s = C0[mi, ni] if C0 is not None else None
    ratio = checks.error_ratio(got, Cref, Sabs, g.K, g.alpha, g.beta, C0s, mode=_bound_mode(mode))
    relf = checks.rel_frobenius(got, Cref)
    return ratio, relf, dC, (A, B, C0)


def test_square256_full_and_more_accurate_than_simt(emu):
    g = W.WORKLOADS["square256_uniform"]
    A, B, _ = W.generate(g)
    Cref, Sabs = oracle.gemm_ref(A, B)
    errs = {}
    for mode in MODES:
        C = _run(emu, A, B, mode=mode)
        assert checks.error_ratio(C, Cref, Sabs, g.K, 1.0, 0.0, mode=_bound_mode(mode)) <= 1.0
        errs[mode] = checks.rel_frobenius(C, Cref)
        assert errs[mode] <= checks.FROBENIUS_TOL
    # the pages: BF16x9 matches or beats native FP32 against an FP64 reference
    assert errs["bf16x9"] <= errs["fp32_simt"]


@pytest.mark.parametrize("name", ["mlip192_k256_n256", "mlip192_k256_n1024", "mlip192_k1024_n256"])
@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
def test_mlip192_every_element(emu, name, mode):
    g = W.WORKLOADS[name]
    A, B, _ = W.generate(g)
    C = _run(emu, A, B, transB=g.transB, mode=mode)
    Cref, Sabs = oracle.gemm_ref(A, B, transB=g.transB)
    assert checks.error_ratio(C, Cref, Sabs, g.K, 1.0, 0.0, mode=mode) <= 1.0
    assert checks.rel_frobenius(C, Cref) <= checks.FROBENIUS_TOL


@pytest.mark.parametrize("name", ["mlip17280_k256_n256", "mlip17280_k256_n1024",
                                  "mlip17280_k1024_n256"])
def test_mlip17280_sampled(emu, name):
    ratio, relf, _, _ = _sampled_check(emu, W.WORKLOADS[name], "bf16x9")
    assert ratio <= 1.0 and relf <= checks.FROBENIUS_TOL, (ratio, relf)


def test_stress4096_alpha_beta_sampled(emu):
    ratio, _, _, _ = _sampled_check(emu, W.WORKLOADS["stress4096"], "bf16x9")
    assert ratio <= 1.0, ratio


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
def test_square8192_sampled(emu, mode):
    ratio, relf, _, _ = _sampled_check(emu, W.WORKLOADS["square8192_normal"], mode)
    assert ratio <= 1.0 and relf <= checks.FROBENIUS_TOL, (ratio, relf)


def test_square8192_n_major_b_same_bits_as_k_major(emu):
    """The benchmark's configuration (8192^3, B stored K x N, which BF16x9
    reads as N-major pieces) gives the same bits as the same product with B
    stored N x K (K-major pieces), on every output; the sampled check above
    holds it to the oracle."""
    import torch
    g = W.WORKLOADS["square8192_normal"]
    A, B, _ = W.generate(g)
    dA = to_dev(A)
    C1 = torch.empty((g.M, g.N), device="cuda")
    C2 = torch.empty((g.M, g.N), device="cuda")
    emu.emu_sgemm(dA, to_dev(B), C1)
    emu.emu_sgemm(dA, to_dev(np.ascontiguousarray(B.T)), C2, transB=True)
    torch.cuda.synchronize()
    assert torch.equal(C1.view(torch.int32), C2.view(torch.int32))
    assert torch.isfinite(C1).all()


def test_bf16x9_at_least_as_accurate_as_fp32_at_long_k(emu):
    """The pages: BF16x9 matches or beats native FP32 against an FP64
    reference -- here at K = 8192, where accumulation error dominates."""
    g = W.Gemm("long_k", 512, 512, 8192, dist="normal", seed=77)
    _, rel9, _, _ = _sampled_check(emu, g, "bf16x9")
    _, rel32, _, _ = _sampled_check(emu, g, "fp32_simt")
    assert rel9 <= rel32, (rel9, rel32)


# ------------------------------------------------------------ edge cases --

def test_k_zero_and_alpha_zero(emu):
    import torch
    r = W.rng(3)
    C0 = W.uniform(r, (70, 90))
    for mode in MODES:
        dC = to_dev(C0)
        emu.emu_sgemm(torch.empty((70, 0), device="cuda"), torch.empty((0, 90), device="cuda"), dC,
                      beta=0.5, mode=mode)
        torch.cuda.synchronize()
        assert np.array_equal(dC.cpu().numpy(), np.float32(0.5) * C0)
        A = torch.full((70, 30), float("nan"), device="cuda")
        B = torch.ones((30, 90), device="cuda")
        dC = to_dev(C0)
        emu.emu_sgemm(A, B, dC, alpha=0.0, beta=2.0, mode=mode)   # A, B not read
        torch.cuda.synchronize()
        assert np.array_equal(dC.cpu().numpy(), 2 * C0)


def test_beta_zero_does_not_read_c(emu):
    import torch
    A = torch.ones((40, 20), device="cuda")
    B = torch.ones((20, 50), device="cuda")
    for mode in MODES:
        C = torch.full((40, 50), float("nan"), device="cuda")
        emu.emu_sgemm(A, B, C, beta=0.0, mode=mode)
        torch.cuda.synchronize()
        assert torch.all(C == 20), mode


def test_host_entry_point_matches_device_path(emu):
    r = W.rng(17)
    A = W.normal(r, (300, 200))
    B = W.normal(r, (200, 260))
    C0 = W.normal(r, (300, 260))
    dev = _run(emu, A, B, alpha=0.5, beta=1.0, C0=C0)
    host = emu.emu_sgemm_host(A, B, C0.copy(), alpha=0.5, beta=1.0)
    assert np.array_equal(dev, host)


@pytest.mark.parametrize("transA,transB,beta,mode",
                         [(0, 0, 0.0, "bf16x9"), (1, 1, 0.5, "bf16x9"), (0, 1, -1.0, "tf32x3"),
                          (1, 0, 0.0, "fp32_simt")])
def test_host_entry_pipelined_rows_match_one_call(emu, transA, transB, beta, mode):
    """Large enough for the chunked copy/compute pipeline (row chunks of C on
    three streams): row chunks of C are computed independently by the same
    kernels, so the result matches the one-call device result within the
    accuracy bound -- and bit for bit where no K range is split (the SIMT
    kernel); the GEMM's stream-K tail depends on the tile count, so a chunk
    and the whole call may sum a tile's K blocks in different groupings."""
    M, N, K = 8300, 1024, 1024                       # ragged last chunk
    r = W.rng(18 + transA + 2 * transB)
    A = W.normal(r, (K, M) if transA else (M, K))
    B = W.normal(r, (N, K) if transB else (K, N))
    C0 = W.normal(r, (M, N))
    dev = _run(emu, A, B, transA, transB, alpha=0.75, beta=beta, C0=C0, mode=mode)
    host = emu.emu_sgemm_host(A, B, C0.copy(), transA=transA, transB=transB, alpha=0.75,
                              beta=beta, mode=mode)
    mi, ni = W.sample_pairs(M, N, 1024, seed=3)
    Cref, Sabs = oracle.gemm_ref(A, B, transA, transB, 0.75, beta, C0, pairs=(mi, ni))
    for C in (host, dev):
        assert checks.error_ratio(C[mi, ni], Cref, Sabs, K, 0.75, beta, C0[mi, ni],
                                  mode=_bound_mode(mode)) <= 1.0
    bound = checks.elementwise_bound(K, 0.75, beta, Sabs, C0[mi, ni], mode=_bound_mode(mode))
    assert np.all(np.abs(host[mi, ni].astype(np.float64) - dev[mi, ni]) <= 2 * bound)
    if mode == "fp32_simt":
        assert np.array_equal(dev, host)


def _profiled(emu, fn):
    """Run fn with the launch counters on; returns (result, launches by kind)."""
    emu.emu_profile_enable(True)
    try:
        out = fn()
        counts = {k: emu.emu_profile_read(k)[0] for k in ("split", "gemm_tc", "gemm_fused")}
    finally:
        emu.emu_profile_enable(False)
    return out, counts


@pytest.mark.parametrize("transA,transB,beta,mode",
                         [(0, 0, 0.0, "bf16x9"), (1, 1, 0.5, "bf16x9"), (0, 1, -1.0, "tf32x3"),
                          (1, 0, 1.0, "bf16x3"), (0, 0, 0.0, "tf32"), (0, 1, 0.25, "tf32x3_oy")])
def test_host_entry_column_panels(emu, transA, transB, beta, mode):
    """A wide op(B) crosses to the device in column panels, each multiplied by
    op(A)'s first 2048 rows as it lands; the rest of op(A) follows in row
    chunks.  M = 5000, N = 2600 (panels of 1024, 1024 and 552 columns), K =
    1700 (B is 17.7 MB): three panel GEMMs and two row-chunk GEMMs, every
    split one launch (A's first chunk, three panels, two chunks)."""
    M, N, K = 5000, 2600, 1700
    r = W.rng(40 + transA + 2 * transB)
    A = W.normal(r, (K, M) if transA else (M, K))
    B = W.normal(r, (N, K) if transB else (K, N))
    C0 = W.normal(r, (M, N))
    host, counts = _profiled(emu, lambda: emu.emu_sgemm_host(
        A, B, C0.copy(), transA=transA, transB=transB, alpha=0.75, beta=beta, mode=mode))
    assert counts == {"split": 6, "gemm_tc": 5, "gemm_fused": 0}, counts
    dev = _run(emu, A, B, transA, transB, alpha=0.75, beta=beta, C0=C0, mode=mode)
    bmode = mode if mode in checks.MODE_EXTRA else "bf16x9"
    mi, ni = W.sample_pairs(M, N, 2048, seed=7)
    # every panel and chunk boundary is sampled too
    edges = np.array([0, 2047, 2048, 2049, 3583, 3584, 4999])
    cols = np.array([0, 1023, 1024, 2047, 2048, 2599])
    mi = np.concatenate([mi, np.repeat(edges, cols.size)])
    ni = np.concatenate([ni, np.tile(cols, edges.size)])
    Cref, Sabs = oracle.gemm_ref(A, B, transA, transB, 0.75, beta, C0, pairs=(mi, ni))
    for C in (host, dev):
        assert checks.error_ratio(C[mi, ni], Cref, Sabs, K, 0.75, beta, C0[mi, ni],
                                  mode=bmode) <= 1.0
    bound = checks.elementwise_bound(K, 0.75, beta, Sabs, C0[mi, ni], mode=bmode)
    assert np.all(np.abs(host[mi, ni].astype(np.float64) - dev[mi, ni]) <= 2 * bound)
    assert np.all(np.isfinite(host))


def test_host_entry_column_panels_wide_b(emu):
    """N = 70000 > 64 panels of 1024: the panels widen (to 1280 columns) and
    every column of C is still written."""
    import torch
    M, N, K = 600, 70000, 64
    r = W.rng(44)
    A = W.normal(r, (M, K))
    B = W.normal(r, (K, N))
    host, counts = _profiled(emu, lambda: emu.emu_sgemm_host(A, B))
    assert counts["gemm_tc"] == 55, counts
    dev = _run(emu, A, B)
    mi, ni = W.sample_pairs(M, N, 4096, seed=8)
    Cref, Sabs = oracle.gemm_ref(A, B, pairs=(mi, ni))
    assert checks.error_ratio(host[mi, ni], Cref, Sabs, K, 1.0, 0.0) <= 1.0
    assert np.all(np.isfinite(host))
    assert np.allclose(host, dev, rtol=0, atol=1e-5 * float(np.abs(dev).max()))


@pytest.mark.parametrize("path", ["auto", "fused_tmem"])
def test_host_entry_pipelined_fused_shape(emu, path):
    """N = 256 rows of an MLIP layer: an on-chip path in every chunk (AUTO
    takes the shared-memory one), B's pieces split once and reused."""
    g = W.WORKLOADS["mlip192_k256_n256"]
    M = 70000
    r = W.rng(19)
    A = W.normal(r, (M, g.K))
    B = W.normal(r, (g.N, g.K), std=g.K ** -0.5)
    old = emu.emu_get_path()
    emu.emu_set_path(path)
    try:
        dev = _run(emu, A, B, transB=True)
        host = emu.emu_sgemm_host(A, B, transB=True)
    finally:
        emu.emu_set_path(old)
    # the one call splits its last wave along K, the two chunks do not: the
    # results agree within the accuracy bound, element by element
    mi, ni = W.sample_pairs(M, g.N, 2048, seed=4)
    Cref, Sabs = oracle.gemm_ref(A, B, transB=True, pairs=(mi, ni))
    for C in (host, dev):
        assert checks.error_ratio(C[mi, ni], Cref, Sabs, g.K, 1.0, 0.0) <= 1.0
    assert np.allclose(host, dev, rtol=0, atol=4e-5 * float(np.abs(dev).max()))


def test_bounded_wait_reports_timeout_and_context_survives(emu):
    emu.emu_clear_device_error()
    assert emu.emu_selftest_timeout(2000) == -5          # EMU_ERR_TIMEOUT
    emu.emu_clear_device_error()
    assert emu.emu_get_last_device_error() == 0
    C = _run(emu, np.eye(8, dtype=np.float32), np.ones((8, 8), np.float32))
    assert np.all(C == 1)


def test_no_device_error_recorded(emu):
    assert emu.emu_get_last_device_error() == 0


# ------------------------------------------------------ the on-chip paths --
# EMU_PATH_FUSED: the GEMM kernel's split warps read FP32 A and store its
# pieces into the shared-memory stages (256-wide tiles); EMU_PATH_FUSED_TMEM:
# A is loaded as FP32 and split into tensor memory (128-wide tiles).  Both
# take BF16x9 with K-major A with 16-byte-aligned rows; otherwise the call
# falls back to the two-pass path.

ON_CHIP = ["fused", "fused_tmem"]


class _fused_path:
    def __init__(self, emu, path="fused"):
        self.emu = emu
        self.path = path

    def __enter__(self):
        self.old = self.emu.emu_get_path()
        self.emu.emu_set_path(self.path)

    def __exit__(self, *exc):
        self.emu.emu_set_path(self.old)


@pytest.mark.parametrize("shape", SHAPES + [(1000, 700, 300), (257, 129, 4096)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("transB", [0, 1])
@pytest.mark.parametrize("path,mode", [("fused", "bf16x9"), ("fused_tmem", "bf16x9"),
                                       ("fused", "tf32x3")])
def test_fused_path_every_element(emu, shape, transB, path, mode):
    M, N, K = shape
    r = W.rng(M * 11 + N * 5 + K + transB)
    A = W.normal(r, (M, K))
    B = W.normal(r, (N, K) if transB else (K, N))
    C0 = W.uniform(r, (M, N))
    with _fused_path(emu, path):
        C = _run(emu, A, B, False, transB, 1.5, -0.75, C0, mode)
    Cref, Sabs = oracle.gemm_ref(A, B, False, transB, 1.5, -0.75, C0)
    assert checks.error_ratio(C, Cref, Sabs, K, 1.5, -0.75, C0, mode=mode) <= 1.0
    C2 = _run(emu, A, B, False, transB, 1.5, -0.75, C0, mode)          # two-pass
    bound = checks.elementwise_bound(K, 1.5, -0.75, Sabs, C0, mode=mode)
    assert np.all(np.abs(C.astype(np.float64) - C2) <= bound)
    if mode == "tf32x3" and K >= 32:
        # the same pieces and the same K blocks: the same bits as two-pass
        # unless a split tail groups the blocks differently
        assert np.mean(C == C2) > 0.5


@pytest.mark.parametrize("path", ON_CHIP)
def test_fused_path_identity_is_exact_and_falls_back_when_needed(emu, path):
    X = W.normal(W.rng(31), (256, 256))
    I = np.eye(256, dtype=np.float32)
    with _fused_path(emu, path):
        assert np.array_equal(_run(emu, I, X), X)
        assert np.array_equal(_run(emu, X, I), X)
        # transposed A and a misaligned row stride take the two-pass path
        assert np.array_equal(_run(emu, I, X, transA=True), X)
        C = _run(emu, X[:, :255].copy(), np.ones((255, 64), np.float32))
        Cref, Sabs = oracle.gemm_ref(X[:, :255].copy(), np.ones((255, 64), np.float32))
        assert checks.error_ratio(C, Cref, Sabs, 255, 1.0, 0.0) <= 1.0


@pytest.mark.parametrize("name", ["mlip17280_k256_n256", "mlip17280_k1024_n256",
                                  "mlip17280_k256_n1024"])
@pytest.mark.parametrize("path", ON_CHIP)
def test_fused_path_mlip17280_sampled(emu, name, path):
    with _fused_path(emu, path):
        ratio, relf, _, _ = _sampled_check(emu, W.WORKLOADS[name], "bf16x9")
    assert ratio <= 1.0 and relf <= checks.FROBENIUS_TOL, (ratio, relf)


@pytest.mark.parametrize("path", ON_CHIP)
def test_fused_path_square8192_sampled(emu, path):
    with _fused_path(emu, path):
        ratio, relf, _, _ = _sampled_check(emu, W.WORKLOADS["square8192_normal"], "bf16x9")
    assert ratio <= 1.0 and relf <= checks.FROBENIUS_TOL, (ratio, relf)


def test_no_device_error_after_fused(emu):
    assert emu.emu_get_last_device_error() == 0


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3", "tf32x3_oy", "bf16x3", "tf32", "fp32_simt"])
def test_subnormal_operands_through_the_tensor_core(emu, mode):
    """FP32 subnormals in B (every element), identity A, and the transpose:
    BF16x9 and SIMT reproduce B exactly, so the tensor core neither flushes
    subnormal BF16 pieces nor subnormal FP32 partial sums; every mode equals
    the oracle's emulation of the same mode bit for bit (one nonzero product
    per output, so no rounding order is involved)."""
    r = W.rng(77)
    u = r.integers(1, 1 << 23, (256, 256)).astype(np.uint32) | \
        (r.integers(0, 2, (256, 256)).astype(np.uint32) << 31)
    Bs = u.view(np.float32)
    I = np.eye(256, dtype=np.float32)
    emul = {"bf16x9": oracle.gemm_bf16x9, "tf32x3": oracle.gemm_tf32x3,
            "tf32x3_oy": oracle.gemm_tf32x3_oy, "bf16x3": oracle.gemm_bf16x3,
            "tf32": oracle.gemm_tf32, "fp32_simt": oracle.gemm_fp32}[mode]
    for X, Y in ((I, Bs), (Bs, I)):
        C = _run(emu, X, Y, mode=mode)
        assert np.array_equal(C.view(np.uint32), emul(X, Y).view(np.uint32))
        if mode in ("bf16x9", "fp32_simt"):
            assert np.array_equal(C.view(np.uint32), u)


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3", "tf32x3_oy", "bf16x3", "tf32"])
def test_subnormal_operand_products_within_the_tensor_core_term(emu, mode):
    """K = 1, so every output is one product a b: 4096 values of a with
    exponents spread over 2^-149 .. 2^-100 (FP32 subnormals below 2^-126)
    times 64 normal b.  BF16x9 keeps a's bits in its pieces, but products
    with a subnormal a come out up to tens of ulps off (the tensor core's
    truncating, scaled accumulation), while from 2^-126 up they stay within
    two ulps (one truncation and the final rounding).  Every mode meets the element-wise bound with the operands'
    absolute term (MODE_SUB_ABS + TC_SUB_ABS), and for BF16x9 some product
    exceeds the bound without TC_SUB_ABS: the term is needed."""
    r = np.random.default_rng(5)
    M, N = 4096, 64
    e = r.uniform(-149, -100, M)
    a = (np.exp2(e) * r.choice([-1, 1], M)).astype(np.float32).reshape(M, 1)
    b = (r.uniform(1, 2, N) * np.exp2(r.integers(-20, 21, N)) *
         r.choice([-1, 1], N)).astype(np.float32).reshape(1, N)
    C = _run(emu, a, b, mode=mode)
    Cref, Sabs = oracle.gemm_ref(a, b)
    S1 = checks.operand_l1(a, b)
    bmode = mode if mode in checks.MODE_EXTRA else "bf16x9"
    assert checks.error_ratio(C, Cref, Sabs, 1, 1.0, 0.0, mode=bmode, S1=S1) <= 1.0
    if mode == "bf16x9":
        err = np.abs(C.astype(np.float64) - Cref)
        normal = np.abs(a[:, 0]) >= 2.0 ** -126
        ulp = np.maximum(np.exp2(np.floor(np.log2(np.abs(Cref))) - 23), 2.0 ** -149)
        assert np.all(err[normal] <= 2 * ulp[normal])
        without = (checks.elementwise_bound(1, 1.0, 0.0, Sabs, mode="bf16x9") +
                   checks.MODE_SUB_ABS["bf16x9"] * S1)
        assert np.any(err > without)


@pytest.mark.parametrize("shape", [(256, 256, 4096), (1024, 1024, 1024), (300, 513, 1000),
                                   (4096, 4096, 512)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3", "bf16x3"])
def test_tail_split_shapes(emu, shape, mode):
    """Shapes whose last round of tiles runs split along K (its K blocks
    shared by several clusters: 1 tile in 13 parts, 16 tiles over 76, 6
    tiles over 48, the last 28 of 256 tiles over 76): within the
    bound, every element where the oracle is fast enough, and the same bits
    on a second call (the reduction order is fixed)."""
    M, N, K = shape
    r = W.rng(M + 3 * N + 7 * K)
    A, B = W.normal(r, (M, K)), W.normal(r, (K, N))
    C1 = _run(emu, A, B, mode=mode)
    C2 = _run(emu, A, B, mode=mode)
    assert np.array_equal(C1, C2)
    bm = mode if mode in ("tf32x3", "bf16x3") else "bf16x9"
    if M * N * K <= (1 << 30):
        Cref, Sabs = oracle.gemm_ref(A, B)
        assert checks.error_ratio(C1, Cref, Sabs, K, 1.0, 0.0, mode=bm) <= 1.0
    else:
        mi, ni = W.sample_pairs(M, N, 2048, seed=8)
        Cref, Sabs = oracle.gemm_ref(A, B, pairs=(mi, ni))
        assert checks.error_ratio(C1[mi, ni], Cref, Sabs, K, 1.0, 0.0, mode=bm) <= 1.0


@pytest.mark.parametrize("shape,transB,path", [
    ((1536, 512, 700), True, "twopass"),      # BF16x9: 12 tiles of 11 blocks, 5 parts each
    ((4864, 512, 700), False, "twopass"),     # 38 tiles of 11 blocks, 2 parts each
    ((300, 384, 4100), True, "auto"),         # 4 tiles of 65 blocks (last one ragged), 13 parts
    ((12288, 256, 1024), False, "twopass"),   # 48 tiles of 16 blocks, stream-K over 76
    ((12288, 256, 4096), True, "twopass"),    # 48 tiles of 64 blocks, stream-K in every mode
    ((12288, 256, 1024), False, "fused_tmem"),  # 96 tiles: 20 left over, 3 parts each
    ((12288, 256, 1024), False, "fused"),     # 48 tiles of 16 blocks, stream-K over 76
    ((1536, 512, 700), True, "fused"),        # 12 tiles of 11 blocks, 5 parts each
], ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else str(v))
@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3", "bf16x3", "tf32", "tf32x3_oy"])
def test_tail_parts_with_alpha_beta(emu, shape, transB, path, mode):
    """Split tails -- equal parts inside a tile, and stream-K ranges that
    start and end inside tiles so that a tile is summed by two or more
    clusters -- with alpha, beta and C0 applied once by the tile's owner:
    within each mode's bound on every element (sampled on the largest
    shapes) and the same bits on a second call."""
    if (path == "fused_tmem" and mode != "bf16x9") or (path == "fused" and mode not in ("bf16x9", "tf32x3")):
        pytest.skip("on-chip splits: BF16x9 (both kernels) and TF32x3 (shared memory)")
    M, N, K = shape
    r = W.rng(M + 5 * N + 11 * K)
    A = W.normal(r, (M, K))
    B = W.normal(r, (N, K) if transB else (K, N), std=K ** -0.5)
    C0 = W.uniform(r, (M, N))
    emu.emu_set_path(path)
    try:
        C1 = _run(emu, A, B, False, transB, alpha=1.5, beta=0.5, C0=C0, mode=mode)
        C2 = _run(emu, A, B, False, transB, alpha=1.5, beta=0.5, C0=C0, mode=mode)
    finally:
        emu.emu_set_path("auto")
    assert np.array_equal(C1, C2)
    assert emu.emu_get_last_device_error() == 0
    if M * N * K <= (1 << 30):
        Cref, Sabs = oracle.gemm_ref(A, B, False, transB, 1.5, 0.5, C0)
        assert checks.error_ratio(C1, Cref, Sabs, K, 1.5, 0.5, C0, mode=mode) <= 1.0
    else:
        mi, ni = W.sample_pairs(M, N, 4096, seed=12)
        Cref, Sabs = oracle.gemm_ref(A, B, False, transB, 1.5, 0.5, C0, pairs=(mi, ni))
        assert checks.error_ratio(C1[mi, ni], Cref, Sabs, K, 1.5, 0.5, C0[mi, ni],
                                  mode=mode) <= 1.0


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
def test_non_finite_operands_follow_the_split(emu, mode):
    """Infinities and NaNs: the split keeps +-inf as (x, +0, +0) and NaN as NaN
    pieces, so an output that meets an infinity is formed from products such
    as inf * 0 and inf * (opposite-signed residual): it comes out NaN or
    +-inf exactly as the oracle's emulation of the same method says, which is
    not always what a plain FP32 dot product gives (the emulation is not
    IEEE-754 arithmetic).  The outputs that meet no special value stay
    within the bound."""
    r = W.rng(91)
    A, B = W.normal(r, (70, 64)), W.normal(r, (64, 90))
    A[3, 5], A[10, 7], A[11, 7] = np.inf, -np.inf, 1.0       # row 11 finite except a clean 1.0
    A[20, 9] = np.nan
    B[5, 20], B[30, 40], B[7, 60] = np.nan, np.inf, 0.0
    C = _run(emu, A, B, mode=mode)
    emul = {"bf16x9": oracle.gemm_bf16x9, "tf32x3": oracle.gemm_tf32x3}[mode](A, B)
    assert np.array_equal(np.isnan(C), np.isnan(emul))
    assert np.array_equal(np.isposinf(C), np.isposinf(emul))
    assert np.array_equal(np.isneginf(C), np.isneginf(emul))
    fin = np.isfinite(emul)
    assert fin.sum() > 0.9 * fin.size
    Af, Bf = np.nan_to_num(A, nan=0.0, posinf=0.0, neginf=0.0), np.nan_to_num(B, nan=0.0, posinf=0.0, neginf=0.0)
    Cref, Sabs = oracle.gemm_ref(Af, Bf)
    clean_rows = np.all(np.isfinite(A), axis=1)
    clean_cols = np.all(np.isfinite(B), axis=0)
    m = np.outer(clean_rows, clean_cols)
    assert checks.error_ratio(C[m], Cref[m], Sabs[m], 64, 1.0, 0.0, mode=mode) <= 1.0


@pytest.mark.parametrize("path", ["auto", "fused", "fused_tmem", "twopass"])
def test_misaligned_operands_and_long_k(emu, path):
    """Operands that start 4 bytes past a 16-byte boundary (the fused path and
    the 16-byte split kernels must step aside), C likewise, and a one-tile
    GEMM with K = 65536 whose K blocks are shared by 16 clusters."""
    import torch
    emu.emu_set_path(path)
    try:
        r = W.rng(97)
        M, N, K = 4100, 200, 300
        A = W.normal(r, (M, K + 1))[:, 1:]
        B = W.normal(r, (N, K + 1))[:, 1:]
        dAbig, dBbig = to_dev(W.normal(W.rng(1), (M, K + 1))), to_dev(W.normal(W.rng(2), (N, K + 1)))
        dAbig[:, 1:] = to_dev(np.ascontiguousarray(A))
        dBbig[:, 1:] = to_dev(np.ascontiguousarray(B))
        Cbig = torch.zeros((M, N + 1), device="cuda")
        emu.emu_sgemm(dAbig[:, 1:], dBbig[:, 1:], Cbig[:, 1:], transB=True)
        torch.cuda.synchronize()
        mi, ni = W.sample_pairs(M, N, 2048, seed=9)
        Cref, Sabs = oracle.gemm_ref(A, B, transB=True, pairs=(mi, ni))
        got = Cbig[:, 1:].cpu().numpy()[mi, ni]
        assert checks.error_ratio(got, Cref, Sabs, K, 1.0, 0.0) <= 1.0
        assert torch.all(Cbig[:, 0] == 0)
        # long K on one tile
        A2, B2 = W.normal(r, (64, 65536)), W.normal(r, (65536, 48))
        C2 = _run(emu, A2, B2)
        Cref2, Sabs2 = oracle.gemm_ref(A2, B2)
        assert checks.error_ratio(C2, Cref2, Sabs2, 65536, 1.0, 0.0) <= 1.0
    finally:
        emu.emu_set_path("auto")


@pytest.mark.parametrize("path,mode,M,K", [("twopass", "bf16x9", 300, 200),
                                           ("twopass", "tf32x3", 300, 200),
                                           ("fused", "bf16x9", 4200, 130),
                                           ("fused_tmem", "bf16x9", 4200, 130),
                                           ("twopass", "bf16x9", 1536, 700)])
def test_c_columns_past_n_are_untouched(emu, path, mode, M, K):
    """C as the first N columns of a wider matrix (ldc = 64, a multiple of
    four, so the epilogue's bulk tensor stores run): columns N..63 keep their
    values for every N = 1..33, beta = 0 and 1, and columns < N are right.
    A bulk store clips at the edge of its map in 16-byte units, so the
    library maps C only up to N & ~3 and stores the rest per lane.  The last
    shape splits its last round along K (parts summed by the tile's owner)."""
    import torch
    old = emu.emu_get_path()
    emu.emu_set_path(path)
    try:
        for N in list(range(1, 18)) + [21, 30, 31, 33]:
            r = W.rng(N + M)
            A = W.normal(r, (M, K))
            B = W.normal(r, (K, N), std=K ** -0.5)
            C0 = W.normal(r, (M, 64))
            for beta in (0.0, 1.0):
                Cs = to_dev(C0)
                emu.emu_sgemm(to_dev(A), to_dev(B), Cs[:, :N], beta=beta, mode=mode)
                torch.cuda.synchronize()
                got = Cs.cpu().numpy()
                assert np.array_equal(got[:, N:], C0[:, N:]), (N, beta)
                mi, ni = W.sample_pairs(M, N, 512, seed=N)
                Cref, Sabs = oracle.gemm_ref(A, B, beta=beta, C0=np.ascontiguousarray(C0[:, :N]),
                                             pairs=(mi, ni))
                assert checks.error_ratio(got[mi, ni], Cref, Sabs, K, 1.0, beta, C0[mi, ni],
                                          mode=_bound_mode(mode)) <= 1.0, (N, beta)
    finally:
        emu.emu_set_path(old)


@pytest.mark.parametrize("path,mode", [("fused", "bf16x9"), ("fused", "tf32x3"),
                                       ("fused_tmem", "bf16x9")])
@pytest.mark.parametrize("K", [129, 130, 131, 257, 1023])
def test_on_chip_split_does_not_read_past_k(emu, path, mode, K):
    """A is read as FP32 by the GEMM kernel (TMA into shared memory, or
    16-byte loads by the split warps): with K = 4k + 1..3 and NaN in the
    padding of A's rows (lda a multiple of 4, so the on-chip path runs), the
    result is finite and within the bound."""
    import torch
    M, N = 4200, 200 if path == "fused" else 100
    lda = (K + 3) // 4 * 4 + 4
    r = W.rng(K + N)
    A = W.normal(r, (M, K))
    B = W.normal(r, (N, K), std=K ** -0.5)
    S = torch.full((M, lda), float("nan"), device="cuda")
    S[:, :K] = to_dev(A)
    C = torch.empty(M, N, device="cuda")
    old = emu.emu_get_path()
    emu.emu_set_path(path)
    try:
        emu.emu_profile_enable(True)
        emu.emu_sgemm(S[:, :K], to_dev(B), C, transB=True, mode=mode)
        torch.cuda.synchronize()
        ran = emu.emu_profile_read("gemm_fused")[0]
        emu.emu_profile_enable(False)
    finally:
        emu.emu_set_path(old)
    assert ran == 1
    got = C.cpu().numpy()
    assert np.all(np.isfinite(got))
    mi, ni = W.sample_pairs(M, N, 2048, seed=K)
    Cref, Sabs = oracle.gemm_ref(A, B, transB=True, pairs=(mi, ni))
    assert checks.error_ratio(got[mi, ni], Cref, Sabs, K, 1.0, 0.0, mode=_bound_mode(mode)) <= 1.0


@pytest.mark.parametrize("shape", [(256, 256, 1105920, 1), (256, 256, 100000, 0),
                                   (512, 256, 65536, 1), (300, 200, 50000, 0)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
def test_deep_k_tiles_spread_over_every_cluster(emu, shape, mode):
    """Weight-gradient shapes (dW = dY^T X over 1.1M rows is one 256 x 256
    tile of 17,280 K blocks): the few tiles are cut into many more than 8
    parts, every resident cluster takes some, and each tile's owner adds all
    of its parts in K order -- within the bound against the oracle on
    sampled outputs, with alpha and beta, and the same bits on a second
    call."""
    import torch
    M, N, K, tA = shape
    r = W.rng(M + N + K)
    A = W.normal(r, (K, M) if tA else (M, K))
    B = W.normal(r, (K, N), std=K ** -0.5)
    C0 = W.uniform(r, (M, N))
    dA, dB = to_dev(A), to_dev(B)
    outs = []
    for _ in range(2):
        C = to_dev(C0)
        emu.emu_sgemm(dA, dB, C, transA=bool(tA), alpha=0.75, beta=0.5, mode=mode)
        torch.cuda.synchronize()
        outs.append(C.cpu().numpy())
    assert np.array_equal(outs[0], outs[1])
    assert emu.emu_get_last_device_error() == 0
    mi, ni = W.sample_pairs(M, N, 768, seed=K)
    Cref, Sabs = oracle.gemm_ref(A, B, tA, False, 0.75, 0.5, C0, pairs=(mi, ni))
    assert checks.error_ratio(outs[0][mi, ni], Cref, Sabs, K, 0.75, 0.5, C0[mi, ni],
                              mode=_bound_mode(mode)) <= 1.0
