"""GPU parity of the two cheaper rungs of the accuracy ladder -- two BF16
pieces with three products (BF16x3) and single-pass TF32 -- and of the
Ootomo-Yokota variant of TF32x3 (residual scaled by 2^11) against the CPU
oracle.

Two criteria per result: the element-wise bound against the FP64 reference,
with the rung's own representation term (2^-16 |alpha| S_abs for BF16x3,
2^-10 + 2^-21 for TF32, 2^-20 for the Ootomo-Yokota TF32x3), and closeness to the oracle's emulation of the same
rung, which keeps the same products: the two differ only in summation order,
so |C_gpu - C_oracle| <= 2 (2K + 2) 2^-24 |alpha| S_abs + 2^-22 |beta C0|.
The second catches a wrong piece or a wrong product that the looser first
bound would let through."""
import numpy as np
import pytest

import oracle
from oracle import checks
from fp32_emulated_gemm_split_gb300 import workloads as W
from gpu_util import emu_module, to_dev

pytestmark = pytest.mark.gpu

RUNGS = {"bf16x3": oracle.gemm_bf16x3, "tf32": oracle.gemm_tf32,
         "tf32x3_oy": oracle.gemm_tf32x3_oy}


@pytest.fixture(scope="module")
def emu():
    return emu_module()


def _run(emu, A, B, transA=False, transB=False, alpha=1.0, beta=0.0, C0=None, mode="bf16x3",
         noalloc=False):
    import torch
    M = A.shape[1] if transA else A.shape[0]
    N = B.shape[0] if transB else B.shape[1]
    dC = to_dev(C0) if C0 is not None else torch.full((M, N), float("nan"), device="cuda")
    fn = emu.emu_sgemm_noalloc if noalloc else emu.emu_sgemm
    fn(to_dev(A), to_dev(B), dC, transA=transA, transB=transB, alpha=alpha, beta=beta, mode=mode)
    torch.cuda.synchronize()
    return dC.cpu().numpy()


def _same_rung_ratio(C, Cemu, Sabs, K, alpha, beta, C0):
    tol = 2 * (2 * K + 2) * checks.U * abs(alpha) * np.asarray(Sabs, np.float64)
    if beta != 0.0:
        tol = tol + 4 * checks.U * abs(beta) * np.abs(np.asarray(C0, np.float64))
    tol = tol + (18 * K + 8) * checks.SUB
    d = np.abs(np.asarray(C, np.float64) - np.asarray(Cemu, np.float64))
    return float(np.max(d / tol)) if d.size else 0.0


def test_identity_keeps_exactly_the_rungs_pieces(emu):
    X = W.normal(W.rng(71), (256, 320))
    I = np.eye(256, dtype=np.float32)
    for mode, fn in RUNGS.items():
        assert np.array_equal(_run(emu, I, X, mode=mode), fn(I, X)), mode


SHAPES = [(1, 1, 1), (7, 13, 5), (129, 257, 65), (300, 513, 1000), (64, 40, 2048)]


@pytest.mark.parametrize("mode", list(RUNGS))
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("transA,transB", [(0, 0), (1, 1), (0, 1)])
def test_ragged_shapes_every_element(emu, mode, shape, transA, transB):
    M, N, K = shape
    r = W.rng(3 * M + 5 * N + K + 2 * transA + transB + 11)
    A = W.uniform(r, (K, M) if transA else (M, K))
    B = W.uniform(r, (N, K) if transB else (K, N))
    C0 = W.uniform(r, (M, N))
    C = _run(emu, A, B, transA, transB, 1.5, -0.75, C0, mode)
    Cref, Sabs = oracle.gemm_ref(A, B, transA, transB, 1.5, -0.75, C0)
    assert checks.error_ratio(C, Cref, Sabs, K, 1.5, -0.75, C0, mode=mode) <= 1.0
    Cemu = RUNGS[mode](A, B, transA, transB, 1.5, -0.75, C0)
    assert _same_rung_ratio(C, Cemu, Sabs, K, 1.5, -0.75, C0) <= 1.0


def test_ladder_order_on_mlip192(emu):
    g = W.WORKLOADS["mlip192_k256_n256"]
    A, B, C0 = W.generate(g)
    Cref, Sabs = oracle.gemm_ref(A, B)
    err = {m: checks.rel_frobenius(_run(emu, A, B, mode=m), Cref)
           for m in ("bf16x9", "tf32x3", "tf32x3_oy", "bf16x3", "tf32")}
    assert err["bf16x9"] <= checks.FROBENIUS_TOL and err["tf32x3"] <= checks.FROBENIUS_TOL
    assert err["tf32x3_oy"] <= checks.FROBENIUS_TOL
    assert err["tf32"] > err["bf16x3"] > 5 * max(err["bf16x9"], err["tf32x3"])
    mi, ni = W.sample_pairs(g.M, g.N, 4096, seed=6)
    for m in ("bf16x3", "tf32", "tf32x3_oy"):
        C = _run(emu, A, B, mode=m)[mi, ni]
        Cemu = RUNGS[m](A, B, pairs=(mi, ni))
        assert _same_rung_ratio(C, Cemu, Sabs[mi, ni], g.K, 1.0, 0.0, None) <= 1.0


@pytest.mark.parametrize("mode", list(RUNGS))
def test_square8192_sampled(emu, mode):
    import torch
    g = W.with_mode(W.WORKLOADS["square8192_normal"], mode)
    A, B, C0 = W.generate(g)
    dC = torch.empty((g.M, g.N), device="cuda")
    emu.emu_sgemm(to_dev(A), to_dev(B), dC, alpha=g.alpha, beta=0.0, mode=mode)
    torch.cuda.synchronize()
    mi, ni = W.sample_pairs(g.M, g.N, 2048, seed=5)
    C = dC.cpu().numpy()[mi, ni]
    Cref, Sabs = oracle.gemm_ref(A, B, alpha=g.alpha, pairs=(mi, ni))
    assert checks.error_ratio(C, Cref, Sabs, g.K, g.alpha, 0.0, mode=mode) <= 1.0
    Cemu = RUNGS[mode](A, B, alpha=g.alpha, pairs=(mi, ni))
    assert _same_rung_ratio(C, Cemu, Sabs, g.K, g.alpha, 0.0, None) <= 1.0


def test_noalloc_entry_takes_the_rungs(emu):
    r = W.rng(72)
    A = W.uniform(r, (300, 200))
    B = W.uniform(r, (200, 260))
    for mode, fn in RUNGS.items():
        C = _run(emu, A, B, mode=mode, noalloc=True)
        Cref, Sabs = oracle.gemm_ref(A, B)
        assert _same_rung_ratio(C, fn(A, B), Sabs, 200, 1.0, 0.0, None) <= 1.0, mode


def test_no_device_error_after_the_rungs(emu):
    assert emu.emu_get_last_device_error() == 0


def test_oy_on_wide_exponent_data_every_element(emu):
    """Values from 2^-30 to 2^30, zeros and subnormals (the stress recipe)."""
    r = W.rng(73)
    A = W.stress(r, (300, 700))
    B = W.stress(r, (700, 260))
    C0 = W.uniform(r, (300, 260))
    C = _run(emu, A, B, alpha=1.5, beta=0.5, C0=C0, mode="tf32x3_oy")
    Cref, Sabs = oracle.gemm_ref(A, B, alpha=1.5, beta=0.5, C0=C0)
    assert checks.error_ratio(C, Cref, Sabs, 700, 1.5, 0.5, C0, mode="tf32x3_oy") <= 1.0
    Cemu = oracle.gemm_tf32x3_oy(A, B, alpha=1.5, beta=0.5, C0=C0)
    assert _same_rung_ratio(C, Cemu, Sabs, 700, 1.5, 0.5, C0) <= 1.0
