"""Seeded random GEMMs through every entry point, mode and path.

Each case draws a shape (log-uniform, 1..6000 rows, 1..1500 columns, 0..2500
deep), transposes, alpha, beta, padded leading dimensions of A, B and C, a
mode, a path (emu_set_path) and an entry point (emu_sgemm, emu_sgemm_bsplit
on B split once, emu_sgemm_host on host buffers, emu_sgemm_noalloc where its
64 MiB array holds the pieces).  The result must meet the mode's element-wise
bound against the oracle's FP64 product on sampled outputs (every corner and
tile edge included), every output must be finite, and the padding columns of
C and 33 rows below it must keep the values they had: the kernels write
nothing outside C.

Bound: "Limitations and decision criteria" of the NVIDIA blog post (BF16x9
matches FP32 accuracy); the cheaper rungs by their piece error (oracle.checks).
"""
import numpy as np
import pytest

import oracle
from oracle import checks
from fp32_emulated_gemm_split_gb300 import workloads as W
from gpu_util import emu_module

pytestmark = pytest.mark.gpu

MODES = ["bf16x9", "tf32x3", "tf32x3_oy", "bf16x3", "tf32", "fp32_simt"]
PATHS = ["auto", "twopass", "fused", "fused_tmem"]
ENTRIES = ["sgemm", "bsplit", "host", "noalloc"]
PIECE_BYTES = {"bf16x9": 6, "tf32x3": 8, "tf32x3_oy": 8, "bf16x3": 4, "tf32": 4, "fp32_simt": 0}
NCASES = 48
SENTINEL = 7.25
ROWS_BELOW = 33         # sentinel rows under C: more than one 32-row store box


@pytest.fixture(scope="module")
def emu():
    return emu_module()


def _draw(i):
    r = np.random.Generator(np.random.PCG64(4242 + i))
    M = int(np.exp(r.uniform(0, np.log(6000))))
    N = int(np.exp(r.uniform(0, np.log(1500))))
    K = 0 if r.random() < 0.04 else int(np.exp(r.uniform(0, np.log(2500))))
    c = dict(M=M, N=N, K=K, tA=int(r.integers(0, 2)), tB=int(r.integers(0, 2)),
             mode=MODES[int(r.integers(0, len(MODES)))], path=PATHS[int(r.integers(0, len(PATHS)))],
             entry=ENTRIES[int(r.integers(0, len(ENTRIES)))],
             alpha=float([1.0, -0.75, 2.0 ** int(r.integers(-20, 21))][int(r.integers(0, 3))]),
             beta=float([0.0, 0.0, 1.0, 0.5, -2.0][int(r.integers(0, 5))]),
             pads=[int(v) for v in r.integers(0, 9, 3)],
             offs=[int(v) for v in r.integers(0, 4, 3)] if r.random() < 0.5 else [0, 0, 0])
    # the host-buffer entry point takes contiguous arrays; the split-B entry
    # point needs a tensor-core mode and some depth; noalloc a fitting problem
    if c["entry"] == "host":
        c["pads"] = [0, 0, 0]
        c["offs"] = [0, 0, 0]
    if c["entry"] == "bsplit" and (c["mode"] == "fp32_simt" or K == 0):
        c["entry"] = "sgemm"
    ldp = max((K + 7) // 8 * 8, 8)
    if c["entry"] == "noalloc" and PIECE_BYTES[c["mode"]] * (M + N) * ldp > (64 << 20):
        c["entry"] = "sgemm"
    return c, r


def _padded(torch, X, pad, off=0):
    """A device copy of X whose rows are `pad` elements longer and which
    starts `off` elements into its allocation (a strided view; off = 1..3
    leaves its base off the 16-byte grid), NaN around it."""
    rows, cols = X.shape
    S = torch.full((rows + 1, cols + pad + off), float("nan"), device="cuda")
    S[:rows, off:off + cols] = torch.from_numpy(np.ascontiguousarray(X)).cuda()
    return S[:rows, off:off + cols]


@pytest.mark.parametrize("i", range(NCASES))
def test_random_gemm(emu, i):
    _random_gemm(emu, i, _draw, "normal")


@pytest.mark.parametrize("i", range(24))
def test_random_gemm_wide_exponents(emu, i):
    """The same draws with the stress distribution in A, B and C0: exponents
    over 2^-30..2^30, 1 % zeros and 0.1 % FP32 subnormals, so that products
    span 2^120 and some fall among the subnormals."""
    _random_gemm(emu, 500 + i, _draw, "stress")


def _random_gemm(emu, i, draw, dist):
    import torch
    c, r = draw(i)
    M, N, K, tA, tB = c["M"], c["N"], c["K"], c["tA"], c["tB"]
    if dist == "stress":
        A = W.stress(r, (K, M) if tA else (M, K))
        B = W.stress(r, (N, K) if tB else (K, N))
        C0 = W.stress(r, (M, N))
    else:
        A = W.normal(r, (K, M) if tA else (M, K))
        B = W.normal(r, (N, K) if tB else (K, N), std=max(K, 1) ** -0.5)
        C0 = W.normal(r, (M, N))
    old = emu.emu_get_path()
    emu.emu_set_path(c["path"])
    try:
        if c["entry"] == "host":
            C = emu.emu_sgemm_host(A, B, C0.copy(), transA=bool(tA), transB=bool(tB),
                                   alpha=c["alpha"], beta=c["beta"], mode=c["mode"])
            pad_ok = True
        else:
            dA = _padded(torch, A, c["pads"][0], c["offs"][0])
            dB = _padded(torch, B, c["pads"][1], c["offs"][1])
            oc = c["offs"][2]
            Cs = torch.full((M + ROWS_BELOW, N + c["pads"][2] + oc), SENTINEL, device="cuda")
            Cs[:M, oc:oc + N] = torch.from_numpy(C0).cuda()
            dC = Cs[:M, oc:oc + N]
            kw = dict(alpha=c["alpha"], beta=c["beta"], mode=c["mode"])
            if c["entry"] == "bsplit":
                P = emu.emu_split_b(dB, transB=bool(tB), mode=c["mode"])
                emu.emu_sgemm_bsplit(dA, P, dC, transA=bool(tA), **kw)
            elif c["entry"] == "noalloc":
                emu.emu_sgemm_noalloc(dA, dB, dC, transA=bool(tA), transB=bool(tB), **kw)
            else:
                emu.emu_sgemm(dA, dB, dC, transA=bool(tA), transB=bool(tB), **kw)
            torch.cuda.synchronize()
            full = Cs.cpu().numpy()
            C = np.ascontiguousarray(full[:M, oc:oc + N])
            pad_ok = bool(np.all(full[:M, :oc] == np.float32(SENTINEL)) and
                          np.all(full[:M, oc + N:] == np.float32(SENTINEL)) and
                          np.all(full[M:] == np.float32(SENTINEL)))
    finally:
        emu.emu_set_path(old)
    assert pad_ok, f"case {i}: C written outside its {N} columns ({c})"
    _check(c, i, A, B, C0, C)


def _check(c, i, A, B, C0, C):
    M, N, K, tA, tB = c["M"], c["N"], c["K"], c["tA"], c["tB"]
    assert np.all(np.isfinite(C)), f"case {i}: non-finite output ({c})"
    if K == 0:              # C = beta C0, one exact FP32 product per element
        assert np.array_equal(C, np.float32(c["beta"]) * C0), f"case {i} ({c})"
        return
    mi, ni = W.sample_pairs(M, N, 2048, seed=i)
    rows = np.array(sorted({0, M - 1, min(255, M - 1), min(256, M - 1), M // 2}))
    cols = np.array(sorted({0, N - 1, min(127, N - 1), min(128, N - 1), min(255, N - 1),
                            min(256, N - 1)}))
    mi = np.concatenate([mi, np.repeat(rows, cols.size)])
    ni = np.concatenate([ni, np.tile(cols, rows.size)])
    Cref, Sabs = oracle.gemm_ref(A, B, tA, tB, c["alpha"], c["beta"], C0, pairs=(mi, ni))
    bmode = c["mode"] if c["mode"] in checks.MODE_EXTRA else "bf16x9"
    S1 = checks.operand_l1(A, B, tA, tB, pairs=(mi, ni))     # for subnormal operands
    ratio = checks.error_ratio(C[mi, ni], Cref, Sabs, K, c["alpha"], c["beta"], C0[mi, ni],
                               mode=bmode, S1=S1)
    assert ratio <= 1.0, f"case {i}: error ratio {ratio} ({c})"


def _draw_on_chip(i):
    """Shapes for the on-chip split paths and the K-split last round: many
    rows, at most 256 columns (or a ragged width above), K-major A."""
    r = np.random.Generator(np.random.PCG64(9191 + i))
    M = int(r.integers(4096, 20001))
    N = int(r.integers(1, 257)) if r.random() < 0.75 else int(r.integers(257, 700))
    K = int(np.exp(r.uniform(np.log(8), np.log(1200))))
    c = dict(M=M, N=N, K=K, tA=0, tB=int(r.integers(0, 2)),
             mode=["bf16x9", "tf32x3"][int(r.integers(0, 2))],
             path=PATHS[int(r.integers(0, len(PATHS)))],
             entry=["sgemm", "bsplit"][int(r.integers(0, 2))],
             alpha=float([1.0, -0.75, 0.5][int(r.integers(0, 3))]),
             beta=float([0.0, 1.0, 0.5][int(r.integers(0, 3))]),
             pads=[int(v) for v in r.integers(0, 9, 3)],
             offs=[int(v) for v in r.integers(0, 4, 3)] if r.random() < 0.3 else [0, 0, 0])
    return c, r


@pytest.mark.parametrize("i", range(24))
def test_random_gemm_on_chip_shapes(emu, i):
    import torch
    c, r = _draw_on_chip(i)
    M, N, K, tB = c["M"], c["N"], c["K"], c["tB"]
    A = W.normal(r, (M, K))
    B = W.normal(r, (N, K) if tB else (K, N), std=K ** -0.5)
    C0 = W.normal(r, (M, N))
    old = emu.emu_get_path()
    emu.emu_set_path(c["path"])
    try:
        dA = _padded(torch, A, c["pads"][0], c["offs"][0])
        dB = _padded(torch, B, c["pads"][1], c["offs"][1])
        oc = c["offs"][2]
        Cs = torch.full((M + ROWS_BELOW, N + c["pads"][2] + oc), SENTINEL, device="cuda")
        Cs[:M, oc:oc + N] = torch.from_numpy(C0).cuda()
        dC = Cs[:M, oc:oc + N]
        kw = dict(alpha=c["alpha"], beta=c["beta"], mode=c["mode"])
        if c["entry"] == "bsplit":
            P = emu.emu_split_b(dB, transB=bool(tB), mode=c["mode"])
            emu.emu_sgemm_bsplit(dA, P, dC, **kw)
        else:
            emu.emu_sgemm(dA, dB, dC, transB=bool(tB), **kw)
        torch.cuda.synchronize()
        full = Cs.cpu().numpy()
    finally:
        emu.emu_set_path(old)
    assert np.all(full[:M, :oc] == np.float32(SENTINEL)), f"case {i} ({c})"
    assert np.all(full[:M, oc + N:] == np.float32(SENTINEL)), f"case {i} ({c})"
    assert np.all(full[M:] == np.float32(SENTINEL)), f"case {i}: rows past M written ({c})"
    _check(c, i, A, B, C0, np.ascontiguousarray(full[:M, oc:oc + N]))


def test_no_device_error_after_fuzz(emu):
    assert emu.emu_get_last_device_error() == 0
