"""GPU pins of the nine BF16x9 products: each of a_i b_j must be formed.

The inputs (tests/band_cases.py) put one-piece values on one side and
three-piece values on the other, so that every output is a sum of a few
products a_i b_j that each leave their own bits, every partial sum is exact
in FP32, and the exact product is the only correct answer.  The CPU tests in
tests/test_band_pins.py show that leaving out any single product, or keeping
six or eight of the nine, changes most nonzero outputs.  Here the GPU result
must equal the exact product bit for bit -- on every output -- and the
oracle's BF16x9 emulation on sampled outputs, on the two-pass path, on both
on-chip split paths, inside stream-K tails (a tile's K blocks summed by
several clusters), through the host-buffer entry point and with a
power-of-two alpha.  The cheaper rungs and TF32x3 are pinned the same way on
the first-piece kinds, against the oracle's emulation of the same rung.

Method: "Blackwell의 BF16x9" section of the discuss.pytorch.kr page; Figure 1
caption (BF16x9) and Figure 2 (TF32x3) of the NVIDIA blog post.
"""
import numpy as np
import pytest

import band_cases as BC
import oracle
from fp32_emulated_gemm_split_gb300 import workloads as W
from gpu_util import emu_module, to_dev

pytestmark = pytest.mark.gpu

PATHS = ["twopass", "fused", "fused_tmem"]
# (M, N, K, transA, transB); the on-chip paths need op(A) = A (transA = 0)
SMALL = [(300, 513, 1000, 0, 0), (129, 257, 200, 0, 1), (200, 136, 64, 0, 0)]
TAIL = [(1536, 512, 700, 0, 1),      # 12 tiles of 11 K blocks, shared by 5 clusters each
        (12288, 256, 1024, 0, 0)]    # 48 tiles of 16 K blocks, stream-K over 76 clusters


@pytest.fixture(scope="module")
def emu():
    return emu_module()


class _on_path:
    def __init__(self, emu, path):
        self.emu, self.path = emu, path

    def __enter__(self):
        self.old = self.emu.emu_get_path()
        self.emu.emu_set_path(self.path)

    def __exit__(self, *exc):
        self.emu.emu_set_path(self.old)


def _gemm(emu, A, B, tA, tB, mode="bf16x9", alpha=1.0, path="auto"):
    """GPU result (C pre-filled with NaN, beta = 0) and the GEMM kernel kind
    that ran ("gemm_tc" two-pass, "gemm_fused" on-chip split)."""
    import torch
    M = A.shape[1] if tA else A.shape[0]
    N = B.shape[0] if tB else B.shape[1]
    dA, dB = to_dev(A), to_dev(B)
    C = torch.full((M, N), float("nan"), device="cuda")
    with _on_path(emu, path):
        emu.emu_profile_enable(True)
        emu.emu_sgemm(dA, dB, C, transA=bool(tA), transB=bool(tB), alpha=alpha, mode=mode)
        torch.cuda.synchronize()
        ran = [k for k in ("gemm_tc", "gemm_fused") if emu.emu_profile_read(k)[0] > 0]
        emu.emu_profile_enable(False)
    return C.cpu().numpy(), ran


def _expect_kernel(path, mode, ran):
    want = "gemm_fused" if path in ("fused", "fused_tmem") and mode == "bf16x9" else "gemm_tc"
    assert ran == [want], (path, ran)


def _check_oracle_sample(A, B, tA, tB, C, alpha=1.0, n=1024, fn=oracle.gemm_bf16x9):
    M, N = C.shape
    mi, ni = W.sample_pairs(M, N, n, seed=M + N)
    want = fn(A, B, tA, tB, alpha=alpha, pairs=(mi, ni))
    assert np.array_equal(C[mi, ni].view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("kind", BC.KINDS)
def test_every_product_formed(emu, kind, path, shape):
    M, N, K, tA, tB = shape
    A, B = BC.make(kind, M, N, K, tA, tB, seed=M * 3 + N + K)
    E = BC.exact(A, B, tA, tB).astype(np.float32)
    C, ran = _gemm(emu, A, B, tA, tB, path=path)
    _expect_kernel(path, "bf16x9", ran)
    assert np.array_equal(C.view(np.uint32), E.view(np.uint32))
    _check_oracle_sample(A, B, tA, tB, C)


@pytest.mark.parametrize("shape", TAIL, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("kind", ["a1", "a2", "b1", "b2"])
def test_every_product_formed_in_split_tails(emu, kind, path, shape):
    """Stream-K tails add FP32 sums of K ranges held by different clusters:
    still exact, so still bit for bit; the same bits on a second call."""
    M, N, K, tA, tB = shape
    A, B = BC.make(kind, M, N, K, tA, tB, seed=M + 7 * N + K)
    E = BC.exact(A, B, tA, tB).astype(np.float32)
    C1, ran = _gemm(emu, A, B, tA, tB, path=path)
    _expect_kernel(path, "bf16x9", ran)
    assert np.array_equal(C1.view(np.uint32), E.view(np.uint32))
    C2, _ = _gemm(emu, A, B, tA, tB, path=path)
    assert np.array_equal(C1.view(np.uint32), C2.view(np.uint32))
    _check_oracle_sample(A, B, tA, tB, C1, n=512)
    assert emu.emu_get_last_device_error() == 0


@pytest.mark.parametrize("path", ["twopass", "fused"])
@pytest.mark.parametrize("kind", ["a2", "b2"])
def test_every_product_formed_4096x4096x512(emu, kind, path):
    """256 tiles on 76 clusters: three full rounds and a last round of 28
    tiles whose K blocks all clusters share."""
    A, B = BC.make(kind, 4096, 4096, 512, seed=41)
    E = BC.exact(A, B).astype(np.float32)
    C, ran = _gemm(emu, A, B, 0, 0, path=path)
    _expect_kernel(path, "bf16x9", ran)
    assert np.array_equal(C.view(np.uint32), E.view(np.uint32))
    _check_oracle_sample(A, B, 0, 0, C, n=512)


def test_power_of_two_alpha_is_exact(emu):
    A, B = BC.make("a2", 300, 260, 700, seed=5)
    C, _ = _gemm(emu, A, B, 0, 0, alpha=2.0 ** 64)
    E = np.ldexp(BC.exact(A, B), 64).astype(np.float32)
    assert np.array_equal(C.view(np.uint32), E.view(np.uint32))


@pytest.mark.parametrize("kind", ["a2", "b1"])
def test_host_entry_point_pipelined(emu, kind):
    """emu_sgemm_host on a problem large enough for its row-chunk pipeline
    (B's pieces split once, reused by every chunk)."""
    A, B = BC.make(kind, 8300, 1024, 1024, 0, 1, seed=6)
    E = BC.exact(A, B, 0, 1).astype(np.float32)
    C = emu.emu_sgemm_host(A, B, transB=True)
    assert np.array_equal(C.view(np.uint32), E.view(np.uint32))


@pytest.mark.parametrize("kind,transA,transB", [("a2", 0, 0), ("b1", 0, 1), ("b2", 0, 0),
                                                ("a2", 1, 0), ("b1", 1, 1)])
def test_host_entry_point_column_panels(emu, kind, transA, transB):
    """emu_sgemm_host with a wide op(B) (3000 x 2304 x 1900, B 17.5 MB): B's
    column panels are split into their rows (or, B stored K x N, into their
    columns of B's N-major pieces) as they land and multiplied by op(A)'s
    first 2048 rows (M-major pieces when A is stored K x M); the remaining
    rows then use the whole of B's pieces.  Exact, so bit for bit on every
    output."""
    A, B = BC.make(kind, 3000, 2304, 1900, transA, transB, seed=8 + transB + 2 * transA)
    E = BC.exact(A, B, transA, transB).astype(np.float32)
    emu.emu_profile_enable(True)
    try:
        C = emu.emu_sgemm_host(A, B, transA=bool(transA), transB=bool(transB))
        launches = emu.emu_profile_read("gemm_tc")[0]
    finally:
        emu.emu_profile_enable(False)
    assert launches == 3 + 2, launches          # three panels, two more row chunks
    assert np.array_equal(C.view(np.uint32), E.view(np.uint32))


@pytest.mark.parametrize("kind", ["a2", "b1"])
def test_host_entry_point_n_major_column_panels(emu, kind):
    """emu_sgemm_host with B stored K x N and K >= 4 N (600 x 2304 x 9300,
    B 86 MB): each column panel of B is split row-wise into its columns of
    B's N-major pieces as it lands and multiplied by all 600 rows of op(A)
    (three panels, no later row chunk).  Exact, so bit for bit on every
    output."""
    A, B = BC.make(kind, 600, 2304, 9300, 0, 0, seed=12)
    E = BC.exact(A, B, 0, 0).astype(np.float32)
    emu.emu_profile_enable(True)
    try:
        C = emu.emu_sgemm_host(A, B)
        launches = emu.emu_profile_read("gemm_tc")[0]
    finally:
        emu.emu_profile_enable(False)
    assert launches == 3, launches
    assert np.array_equal(C.view(np.uint32), E.view(np.uint32))


def test_host_entry_point_n_major_column_panels_bf16x3(emu):
    """The same panels in BF16x3, which keeps N-major pieces only for deep K
    (here K = 9300 >= 4 N): with a first-piece A every result is the exact
    sum of the rung's products, so bit for bit the oracle's BF16x3."""
    A, B = BC.make("a0", 600, 2304, 9300, 0, 0, seed=13)
    emu.emu_profile_enable(True)
    try:
        C = emu.emu_sgemm_host(A, B, mode="bf16x3")
        launches = emu.emu_profile_read("gemm_tc")[0]
    finally:
        emu.emu_profile_enable(False)
    assert launches == 3, launches
    _check_oracle_sample(A, B, 0, 0, C, n=2048, fn=oracle.gemm_bf16x3)


LADDER = {"tf32x3": oracle.gemm_tf32x3, "tf32x3_oy": oracle.gemm_tf32x3_oy,
          "bf16x3": oracle.gemm_bf16x3, "tf32": oracle.gemm_tf32}


@pytest.mark.parametrize("shape", SMALL + [(1536, 512, 700, 0, 1)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("mode", list(LADDER))
@pytest.mark.parametrize("kind", ["a0", "b0"])
def test_ladder_modes_form_their_products(emu, kind, mode, shape):
    """With a first-piece operand every rung's result is the exact sum of the
    products it keeps (TF32x3: the exact product), so it is compared bit for
    bit with the oracle's emulation of the same rung on every output."""
    M, N, K, tA, tB = shape
    A, B = BC.make(kind, M, N, K, tA, tB, seed=M + N + 3 * K)
    C, ran = _gemm(emu, A, B, tA, tB, mode=mode)
    _expect_kernel("twopass", mode, ran)
    want = LADDER[mode](A, B, tA, tB)
    assert np.array_equal(C.view(np.uint32), want.view(np.uint32))
    if mode in ("tf32x3", "tf32x3_oy"):
        assert np.array_equal(C, BC.exact(A, B, tA, tB).astype(np.float32))


@pytest.mark.parametrize("shape", SMALL + [(12288, 256, 1024, 0, 1), (1536, 512, 700, 0, 1)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("kind", ["a0", "b0"])
def test_tf32x3_on_chip_forms_its_products(emu, kind, shape):
    """TF32x3 with A split in shared memory by the GEMM kernel: the exact
    product, bit for bit, with the on-chip kernel asserted to have run."""
    M, N, K, tA, tB = shape
    A, B = BC.make(kind, M, N, K, tA, tB, seed=M + 5 * N + K)
    C, ran = _gemm(emu, A, B, tA, tB, mode="tf32x3", path="fused")
    assert ran == ["gemm_fused"], ran
    E = BC.exact(A, B, tA, tB).astype(np.float32)
    assert np.array_equal(C.view(np.uint32), E.view(np.uint32))
    _check_oracle_sample(A, B, tA, tB, C, fn=oracle.gemm_tf32x3)
