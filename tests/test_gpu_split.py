"""GPU parity of the split/pack kernels: the pieces written by the CUDA path
must equal the oracle's bit for bit (x = x0 + 2^-8 x1 + 2^-16 x2 with
nearest-even rounding, "Blackwell의 BF16x9" section of the discuss.pytorch.kr
page; x = hi + lo in TF32, Figure 2 of the NVIDIA blog post)."""
import numpy as np
import pytest

import oracle
from fp32_emulated_gemm_split_gb300 import workloads as W
from gpu_util import bits16, emu_module, stratified_patterns, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def emu():
    return emu_module()


def _check_bf16(emu, X, trans=False, ldp=None, cols_slice=None):
    Xd = to_dev(X)
    if cols_slice is not None:          # a strided, misaligned view on both sides
        X, Xd = X[:, cols_slice], Xd[:, cols_slice]
    P = emu.emu_split_bf16x3(Xd, trans=trans, ldp=ldp)
    Q = oracle.split_bf16x3(X, trans=trans)
    cols = Q[0].shape[1]
    for i, (p, q) in enumerate(zip(P, Q)):
        got = bits16(p)[:, :cols]
        bad = np.nonzero(got != q)
        assert bad[0].size == 0, (f"piece {i}: {bad[0].size} mismatches, first at {bad[0][0]},{bad[1][0]}: "
                                  f"gpu 0x{got[bad][0]:04x} oracle 0x{q[bad][0]:04x}")


def _check_tf32(emu, X, trans=False, ldp=None, cols_slice=None):
    Xd = to_dev(X)
    if cols_slice is not None:
        X, Xd = X[:, cols_slice], Xd[:, cols_slice]
    hi, lo = emu.emu_split_tf32x2(Xd, trans=trans, ldp=ldp)
    h, l = oracle.split_tf32x2(X, trans=trans)
    cols = h.shape[1]
    assert np.array_equal(hi.cpu().numpy()[:, :cols].view(np.uint32), h.view(np.uint32))
    assert np.array_equal(lo.cpu().numpy()[:, :cols].view(np.uint32), l.view(np.uint32))


def _check_tf32_scaled(emu, X, trans=False):
    hi, lo = emu.emu_split_tf32x2(to_dev(X), trans=trans, scaled=True)
    h, l = oracle.split_tf32x2s(X, trans=trans)
    cols = h.shape[1]
    assert np.array_equal(hi.cpu().numpy()[:, :cols].view(np.uint32), h.view(np.uint32))
    assert np.array_equal(lo.cpu().numpy()[:, :cols].view(np.uint32), l.view(np.uint32))


def test_tf32x2_scaled_residual_bit_patterns(emu):
    """The Ootomo-Yokota split: residual times 2^11 before its rounding."""
    x = stratified_patterns()
    _check_tf32_scaled(emu, x.reshape(-1, 4096))
    X = stratified_patterns(low_per_high=8, n_random=0)[: 1 << 19].reshape(512, 1024)
    _check_tf32_scaled(emu, X, trans=True)
    _check_tf32_scaled(emu, W.stress(W.rng(8), (37, 53)), trans=True)
    _check_tf32_scaled(emu, W.stress(W.rng(9), (37, 53)))


def test_bf16x3_stratified_bit_patterns(emu):
    x = stratified_patterns()
    _check_bf16(emu, x.reshape(-1, 4096))            # vectorised row path


def test_tf32x2_stratified_bit_patterns(emu):
    x = stratified_patterns()
    _check_tf32(emu, x.reshape(-1, 4096))


def test_bf16x3_transposed_and_scalar_paths(emu):
    x = stratified_patterns(low_per_high=8, n_random=0)[: 1 << 19]
    X = x.reshape(512, 1024)
    _check_bf16(emu, X, trans=True)                  # shared-memory transpose path
    _check_bf16(emu, X, cols_slice=slice(3, 1000))    # misaligned rows: scalar path
    _check_bf16(emu, X, trans=True, cols_slice=slice(5, 1001))
    _check_tf32(emu, X, trans=True)
    _check_tf32(emu, X, cols_slice=slice(1, 998))


@pytest.mark.parametrize("shape,trans", [((1, 1), False), ((37, 53), False), ((37, 53), True),
                                         ((65, 129), True), ((130, 72), False), ((3, 8), True)])
def test_ragged_shapes(emu, shape, trans):
    X = W.stress(W.rng(7), shape)
    _check_bf16(emu, X, trans=trans)
    _check_bf16(emu, X, trans=trans, ldp=(X.shape[0] if trans else X.shape[1]) + 13)
    _check_tf32(emu, X, trans=trans)


@pytest.mark.parametrize("name", ["square256_uniform", "mlip192_k256_n1024", "mlip192_k1024_n256",
                                  "stress4096"])
def test_workload_operands_as_the_gemm_packs_them(emu, name):
    g = W.WORKLOADS[name]
    A, B, _ = W.generate(g)
    _check_bf16(emu, A, trans=g.transA)
    _check_bf16(emu, B, trans=not g.transB)          # op(B)^T, K-major
    _check_tf32(emu, A, trans=g.transA)


def test_square8192_operands(emu):
    g = W.WORKLOADS["square8192_normal"]
    A, B, _ = W.generate(g)
    _check_bf16(emu, A)
    _check_bf16(emu, B, trans=True)
    _check_tf32(emu, B, trans=True)                  # vectorised TF32 transpose
    _check_tf32_scaled(emu, B, trans=True)


@pytest.mark.parametrize("cols", [8, 64])
def test_transposed_more_op_row_tiles_than_the_grid(emu, cols):
    """op(X) = X^T with more 64-row tiles of op rows than a grid's y extent
    (65535): the transposed kernels loop over the rest.  cols = 64 runs the
    vectorised kernels (whole tiles), cols = 8 the ragged ones; the last
    tiles are the ones past the first pass."""
    rows = 65536 * 64 + (64 if cols == 64 else 36)
    X = W.normal(W.rng(12), (cols, rows))              # stored cols x rows: op(X) is rows x cols
    _check_bf16(emu, X, trans=True)
    _check_tf32(emu, X, trans=True)
