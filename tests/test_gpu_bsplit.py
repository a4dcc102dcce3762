"""emu_sgemm_bsplit: the GEMM with op(B) given as its split pieces (a linear
layer's weight split once and reused, the way the blog post's MLIP layers
apply one weight to every batch of edge tokens, Figure 3).

* Same kernels, same pieces: the result equals emu_sgemm's for the same B,
  bit for bit, in every mode and on every path.
* The nine-product band pins hold through it (exact results).
* Runs of calls on one stream overlap each kernel's start with the end of
  the one before (programmatic dependent launch): a chain of layers whose
  output is the next layer's input, with ping-pong buffers (each call
  overwrites the buffer the call before it read), must give the same bits as
  the same chain with the device synchronised between calls.
"""
import numpy as np
import pytest

import band_cases as BC
import oracle
from oracle import checks
from fp32_emulated_gemm_split_gb300 import workloads as W
from gpu_util import emu_module, to_dev

pytestmark = pytest.mark.gpu

MODES = ["bf16x9", "bf16x3", "tf32x3", "tf32x3_oy", "tf32"]


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


SHAPES = [(300, 513, 1000, 0, 0), (129, 257, 200, 1, 1), (4100, 200, 300, 0, 1),
          (12288, 256, 256, 0, 1), (1536, 512, 700, 0, 0)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("path", ["auto", "twopass", "fused", "fused_tmem"])
@pytest.mark.parametrize("mode", MODES)
def test_same_bits_as_emu_sgemm(emu, mode, path, shape):
    import torch
    if (path == "fused_tmem" and mode != "bf16x9") or (path == "fused" and mode not in ("bf16x9", "tf32x3")):
        pytest.skip("on-chip splits: BF16x9 (both kernels) and TF32x3 (shared memory)")
    M, N, K, tA, tB = shape
    r = W.rng(M + N + K + tA)
    A = to_dev(W.normal(r, (K, M) if tA else (M, K)))
    B = to_dev(W.normal(r, (N, K) if tB else (K, N), std=K ** -0.5))
    C0 = to_dev(W.uniform(r, (M, N)))
    with _on_path(emu, path):
        ref = C0.clone()
        emu.emu_sgemm(A, B, ref, transA=bool(tA), transB=bool(tB), alpha=1.5, beta=-0.5, mode=mode)
        P = emu.emu_split_b(B, transB=bool(tB), mode=mode)
        out = C0.clone()
        emu.emu_sgemm_bsplit(A, P, out, transA=bool(tA), alpha=1.5, beta=-0.5, mode=mode)
        torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int32), ref.view(torch.int32))
    if M * N * K <= (1 << 28):
        An, Bn, C0n = A.cpu().numpy(), B.cpu().numpy(), C0.cpu().numpy()
        Cref, Sabs = oracle.gemm_ref(An, Bn, tA, tB, 1.5, -0.5, C0n)
        assert checks.error_ratio(out.cpu().numpy(), Cref, Sabs, K, 1.5, -0.5, C0n,
                                  mode=mode) <= 1.0


@pytest.mark.parametrize("path", ["auto", "twopass", "fused", "fused_tmem"])
@pytest.mark.parametrize("kind", ["a2", "b1", "b2"])
def test_nine_products_formed(emu, kind, path):
    import torch
    M, N, K = 4096, 256, 700
    A, B = BC.make(kind, M, N, K, 0, 1, seed=31)
    E = BC.exact(A, B, 0, 1).astype(np.float32)
    with _on_path(emu, path):
        P = emu.emu_split_b(to_dev(B), transB=True)
        out = torch.full((M, N), float("nan"), device="cuda")
        emu.emu_sgemm_bsplit(to_dev(A), P, out)
        torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy().view(np.uint32), E.view(np.uint32))


def test_one_kernel_per_call_on_the_fused_path(emu):
    """BF16x9, K-major A, N <= 256, M >= 4096: one launch, the fused GEMM."""
    import torch
    A = torch.randn(12288, 256, device="cuda")
    B = torch.randn(256, 256, device="cuda")
    P = emu.emu_split_b(B, transB=True)
    C = torch.empty(12288, 256, device="cuda")
    emu.emu_profile_enable(True)
    emu.emu_sgemm_bsplit(A, P, C)
    torch.cuda.synchronize()
    counts = {k: emu.emu_profile_read(k)[0] for k in ("split", "gemm_tc", "gemm_fused")}
    emu.emu_profile_enable(False)
    assert counts == {"split": 0, "gemm_tc": 0, "gemm_fused": 1}, counts


@pytest.mark.parametrize("M,D,mode", [(12288, 256, "bf16x9"), (12288, 128, "bf16x9"),
                                       (6144, 1024, "bf16x9"), (12288, 256, "tf32x3"),
                                       (12288, 256, "bf16x3")])
def test_chain_of_layers_back_to_back(emu, M, D, mode):
    """Eight D x D layers: layer i reads the buffer layer i-1 wrote and
    overwrites the one layer i-1 read.  Run back to back, the chain gives the
    bits it gives with the device synchronised after every call (on the
    fused path for D = 256, the tensor-memory one for D = 128, two-pass for
    D = 1024 and the other modes)."""
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(7 + D)
    Ws = [torch.randn(D, D, generator=g, device="cuda").mul_(D ** -0.5) for _ in range(8)]
    Ps = [emu.emu_split_b(w, transB=True, mode=mode) for w in Ws]
    X0 = torch.randn(M, D, generator=g, device="cuda")

    def run(sync):
        bufs = [X0.clone(), torch.empty(M, D, device="cuda")]
        torch.cuda.synchronize()
        for i, P in enumerate(Ps):
            emu.emu_sgemm_bsplit(bufs[i % 2], P, bufs[(i + 1) % 2], mode=mode)
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return bufs[len(Ps) % 2].clone()

    want = run(True)
    for _ in range(3):
        got = run(False)
        assert torch.equal(got.view(torch.int32), want.view(torch.int32))
    assert torch.isfinite(want).all() and want.abs().max() > 0
    assert emu.emu_get_last_device_error() == 0


def test_bad_pieces_are_rejected(emu):
    import torch
    A = torch.randn(64, 32, device="cuda")
    P = emu.emu_split_b(torch.randn(32, 48, device="cuda"))
    C = torch.full((64, 48), 3.0, device="cuda")
    L = emu.lib()
    h = torch.cuda.current_stream().cuda_stream
    # misaligned base, row stride not a multiple of 8, FP32 SIMT
    assert L.emu_sgemm_bsplit(0, 64, 48, 32, 1.0, A.data_ptr(), 32, P.data_ptr() + 2, 32, 0.0,
                              C.data_ptr(), 48, 0, h) == -1
    assert L.emu_sgemm_bsplit(0, 64, 48, 32, 1.0, A.data_ptr(), 32, P.data_ptr(), 36, 0.0,
                              C.data_ptr(), 48, 0, h) == -1
    assert L.emu_sgemm_bsplit(0, 64, 48, 32, 1.0, A.data_ptr(), 32, P.data_ptr(), 32, 0.0,
                              C.data_ptr(), 48, 2, h) == -1
    torch.cuda.synchronize()
    assert torch.all(C == 3.0)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("K", [1001, 1005, 1007, 64 + 3])
def test_padding_columns_of_the_pieces_are_not_read(emu, mode, K):
    """Columns K..ldbp-1 of the pieces hold NaN (BF16 0x7FC0, FP32 NaN): the
    tensor copies clip at K, so the result is finite and equal, bit for bit,
    to the same call on zero-padded pieces."""
    import torch
    r = W.rng(K)
    M, N = 700, 300
    A = to_dev(W.normal(r, (M, K)))
    B = to_dev(W.normal(r, (N, K), std=K ** -0.5))
    P = emu.emu_split_b(B, transB=True, mode=mode)
    ref = torch.empty(M, N, device="cuda")
    emu.emu_sgemm_bsplit(A, P, ref, mode=mode)
    Q = P.clone()
    if Q.dtype == torch.int16:
        Q[:, :, K:] = 0x7FC0
    else:
        Q[:, :, K:] = float("nan")
    out = torch.empty(M, N, device="cuda")
    emu.emu_sgemm_bsplit(A, Q, out, mode=mode)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    assert torch.equal(out.view(torch.int32), ref.view(torch.int32))
