"""emu_sgemm_noalloc: the GEMM for callers that cannot let the library
allocate device memory (their memory belongs to another allocator or a fixed
budget, or they cannot take cudaMalloc's device-wide synchronisation).  It
must give results within the same accuracy bound as emu_sgemm while keeping
the split pieces in the library's fixed 64 MiB device array, and once its
first call on the device has returned it must not change the device's free
memory.  This file is collected last on purpose: a run that stops at its
first failure has run every other test before it."""
import numpy as np
import pytest

import band_cases as BC
import oracle
from oracle import checks
from fp32_emulated_gemm_split_gb300 import workloads as W
from gpu_util import emu_module, to_dev

pytestmark = pytest.mark.gpu

LIMIT = 64 << 20


@pytest.fixture(scope="module")
def emu():
    return emu_module()


def _noalloc(emu, dA, dB, C, c):
    """The C entry point itself, through ctypes; returns its status."""
    import torch
    L = emu.lib()
    return L.emu_sgemm_noalloc(int(c["transA"]), int(c["transB"]), c["M"], c["N"], c["K"],
                               c["alpha"], dA.data_ptr(), max(dA.shape[1], 1), dB.data_ptr(),
                               max(dB.shape[1], 1), c["beta"], C.data_ptr(), c["N"],
                               emu.MODE[c["mode"]], torch.cuda.current_stream().cuda_stream)


def _operands(c, seed):
    r = W.rng(seed)
    A = W.normal(r, (c["K"], c["M"]) if c["transA"] else (c["M"], c["K"]))
    B = W.normal(r, (c["N"], c["K"]) if c["transB"] else (c["K"], c["N"]))
    C0 = W.normal(r, (c["M"], c["N"]))
    return A, B, C0


def _bound_mode(mode):
    return mode if mode in checks.MODE_EXTRA else "bf16x9"


# Different problems back to back: a call must not be affected by what the
# one before it left in the shared array.
CASES = [
    dict(M=1000, N=700, K=300, transA=False, transB=False, alpha=1.25, beta=0.5, mode="bf16x9"),
    dict(M=513, N=257, K=1029, transA=True, transB=True, alpha=1.0, beta=0.0, mode="tf32x3"),
    dict(M=300, N=512, K=200, transA=False, transB=True, alpha=-0.5, beta=0.25, mode="bf16x3"),
    dict(M=260, N=300, K=96, transA=True, transB=False, alpha=1.0, beta=0.0, mode="tf32"),
    dict(M=200, N=384, K=520, transA=False, transB=False, alpha=1.0, beta=1.0, mode="tf32x3_oy"),
    dict(M=129, N=65, K=77, transA=False, transB=True, alpha=2.0, beta=-1.0, mode="fp32_simt"),
]


def test_matches_emu_sgemm_call_after_call(emu):
    import torch
    for i, c in enumerate(CASES):
        A, B, C0 = _operands(c, 900 + i)
        dA, dB = to_dev(A), to_dev(B)
        ref = to_dev(C0)
        emu.emu_sgemm(dA, dB, ref, transA=c["transA"], transB=c["transB"], alpha=c["alpha"],
                      beta=c["beta"], mode=c["mode"])
        out = to_dev(C0)
        st = _noalloc(emu, dA, dB, out, c)
        assert st == 0, emu.emu_status_string(st)
        torch.cuda.synchronize()
        got, want = out.cpu().numpy(), ref.cpu().numpy()
        mode = _bound_mode(c["mode"])
        Cref, Sabs = oracle.gemm_ref(A, B, c["transA"], c["transB"], c["alpha"], c["beta"], C0)
        bound = checks.elementwise_bound(c["K"], c["alpha"], c["beta"], Sabs, C0, mode)
        assert np.all(np.abs(got.astype(np.float64) - want) <= bound), c["mode"]   # vs emu_sgemm
        assert checks.error_ratio(got, Cref, Sabs, c["K"], c["alpha"], c["beta"], C0, mode) <= 1.0
    assert emu.emu_get_last_device_error() == 0


def test_k_zero_and_alpha_zero_scale_c(emu):
    import torch
    C0 = W.uniform(W.rng(3), (70, 90))
    A = torch.full((70, 30), float("nan"), device="cuda")      # not read
    B = torch.ones((30, 90), device="cuda")
    for c in (dict(M=70, N=90, K=0, transA=False, transB=False, alpha=1.0, beta=0.5, mode="bf16x9"),
              dict(M=70, N=90, K=30, transA=False, transB=False, alpha=0.0, beta=0.5, mode="tf32x3")):
        out = to_dev(C0)
        assert _noalloc(emu, A, B, out, c) == 0
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), np.float32(0.5) * C0)


def test_nine_products_formed(emu):
    """The band pins of tests/test_gpu_band_pins.py through this entry point:
    every output equals the exact product bit for bit."""
    import torch
    for kind in ("a2", "b2"):
        A, B = BC.make(kind, 300, 513, 1000, seed=17)
        E = BC.exact(A, B).astype(np.float32)
        out = torch.full(E.shape, float("nan"), device="cuda")
        c = dict(M=300, N=513, K=1000, transA=False, transB=False, alpha=1.0, beta=0.0,
                 mode="bf16x9")
        assert _noalloc(emu, to_dev(A), to_dev(B), out, c) == 0
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy().view(np.uint32), E.view(np.uint32))


def test_problem_exactly_at_the_limit(emu):
    """TF32X3 keeps 2 pieces x 4 bytes x K per row of op(A) and op(B)^T:
    (4096 + 4096) x 8 x 1024 bytes is the array's 64 MiB exactly; one more
    column of C is refused."""
    import torch
    c = dict(M=4096, N=4096, K=1024, transA=False, transB=False, alpha=1.0, beta=0.0,
             mode="tf32x3")
    assert (c["M"] + c["N"]) * 8 * c["K"] == LIMIT
    A, B, _ = _operands(c, 77)
    dA, dB = to_dev(A), to_dev(B)
    out = torch.empty((4096, 4096), device="cuda")
    assert _noalloc(emu, dA, dB, out, c) == 0
    torch.cuda.synchronize()
    mi, ni = W.sample_pairs(4096, 4096, 2048, seed=5)
    Cref, Sabs = oracle.gemm_ref(A, B, pairs=(mi, ni))
    assert checks.error_ratio(out.cpu().numpy()[mi, ni], Cref, Sabs, 1024, 1.0, 0.0,
                              mode="tf32x3") <= 1.0
    B1 = to_dev(W.normal(W.rng(78), (1024, 4097)))
    out1 = torch.full((4096, 4097), 7.0, device="cuda")
    c1 = dict(c, N=4097)
    assert _noalloc(emu, dA, B1, out1, c1) == -1               # EMU_ERR_INVALID_VALUE
    torch.cuda.synchronize()
    assert torch.all(out1 == 7.0)


def test_rejects_a_problem_larger_than_the_array(emu):
    import torch
    A = torch.ones((4096, 4096), device="cuda")
    C = torch.full((4096, 4096), 7.0, device="cuda")
    # 6 * (4096 + 4096) * 4096 bytes = 192 MiB of pieces > 64 MiB
    with pytest.raises(emu.EmuError) as e:
        emu.emu_sgemm_noalloc(A, A, C)
    assert e.value.status == -1
    # sizes whose byte counts would wrap a 64-bit product are refused too
    L = emu.lib()
    big = (1 << 31) - 1
    st = L.emu_sgemm_noalloc(0, 0, 1 << 30, 1 << 30, big, 1.0, A.data_ptr(), big,
                             A.data_ptr(), 1 << 30, 0.0, C.data_ptr(), 1 << 30,
                             emu.MODE["tf32x3"], torch.cuda.current_stream().cuda_stream)
    assert st == -1
    torch.cuda.synchronize()
    assert torch.all(C == 7.0)              # nothing was launched


def test_calls_after_the_first_allocate_nothing(emu):
    """After one call per mode (the first call on the device resolves the
    array and each kernel's first launch loads it), further calls of every
    mode leave the device's free memory and torch's allocator unchanged."""
    import torch
    cases = [dict(c) for c in CASES] + [
        dict(M=70, N=90, K=0, transA=False, transB=False, alpha=1.0, beta=0.5, mode="bf16x9")]
    bufs = []
    for i, c in enumerate(cases):
        A, B, C0 = _operands(c, 950 + i)
        bufs.append((to_dev(A), to_dev(B), to_dev(C0)))
    torch.cuda.synchronize()
    for (dA, dB, dC), c in zip(bufs, cases):
        assert _noalloc(emu, dA, dB, dC, c) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    reserved0, allocated0 = torch.cuda.memory_reserved(), torch.cuda.memory_allocated()
    for _ in range(3):
        for (dA, dB, dC), c in zip(bufs, cases):
            assert _noalloc(emu, dA, dB, dC, c) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_reserved() == reserved0
    assert torch.cuda.memory_allocated() == allocated0
    assert emu.emu_get_last_device_error() == 0
