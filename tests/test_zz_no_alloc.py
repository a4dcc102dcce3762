"""emu_sgemm_noalloc: the GEMM for callers that cannot let the library
allocate device memory (their memory belongs to another allocator or a fixed
budget, or they cannot take cudaMalloc's device-wide synchronisation).  It
must give the same results as emu_sgemm while keeping the split pieces in the
library's fixed 64 MiB device array.  This file is collected last on purpose:
a run that stops at its first failure has run every other test before it."""
import ctypes

import numpy as np
import pytest

import oracle
from oracle import checks
from fp32_emulated_gemm_split_gb300 import workloads as W
from gpu_util import emu_module, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def emu():
    return emu_module()


# Two different problems back to back: the second call must not be affected
# by what the first one left in the shared array.
CASES = [
    dict(M=1000, N=700, K=300, transA=False, transB=False, alpha=1.25, beta=0.5, mode="bf16x9"),
    dict(M=513, N=257, K=1029, transA=True, transB=True, alpha=1.0, beta=0.0, mode="tf32x3"),
]


def test_matches_emu_sgemm_on_two_calls_in_a_row(emu):
    import torch
    for i, c in enumerate(CASES):
        r = W.rng(900 + i)
        A = W.normal(r, (c["K"], c["M"]) if c["transA"] else (c["M"], c["K"]))
        B = W.normal(r, (c["N"], c["K"]) if c["transB"] else (c["K"], c["N"]))
        C0 = W.normal(r, (c["M"], c["N"]))
        dA, dB = to_dev(A), to_dev(B)
        ref = to_dev(C0)
        emu.emu_sgemm(dA, dB, ref, transA=c["transA"], transB=c["transB"], alpha=c["alpha"],
                      beta=c["beta"], mode=c["mode"])
        out = to_dev(C0)
        L = emu.lib()           # the C entry point itself, through ctypes
        st = L.emu_sgemm_noalloc(int(c["transA"]), int(c["transB"]), c["M"], c["N"], c["K"],
                                 c["alpha"], dA.data_ptr(), dA.shape[1], dB.data_ptr(),
                                 dB.shape[1], c["beta"], out.data_ptr(), c["N"],
                                 emu.MODE[c["mode"]], torch.cuda.current_stream().cuda_stream)
        assert st == 0, emu.emu_status_string(st)
        torch.cuda.synchronize()
        got, want = out.cpu().numpy(), ref.cpu().numpy()
        Cref, Sabs = oracle.gemm_ref(A, B, c["transA"], c["transB"], c["alpha"], c["beta"], C0)
        mode = "tf32x3" if c["mode"] == "tf32x3" else "bf16x9"
        bound = checks.elementwise_bound(c["K"], c["alpha"], c["beta"], Sabs, C0, mode)
        assert np.all(np.abs(got.astype(np.float64) - want) <= bound)     # vs emu_sgemm
        assert checks.error_ratio(got, Cref, Sabs, c["K"], c["alpha"], c["beta"], C0, mode) <= 1.0
    assert emu.emu_get_last_device_error() == 0


def test_rejects_a_problem_larger_than_the_array(emu):
    import torch
    A = torch.ones((4096, 4096), device="cuda")
    C = torch.full((4096, 4096), 7.0, device="cuda")
    # 6 * (4096 + 4096) * 4096 bytes = 192 MiB of pieces > 64 MiB
    with pytest.raises(emu.EmuError) as e:
        emu.emu_sgemm_noalloc(A, A, C)
    assert e.value.status == -1
    torch.cuda.synchronize()
    assert torch.all(C == 7.0)              # nothing was launched
