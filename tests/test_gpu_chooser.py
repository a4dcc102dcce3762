"""The PERFORMANT strategy on the GPU: the call runs the kernel the chooser
names (seen through the library's per-kind launch counters) and the result
meets the accuracy bound either way."""
import numpy as np
import pytest

import oracle
from oracle import checks
from fp32_emulated_gemm_split_gb300 import workloads as W
from gpu_util import emu_module, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def emu():
    m = emu_module()
    yield m
    m.emu_set_strategy("eager")
    m.emu_profile_enable(False)


@pytest.mark.parametrize("shape", [(64, 64, 16), (1000, 700, 8), (1024, 1024, 1024), (300, 260, 700)])
def test_performant_runs_the_chosen_kernel(emu, shape):
    import torch
    M, N, K = shape
    r = W.rng(M + N + K)
    A, B = W.uniform(r, (M, K)), W.uniform(r, (K, N))
    emu.emu_set_strategy("performant")
    want = emu.emu_choose_mode(M, N, K, "bf16x9")
    emu.emu_profile_enable(True)          # resets the counters
    C = torch.empty((M, N), device="cuda")
    emu.emu_sgemm(to_dev(A), to_dev(B), C, mode="bf16x9")
    torch.cuda.synchronize()
    n_simt, _ = emu.emu_profile_read("gemm_simt")
    n_tc = emu.emu_profile_read("gemm_tc")[0] + emu.emu_profile_read("gemm_fused")[0]
    emu.emu_profile_enable(False)
    emu.emu_set_strategy("eager")
    assert (n_simt, n_tc) == ((1, 0) if want == "fp32_simt" else (0, 1))
    Cref, Sabs = oracle.gemm_ref(A, B)
    assert checks.error_ratio(C.cpu().numpy(), Cref, Sabs, K, 1.0, 0.0) <= 1.0


def test_both_choices_occur(emu):
    assert emu.emu_choose_mode(64, 64, 16, "bf16x9", "performant") == "fp32_simt"
    assert emu.emu_choose_mode(1024, 1024, 1024, "bf16x9", "performant") == "bf16x9"
