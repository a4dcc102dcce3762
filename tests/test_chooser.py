"""The PERFORMANT strategy's host-side choice between an emulated mode and
the FP32 SIMT kernel (no GPU needed: the SM count is passed in)."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def emu():
    from fp32_emulated_gemm_split_gb300 import _build
    _build.build()
    import fp32_emulated_gemm_split_gb300 as emu
    return emu


SHAPES = [(1, 1, 1), (64, 64, 16), (256, 256, 256), (1024, 1024, 16), (12288, 256, 256),
          (8192, 8192, 8192), (64, 64, 4096)]
TC_MODES = ["bf16x9", "tf32x3", "tf32x3_oy", "bf16x3", "tf32"]


@pytest.mark.parametrize("mode", TC_MODES + ["fp32_simt"])
def test_eager_runs_what_is_asked(emu, mode):
    for s in SHAPES:
        assert emu.emu_choose_mode(*s, mode, "eager", 152) == mode


def test_performant_keeps_emulation_for_large_gemms(emu):
    for s in [(8192, 8192, 8192), (4096, 4096, 4096), (12288, 256, 256), (1105920, 256, 256)]:
        for mode in TC_MODES:
            assert emu.emu_choose_mode(*s, mode, "performant", 152) == mode, (s, mode)


def test_performant_takes_simt_for_tiny_k(emu):
    # with a handful of K steps the split launches cost more than the whole SIMT GEMM
    assert emu.emu_choose_mode(64, 64, 16, "bf16x9", "performant", 152) == "fp32_simt"
    assert emu.emu_choose_mode(1024, 1024, 8, "bf16x9", "performant", 152) == "fp32_simt"
    assert emu.emu_choose_mode(64, 64, 16, "fp32_simt", "performant", 152) == "fp32_simt"


def test_choice_follows_the_estimates(emu):
    for s in SHAPES + [(300, 500, 40), (2000, 100, 33)]:
        tc = emu.emu_predict_us(*s, "bf16x9", 152)
        simt = emu.emu_predict_us(*s, "fp32_simt", 152)
        assert tc > 0 and simt > 0
        want = "fp32_simt" if simt < tc else "bf16x9"
        assert emu.emu_choose_mode(*s, "bf16x9", "performant", 152) == want


def test_estimates_grow_with_work(emu):
    for mode in TC_MODES + ["fp32_simt"]:
        t = [emu.emu_predict_us(4096, 4096, k, mode, 152) for k in (64, 256, 1024, 4096)]
        assert all(a < b for a, b in zip(t, t[1:])), mode
        t = [emu.emu_predict_us(m, 4096, 1024, mode, 152) for m in (256, 4096, 65536)]
        assert all(a < b for a, b in zip(t, t[1:])), mode
    # fewer SMs: more waves
    assert emu.emu_predict_us(8192, 8192, 1024, "bf16x9", 76) > emu.emu_predict_us(8192, 8192, 1024, "bf16x9", 152)


def test_invalid_arguments(emu):
    L = emu.lib()
    assert L.emu_choose_mode(4, 4, 4, 9, 1, 152) == -1
    assert L.emu_choose_mode(-1, 4, 4, 0, 1, 152) == -1
    assert L.emu_choose_mode(4, 4, 4, 0, 7, 152) == -1
    assert L.emu_predict_us(4, 4, 4, 0, 0) == -1.0
    assert L.emu_set_strategy(2) == -1


def test_strategy_roundtrip_and_environment(emu):
    assert emu.emu_get_strategy() == "eager"
    emu.emu_set_strategy("performant")
    assert emu.emu_get_strategy() == "performant"
    emu.emu_set_strategy("eager")
    code = ("import fp32_emulated_gemm_split_gb300 as e; print(e.emu_get_strategy())")
    env = dict(os.environ, EMU_SGEMM_STRATEGY="performant")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                         text=True, check=True)
    assert out.stdout.strip() == "performant"
