"""Helpers for the GPU parity tests (imported only by tests marked gpu)."""
import numpy as np
import pytest


def emu_module():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    from fp32_emulated_gemm_split_gb300 import _build
    _build.build()
    import fp32_emulated_gemm_split_gb300 as emu
    emu.lib()
    return emu


def to_dev(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def bits16(t):
    return t.cpu().numpy().view(np.uint16)


def stratified_patterns(low_per_high=64, n_random=1 << 20, seed=99):
    """Every one of the 2^16 sign/exponent/top-mantissa patterns combined with
    `low_per_high` low halves (including 0x0000, 0x8000, 0x7FFF, 0xFFFF), plus
    uniformly random patterns: float32 array of length a multiple of 64."""
    r = np.random.Generator(np.random.PCG64(seed))
    lows = np.concatenate([np.array([0x0000, 0x8000, 0x7FFF, 0xFFFF, 0x0001, 0x7FFE, 0x8001, 0x4000],
                                    np.uint32),
                           r.integers(0, 1 << 16, low_per_high - 8).astype(np.uint32)])
    highs = np.arange(1 << 16, dtype=np.uint32)
    u = (highs[:, None] << 16 | lows[None, :]).ravel()
    u = np.concatenate([u, r.integers(0, 1 << 32, n_random, dtype=np.uint64).astype(np.uint32)])
    u = u[: len(u) // 64 * 64]
    return u.view(np.float32)
