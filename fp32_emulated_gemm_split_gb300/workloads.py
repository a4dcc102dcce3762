"""Seeded synthetic inputs for the emulated-FP32 GEMM workloads.

This module only draws random numbers; it holds none of the method's
arithmetic, so both the CUDA path's tests and the CPU oracle can take their
inputs from it.  Every generator uses numpy's PCG64 with a fixed seed.

The workloads stand in for the ones the pages measure ("Unlocking Tensor Core
Performance for Machine Learning Interatomic Potentials", Figure 3: the PET
model's large GEMMs on a 192-atom water box and a 17,280-atom supercell, plus
square 4096^3 and 8192^3 GEMMs).  No model, checkpoint or dataset is used:
the MLIP layers are linear layers over 64 edge tokens per atom with
activations drawn from N(0, 1) and weights from N(0, 1/K).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np

EDGE_TOKENS_PER_ATOM = 64
# (N, K) of the three layer GEMMs: K=256 -> N=256, K=256 -> N=1024, K=1024 -> N=256.
MLIP_LAYERS = ((256, 256), (1024, 256), (256, 1024))


@dataclass(frozen=True)
class Gemm:
    """One GEMM C = alpha * op(A) op(B) + beta * C0 (row-major storage).

    ``transB=True`` stores B as an N x K weight matrix, the layout of a linear
    layer's weight (y = x W^T)."""
    name: str
    M: int
    N: int
    K: int
    transA: bool = False
    transB: bool = False
    alpha: float = 1.0
    beta: float = 0.0
    dist: str = "normal"      # "uniform" | "normal" | "mlip" | "stress"
    seed: int = 1
    mode: str = "bf16x9"
    extra: dict = field(default_factory=dict, compare=False)

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K


def _mlip(atoms: int, seed: int):
    M = atoms * EDGE_TOKENS_PER_ATOM
    return [Gemm(f"mlip{atoms}_k{K}_n{N}", M, N, K, transB=True, dist="mlip",
                 seed=seed * 100 + i) for i, (N, K) in enumerate(MLIP_LAYERS)]


WORKLOADS = {
    g.name: g for g in [
        Gemm("square256_uniform", 256, 256, 256, dist="uniform", seed=1),
        *_mlip(192, 2),
        *_mlip(17280, 3),
        Gemm("stress4096", 4096, 4096, 4096, alpha=1.5, beta=0.5, dist="stress", seed=4),
        Gemm("square8192_normal", 8192, 8192, 8192, dist="normal", seed=5),
        Gemm("square8192_normal_tf32x3", 8192, 8192, 8192, dist="normal", seed=5,
             mode="tf32x3"),
    ]
}


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def uniform(r: np.random.Generator, shape, lo=-1.0, hi=1.0) -> np.ndarray:
    return r.uniform(lo, hi, size=shape).astype(np.float32)


def normal(r: np.random.Generator, shape, std=1.0) -> np.ndarray:
    x = r.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def stress(r: np.random.Generator, shape) -> np.ndarray:
    """sign * m * 2^e with m ~ U[1, 2), e ~ U{-30..30}; 1% exact zeros and
    0.1% FP32 subnormals (random nonzero mantissa, exponent field 0)."""
    n = int(np.prod(shape))
    sign = np.where(r.random(n) < 0.5, -1.0, 1.0)
    m = r.uniform(1.0, 2.0, n)
    e = r.integers(-30, 31, n)
    x = (sign * np.ldexp(m, e)).astype(np.float32)
    u = r.random(n)
    x[u < 0.01] = 0.0
    sub = (u >= 0.01) & (u < 0.011)
    bits = r.integers(1, 1 << 23, n, dtype=np.uint32) | (sign < 0).astype(np.uint32) << 31
    x[sub] = bits[sub].view(np.float32)
    return x.reshape(shape)


def _draw(r, dist, shape, K):
    if dist == "uniform":
        return uniform(r, shape)
    if dist == "normal":
        return normal(r, shape)
    if dist == "stress":
        return stress(r, shape)
    raise ValueError(dist)


def generate(g: Gemm):
    """Return (A, B, C0) as float32 arrays in the stored layout (C0 is None
    when beta == 0)."""
    r = rng(g.seed)
    a_shape = (g.K, g.M) if g.transA else (g.M, g.K)
    b_shape = (g.N, g.K) if g.transB else (g.K, g.N)
    if g.dist == "mlip":
        B = normal(r, b_shape, std=1.0 / np.sqrt(g.K))
        ra = rng(g.seed * 7919 + 1)
        A = normal(ra, a_shape)
        return A, B, None
    A = _draw(r, g.dist, a_shape, g.K)
    B = _draw(r, g.dist, b_shape, g.K)
    C0 = uniform(r, (g.M, g.N)) if g.beta != 0.0 else None
    return A, B, C0


def sample_pairs(M: int, N: int, n: int, seed: int = 12345):
    """Output positions for sampled checks: n random (m, n) pairs plus the
    first and last row and column corners."""
    r = rng(seed)
    mi = r.integers(0, M, n)
    ni = r.integers(0, N, n)
    edge_m = np.array([0, 0, M - 1, M - 1, M // 2], np.int64)
    edge_n = np.array([0, N - 1, 0, N - 1, N // 2], np.int64)
    return (np.concatenate([mi, edge_m]).astype(np.int64),
            np.concatenate([ni, edge_n]).astype(np.int64))


def with_mode(g: Gemm, mode: str) -> Gemm:
    return replace(g, mode=mode)
