"""CPU oracle for the emulated-FP32 GEMM (BF16x9 and TF32x3).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU-baseline leg
of the benchmark may use this package; the library's product path never
imports it and shares no code with it.

The arithmetic lives in ``emu_oracle.c`` (plain loops, FP64 reference, FP32
emulation written from the method's definition); this module compiles it with
gcc on first use and marshals numpy arrays.  See the header of the C file for
the passages it follows and the readings it takes.

Matrices are row major numpy arrays of float32 with unit column stride; the
row stride of the array is the leading dimension.  ``op(X)`` is ``X`` or
``X.T`` as selected by the ``trans`` flags.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "emu_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, f"liboracle.{platform.machine()}.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off: every FP32 product and sum must be rounded on its own
# (gcc contracts a*b+c into an FMA by default on aarch64).
CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
          "-fPIC", "-shared"]


def compile_c(src: str, out: str) -> str:
    """Compile one C file of the oracle into a shared library at ``out``."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, src, "-o", tmp, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build`` (idempotent)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_c(_SRC, _LIB_PATH)


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


_i64 = ctypes.c_int64
_int = ctypes.c_int
_f32 = ctypes.c_float
_vp = ctypes.c_void_p


def _declare(L: ctypes.CDLL) -> ctypes.CDLL:
    L.oracle_bf16_rne.argtypes = [_f32]
    L.oracle_bf16_rne.restype = ctypes.c_uint16
    L.oracle_tf32_rne_bits.argtypes = [_f32]
    L.oracle_tf32_rne_bits.restype = ctypes.c_uint32
    L.oracle_split_bf16x3.argtypes = [_vp, _i64, _i64, _i64, _int, _vp, _vp, _vp]
    L.oracle_split_bf16x3.restype = None
    L.oracle_split_tf32x2.argtypes = [_vp, _i64, _i64, _i64, _int, _vp, _vp]
    L.oracle_split_tf32x2.restype = None
    L.oracle_split_tf32x2s.argtypes = [_vp, _i64, _i64, _i64, _int, _vp, _vp]
    L.oracle_split_tf32x2s.restype = None
    L.oracle_split_bf16x3_vec.argtypes = [_vp, _i64, _vp, _vp, _vp]
    L.oracle_split_bf16x3_vec.restype = None
    L.oracle_split_tf32x2_vec.argtypes = [_vp, _i64, _vp, _vp]
    L.oracle_split_tf32x2_vec.restype = None
    gemm_args = [_int, _int, _i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64,
                 _f32, _vp, _i64, _vp, _vp, _i64]
    L.oracle_gemm_f64.argtypes = gemm_args + [_vp, _vp]
    L.oracle_gemm_f64.restype = None
    L.oracle_gemm_bf16x9.argtypes = gemm_args + [_vp, _vp]
    L.oracle_gemm_bf16x9.restype = None
    L.oracle_gemm_tf32x3.argtypes = gemm_args + [_vp, _vp]
    L.oracle_gemm_tf32x3.restype = None
    L.oracle_gemm_fp32.argtypes = gemm_args + [_vp]
    L.oracle_gemm_fp32.restype = None
    for name in ("oracle_gemm_bf16x3", "oracle_gemm_tf32", "oracle_gemm_tf32x3_oy"):
        getattr(L, name).argtypes = gemm_args + [_vp]
        getattr(L, name).restype = None
    L.oracle_max_threads.argtypes = []
    L.oracle_max_threads.restype = _int
    return L


def load(path: str) -> ctypes.CDLL:
    """Load another build of the oracle's C file (the tests use this to show
    that a deliberately broken copy fails the pins)."""
    return _declare(ctypes.CDLL(path))


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data


def _mat(X):
    X = np.asarray(X)
    if X.dtype != np.float32 or X.ndim != 2:
        raise TypeError("expected a 2-D float32 array")
    if X.strides[1] != 4:
        X = np.ascontiguousarray(X)
    ld = X.strides[0] // 4 if X.shape[0] > 1 else max(X.shape[1], 1)
    return X, ld


# --------------------------------------------------------------------------
# Splits
# --------------------------------------------------------------------------

def split_bf16x3(X, trans: bool = False, L=None):
    """Three BF16 planes (uint16 bit patterns) of op(X): x = x0 + 2^-8 x1 + 2^-16 x2."""
    X, ld = _mat(X)
    rows, cols = (X.shape[1], X.shape[0]) if trans else X.shape
    P = [np.empty((rows, cols), np.uint16) for _ in range(3)]
    (L or lib()).oracle_split_bf16x3(_ptr(X), rows, cols, ld, int(trans), *(_ptr(p) for p in P))
    return tuple(P)


def split_tf32x2(X, trans: bool = False, L=None):
    """TF32 hi / lo planes (float32 with the low 13 bits zero) of op(X)."""
    X, ld = _mat(X)
    rows, cols = (X.shape[1], X.shape[0]) if trans else X.shape
    hi = np.empty((rows, cols), np.float32)
    lo = np.empty((rows, cols), np.float32)
    (L or lib()).oracle_split_tf32x2(_ptr(X), rows, cols, ld, int(trans), _ptr(hi), _ptr(lo))
    return hi, lo


def split_tf32x2s(X, trans: bool = False, L=None):
    """TF32 hi and 2^11-scaled lo planes of op(X) (the Ootomo-Yokota split)."""
    X, ld = _mat(X)
    rows, cols = (X.shape[1], X.shape[0]) if trans else X.shape
    hi = np.empty((rows, cols), np.float32)
    lo = np.empty((rows, cols), np.float32)
    (L or lib()).oracle_split_tf32x2s(_ptr(X), rows, cols, ld, int(trans), _ptr(hi), _ptr(lo))
    return hi, lo


def bf16_bits_to_f32(P):
    """BF16 bit patterns (uint16) -> float32 values."""
    return (np.asarray(P, np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# GEMMs
# --------------------------------------------------------------------------

def _gemm_setup(A, B, transA, transB, C0, beta, pairs):
    A, lda = _mat(A)
    B, ldb = _mat(B)
    M, K = (A.shape[1], A.shape[0]) if transA else A.shape
    K2, N = (B.shape[1], B.shape[0]) if transB else B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    ldc0 = 1
    if beta != 0.0:
        C0, ldc0 = _mat(C0)
        if C0.shape != (M, N):
            raise ValueError("C0 must be M x N")
    else:
        C0 = None
    if pairs is None:
        mi = np.repeat(np.arange(M, dtype=np.int64), N)
        ni = np.tile(np.arange(N, dtype=np.int64), M)
        full = True
    else:
        mi = np.ascontiguousarray(pairs[0], dtype=np.int64)
        ni = np.ascontiguousarray(pairs[1], dtype=np.int64)
        full = False
    return A, lda, B, ldb, C0, ldc0, M, N, K, mi, ni, full


def _common_args(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C0, ldc0, mi, ni):
    return (int(transA), int(transB), M, N, K, float(alpha), _ptr(A), lda, _ptr(B), ldb,
            float(beta), _ptr(C0), ldc0, _ptr(mi), _ptr(ni), mi.size)


def gemm_ref(A, B, transA=False, transB=False, alpha=1.0, beta=0.0, C0=None, pairs=None, L=None):
    """FP64 reference C_ref and S_abs = sum_k |a||b|.

    With ``pairs=(mi, ni)`` only those outputs are computed (1-D results),
    otherwise full M x N arrays are returned."""
    A, lda, B, ldb, C0, ldc0, M, N, K, mi, ni, full = _gemm_setup(A, B, transA, transB, C0, beta, pairs)
    Cref = np.empty(mi.size, np.float64)
    Sabs = np.empty(mi.size, np.float64)
    (L or lib()).oracle_gemm_f64(*_common_args(transA, transB, M, N, K, alpha, A, lda, B, ldb,
                                        beta, C0, ldc0, mi, ni), _ptr(Cref), _ptr(Sabs))
    if full:
        return Cref.reshape(M, N), Sabs.reshape(M, N)
    return Cref, Sabs


def _emu(fn, nb, A, B, transA, transB, alpha, beta, C0, pairs, with_bands):
    A, lda, B, ldb, C0, ldc0, M, N, K, mi, ni, full = _gemm_setup(A, B, transA, transB, C0, beta, pairs)
    C = np.empty(mi.size, np.float32)
    bands = np.empty((mi.size, nb), np.float64) if with_bands else None
    fn(*_common_args(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C0, ldc0, mi, ni),
       _ptr(C), _ptr(bands))
    if full:
        C = C.reshape(M, N)
        if with_bands:
            bands = bands.reshape(M, N, nb)
    return (C, bands) if with_bands else C


def gemm_bf16x9(A, B, transA=False, transB=False, alpha=1.0, beta=0.0, C0=None,
                pairs=None, with_bands=False, L=None):
    """CPU BF16x9 emulation (FP32 result).  ``with_bands`` also returns the
    five unscaled band sums sum_{i+j=b} a_i b_j in FP64."""
    return _emu((L or lib()).oracle_gemm_bf16x9, 5, A, B, transA, transB, alpha, beta, C0,
                pairs, with_bands)


def gemm_tf32x3(A, B, transA=False, transB=False, alpha=1.0, beta=0.0, C0=None,
                pairs=None, with_bands=False, L=None):
    """CPU TF32x3 emulation (FP32 result).  ``with_bands`` also returns
    [sum hi*hi, sum (hi*lo + lo*hi)] in FP64."""
    return _emu((L or lib()).oracle_gemm_tf32x3, 2, A, B, transA, transB, alpha, beta, C0,
                pairs, with_bands)


def _plain(fn_name, A, B, transA, transB, alpha, beta, C0, pairs, L):
    A, lda, B, ldb, C0, ldc0, M, N, K, mi, ni, full = _gemm_setup(A, B, transA, transB, C0, beta, pairs)
    C = np.empty(mi.size, np.float32)
    getattr(L or lib(), fn_name)(*_common_args(transA, transB, M, N, K, alpha, A, lda, B, ldb,
                                               beta, C0, ldc0, mi, ni), _ptr(C))
    return C.reshape(M, N) if full else C


def gemm_fp32(A, B, transA=False, transB=False, alpha=1.0, beta=0.0, C0=None, pairs=None, L=None):
    """Plain FP32 GEMM: sequential accumulation, product and sum rounded separately."""
    return _plain("oracle_gemm_fp32", A, B, transA, transB, alpha, beta, C0, pairs, L)


def gemm_bf16x3(A, B, transA=False, transB=False, alpha=1.0, beta=0.0, C0=None, pairs=None, L=None):
    """Two BF16 pieces, three products (a0 b0, a0 b1, a1 b0), band 1 first."""
    return _plain("oracle_gemm_bf16x3", A, B, transA, transB, alpha, beta, C0, pairs, L)


def gemm_tf32x3_oy(A, B, transA=False, transB=False, alpha=1.0, beta=0.0, C0=None, pairs=None,
                   L=None):
    """TF32x3 with the 2^11-scaled residual (Ootomo-Yokota correction)."""
    return _plain("oracle_gemm_tf32x3_oy", A, B, transA, transB, alpha, beta, C0, pairs, L)


def gemm_tf32(A, B, transA=False, transB=False, alpha=1.0, beta=0.0, C0=None, pairs=None, L=None):
    """Single-pass TF32: one product of the leading TF32 pieces."""
    return _plain("oracle_gemm_tf32", A, B, transA, transB, alpha, beta, C0, pairs, L)
