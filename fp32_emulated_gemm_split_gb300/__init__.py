"""Python binding of libemusgemm: FP32 GEMM emulated on GB300 tensor cores.

The functions below have the names of the C entry points declared in
``include/emu_sgemm.h`` and only marshal arguments: every step of the
computation runs in the library's CUDA kernels.  There is no fallback: if the
library has not been built, or the GPU is not a GB300 (sm_103a), the calls
raise.

Tensors are ``torch.float32`` CUDA tensors in row-major storage (unit stride
along rows); a tensor whose *rows* have unit stride (a transposed view) is
passed as the stored matrix with the ``trans`` flag flipped.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

MODE = {"bf16x9": 0, "tf32x3": 1, "fp32_simt": 2, "bf16x3": 3, "tf32": 4, "tf32x3_oy": 5}
PATH = {"auto": 0, "twopass": 1, "fused": 2, "fused_tmem": 3}
PROFILE_KIND = {"split": 0, "gemm_tc": 1, "gemm_fused": 2, "gemm_simt": 3, "scale": 4}

_lib = None


class EmuError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = ""
        if status in (-3, -4, -6):
            detail = f", CUDA: {emu_last_cuda_error()}"
        super().__init__(f"{where}: {emu_status_string(status)} ({status}){detail}")


def lib() -> ctypes.CDLL:
    """Load the in-tree libemusgemm; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB_PATH):
            raise RuntimeError(
                f"libemusgemm is not built ({_build.LIB_PATH} is missing); run "
                "`python -c 'import __graft_entry__ as g; g.build()'` first")
        _lib = _declare(ctypes.CDLL(_build.LIB_PATH))
    return _lib


_i64, _int, _f32, _vp, _f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_double


def _declare(L):
    gemm = [_int, _int, _i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64, _int, _vp]
    for name in ("emu_sgemm", "emu_sgemm_host"):
        getattr(L, name).argtypes = gemm
        getattr(L, name).restype = _int
    L.emu_sgemm_noalloc.argtypes = gemm
    L.emu_sgemm_noalloc.restype = _int
    L.emu_sgemm_bsplit.argtypes = [_int, _i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp,
                                   _i64, _int, _vp]
    L.emu_sgemm_bsplit.restype = _int
    L.emu_split_bf16x3.argtypes = [_vp, _i64, _i64, _i64, _int, _vp, _vp, _vp, _i64, _vp]
    L.emu_split_bf16x3.restype = _int
    L.emu_split_tf32x2.argtypes = [_vp, _i64, _i64, _i64, _int, _vp, _vp, _i64, _vp]
    L.emu_split_tf32x2.restype = _int
    L.emu_set_strategy.argtypes = [_int]
    L.emu_set_strategy.restype = _int
    L.emu_get_strategy.argtypes = []
    L.emu_get_strategy.restype = _int
    L.emu_choose_mode.argtypes = [_i64, _i64, _i64, _int, _int, _int]
    L.emu_choose_mode.restype = _int
    L.emu_predict_us.argtypes = [_i64, _i64, _i64, _int, _int]
    L.emu_predict_us.restype = ctypes.c_double
    L.emu_split_tf32x2_scaled.argtypes = [_vp, _i64, _i64, _i64, _int, _vp, _vp, _i64, _vp]
    L.emu_split_tf32x2_scaled.restype = _int
    L.emu_set_path.argtypes = [_int]
    L.emu_set_path.restype = _int
    L.emu_get_path.argtypes = []
    L.emu_get_path.restype = _int
    L.emu_workspace_size.argtypes = [_i64, _i64, _i64, _int]
    L.emu_workspace_size.restype = ctypes.c_size_t
    for name in ("emu_get_last_device_error", "emu_clear_device_error", "emu_shutdown"):
        getattr(L, name).argtypes = []
        getattr(L, name).restype = _int
    L.emu_selftest_timeout.argtypes = [_int, _vp]
    L.emu_selftest_timeout.restype = _int
    L.emu_profile_enable.argtypes = [_int]
    L.emu_profile_enable.restype = _int
    L.emu_profile_read.argtypes = [_int, ctypes.POINTER(_i64), ctypes.POINTER(_f64)]
    L.emu_profile_read.restype = _int
    L.emu_status_string.argtypes = [_int]
    L.emu_status_string.restype = ctypes.c_char_p
    L.emu_last_cuda_error.argtypes = []
    L.emu_last_cuda_error.restype = ctypes.c_char_p
    L.emu_version.argtypes = []
    L.emu_version.restype = _int
    return L


def _check(status: int, where: str) -> None:
    if status != 0:
        raise EmuError(status, where)


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _stored(X, trans: bool):
    """(tensor whose rows are contiguous, trans flag, leading dimension)."""
    import torch
    if X.dtype != torch.float32 or X.dim() != 2:
        raise TypeError("expected a 2-D float32 tensor")
    if X.stride(1) == 1 or X.size(1) <= 1:
        ld = X.stride(0) if X.size(0) > 1 else max(X.size(1), 1)
        return X, bool(trans), max(ld, X.size(1), 1)
    if X.stride(0) == 1:
        Xt = X.t()
        ld = Xt.stride(0) if Xt.size(0) > 1 else max(Xt.size(1), 1)
        return Xt, not trans, max(ld, Xt.size(1), 1)
    raise ValueError("matrix needs unit stride along rows or columns")


def _mode(mode) -> int:
    return MODE[mode] if isinstance(mode, str) else int(mode)


# ------------------------------------------------------------------- GEMM --

def emu_sgemm(A, B, C=None, *, transA=False, transB=False, alpha=1.0, beta=0.0,
              mode="bf16x9", stream=None):
    """C = alpha * op(A) @ op(B) + beta * C on the current CUDA stream; returns C.

    A, B (and C) are float32 CUDA tensors; C is allocated when not given (then
    beta must be 0)."""
    import torch
    As, tA, lda = _stored(A, transA)
    Bs, tB, ldb = _stored(B, transB)
    M, K = (As.size(1), As.size(0)) if tA else (As.size(0), As.size(1))
    K2, N = (Bs.size(1), Bs.size(0)) if tB else (Bs.size(0), Bs.size(1))
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C")
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    if C.dim() != 2 or C.shape != (M, N) or C.dtype != torch.float32 or (C.stride(1) != 1 and N > 1):
        raise ValueError("C must be an M x N float32 tensor with unit row stride")
    ldc = C.stride(0) if M > 1 else max(N, 1)
    st = lib().emu_sgemm(int(tA), int(tB), M, N, K, float(alpha), As.data_ptr(), lda,
                         Bs.data_ptr(), ldb, float(beta), C.data_ptr(), max(ldc, N, 1),
                         _mode(mode), _stream_handle(stream))
    _check(st, "emu_sgemm")
    return C


def emu_sgemm_noalloc(A, B, C, *, transA=False, transB=False, alpha=1.0, beta=0.0,
                      mode="bf16x9", stream=None):
    """emu_sgemm without any device allocation by the library: the split
    pieces go to a fixed 64 MiB device array instead of a workspace grown with
    cudaMalloc (for callers that cannot allocate).  C must be given; a
    problem whose pieces do not fit raises EmuError(EMU_ERR_INVALID_VALUE).
    Calls that overlap on the GPU share that array and must be serialised."""
    As, tA, lda = _stored(A, transA)
    Bs, tB, ldb = _stored(B, transB)
    M, K = (As.size(1), As.size(0)) if tA else (As.size(0), As.size(1))
    K2, N = (Bs.size(1), Bs.size(0)) if tB else (Bs.size(0), Bs.size(1))
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if C.dim() != 2 or C.shape != (M, N) or (C.stride(1) != 1 and N > 1):
        raise ValueError("C must be an M x N float32 tensor with unit row stride")
    ldc = C.stride(0) if M > 1 else max(N, 1)
    st = lib().emu_sgemm_noalloc(int(tA), int(tB), M, N, K, float(alpha), As.data_ptr(), lda,
                                 Bs.data_ptr(), ldb, float(beta), C.data_ptr(), max(ldc, N, 1),
                                 _mode(mode), _stream_handle(stream))
    _check(st, "emu_sgemm_noalloc")
    return C


PIECES = {"bf16x9": 3, "bf16x3": 2, "tf32x3": 2, "tf32x3_oy": 2, "tf32": 1}


def emu_split_b(B, transB=False, mode="bf16x9", stream=None):
    """The pieces of op(B)^T that emu_sgemm_bsplit takes, as one CUDA tensor
    of shape (pieces, N, ldp) (int16 BF16 bits for the BF16 modes, float32
    for the TF32 ones; ldp = K rounded up to 8), split by the library's own
    split kernels."""
    import torch
    m = mode if isinstance(mode, str) else {v: k for k, v in MODE.items()}[int(mode)]
    Bs, tB, ldb = _stored(B, transB)
    K, N = (Bs.size(1), Bs.size(0)) if tB else (Bs.size(0), Bs.size(1))
    ldp = max((K + 7) // 8 * 8, 8)
    tf32 = m.startswith("tf32")
    P = torch.zeros((3 if not tf32 else 2, N, ldp),
                    dtype=torch.float32 if tf32 else torch.int16, device=B.device)
    h = _stream_handle(stream)
    if N > 0 and K > 0:
        if tf32:
            name = "emu_split_tf32x2_scaled" if m == "tf32x3_oy" else "emu_split_tf32x2"
            st = getattr(lib(), name)(Bs.data_ptr(), N, K, ldb, int(not tB), P[0].data_ptr(),
                                      P[1].data_ptr(), ldp, h)
        else:
            st = lib().emu_split_bf16x3(Bs.data_ptr(), N, K, ldb, int(not tB), P[0].data_ptr(),
                                        P[1].data_ptr(), P[2].data_ptr(), ldp, h)
        _check(st, "emu_split_b")
    return P[:PIECES[m]]


def emu_sgemm_bsplit(A, Bp, C=None, *, transA=False, alpha=1.0, beta=0.0, mode="bf16x9",
                     stream=None):
    """C = alpha * op(A) @ op(B) + beta * C with op(B) given by its pieces
    (``emu_split_b``): a (pieces, N, ldp) CUDA tensor."""
    import torch
    As, tA, lda = _stored(A, transA)
    M, K = (As.size(1), As.size(0)) if tA else (As.size(0), As.size(1))
    if Bp.dim() != 3 or not Bp.is_contiguous():
        raise ValueError("Bp must be a contiguous (pieces, N, ldp) tensor")
    N, ldp = Bp.size(1), Bp.size(2)
    if ldp < K:
        raise ValueError("Bp's rows are shorter than K")
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C")
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    if C.dim() != 2 or C.shape != (M, N) or C.dtype != torch.float32 or (C.stride(1) != 1 and N > 1):
        raise ValueError("C must be an M x N float32 tensor with unit row stride")
    ldc = C.stride(0) if M > 1 else max(N, 1)
    st = lib().emu_sgemm_bsplit(int(tA), M, N, K, float(alpha), As.data_ptr(), lda,
                                Bp.data_ptr(), ldp, float(beta), C.data_ptr(), max(ldc, N, 1),
                                _mode(mode), _stream_handle(stream))
    _check(st, "emu_sgemm_bsplit")
    return C


def emu_sgemm_host(A, B, C=None, *, transA=False, transB=False, alpha=1.0, beta=0.0,
                   mode="bf16x9", stream=None):
    """emu_sgemm on host (numpy float32, row-major) buffers; returns C (numpy).

    The library copies the operands to the GPU, runs the GEMM, copies C back
    and synchronises before returning."""
    import numpy as np
    A = np.ascontiguousarray(A, np.float32)
    B = np.ascontiguousarray(B, np.float32)
    M, K = (A.shape[1], A.shape[0]) if transA else A.shape
    K2, N = (B.shape[1], B.shape[0]) if transB else B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C")
        C = np.empty((M, N), np.float32)
    elif C.dtype != np.float32 or not C.flags.c_contiguous or C.shape != (M, N):
        raise ValueError("C must be a C-contiguous M x N float32 array")
    st = lib().emu_sgemm_host(int(transA), int(transB), M, N, K, float(alpha),
                              A.ctypes.data, max(A.shape[1], 1), B.ctypes.data,
                              max(B.shape[1], 1), float(beta), C.ctypes.data, max(N, 1),
                              _mode(mode), _stream_handle(stream))
    _check(st, "emu_sgemm_host")
    return C


# ----------------------------------------------------------------- splits --

def emu_split_bf16x3(X, trans=False, ldp=None, stream=None):
    """Three BF16 pieces of op(X) as int16 CUDA tensors (bit patterns), each
    rows x ldp (columns past op(X)'s are left as allocated)."""
    import torch
    Xs, t, ld = _stored(X, trans)
    rows, cols = (Xs.size(1), Xs.size(0)) if t else (Xs.size(0), Xs.size(1))
    ldp = cols if ldp is None else ldp
    P = [torch.zeros((rows, max(ldp, 1)), dtype=torch.int16, device=X.device) for _ in range(3)]
    st = lib().emu_split_bf16x3(Xs.data_ptr(), rows, cols, ld, int(t), P[0].data_ptr(),
                                P[1].data_ptr(), P[2].data_ptr(), max(ldp, 1),
                                _stream_handle(stream))
    _check(st, "emu_split_bf16x3")
    return tuple(P)


def emu_split_tf32x2(X, trans=False, ldp=None, stream=None, scaled=False):
    """TF32 hi / lo pieces of op(X) as float32 CUDA tensors (rows x ldp);
    scaled=True gives the 2^11-scaled residual (emu_split_tf32x2_scaled)."""
    import torch
    Xs, t, ld = _stored(X, trans)
    rows, cols = (Xs.size(1), Xs.size(0)) if t else (Xs.size(0), Xs.size(1))
    ldp = cols if ldp is None else ldp
    hi = torch.zeros((rows, max(ldp, 1)), dtype=torch.float32, device=X.device)
    lo = torch.zeros_like(hi)
    name = "emu_split_tf32x2_scaled" if scaled else "emu_split_tf32x2"
    st = getattr(lib(), name)(Xs.data_ptr(), rows, cols, ld, int(t), hi.data_ptr(),
                              lo.data_ptr(), max(ldp, 1), _stream_handle(stream))
    _check(st, name)
    return hi, lo


# ------------------------------------------------------------ the rest --

def emu_set_path(path) -> None:
    _check(lib().emu_set_path(PATH[path] if isinstance(path, str) else int(path)), "emu_set_path")


STRATEGY = {"eager": 0, "performant": 1}


def emu_set_strategy(strategy) -> None:
    """'eager' (every call runs the mode it asks for) or 'performant' (the FP32
    SIMT kernel where it is predicted faster than the emulation)."""
    v = STRATEGY[strategy] if isinstance(strategy, str) else int(strategy)
    _check(lib().emu_set_strategy(v), "emu_set_strategy")


def emu_get_strategy() -> str:
    return {0: "eager", 1: "performant"}[lib().emu_get_strategy()]


def emu_choose_mode(M, N, K, mode="bf16x9", strategy=None, sms=0) -> str:
    """The mode emu_sgemm would run for this shape (sms 0: the current GPU's)."""
    st = -1 if strategy is None else (STRATEGY[strategy] if isinstance(strategy, str) else int(strategy))
    v = lib().emu_choose_mode(M, N, K, _mode(mode), st, sms)
    if v < 0:
        raise EmuError(-1, "emu_choose_mode")
    return {m: n for n, m in MODE.items()}[v]


def emu_predict_us(M, N, K, mode="bf16x9", sms=152) -> float:
    return float(lib().emu_predict_us(M, N, K, _mode(mode), sms))


def emu_get_path() -> str:
    v = lib().emu_get_path()
    return {0: "auto", 1: "twopass", 2: "fused", 3: "fused_tmem"}[v]


def emu_workspace_size(M, N, K, mode="bf16x9") -> int:
    return int(lib().emu_workspace_size(M, N, K, _mode(mode)))


def emu_get_last_device_error() -> int:
    return int(lib().emu_get_last_device_error())


def emu_clear_device_error() -> None:
    _check(lib().emu_clear_device_error(), "emu_clear_device_error")


def emu_selftest_timeout(limit_us=1000, stream=None) -> int:
    return int(lib().emu_selftest_timeout(int(limit_us), _stream_handle(stream)))


def emu_profile_enable(on=True) -> None:
    _check(lib().emu_profile_enable(int(bool(on))), "emu_profile_enable")


def emu_profile_read(kind) -> tuple[int, float]:
    n = ctypes.c_int64(0)
    ms = ctypes.c_double(0.0)
    k = PROFILE_KIND[kind] if isinstance(kind, str) else int(kind)
    _check(lib().emu_profile_read(k, ctypes.byref(n), ctypes.byref(ms)), "emu_profile_read")
    return int(n.value), float(ms.value)


def emu_last_cuda_error() -> str:
    return lib().emu_last_cuda_error().decode()


def emu_status_string(status: int) -> str:
    return lib().emu_status_string(int(status)).decode()


def emu_shutdown() -> None:
    _check(lib().emu_shutdown(), "emu_shutdown")


def emu_version() -> int:
    return int(lib().emu_version())
