"""Pins for the oracle's BF16 three-way split and TF32 two-way split.

The split is fixed by the pages: x = x0 + 2^-8 x1 + 2^-16 x2 with three BF16
pieces ("Blackwell의 BF16x9" section of the discuss.pytorch.kr page; Figure 1
caption of the NVIDIA blog post), and x = hi + lo with two TF32 pieces and no
scaling (Figure 2 of the NVIDIA blog post).  Rounding is the reading
"nearest, ties to even".  Each test checks the oracle against something other
than itself: an exhaustive brute-force check over all 2^32 FP32 patterns
(tests/split_exhaustive.c), torch's own float->bfloat16 conversion, and a
numpy rint-based TF32 rounding.
"""
import ctypes
import os
import platform
import subprocess

import numpy as np
import pytest
import torch

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _checker():
    src = os.path.join(HERE, "split_exhaustive.c")
    out_dir = os.path.join(HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, f"libsplitcheck.{platform.machine()}.so")
    if not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
        tmp = so + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off",
                               "-fPIC", "-shared", src, "-o", tmp, "-lm"])
        os.replace(tmp, so)
    L = ctypes.CDLL(so)
    for name in ("check_bf16x3_exhaustive", "check_tf32x2_exhaustive"):
        fn = getattr(L, name)
        fn.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]
        fn.restype = ctypes.c_int64
    return L


def test_bf16x3_split_exhaustive_all_fp32_patterns():
    L = _checker()
    fn = ctypes.cast(oracle.lib().oracle_split_bf16x3_vec, ctypes.c_void_p).value
    first = ctypes.c_uint32(0)
    fails = L.check_bf16x3_exhaustive(fn, ctypes.byref(first))
    assert fails == 0, f"{fails} patterns fail, first 0x{first.value:08x}"


def test_tf32x2_split_exhaustive_all_fp32_patterns():
    L = _checker()
    fn = ctypes.cast(oracle.lib().oracle_split_tf32x2_vec, ctypes.c_void_p).value
    first = ctypes.c_uint32(0)
    fails = L.check_tf32x2_exhaustive(fn, ctypes.byref(first))
    assert fails == 0, f"{fails} patterns fail, first 0x{first.value:08x}"


def _random_patterns(n, seed=7):
    r = np.random.Generator(np.random.PCG64(seed))
    u = r.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    return u.view(np.float32)


def test_x0_agrees_with_torch_bfloat16_conversion():
    x = _random_patterns(1 << 22)
    u = x.view(np.uint32)
    finite = (u & 0x7F800000) != 0x7F800000
    # torch rounds values at or above the BF16 overflow threshold to inf,
    # where the reading truncates: compare those separately below.
    below = (u & 0x7FFFFFFF) < 0x7F7F8000
    keep = finite & below
    xs = x[keep]
    p0, _, _ = oracle.split_bf16x3(xs.reshape(1, -1))
    ref = torch.from_numpy(xs.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(p0.ravel(), ref)


def test_overflow_nan_inf_and_signed_zero_readings():
    vals = np.array([0x7F7F8000, 0x7F7FFFFF, 0xFF7FC000, 0x7F800000, 0xFF800000,
                     0x7FC00001, 0xFFFFFFFF, 0x00000000, 0x80000000, 0x3F800000,
                     0xBF800000], np.uint32).view(np.float32)
    p0, p1, p2 = (p.ravel() for p in oracle.split_bf16x3(vals.reshape(1, -1)))
    assert list(p0[:3]) == [0x7F7F, 0x7F7F, 0xFF7F]          # truncated, not inf
    assert list(p0[3:5]) == [0x7F80, 0xFF80] and list(p1[3:5]) == [0, 0] and list(p2[3:5]) == [0, 0]
    assert list(p0[5:7]) == [0x7FC0, 0x7FC0] and list(p2[5:7]) == [0x7FC0, 0x7FC0]
    assert list(p0[7:9]) == [0x0000, 0x8000] and list(p1[7:9]) == [0, 0]
    assert list(p0[9:]) == [0x3F80, 0xBF80] and list(p1[9:]) == [0, 0] and list(p2[9:]) == [0, 0]
    # the pieces of the truncated values still add up to x exactly
    f = oracle.bf16_bits_to_f32
    rec = f(p0[:3]).astype(np.float64) + np.ldexp(f(p1[:3]), -8) + np.ldexp(f(p2[:3]), -16)
    assert np.array_equal(rec, vals[:3].astype(np.float64))


def test_tf32_hi_agrees_with_rint_rounding():
    r = np.random.Generator(np.random.PCG64(11))
    x = (r.standard_normal(1 << 20) * np.exp2(r.integers(-60, 60, 1 << 20))).astype(np.float32)
    x = x[x != 0]
    hi, lo = oracle.split_tf32x2(x.reshape(1, -1))
    xd = x.astype(np.float64)
    e = np.floor(np.log2(np.abs(xd)))
    ulp = np.exp2(e - 10)
    hi_ref = np.rint(xd / ulp) * ulp          # numpy rint: ties to even
    assert np.array_equal(hi.ravel().astype(np.float64), hi_ref)
    res = xd - hi.ravel()
    nz = res != 0
    e2 = np.floor(np.log2(np.abs(res[nz])))
    ulp2 = np.exp2(e2 - 10)
    lo_ref = np.rint(res[nz] / ulp2) * ulp2
    assert np.array_equal(lo.ravel()[nz].astype(np.float64), lo_ref)
    assert np.all(lo.ravel()[~nz] == 0)


def test_bf16_pieces_agree_with_rint_rounding():
    """x0 and x1 are the nearest BF16 values (numpy rint, ties to even) of x and
    of 2^8 (x - x0); x2 carries the rest exactly."""
    r = np.random.Generator(np.random.PCG64(12))
    x = (r.standard_normal(1 << 20) * np.exp2(r.integers(-40, 40, 1 << 20))).astype(np.float32)
    x = x[x != 0]
    p0, p1, p2 = (oracle.bf16_bits_to_f32(p).ravel().astype(np.float64)
                  for p in oracle.split_bf16x3(x.reshape(1, -1)))
    xd = x.astype(np.float64)

    def rint_bf16(v):
        out = np.zeros_like(v)
        nz = v != 0
        ulp = np.exp2(np.floor(np.log2(np.abs(v[nz]))) - 7)
        out[nz] = np.rint(v[nz] / ulp) * ulp
        return out

    assert np.array_equal(p0, rint_bf16(xd))
    v1 = (xd - p0) * 256.0
    assert np.array_equal(p1, rint_bf16(v1))
    assert np.array_equal(p2, (v1 - p1) * 256.0)


def test_split_of_transposed_operand():
    r = np.random.Generator(np.random.PCG64(3))
    X = r.standard_normal((37, 53)).astype(np.float32)
    a = oracle.split_bf16x3(X, trans=True)
    b = oracle.split_bf16x3(np.ascontiguousarray(X.T))
    for pa, pb in zip(a, b):
        assert np.array_equal(pa, pb)
    # a row stride larger than the row length (a view of a wider array)
    W = r.standard_normal((37, 80)).astype(np.float32)
    c = oracle.split_bf16x3(W[:, 5:58])
    d = oracle.split_bf16x3(np.ascontiguousarray(W[:, 5:58]))
    for pc, pd in zip(c, d):
        assert np.array_equal(pc, pd)
    h1, l1 = oracle.split_tf32x2(X, trans=True)
    h2, l2 = oracle.split_tf32x2(np.ascontiguousarray(X.T))
    assert np.array_equal(h1, h2) and np.array_equal(l1, l2)
