"""The C ABI library without a GPU: it builds, loads, exports every entry
point that include/*.h declares, and rejects bad arguments on the host
before anything is launched."""
import ctypes
import glob
import os
import re

import pytest

from fp32_emulated_gemm_split_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def emu():
    _build.build()
    import fp32_emulated_gemm_split_gb300 as m
    m.lib()
    return m


def _declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"\b(emu_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_gemm_entry_point():
    names = _declared_symbols()
    assert "emu_sgemm" in names and "emu_split_bf16x3" in names and len(names) >= 10


def test_library_exports_every_declared_symbol(emu):
    L = ctypes.CDLL(_build.LIB_PATH)
    missing = [n for n in _declared_symbols() if not hasattr(L, n)]
    assert not missing, missing


def test_status_strings_and_version(emu):
    assert emu.emu_status_string(0) == "EMU_OK"
    assert emu.emu_status_string(-5) == "EMU_ERR_TIMEOUT"
    assert emu.emu_version() >= 100


def _sgemm(L, transA=0, transB=0, M=4, N=4, K=4, lda=4, ldb=4, ldc=4, mode=0,
           A=1, B=1, C=1):
    return L.emu_sgemm(transA, transB, M, N, K, 1.0, A, lda, B, ldb, 0.0, C, ldc, mode, None)


@pytest.mark.parametrize("kw", [
    dict(M=-1), dict(N=-2), dict(K=-1), dict(transA=2), dict(transB=-1), dict(mode=7), dict(mode=6), dict(mode=-1),
    dict(lda=3), dict(ldb=3), dict(ldc=3), dict(transA=1, M=8, lda=4),
    dict(transB=1, K=8, ldb=4), dict(C=None), dict(A=None), dict(B=None),
    dict(M=1 << 31),
])
def test_bad_arguments_are_rejected_on_the_host(emu, kw):
    # the pointers are never dereferenced: the checks run before any CUDA call
    assert _sgemm(emu.lib(), **kw) == -1


def test_empty_problem_is_a_noop_without_touching_the_device(emu):
    L = emu.lib()
    assert L.emu_sgemm(0, 0, 0, 5, 3, 1.0, None, 3, None, 5, 0.0, None, 5, 0, None) == 0
    assert L.emu_sgemm(0, 0, 5, 0, 3, 1.0, None, 3, None, 1, 0.0, None, 1, 0, None) == 0


def test_split_argument_checks(emu):
    L = emu.lib()
    assert L.emu_split_bf16x3(1, 4, 4, 3, 0, 1, 1, 1, 4, None) == -1      # ld < cols
    assert L.emu_split_bf16x3(1, 4, 4, 4, 0, 1, 1, 1, 3, None) == -1      # ldp < cols
    assert L.emu_split_bf16x3(1, 4, 4, 4, 2, 1, 1, 1, 4, None) == -1      # bad trans
    assert L.emu_split_bf16x3(1, 4, 4, 4, 0, 1, 1, None, 4, None) == -1   # missing piece
    assert L.emu_split_bf16x3(None, 0, 4, 4, 0, None, None, None, 4, None) == 0   # empty
    assert L.emu_split_tf32x2(1, 8, 4, 4, 1, 1, 1, 4, None) == -1         # trans: ld < rows


def test_path_selection_and_workspace_size(emu):
    assert emu.lib().emu_set_path(5) == -1
    emu.emu_set_path("twopass")
    assert emu.emu_get_path() == "twopass"
    emu.emu_set_path("auto")
    # B's pieces first (region rounded up to 1 KB), then A's.  K-major: rows
    # of op(A) and op(B)^T, K = 13 padded to 16 elements.  BF16x9 keeps an
    # operand stored with K as its row index M- or N-major (13 rows of M or
    # N padded to 64): the larger for A (13 x 128 > 100 x 16), not for B
    # (13 x 64 < 60 x 16).  The other modes stay K-major here (BF16x3 goes
    # M- or N-major only when K is at least 4 times M or N)
    kib = lambda x: (x + 1023) // 1024 * 1024
    assert emu.emu_workspace_size(100, 60, 13, "bf16x9") == kib(3 * 2 * 16 * 60) + 3 * 2 * 13 * 128
    assert emu.emu_workspace_size(100, 60, 13, "tf32x3") == kib(2 * 4 * 16 * 60) + 2 * 4 * 16 * 100
    # the cheaper rungs: two BF16 pieces, one TF32 piece
    assert emu.emu_workspace_size(100, 60, 13, "bf16x3") == kib(2 * 2 * 16 * 60) + 2 * 2 * 16 * 100
    assert emu.emu_workspace_size(100, 60, 13, "tf32") == kib(1 * 4 * 16 * 60) + 1 * 4 * 16 * 100
    assert emu.emu_workspace_size(100, 60, 13, "tf32x3_oy") == emu.emu_workspace_size(100, 60, 13, "tf32x3")
    # one row and one column, K = 1000: the BF16 modes may keep M- and N-major
    # pieces (1000 rows of one 64-element chunk), the larger; TF32 K-major
    # ones (1000 elements)
    assert emu.emu_workspace_size(1, 1, 1000, "bf16x3") == kib(2 * 2 * 1000 * 64) + 2 * 2 * 1000 * 64
    assert emu.emu_workspace_size(1, 1, 1000, "bf16x9") == kib(3 * 2 * 1000 * 64) + 3 * 2 * 1000 * 64
    assert emu.emu_workspace_size(1, 1, 1000, "tf32x3") == kib(2 * 4 * 1000) + 2 * 4 * 1000
    assert emu.lib().emu_workspace_size(100, 60, 13, 6) == 0
    assert emu.emu_workspace_size(100, 60, 13, "fp32_simt") == 0
    assert emu.emu_workspace_size(0, 60, 13, "bf16x9") == 0


def test_profile_read_rejects_bad_kind(emu):
    n = ctypes.c_int64()
    ms = ctypes.c_double()
    assert emu.lib().emu_profile_read(9, ctypes.byref(n), ctypes.byref(ms)) == -1


def _build_c_client(tmp_path):
    import subprocess
    from fp32_emulated_gemm_split_gb300 import _build
    lib = _build.LIB_PATH
    libdir = os.path.dirname(lib)
    name = os.path.basename(lib)
    exe = str(tmp_path / "c_client")
    # link the library by its file name (it carries the machine in its name)
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c_client.c"), "-o", exe,
           "-L" + libdir, "-l:" + name, "-Wl,-rpath," + libdir, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_c_client_compiles_and_links_against_the_header_and_library(emu, tmp_path):
    """The header is plain C and every entry point the client uses links."""
    assert os.path.exists(_build_c_client(tmp_path))


@pytest.mark.gpu
def test_c_client_runs(emu, tmp_path):
    import subprocess
    exe = _build_c_client(tmp_path)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.startswith("ok ")


def _bsplit(L, transA=0, M=4, N=4, K=4, lda=4, ldbp=8, ldc=4, mode=0, A=1, Bp=16, C=1):
    return L.emu_sgemm_bsplit(transA, M, N, K, 1.0, A, lda, Bp, ldbp, 0.0, C, ldc, mode, None)


@pytest.mark.parametrize("kw", [
    dict(M=-1), dict(K=-1), dict(transA=2), dict(mode=2), dict(mode=6), dict(lda=3),
    dict(ldbp=3), dict(ldbp=12), dict(ldc=3), dict(Bp=None), dict(Bp=8), dict(A=None),
    dict(C=None), dict(N=1 << 31),
])
def test_bsplit_bad_arguments_are_rejected_on_the_host(emu, kw):
    """emu_sgemm_bsplit: FP32_SIMT has no pieces, the pieces' rows must be a
    multiple of 8 elements and their base 16-byte aligned (TMA), ldbp >= K;
    nothing is launched or dereferenced."""
    assert _bsplit(emu.lib(), **kw) == -1


def test_bsplit_empty_problem_is_a_noop(emu):
    L = emu.lib()
    assert L.emu_sgemm_bsplit(0, 0, 5, 3, 1.0, None, 3, None, 8, 0.0, None, 5, 0, None) == 0
    assert L.emu_sgemm_bsplit(0, 5, 0, 3, 1.0, None, 3, None, 8, 0.0, None, 1, 0, None) == 0
