"""fp64 CPU oracle for C = alpha*A*B + beta*C (row-major FP32 inputs).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may use this package; the product library
never does, and this package imports nothing from it.

The arithmetic lives in ``sgemm_ref.c`` (a plain fp64 triple loop, the
definition written out; see its header for the pages it follows and the
readings taken where they are silent).  This module only compiles it with
gcc and marshals numpy arrays into it.

Pinned by ``tests/test_oracle.py``: exact rational brute force on tiny shapes,
integer-valued inputs against exact integer products, identity, permutation
and all-ones closed forms, the beta/alpha/K quick-return semantics, a
hand-worked example under ``tests/golden/``, and a cross-check against an
fp64 library matmul.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sgemm_ref.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_sgemm.so")

_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_f64 = ctypes.c_double
_pf = ctypes.POINTER(ctypes.c_float)
_pd = ctypes.POINTER(ctypes.c_double)
_pi64 = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library (gcc, OpenMP); returns its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    lib.oracle_sgemm_f64.restype = ctypes.c_int
    lib.oracle_sgemm_f64.argtypes = [
        _i64, _i64, _i64, _f64, _pf, _i64, _pf, _i64, _f64, _pf, _i64,
        _pd, _i64, ctypes.c_int]
    lib.oracle_sgemm_entries_f64.restype = ctypes.c_int
    lib.oracle_sgemm_entries_f64.argtypes = [
        _i64, _f64, _pf, _i64, _pf, _i64, _f64, _pf, _i64, _i64,
        _pi64, _pi64, _pd, ctypes.c_int]
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def load_variant(path: str):
    """Bind another compiled copy of ``sgemm_ref.c`` (the tests compile
    deliberately broken copies to show that the pins catch them)."""
    return _bind(ctypes.CDLL(path))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _fptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.dtype == np.float32 and a.flags.c_contiguous
    return a.ctypes.data_as(_pf)


def _check_operand(name: str, arr: np.ndarray, rows: int, cols: int) -> int:
    if arr.dtype != np.float32 or arr.ndim != 2 or not arr.flags.c_contiguous:
        raise ValueError(f"{name} must be a C-contiguous 2-D float32 array")
    if rows > 0 and (arr.shape[0] < rows or arr.shape[1] < cols):
        raise ValueError(f"{name} of shape {arr.shape} is smaller than {rows}x{cols}")
    return arr.shape[1]


def sgemm_ref(M: int, N: int, K: int, alpha: float, A: np.ndarray,
              B: np.ndarray, beta: float = 0.0, C0: np.ndarray | None = None,
              threads: int = 0, lib=None) -> np.ndarray:
    """fp64 result [M, N] of alpha*A*B + beta*C0.

    A is [M, lda] (lda >= K), B is [K, ldb] (ldb >= N), C0 is [M, ldc] or None
    (allowed only when beta == 0).  Padding columns are never read.
    """
    lda = _check_operand("A", A, M, K) if M > 0 else max(K, 1)
    ldb = _check_operand("B", B, K, N) if K > 0 else max(N, 1)
    ldc = max(N, 1)
    if beta != 0.0:
        if C0 is None:
            raise ValueError("beta != 0 needs C0")
        ldc = _check_operand("C0", C0, M, N)
    out = np.zeros((M, N), dtype=np.float64)
    if M == 0 or N == 0:
        return out
    rc = (lib or _load()).oracle_sgemm_f64(
        M, N, K, float(alpha), _fptr(A), lda, _fptr(B), ldb, float(beta),
        _fptr(C0) if beta != 0.0 else None, ldc,
        out.ctypes.data_as(_pd), N, int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_sgemm_f64 failed with code {rc}")
    return out


def sgemm_ref_entries(K: int, alpha: float, A: np.ndarray, B: np.ndarray,
                      rows: np.ndarray, cols: np.ndarray, beta: float = 0.0,
                      C0: np.ndarray | None = None, threads: int = 0) -> np.ndarray:
    """fp64 values of the selected output entries (rows[t], cols[t])."""
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape or rows.ndim != 1:
        raise ValueError("rows and cols must be 1-D and of equal length")
    M = int(rows.max()) + 1 if rows.size else 0
    N = int(cols.max()) + 1 if cols.size else 0
    lda = _check_operand("A", A, M, K) if M > 0 else max(K, 1)
    ldb = _check_operand("B", B, K, N) if K > 0 else max(N, 1)
    ldc = 1
    if beta != 0.0:
        if C0 is None:
            raise ValueError("beta != 0 needs C0")
        ldc = _check_operand("C0", C0, M, N)
    out = np.zeros(rows.shape[0], dtype=np.float64)
    if rows.size == 0:
        return out
    rc = _load().oracle_sgemm_entries_f64(
        K, float(alpha), _fptr(A), lda, _fptr(B), ldb, float(beta),
        _fptr(C0) if beta != 0.0 else None, ldc, rows.shape[0],
        rows.ctypes.data_as(_pi64), cols.ctypes.data_as(_pi64),
        out.ctypes.data_as(_pd), int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_sgemm_entries_f64 failed with code {rc}")
    return out
