"""The oracle's pins catch plausible mistakes.

Each case below compiles a copy of ``oracle/sgemm_ref.c`` with one planted
mistake (on the CPU, into a temporary directory) and runs a small set of the
pin checks against it: the unmodified source must pass all of them and every
mutant must fail at least one.  The problems are square with padded leading
dimensions, so mutants that transpose an index still read inside the buffers.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from fp32_sgemm_gb300 import inputs

SRC = os.path.join(os.path.dirname(oracle.__file__), "sgemm_ref.c")

MUTANTS = {
    "dropped_beta_term": ("orow[j] = alpha * acc[j] + beta * (double)crow[j];",
                          "orow[j] = alpha * acc[j];"),
    "dropped_alpha": ("orow[j] = alpha * acc[j] + beta * (double)crow[j];",
                      "orow[j] = acc[j] + beta * (double)crow[j];"),
    "wrong_sign": ("acc[j] += a * (double)brow[j];", "acc[j] -= a * (double)brow[j];"),
    "transposed_b": ("acc[j] += a * (double)brow[j];",
                     "acc[j] += a * (double)B[j * ldb + k];"),
    "transposed_a": ("const double a = (double)A[i * lda + k];",
                     "const double a = (double)A[k * lda + i];"),
    "lda_taken_as_k": ("const double a = (double)A[i * lda + k];",
                       "const double a = (double)A[i * K + k];"),
    "ldb_taken_as_n": ("const float *brow = B + k * ldb;", "const float *brow = B + k * N;"),
    "k_loop_short": ("for (int64_t k = 0; k < K; ++k) {\n                        const double a",
                     "for (int64_t k = 0; k < K - 1; ++k) {\n                        const double a"),
    "stale_accumulator": ("for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;",
                          "for (int64_t j = 0; j + 1 < N; ++j) acc[j] = 0.0;"),
    "reads_c_when_beta_zero": ("if (beta != 0.0) {\n                    const float *crow",
                               "if (1) {\n                    const float *crow"),
    "reads_ab_when_alpha_zero": ("const int use_product = (alpha != 0.0 && K > 0);\n    int failed",
                                 "const int use_product = (K > 0);\n    int failed"),
}


def _build_variant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    src = src.replace(old, new, 1)
    cfile = tmp_path / f"{name}.c"
    cfile.write_text(src)
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                    "-ffp-contract=off", str(cfile), "-o", str(so)], check=True)
    return oracle.load_variant(str(so))


def _call(lib, M, N, K, alpha, A, B, beta, C0):
    # Always hands over a C buffer, so a mutant that reads C when beta == 0
    # reads NaN instead of dereferencing NULL.
    out = np.zeros((M, N), np.float64)
    f = ctypes.POINTER(ctypes.c_float)
    rc = lib.oracle_sgemm_f64(M, N, K, alpha, A.ctypes.data_as(f), A.shape[1],
                              B.ctypes.data_as(f), B.shape[1], beta,
                              C0.ctypes.data_as(f), C0.shape[1],
                              out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), N, 2)
    assert rc == 0
    return out


def _checks(lib):
    """Names of the pin checks that this build fails."""
    failed = []
    n, pad = 24, 3
    # Integer inputs, exact against an integer matrix product.
    p = inputs.make_problem(n, n, n, 1003, kind="integer", alpha=0.5, beta=0.25,
                            with_c=True, lda=n + pad, ldb=n + pad, ldc=n + pad)
    want = 0.5 * (p.A[:, :n].astype(np.int64) @ p.B[:, :n].astype(np.int64)) \
        + 0.25 * p.C0[:, :n].astype(np.float64)
    if not np.array_equal(_call(lib, n, n, n, 0.5, p.A, p.B, 0.25, p.C0), want):
        failed.append("integer_exact")
    # Uniform inputs against the library fp64 matmul.
    q = inputs.make_problem(n, n, n, 77, alpha=-0.75, beta=1.5, with_c=True,
                            lda=n + pad, ldb=n + pad, ldc=n + pad)
    want = -0.75 * (q.A[:, :n].astype(np.float64) @ q.B[:, :n].astype(np.float64)) \
        + 1.5 * q.C0[:, :n].astype(np.float64)
    got = _call(lib, n, n, n, -0.75, q.A, q.B, 1.5, q.C0)
    if not (np.isfinite(got).all() and np.abs(got - want).max() < 1e-12):
        failed.append("library_fp64")
    # beta == 0 must not read C (C is NaN here).
    nanc = np.full_like(q.C0, np.nan)
    got = _call(lib, n, n, n, 1.0, q.A, q.B, 0.0, nanc)
    want = q.A[:, :n].astype(np.float64) @ q.B[:, :n].astype(np.float64)
    if not (np.isfinite(got).all() and np.abs(got - want).max() < 1e-12):
        failed.append("beta_zero_nan_c")
    # alpha == 0 must not read A or B (A is NaN here).
    nana = np.full_like(q.A, np.nan)
    got = _call(lib, n, n, n, 0.0, nana, q.B, 1.5, q.C0)
    if not np.array_equal(got, 1.5 * q.C0[:, :n].astype(np.float64)):
        failed.append("alpha_zero_nan_a")
    return failed


def test_unmodified_oracle_passes_every_check(tmp_path):
    shutil.copy(SRC, tmp_path / "orig.c")
    lib = _build_variant(tmp_path, "orig", "int oracle_max_threads", "int oracle_max_threads")
    assert _checks(lib) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    lib = _build_variant(tmp_path, name, old, new)
    assert _checks(lib), f"mutant {name} passed every pin"
