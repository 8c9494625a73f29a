"""Pins of the fp64 oracle against things other than itself.

Each pin is chosen so that a plausible slip in the oracle (a dropped alpha or
beta term, a wrong sign, a transposed operand, a wrong leading dimension, an
off-by-one in a loop bound, reading C when beta == 0) fails at least one test:

  * hand-worked examples (tests/golden/), typed in by hand, not computed;
  * exact rational arithmetic (fractions.Fraction) on tiny shapes;
  * integer-valued inputs against exact integer matrix products;
  * identity, permutation and all-ones closed forms;
  * the BLAS quick-return semantics chosen where the pages are silent;
  * an fp64 library matmul (numpy) as an independent implementation.
"""
import itertools
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from fp32_sgemm_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sgemm_worked_examples.txt")


def _parse_golden(path):
    cases, cur, block = [], None, None
    for raw in open(path):
        line = raw.split("#", 1)[0].strip()
        if not line:
            continue
        tok = line.split()
        if tok[0] == "case":
            cur = {"name": tok[1], "A": [], "B": [], "C0": [], "expected": []}
            cases.append(cur)
        elif tok[0] == "dims":
            cur["M"], cur["N"], cur["K"] = map(int, tok[1:4])
            cur["alpha"], cur["beta"] = float(tok[4]), float(tok[5])
        elif tok[0] in ("A", "B", "C0", "expected"):
            block = tok[0]
        else:
            cur[block].append([float(v) for v in tok])
    return cases


def _f32(rows):
    return np.ascontiguousarray(np.array(rows, dtype=np.float32))


@pytest.mark.parametrize("case", _parse_golden(GOLDEN), ids=lambda c: c["name"])
def test_hand_worked_examples(case):
    M, N, K = case["M"], case["N"], case["K"]
    A, B = _f32(case["A"]), _f32(case["B"])
    assert A.shape == (M, K) and B.shape == (K, N)
    C0 = _f32(case["C0"]) if case["C0"] else np.full((M, N), np.nan, np.float32)
    got = oracle.sgemm_ref(M, N, K, case["alpha"], A, B, case["beta"], C0)
    np.testing.assert_array_equal(got, np.array(case["expected"], dtype=np.float64))


def _exact(M, N, K, alpha, A, B, beta, C0):
    out = [[Fraction(0)] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            s = Fraction(0)
            for k in range(K):
                s += Fraction(float(A[i, k])) * Fraction(float(B[k, j]))
            v = Fraction(alpha) * s
            if beta != 0.0:
                v += Fraction(beta) * Fraction(float(C0[i, j]))
            out[i][j] = v
    return out


_TINY = [(1, 1, 1), (1, 5, 3), (4, 1, 7), (3, 4, 1), (5, 3, 2), (2, 6, 9), (7, 7, 7)]


@pytest.mark.parametrize("M,N,K", _TINY)
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (0.5, 0.25), (-1.75, 3.0)])
def test_brute_force_exact_rationals(M, N, K, alpha, beta):
    p = inputs.make_problem(M, N, K, seed=M * 100 + N * 10 + K, alpha=alpha,
                            beta=beta, with_c=True, lda=K + 2, ldb=N + 1, ldc=N + 3)
    got = oracle.sgemm_ref(M, N, K, alpha, p.A, p.B, beta, p.C0)
    ex = _exact(M, N, K, alpha, p.A, p.B, beta, p.C0)
    for i, j in itertools.product(range(M), range(N)):
        absum = sum(abs(float(p.A[i, k]) * float(p.B[k, j])) for k in range(K))
        bound = (K + 3) * 2.0 ** -52 * (abs(alpha) * absum + abs(beta * float(p.C0[i, j])))
        assert abs(Fraction(got[i, j]) - ex[i][j]) <= Fraction(bound) + Fraction(1, 2 ** 1074)


@pytest.mark.parametrize("M,N,K,lda,ldb", [(37, 53, 61, 61, 53), (128, 128, 128, 128, 128),
                                           (65, 33, 300, 301, 40), (200, 1, 17, 20, 1)])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (0.5, 0.25)])
def test_integer_inputs_match_exact_integer_product(M, N, K, lda, ldb, alpha, beta):
    p = inputs.make_problem(M, N, K, seed=3 + 1000, kind="integer", alpha=alpha,
                            beta=beta, with_c=True, lda=lda, ldb=ldb)
    Ai = p.A[:, :K].astype(np.int64)
    Bi = p.B[:, :N].astype(np.int64)
    exact = Ai @ Bi
    want = alpha * exact.astype(np.float64)
    if beta != 0.0:
        want = want + beta * p.C0[:, :N].astype(np.float64)
    got = oracle.sgemm_ref(M, N, K, alpha, p.A, p.B, beta, p.C0)
    np.testing.assert_array_equal(got, want)


def test_identity_left_and_right():
    n, N = 70, 45
    p = inputs.make_problem(n, N, n, seed=5)
    eye = np.eye(n, dtype=np.float32)
    np.testing.assert_array_equal(oracle.sgemm_ref(n, N, n, 1.0, eye, p.B),
                                  p.B[:, :N].astype(np.float64))
    q = inputs.make_problem(N, n, n, seed=6)
    np.testing.assert_array_equal(oracle.sgemm_ref(N, n, n, 1.0, q.A, eye),
                                  q.A[:, :n].astype(np.float64))


def test_permutation_rows_and_columns():
    n, N = 33, 20
    perm = np.random.default_rng(0).permutation(n)
    P = np.zeros((n, n), np.float32)
    P[np.arange(n), perm] = 1.0
    p = inputs.make_problem(n, N, n, seed=8)
    got = oracle.sgemm_ref(n, N, n, 1.0, P, p.B)
    np.testing.assert_array_equal(got, p.B[perm, :N].astype(np.float64))
    # Right multiplication by P^T permutes columns of A.
    q = inputs.make_problem(N, n, n, seed=9)
    PT = np.ascontiguousarray(P.T)
    got = oracle.sgemm_ref(N, n, n, 1.0, q.A, PT)
    np.testing.assert_array_equal(got, q.A[:, :n][:, perm].astype(np.float64))


@pytest.mark.parametrize("M,N,K", [(3, 5, 7), (64, 48, 1023)])
def test_all_ones_closed_form(M, N, K):
    A = np.ones((M, K), np.float32)
    B = np.ones((K, N), np.float32)
    C0 = inputs.make_problem(M, N, 1, seed=2, with_c=True).C0
    got = oracle.sgemm_ref(M, N, K, 0.5, A, B, 0.25, C0)
    np.testing.assert_array_equal(got, 0.5 * K + 0.25 * C0.astype(np.float64))


def test_beta_zero_does_not_read_c():
    p = inputs.make_problem(9, 11, 13, seed=12)
    C0 = np.full((9, 11), np.nan, np.float32)
    got = oracle.sgemm_ref(9, 11, 13, 1.0, p.A, p.B, 0.0, C0)
    assert np.isfinite(got).all()
    np.testing.assert_array_equal(got, oracle.sgemm_ref(9, 11, 13, 1.0, p.A, p.B))


def test_alpha_zero_and_k_zero_skip_the_product():
    p = inputs.make_problem(6, 8, 5, seed=13, beta=0.5)
    A_nan = np.full_like(p.A, np.nan)
    got = oracle.sgemm_ref(6, 8, 5, 0.0, A_nan, p.B, 0.5, p.C0)
    np.testing.assert_array_equal(got, 0.5 * p.C0.astype(np.float64))
    got = oracle.sgemm_ref(6, 8, 0, 2.0, np.zeros((6, 1), np.float32),
                           np.zeros((0, 8), np.float32), -1.5, p.C0)
    np.testing.assert_array_equal(got, -1.5 * p.C0.astype(np.float64))
    got = oracle.sgemm_ref(6, 8, 0, 2.0, np.zeros((6, 1), np.float32),
                           np.zeros((0, 8), np.float32), 0.0, None)
    np.testing.assert_array_equal(got, np.zeros((6, 8)))


def test_empty_outputs():
    assert oracle.sgemm_ref(0, 5, 3, 1.0, np.zeros((0, 3), np.float32),
                            np.zeros((3, 5), np.float32)).shape == (0, 5)
    assert oracle.sgemm_ref(4, 0, 3, 1.0, np.zeros((4, 3), np.float32),
                            np.zeros((3, 1), np.float32)).shape == (4, 0)


def test_padding_columns_never_read():
    # The generator fills padding with NaN; any read of it would poison the result.
    p = inputs.make_problem(31, 17, 29, seed=14, beta=2.0, lda=37, ldb=21, ldc=19)
    got = oracle.sgemm_ref(31, 17, 29, 1.0, p.A, p.B, 2.0, p.C0)
    assert np.isfinite(got).all()


def test_transposed_operand_would_be_caught():
    # A square case where A.B != B.A and A.B != A^T.B, so swapped or
    # transposed operands in the oracle cannot pass the other pins unnoticed.
    p = inputs.make_problem(16, 16, 16, seed=15)
    ab = oracle.sgemm_ref(16, 16, 16, 1.0, p.A, p.B)
    ba = oracle.sgemm_ref(16, 16, 16, 1.0, p.B, p.A)
    atb = oracle.sgemm_ref(16, 16, 16, 1.0, np.ascontiguousarray(p.A.T), p.B)
    assert np.abs(ab - ba).max() > 0.1 and np.abs(ab - atb).max() > 0.1
    lib = p.A.astype(np.float64) @ p.B.astype(np.float64)
    assert np.abs(ab - lib).max() < 1e-12


@pytest.mark.parametrize("M,N,K", [(1, 384, 257), (129, 131, 127), (384, 256, 512)])
def test_cross_check_library_fp64_matmul(M, N, K):
    p = inputs.make_problem(M, N, K, seed=M + N + K, alpha=-0.75, beta=1.5)
    got = oracle.sgemm_ref(M, N, K, -0.75, p.A, p.B, 1.5, p.C0)
    A64 = p.A[:, :K].astype(np.float64)
    B64 = p.B[:, :N].astype(np.float64)
    want = -0.75 * (A64 @ B64) + 1.5 * p.C0[:, :N].astype(np.float64)
    absum = 0.75 * (np.abs(A64) @ np.abs(B64)) + 1.5 * np.abs(p.C0[:, :N])
    assert np.all(np.abs(got - want) <= 2 * (K + 3) * 2.0 ** -52 * absum + 1e-300)


def test_entries_agree_with_full():
    p = inputs.make_problem(257, 300, 129, seed=16, alpha=0.5, beta=0.25, lda=130, ldb=301)
    full = oracle.sgemm_ref(257, 300, 129, 0.5, p.A, p.B, 0.25, p.C0)
    r, c = inputs.sample_entries(257, 300, 4000, 16)
    ent = oracle.sgemm_ref_entries(129, 0.5, p.A, p.B, r, c, 0.25, p.C0)
    np.testing.assert_array_equal(ent, full[r, c])


def test_threads_do_not_change_the_result():
    p = inputs.make_problem(97, 65, 300, seed=17)
    one = oracle.sgemm_ref(97, 65, 300, 1.0, p.A, p.B, threads=1)
    many = oracle.sgemm_ref(97, 65, 300, 1.0, p.A, p.B, threads=4)
    np.testing.assert_array_equal(one, many)
