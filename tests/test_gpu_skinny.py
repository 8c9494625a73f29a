"""Skinny products (M <= 32 or N <= 32): the HBM-bound streaming kernels vs
the fp64 oracle.  Integer inputs bit exact (the split partial sums are
exact), uniform inputs within the FP32 bound.  Operands TMA can read in
place take the TMA-fed kernels (plan stages == 6); odd pitches and small
shapes take the plain-load kernels (stages == 0): both are covered."""
import itertools

import numpy as np
import pytest

import oracle
from fp32_sgemm_gb300 import inputs
from conftest import fp32_tolerance

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=[0, 1], ids=["ffma", "tf32x3-mode"])
def handle(request):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp32_sgemm_gb300 as m
    m.build()
    h = m.Handle()
    h.set_math_mode(request.param)   # skinny shapes take the FP32 streaming kernels in both modes
    yield h
    h.close()


def _run(h, p):
    A = torch.from_numpy(p.A).cuda()[:, : p.K]
    B = torch.from_numpy(p.B).cuda()[:, : p.N]
    Cb = torch.from_numpy(p.C0 if p.C0 is not None else np.full((p.M, p.N), np.nan, np.float32)).cuda()
    C = Cb[:, : p.N]
    h.gemm(A, B, C, p.alpha, p.beta)
    torch.cuda.synchronize()
    assert h.device_error() == 0
    return Cb.cpu().numpy(), h.plan(A, B, C, p.alpha, p.beta)


def _ref(p):
    return oracle.sgemm_ref(p.M, p.N, p.K, p.alpha, p.A, p.B, p.beta, p.C0)


SMALL = [1, 2, 3, 5, 8, 13, 16, 17, 24, 32]
BIG = [(1000, 129), (4097, 3000), (64, 5)]


@pytest.mark.parametrize("small", SMALL)
@pytest.mark.parametrize("big,K", BIG)
@pytest.mark.parametrize("side", ["m", "n"])
def test_skinny_shapes(handle, small, big, K, side):
    M, N = (small, big) if side == "m" else (big, small)
    pad = 3 if (small + big) % 2 else 0
    for kind in ("integer", "uniform"):
        p = inputs.make_problem(M, N, K, seed=M * 31 + N * 7 + K, kind=kind, alpha=0.75, beta=-0.5,
                                lda=K + pad, ldb=N + pad, ldc=N + 1)
        got, plan = _run(handle, p)
        assert plan["kind"] == 4, plan
        ref = _ref(p)
        if kind == "integer":
            np.testing.assert_array_equal(got[:, :N].astype(np.float64), ref)
        else:
            assert np.all(np.abs(got[:, :N].astype(np.float64) - ref) <= fp32_tolerance(ref))
        assert np.isnan(got[:, N:]).all()


@pytest.mark.parametrize("M,N,K", [(8, 16384, 16384), (16384, 8, 16384), (1, 8192, 12345)])
def test_large_skinny_full(handle, M, N, K):
    p = inputs.make_problem(M, N, K, seed=M + N + K)
    got, plan = _run(handle, p)
    assert plan["kind"] == 4
    ref = _ref(p)
    assert np.all(np.abs(got.astype(np.float64) - ref) <= fp32_tolerance(ref))


def test_beta_zero_never_reads_c(handle):
    p = inputs.make_problem(4, 3000, 700, seed=3)
    got, _ = _run(handle, p)       # C starts as NaN
    assert np.isfinite(got).all()
    ref = _ref(p)
    assert np.all(np.abs(got.astype(np.float64) - ref) <= fp32_tolerance(ref))


def _aligned_problem(M, N, K, seed, kind, alpha=1.0, beta=0.0):
    # Row pitches rounded up to 16 bytes (TMA reads A and B in place).
    r4 = lambda n: (n + 3) // 4 * 4
    return inputs.make_problem(M, N, K, seed=seed, kind=kind, alpha=alpha, beta=beta,
                               with_c=True, lda=r4(K), ldb=r4(N), ldc=N + 1)


@pytest.mark.parametrize("M,N,K", [
    (8, 4096, 1000),        # small M, whole 1024-column blocks, K tail of a k-block
    (3, 3001, 1001),        # small M, ragged last column block
    (16, 2500, 4099),
    (2, 65536, 64),         # 64 blocks of 8 k-blocks: CTA ranges cross blocks
    (1, 300, 16),
    (4097, 8, 1000),        # small N, ragged last 512-row block
    (65539, 3, 48),         # 129 row blocks of 3 k-blocks
    (1000, 16, 2047),
    (600, 5, 16),
    (32, 5000, 777),        # 32-row variant
    (20, 2048, 4096),
    (3000, 32, 999),        # 32-column variant
    (5000, 27, 64),
])
def test_tma_fed_kernels(handle, M, N, K):
    for kind in ("integer", "uniform"):
        p = _aligned_problem(M, N, K, seed=M + 3 * N + 5 * K, kind=kind, alpha=-0.5, beta=2.0)
        got, plan = _run(handle, p)
        assert plan["kind"] == 4 and plan["stages"] == 6, plan
        ref = _ref(p)
        if kind == "integer":
            np.testing.assert_array_equal(got[:, :N].astype(np.float64), ref)
        else:
            assert np.all(np.abs(got[:, :N].astype(np.float64) - ref) <= fp32_tolerance(ref))
        assert np.isnan(got[:, N:]).all(), "ldc padding written"


def test_plain_kernels_for_odd_pitches(handle):
    p = inputs.make_problem(8, 3000, 700, seed=9, kind="integer", lda=701, ldb=3001, ldc=3000)
    got, plan = _run(handle, p)
    assert plan["kind"] == 4 and plan["stages"] == 0, plan
    np.testing.assert_array_equal(got.astype(np.float64), _ref(p))


def test_tma_fed_repeatable_bitwise(handle):
    for M, N in ((8, 20000), (20000, 8)):
        p = _aligned_problem(M, N, 3000, seed=M + N, kind="uniform")
        A = torch.from_numpy(p.A).cuda()[:, :3000]
        B = torch.from_numpy(p.B).cuda()[:, :N]
        first = torch.empty((M, N), device="cuda")
        handle.gemm(A, B, first)
        C = torch.empty_like(first)
        for _ in range(5):
            handle.gemm(A, B, C)
            assert torch.equal(C.view(torch.int32), first.view(torch.int32))
        assert handle.plan(A, B, C)["stages"] == 6
