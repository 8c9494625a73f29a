"""Skinny products (M <= 16 or N <= 16): the HBM-bound streaming kernels vs
the fp64 oracle.  Integer inputs bit exact (the split partial sums are
exact), uniform inputs within the FP32 bound."""
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


SMALL = [1, 2, 3, 5, 8, 13, 16]
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
