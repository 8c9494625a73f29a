"""Sizes past 32-bit element indexing: C with more than 2^31 elements, a
skinny B with more than 2^31 elements, and a strided batch whose C spans
more than 2^31 elements.  Integer-valued operands make every entry exact,
so sampled entries must match the fp64 oracle bit for bit."""
import numpy as np
import pytest

import oracle
from fp32_sgemm_gb300 import inputs

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=[0, 1], ids=["ffma", "tf32x3"])
def handle(request):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp32_sgemm_gb300 as m
    m.build()
    h = m.Handle()
    h.set_math_mode(request.param)
    yield h
    h.close()
    torch.cuda.empty_cache()


def _samples(M, N, count, seed):
    rows, cols = inputs.sample_entries(M, N, count, seed)
    # The corners too: the last row and column are where 32-bit offsets break.
    rows = np.concatenate([rows, [0, M - 1, M - 1, 0]])
    cols = np.concatenate([cols, [0, N - 1, 0, N - 1]])
    return rows, cols


def test_output_past_2_31_elements(handle):
    M = N = 46341                          # M * N = 2,147,488,281 > 2^31
    K = 8
    p = inputs.make_problem(M, N, K, seed=91, kind="integer")
    C = torch.empty((M, N), device="cuda")
    handle.gemm(torch.from_numpy(p.A).cuda(), torch.from_numpy(p.B).cuda(), C)
    rows, cols = _samples(M, N, 16384, 91)
    got = C[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().numpy()
    assert handle.device_error() == 0
    np.testing.assert_array_equal(got.astype(np.float64),
                                  oracle.sgemm_ref_entries(K, 1.0, p.A, p.B, rows, cols))
    del C


@pytest.mark.parametrize("N", [(1 << 27) + 5, (1 << 27) + 8], ids=["plain-loads", "tma"])
def test_skinny_operands_past_2_31_elements(handle, N):
    M, K = 16, 16                          # B and C: 2^31 + 16 * (N - 2^27) elements each
    A_h = inputs.pattern(np.arange(M)[:, None], np.arange(K)[None, :], 1)
    B = torch.empty((K, N), device="cuda")
    k = torch.arange(K, device="cuda")[:, None]
    step = 1 << 24
    for j0 in range(0, N, step):
        j = torch.arange(j0, min(N, j0 + step), device="cuda")[None, :]
        B[:, j0:j0 + j.shape[1]] = inputs.pattern(k, j, 2)
    C = torch.empty((M, N), device="cuda")
    handle.gemm(torch.from_numpy(A_h).cuda(), B, C)
    plan = handle.plan(torch.from_numpy(A_h).cuda(), B, C)
    assert plan["kind"] == 4 and plan["stages"] == (6 if N % 4 == 0 else 0)
    rows, cols = _samples(M, N, 4096, 92)
    got = C[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().numpy()
    assert handle.device_error() == 0
    # The oracle gets the columns of B the samples use, from the same formula.
    B_cols = inputs.pattern(np.arange(K)[:, None], cols[None, :], 2)          # K x samples
    ref = np.array([oracle.sgemm_ref(1, 1, K, 1.0, A_h[r:r + 1], np.ascontiguousarray(B_cols[:, t:t + 1]))[0, 0]
                    for t, r in enumerate(rows)])
    np.testing.assert_array_equal(got.astype(np.float64), ref)
    del B, C


def test_batch_spanning_past_2_31_elements(handle):
    batch, M, N, K = 520, 2048, 2048, 8    # C: 2,181,038,080 elements
    z = np.arange(batch)[:, None, None]
    A_h = inputs.pattern(z * 1000 + np.arange(M)[None, :, None], np.arange(K)[None, None, :], 3)
    B_h = inputs.pattern(z * 1000 + np.arange(K)[None, :, None], np.arange(N)[None, None, :], 4)
    C = torch.empty((batch, M, N), device="cuda")
    handle.gemm_batched(torch.from_numpy(A_h).cuda(), torch.from_numpy(B_h).cuda(), C)
    assert handle.device_error() == 0
    for b in (0, 263, batch - 1):
        rows, cols = _samples(M, N, 2048, 93 + b)
        got = C[b][torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().numpy()
        ref = oracle.sgemm_ref_entries(K, 1.0, np.ascontiguousarray(A_h[b]), np.ascontiguousarray(B_h[b]),
                                       rows, cols)
        np.testing.assert_array_equal(got.astype(np.float64), ref, err_msg=f"batch entry {b}")
    del C
