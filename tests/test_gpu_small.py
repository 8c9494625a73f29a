"""The small-product kernel (plan kind 5: one CTA, or a cluster of up to 8
sharing K, per 32 x 32 block of C) against the fp64 oracle: ragged and
tile-sized shapes, K split over clusters of 1, 2, 4 and 8, all four operand
forms read in place, batches with padded and odd pitches and strides, beta
semantics (C never read when beta == 0), the ldc padding, and the limits
of the automatic choice.  Integer inputs must match bit for bit."""
import numpy as np
import pytest

import oracle
from fp32_sgemm_gb300 import inputs
from conftest import fp32_tolerance

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def handle():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp32_sgemm_gb300 as m
    m.build()
    h = m.Handle()
    yield h
    h.close()


def _stored(rows, cols, ld, batch, bstride, seed, kind, fill=np.nan):
    """[batch, rows, cols] view with row pitch ld and batch stride bstride
    over one NaN-padded device buffer, and the values on the host."""
    span = (batch - 1) * bstride + rows * ld
    flat = np.full(span + 8, fill, np.float32)
    vals = inputs.draw(seed, 0, batch * rows * cols, kind).reshape(batch, rows, cols)
    for z in range(batch):
        for r in range(rows):
            off = z * bstride + r * ld
            flat[off:off + cols] = vals[z, r]
    dev = torch.from_numpy(flat).cuda()
    return torch.as_strided(dev, (batch, rows, cols), (bstride, ld, 1)), vals, dev


def _check(got, ref, kind):
    if kind == "integer":
        np.testing.assert_array_equal(got.astype(np.float64), ref)
    else:
        err = np.abs(got.astype(np.float64) - ref)
        assert np.all(err <= fp32_tolerance(ref)), float(np.max(err / fp32_tolerance(ref)))


def _run(handle, opA, opB, M, N, K, batch, kind, alpha, beta, pad=0, odd=False, seed=0):
    ar, ac = (K, M) if opA else (M, K)
    br, bc = (N, K) if opB else (K, N)
    lda, ldb, ldc = ac + pad, bc + pad, N + pad
    sa = ar * lda + (3 if odd else 0)
    sb = br * ldb + (1 if odd else 0)
    sc = M * ldc + (5 if odd else 0)
    A, Ah, _ = _stored(ar, ac, lda, batch, sa, seed, kind)
    B, Bh, _ = _stored(br, bc, ldb, batch, sb, seed + 1, kind)
    C, C0, cbuf = _stored(M, N, ldc, batch, sc, seed + 2, kind)
    if beta == 0.0:
        C.fill_(float("nan"))                       # never read
    before = cbuf.cpu().numpy().copy()
    handle.gemm_batched(A, B, C, alpha, beta, trans_a=bool(opA), trans_b=bool(opB))
    torch.cuda.synchronize()
    assert handle.device_error() == 0
    got = C.cpu().numpy()
    for z in range(batch):
        opa = np.ascontiguousarray(Ah[z].T if opA else Ah[z])
        opb = np.ascontiguousarray(Bh[z].T if opB else Bh[z])
        c0 = np.ascontiguousarray(C0[z]) if beta != 0.0 else None
        ref = oracle.sgemm_ref(M, N, K, alpha, opa, opb, beta, c0)
        _check(got[z], ref, kind)
    # Nothing outside the C matrices (ldc padding, gaps between batches) changes.
    after = cbuf.cpu().numpy()
    mask = np.ones(after.shape, bool)
    for z in range(batch):
        for r in range(M):
            mask[z * sc + r * ldc: z * sc + r * ldc + N] = False
    assert np.array_equal(after[mask].view(np.uint32), before[mask].view(np.uint32))


SHAPES = [(1, 1, 1), (33, 31, 17), (32, 32, 32), (64, 96, 33), (100, 37, 1), (128, 128, 128),
          (200, 300, 500), (255, 129, 64), (40, 40, 2048)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("kind", ["integer", "uniform"])
def test_shapes(handle, M, N, K, kind):
    # Stored as given when both sides exceed 32 (narrower products take the
    # skinny kernels there); A transposed otherwise, which only this kernel
    # reads in place.
    opA = 0 if min(M, N) > 32 else 1
    if opA == 0:
        A = torch.empty((M, K), device="cuda")
        B = torch.empty((K, N), device="cuda")
        assert handle.plan(A, B, torch.empty((M, N), device="cuda"))["kind"] == 5
    _run(handle, opA, 0, M, N, K, 1, kind, 0.5, 0.25 if kind == "integer" else -1.5, seed=M + N + K)
    _run(handle, opA, 0, M, N, K, 1, kind, 1.0, 0.0, pad=3, seed=M * N + K)


@pytest.mark.parametrize("opA,opB", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("M,N,K,batch,pad,odd", [(70, 45, 100, 3, 4, False), (33, 200, 65, 2, 1, True),
                                                 (8, 8, 300, 5, 0, False), (130, 129, 31, 1, 2, True)])
@pytest.mark.parametrize("kind", ["integer", "uniform"])
def test_operand_forms_and_batches(handle, opA, opB, M, N, K, batch, pad, odd, kind):
    seed = M + 3 * N + 7 * K + 11 * batch + 13 * opA + 17 * opB
    _run(handle, opA, opB, M, N, K, batch, kind, -0.75, 0.5, pad=pad, odd=odd, seed=seed)
    _run(handle, opA, opB, M, N, K, batch, kind, 2.0, 0.0, pad=pad, odd=odd, seed=seed + 100)


def test_automatic_choice_limits(handle):
    def plan(M, N, K, batch=1, **kw):
        A = torch.empty((batch, M, K), device="cuda")
        B = torch.empty((batch, K, N), device="cuda")
        C = torch.empty((batch, M, N), device="cuda")
        if batch == 1:
            return handle.plan(A[0], B[0], C[0], **kw)
        return None
    # 16 blocks of 32 x 32, each shared by a cluster of 4 CTAs (one 32-deep
    # K piece each): as many K ranges as pieces, at most 8, at most 4 CTAs
    # per SM.
    p = plan(128, 128, 128)
    assert p["kind"] == 5 and (p["tile_m"], p["tile_n"], p["ctas"]) == (32, 32, 64)
    assert plan(40, 40, 2048)["ctas"] == 4 * 8
    assert plan(64, 96, 33)["ctas"] == 6 * 2
    assert plan(512, 512, 512)["ctas"] == 256 * 2
    assert plan(512, 512, 512)["kind"] == 5         # 2^27 multiply-adds
    assert plan(1024, 1024, 128)["kind"] == 5
    assert plan(256, 256, 4096)["kind"] == 5        # 2^28, 64 blocks
    assert plan(1025, 512, 64)["kind"] == 1         # a side above 1024
    assert plan(128, 128, 16384)["kind"] == 1       # K above 8192
    assert plan(1024, 1024, 256)["kind"] == 1       # 2^28 in 1024 blocks
    assert plan(1024, 1024, 512)["kind"] == 1       # 2^29
    handle.set_algo(10)                              # a pinned tile configuration
    assert plan(128, 128, 128)["kind"] == 1
    handle.set_algo(0)
    handle.set_schedule(1)                           # a pinned schedule
    assert plan(128, 128, 128)["kind"] == 1
    handle.set_schedule(0)
    handle.set_math_mode(1)                          # 3xTF32 asked for
    assert plan(128, 128, 128)["kind"] == 3
    handle.set_math_mode(0)


def test_many_small_products_one_launch(handle):
    # 500 products of 20 x 50 x 40 in one call: 1000 CTAs of one kernel.
    M, N, K, batch = 20, 50, 40, 500
    A, Ah, _ = _stored(M, K, K, batch, M * K, 3, "integer")
    B, Bh, _ = _stored(K, N, N, batch, K * N, 4, "integer")
    C = torch.empty((batch, M, N), device="cuda")
    handle.gemm_batched(A, B, C, 1.0, 0.0)
    torch.cuda.synchronize()
    got = C.cpu().numpy()
    for z in range(0, batch, 23):
        ref = oracle.sgemm_ref(M, N, K, 1.0, np.ascontiguousarray(Ah[z]), np.ascontiguousarray(Bh[z]))
        np.testing.assert_array_equal(got[z].astype(np.float64), ref)
