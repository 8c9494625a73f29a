"""sgemmStridedBatched vs the fp64 oracle: all four operand forms (A and B
each as stored or transposed), several batch sizes, padded and odd row
pitches, padded and zero batch strides, both arithmetic paths.  The oracle
is applied batch by batch to the explicit op(A), op(B)."""
import itertools

import numpy as np
import pytest

import oracle
from fp32_sgemm_gb300 import inputs
from conftest import fp32_tolerance

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


def _stored(rows, cols, ld, batch, bstride, seed, kind):
    """A [batch, rows, cols] view with row pitch ld and batch stride bstride
    (bstride 0: one matrix shared by every batch entry) over one buffer."""
    nmat = 1 if bstride == 0 else batch
    span = (nmat - 1) * bstride + rows * ld
    flat = np.full(span + 8, np.nan, np.float32)
    vals = inputs.draw(seed, 0, nmat * rows * cols, kind).reshape(nmat, rows, cols)
    for z in range(nmat):
        for r in range(rows):
            off = z * bstride + r * ld
            flat[off:off + cols] = vals[z, r]
    dev = torch.from_numpy(flat).cuda()
    view = torch.as_strided(dev, (batch, rows, cols), (bstride, ld, 1))
    host = np.stack([vals[0 if bstride == 0 else z] for z in range(batch)])
    return view, host


CASES = [
    # opA, opB, M, N, K, batch, pad (row-pitch slack), odd
    (0, 0, 130, 200, 96, 3, 4, False),
    (1, 0, 130, 200, 96, 3, 4, False),
    (0, 1, 130, 200, 96, 3, 4, False),
    (1, 1, 130, 200, 96, 3, 4, False),
    (1, 1, 257, 129, 300, 2, 1, True),
    (0, 1, 64, 64, 64, 7, 0, False),
    (1, 0, 33, 17, 9, 5, 3, True),
]


# algo 0: the automatic choice (in FFMA mode the small-product kernel for
# these sizes, which reads transposed operands in place); 29: the main
# kernel's 256 x 128 tile pinned (transposed operands go through the
# workspace).  In math mode 1 a value above 3 leaves the automatic choice.
@pytest.mark.parametrize("algo", [0, 29])
@pytest.mark.parametrize("opA,opB,M,N,K,batch,pad,odd", CASES)
@pytest.mark.parametrize("kind", ["uniform", "integer"])
def test_forms_and_batches(handle, opA, opB, M, N, K, batch, pad, odd, kind, algo):
    ar, ac = (K, M) if opA else (M, K)
    br, bc = (N, K) if opB else (K, N)
    lda, ldb, ldc = ac + pad, bc + pad, N + pad
    # Batch strides: padded past the matrix (odd ones defeat 16-byte TMA
    # addressing and force the repack path).
    sa = ar * lda + (3 if odd else 16)
    sb = br * ldb + (1 if odd else 8)
    sc = M * ldc + (5 if odd else 4)
    seed = M + 3 * N + 7 * K + 11 * batch + 13 * opA + 17 * opB
    A, Ah = _stored(ar, ac, lda, batch, sa, seed, kind)
    B, Bh = _stored(br, bc, ldb, batch, sb, seed + 1, kind)
    C, C0 = _stored(M, N, ldc, batch, sc, seed + 2, kind)
    alpha, beta = 0.5, -1.25
    handle.set_algo(algo)
    handle.gemm_batched(A, B, C, alpha, beta, trans_a=bool(opA), trans_b=bool(opB))
    handle.set_algo(0)
    torch.cuda.synchronize()
    assert handle.device_error() == 0
    got = C.contiguous().cpu().numpy()
    for z in range(batch):
        opa = np.ascontiguousarray(Ah[z].T if opA else Ah[z])
        opb = np.ascontiguousarray(Bh[z].T if opB else Bh[z])
        ref = oracle.sgemm_ref(M, N, K, alpha, opa, opb, beta, np.ascontiguousarray(C0[z]))
        if kind == "integer":
            np.testing.assert_array_equal(got[z].astype(np.float64), ref, err_msg=f"batch {z}")
        else:
            assert np.all(np.abs(got[z].astype(np.float64) - ref) <= fp32_tolerance(ref)), f"batch {z}"


def test_zero_stride_broadcasts_one_operand(handle):
    M, N, K, batch = 96, 80, 64, 4
    A, Ah = _stored(M, K, K, batch, 0, 5, "integer")        # one A for all
    B, Bh = _stored(K, N, N, batch, K * N, 6, "integer")
    C = torch.empty((batch, M, N), device="cuda")
    handle.gemm_batched(A, B, C)
    torch.cuda.synchronize()
    for z in range(batch):
        ref = oracle.sgemm_ref(M, N, K, 1.0, np.ascontiguousarray(Ah[z]), np.ascontiguousarray(Bh[z]))
        np.testing.assert_array_equal(C[z].cpu().numpy().astype(np.float64), ref)


def test_many_small_matrices(handle):
    # 300 products of 48 x 40 x 72: the tiles of every batch entry share one
    # persistent grid.
    M, N, K, batch = 48, 40, 72, 300
    A, Ah = _stored(M, K, K, batch, M * K, 8, "uniform")
    B, Bh = _stored(K, N, N, batch, K * N, 9, "uniform")
    C = torch.empty((batch, M, N), device="cuda")
    handle.gemm_batched(A, B, C, 2.0, 0.0)
    torch.cuda.synchronize()
    got = C.cpu().numpy()
    for z in range(0, batch, 37):
        ref = oracle.sgemm_ref(M, N, K, 2.0, np.ascontiguousarray(Ah[z]), np.ascontiguousarray(Bh[z]))
        assert np.all(np.abs(got[z].astype(np.float64) - ref) <= fp32_tolerance(ref))


def test_batched_alpha_zero_scales_every_c(handle):
    M, N, K, batch = 20, 30, 10, 3
    C, C0 = _stored(M, N, N + 2, batch, M * (N + 2) + 4, 10, "integer")
    A = torch.full((batch, M, K), float("nan"), device="cuda")
    B = torch.full((batch, K, N), float("nan"), device="cuda")
    handle.gemm_batched(A, B, C, 0.0, 3.0)
    torch.cuda.synchronize()
    for z in range(batch):
        np.testing.assert_array_equal(C[z].cpu().numpy(), 3.0 * C0[z])
