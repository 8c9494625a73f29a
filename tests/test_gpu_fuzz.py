"""Seeded random shapes against the fp64 oracle, through the automatic
kernel choice: sizes from 1 to a few hundred (and a few larger), padded
pitches, transposed operands, batches, alpha and beta from a small set, in
both math modes.  Integer-valued inputs, so every result must match the
oracle bit for bit whichever kernel (small-product, tile, skinny, 3xTF32)
and schedule the library picks."""
import numpy as np
import pytest

import oracle
from fp32_sgemm_gb300 import inputs

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

ALPHAS = (1.0, 0.5, -2.0, 0.25)
BETAS = (0.0, 1.0, -0.5)


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


def _stored(rows, cols, ld, batch, bstride, seed):
    span = (batch - 1) * bstride + rows * ld
    flat = np.full(span + 4, np.nan, np.float32)
    vals = inputs.draw(seed, 0, batch * rows * cols, "integer").reshape(batch, rows, cols)
    for z in range(batch):
        for r in range(rows):
            flat[z * bstride + r * ld: z * bstride + r * ld + cols] = vals[z, r]
    dev = torch.from_numpy(flat).cuda()
    return torch.as_strided(dev, (batch, rows, cols), (bstride, ld, 1)), vals


def _case(rng):
    big = rng.random() < 0.15
    hi = 1500 if big else 300
    M, N, K = (int(rng.integers(1, hi)) for _ in range(3))
    opA, opB = int(rng.integers(0, 2)), int(rng.integers(0, 2))
    batch = 1 if big or rng.random() < 0.5 else int(rng.integers(2, 5))
    pad = int(rng.choice([0, 0, 1, 3, 4]))
    return M, N, K, opA, opB, batch, pad, float(rng.choice(ALPHAS)), float(rng.choice(BETAS))


@pytest.mark.parametrize("chunk", range(6))
def test_random_shapes_bit_exact(handle, chunk):
    rng = np.random.default_rng(20261202 + chunk)
    for case in range(12):
        M, N, K, opA, opB, batch, pad, alpha, beta = _case(rng)
        ar, ac = (K, M) if opA else (M, K)
        br, bc = (N, K) if opB else (K, N)
        lda, ldb, ldc = ac + pad, bc + pad, N + pad
        seed = 1000 * chunk + case
        A, Ah = _stored(ar, ac, lda, batch, ar * lda + pad, seed)
        B, Bh = _stored(br, bc, ldb, batch, br * ldb + pad, seed + 1)
        C, C0 = _stored(M, N, ldc, batch, M * ldc + pad, seed + 2)
        if beta == 0.0:
            C.fill_(float("nan"))
        handle.gemm_batched(A, B, C, alpha, beta, trans_a=bool(opA), trans_b=bool(opB))
        torch.cuda.synchronize()
        assert handle.device_error() == 0
        got = C.cpu().numpy()
        for z in range(batch):
            opa = np.ascontiguousarray(Ah[z].T if opA else Ah[z])
            opb = np.ascontiguousarray(Bh[z].T if opB else Bh[z])
            c0 = np.ascontiguousarray(C0[z]) if beta != 0.0 else None
            ref = oracle.sgemm_ref(M, N, K, alpha, opa, opb, beta, c0)
            np.testing.assert_array_equal(
                got[z].astype(np.float64), ref,
                err_msg=f"M={M} N={N} K={K} opA={opA} opB={opB} batch={batch} pad={pad} "
                        f"alpha={alpha} beta={beta} entry {z}")
