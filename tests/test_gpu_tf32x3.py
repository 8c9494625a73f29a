"""Error-compensated 3xTF32 tensor-core path (math mode 1) vs the fp64 oracle,
through the C ABI: the same FP32 acceptance bound as the FFMA path for
uniform inputs, bit-exact results for integer-valued inputs."""
import itertools

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
    h.set_math_mode(1)
    yield h
    h.close()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _run(h, p, C_init=None):
    A = _dev(p.A)[:, : p.K]
    B = _dev(p.B)[:, : p.N]
    if C_init is None:
        C_init = p.C0 if p.C0 is not None else np.full((p.M, p.N), np.nan, np.float32)
    Cbuf = _dev(C_init)
    h.gemm(A, B, Cbuf[:, : p.N], p.alpha, p.beta)
    torch.cuda.synchronize()
    assert h.device_error() == 0
    return Cbuf.cpu().numpy()


def _ref(p):
    return oracle.sgemm_ref(p.M, p.N, p.K, p.alpha, p.A, p.B, p.beta, p.C0)


def _close(got, ref):
    err = np.abs(got.astype(np.float64) - ref)
    tol = fp32_tolerance(ref)
    assert np.all(err <= tol), f"worst error/tolerance {float(np.max(err / tol)):.3g}"
    return float(np.max(err / tol))


def test_plan_uses_the_tensor_core_kernel(handle):
    A = torch.zeros((256, 64), device="cuda")
    B = torch.zeros((64, 128), device="cuda")
    C = torch.zeros((256, 128), device="cuda")
    plan = handle.plan(A, B, C)
    assert plan["kind"] == 3 and plan["launches"] == 3


@pytest.mark.parametrize("name", ["sgemm_128", "sgemm_1024", "sgemm_4096", "sgemm_4095x4097x1023"])
def test_workloads_uniform_and_integer(handle, name):
    w = inputs.WORKLOADS[name]
    p = inputs.workload_problem(w, "uniform")
    ratio = _close(_run(handle, p)[:, : p.N], _ref(p))
    assert ratio < 0.5
    q = inputs.workload_problem(w, "integer")
    np.testing.assert_array_equal(_run(handle, q)[:, : q.N].astype(np.float64), _ref(q))


def test_8192_sampled(handle):
    w = inputs.WORKLOADS["sgemm_8192"]
    rows, cols = inputs.sample_entries(w.M, w.N, w.samples, w.seed)
    for kind in ("uniform", "integer"):
        p = inputs.workload_problem(w, kind)
        C = torch.empty((w.M, w.N), device="cuda")
        handle.gemm(_dev(p.A), _dev(p.B), C)
        got = C[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().numpy()
        ref = oracle.sgemm_ref_entries(w.K, w.alpha, p.A, p.B, rows, cols)
        if kind == "uniform":
            _close(got, ref)
        else:
            np.testing.assert_array_equal(got.astype(np.float64), ref)
    assert handle.device_error() == 0


def test_small_and_edge_shapes(handle):
    sizes = [1, 3, 8, 31, 33, 127, 129, 200]
    for M, N, K in itertools.product(sizes[::2], sizes[1::2], [1, 5, 32, 33, 100]):
        q = inputs.make_problem(M, N, K, seed=M * 7 + N * 3 + K, kind="integer", alpha=1.0,
                                beta=0.5, with_c=True, lda=K + (M % 3), ldb=N + 1, ldc=N + 2)
        got = _run(handle, q)
        np.testing.assert_array_equal(got[:, :N].astype(np.float64), _ref(q),
                                      err_msg=f"shape {(M, N, K)}")
        assert np.isnan(got[:, N:]).all()
        p = inputs.make_problem(M, N, K, seed=M + N + K, alpha=-1.5, beta=0.25)
        _close(_run(handle, p)[:, :N], _ref(p))


def test_beta_zero_never_reads_c(handle):
    p = inputs.make_problem(300, 260, 100, seed=5)
    got = _run(handle, p, C_init=np.full((300, 260), np.nan, np.float32))
    assert np.isfinite(got).all()
    _close(got, _ref(p))


def test_large_magnitudes_and_mixed_scales(handle):
    # Inputs spread over many binades, where the TF32 residual carries bits
    # that a single TF32 pass would lose.
    rng = np.random.default_rng(3)
    M, N, K = 384, 320, 1000
    A = (rng.uniform(-1, 1, (M, K)) * 2.0 ** rng.integers(-20, 20, (M, K))).astype(np.float32)
    B = (rng.uniform(-1, 1, (K, N)) * 2.0 ** rng.integers(-20, 20, (K, N))).astype(np.float32)
    C = torch.empty((M, N), device="cuda")
    handle.gemm(_dev(A), _dev(B), C)
    got = C.cpu().numpy().astype(np.float64)
    ref = oracle.sgemm_ref(M, N, K, 1.0, A, B)
    # Relative to the magnitude sum, as any FP32 summation is.
    scale = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64))
    assert np.all(np.abs(got - ref) <= 1e-5 * scale + 1e-30)


def test_repeated_calls_bitwise_identical(handle):
    p = inputs.make_problem(1024, 768, 640, seed=10)
    A, B = _dev(p.A), _dev(p.B)
    first = torch.empty((1024, 768), device="cuda")
    handle.gemm(A, B, first)
    C = torch.empty_like(first)
    for _ in range(10):
        handle.gemm(A, B, C)
        assert torch.equal(C.view(torch.int32), first.view(torch.int32))


@pytest.mark.parametrize("config", [1, 2, 3, 4])
@pytest.mark.parametrize("shape", [(1000, 1500, 700), (256, 4097, 333), (4096, 4096, 4096)])
def test_every_tensor_tile_configuration(handle, config, shape):
    M, N, K = shape
    handle.set_algo(config)
    try:
        p = inputs.make_problem(M, N, K, seed=M + N + K + config, alpha=0.5, beta=0.25)
        _close(_run(handle, p)[:, :N], _ref(p))
        q = inputs.make_problem(M, N, K, seed=M + N + K + config + 1000, kind="integer", alpha=0.5,
                                beta=0.25)
        np.testing.assert_array_equal(_run(handle, q)[:, :N].astype(np.float64), _ref(q))
    finally:
        handle.set_algo(0)


def test_plan_at_4096_is_sm_pair_tiles_with_stream_k(handle):
    A = torch.empty((4096, 4096), device="cuda")
    B = torch.empty((4096, 4096), device="cuda")
    C = torch.empty((4096, 4096), device="cuda")
    handle._ensure_workspace(handle.workspace_size(4096, 4096, 4096, A.data_ptr(), 4096, B.data_ptr(), 4096))
    plan = handle.plan(A, B, C)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert (plan["tile_m"], plan["tile_n"]) == (256, 256)
    assert plan["ctas"] % 2 == 0 and plan["ctas"] <= sms
    # Stream-K when the last wave of whole pair tiles would be under half full.
    waves = (4096 // 256) ** 2 / (plan["ctas"] // 2)
    frac = waves - int(waves)
    assert plan["stream_k"] == (1 if 0 < frac < 0.5 else 0)


def test_mid_size_keeps_single_sm_tiles(handle):
    # 16 pair tiles at 1024^3 would leave most SM pairs idle.
    A = torch.empty((1024, 1024), device="cuda")
    plan = handle.plan(A, A, A)
    assert plan["tile_m"] == 128


@pytest.mark.parametrize("schedule", [1, 2])
@pytest.mark.parametrize("config", [1, 3, 4])
@pytest.mark.parametrize("shape", [(1000, 1500, 700), (257, 255, 4000), (2048, 2048, 2048), (130, 4100, 96)])
def test_tensor_schedules(handle, schedule, config, shape):
    # schedule 2 cuts tiles between CTAs (stream-K) and adds the partial
    # tiles in a fixup; schedule 1 keeps whole tiles.
    M, N, K = shape
    handle.set_algo(config)
    handle.set_schedule(schedule)
    try:
        p = inputs.make_problem(M, N, K, seed=M + N + K + 7 * config + schedule, alpha=0.75, beta=-0.5)
        _close(_run(handle, p)[:, :N], _ref(p))
        q = inputs.make_problem(M, N, K, seed=M + N + K + 7 * config + schedule + 1000, kind="integer",
                                alpha=0.75, beta=-0.5)
        np.testing.assert_array_equal(_run(handle, q)[:, :N].astype(np.float64), _ref(q))
    finally:
        handle.set_algo(0)
        handle.set_schedule(0)


def test_stream_k_repeatable_bitwise(handle):
    p = inputs.make_problem(1536, 1280, 2048, seed=77)
    A, B = _dev(p.A), _dev(p.B)
    handle.set_schedule(2)
    try:
        first = torch.empty((1536, 1280), device="cuda")
        handle.gemm(A, B, first)
        assert handle.plan(A, B, first)["stream_k"] == 1
        C = torch.empty_like(first)
        for _ in range(10):
            handle.gemm(A, B, C)
            assert torch.equal(C.view(torch.int32), first.view(torch.int32))
    finally:
        handle.set_schedule(0)
    assert handle.device_error() == 0
    _close(first.cpu().numpy(), _ref(p))


@pytest.mark.parametrize("M,N,K", [(1000, 1500, 700), (512, 384, 260)])
def test_operand_read_in_place_matches_its_copy_bitwise(handle, M, N, K):
    # With lda = K (16-byte aligned rows) A is read in place as its own high
    # part; with lda = K + 1 its truncated high part is copied first.  The
    # tensor core sees the same TF32 values either way.
    p = inputs.make_problem(M, N, K, seed=M + K, alpha=0.75, beta=0.0)
    A = _dev(p.A)
    B = _dev(p.B)
    A_odd = torch.empty((M, K + 1), device="cuda")
    A_odd[:, :K] = A
    C1 = torch.empty((M, N), device="cuda")
    C2 = torch.empty((M, N), device="cuda")
    handle.gemm(A, B, C1, 0.75)
    handle.gemm(A_odd[:, :K], B, C2, 0.75)
    torch.cuda.synchronize()
    assert handle.device_error() == 0
    assert torch.equal(C1.view(torch.int32), C2.view(torch.int32))
    _close(C1.cpu().numpy(), _ref(p))


@pytest.mark.parametrize("schedule", [1, 2])
@pytest.mark.parametrize("opA,opB", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_sm_pair_tile_on_batches_and_transposes(handle, opA, opB, schedule):
    # Configuration 4 (256 x 256 on SM pairs) pinned: three matrices per
    # call, every operand form, whole tiles and stream-K (the K range of a
    # tile cut between pairs, partial tiles added by the rank-matched CTA).
    M, N, K, batch = 300, 520, 700, 3
    ar, ac = (K, M) if opA else (M, K)
    br, bc = (N, K) if opB else (K, N)
    seed = 31 + 2 * opA + opB + 5 * schedule
    A = inputs.draw(seed, 0, batch * ar * ac, "integer").reshape(batch, ar, ac)
    B = inputs.draw(seed + 1, 0, batch * br * bc, "integer").reshape(batch, br, bc)
    C0 = inputs.draw(seed + 2, 0, batch * M * N, "integer").reshape(batch, M, N)
    dA, dB, dC = _dev(A), _dev(B), _dev(C0)
    handle.set_algo(4)
    handle.set_schedule(schedule)
    try:
        handle.gemm_batched(dA, dB, dC, 0.5, -1.25, trans_a=bool(opA), trans_b=bool(opB))
        torch.cuda.synchronize()
    finally:
        handle.set_algo(0)
        handle.set_schedule(0)
    assert handle.device_error() == 0
    got = dC.cpu().numpy()
    for z in range(batch):
        opa = np.ascontiguousarray(A[z].T if opA else A[z])
        opb = np.ascontiguousarray(B[z].T if opB else B[z])
        ref = oracle.sgemm_ref(M, N, K, 0.5, opa, opb, -1.25, np.ascontiguousarray(C0[z]))
        np.testing.assert_array_equal(got[z].astype(np.float64), ref, err_msg=f"batch {z}")


@pytest.mark.parametrize("config", [0, 4])
def test_deep_k_stays_inside_the_bound(handle, config):
    # 64 accumulator chunks of 256 K each, summed in FP32 registers: the
    # tensor core's own accumulation error must not pile up across K.
    M, N, K = 512, 512, 16384
    p = inputs.make_problem(M, N, K, seed=K + config)
    handle.set_algo(config)
    try:
        got = _run(handle, p)
    finally:
        handle.set_algo(0)
    assert _close(got, _ref(p)) < 0.5
