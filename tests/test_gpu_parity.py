"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Uniform inputs must satisfy |C_gpu - C_ref| <= 1e-3 + 1e-3*|C_ref|
elementwise; integer-valued inputs in {-4..4} must match bit for bit (every
FP32 partial sum is exact, so any summation order gives the oracle's value).
"""
import itertools

import numpy as np
import pytest

import oracle
from fp32_sgemm_gb300 import inputs
from conftest import fp32_tolerance

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp32_sgemm_gb300 as m
    m.build()
    return m


@pytest.fixture(scope="module")
def handle(sg):
    return sg.Handle()


def _to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _gpu(sg, handle, p, C_init=None, algo=0, schedule=0):
    """Run the problem on the GPU; returns the full [M, ldc] C buffer on the host."""
    A = _to_dev(p.A)[:, : p.K] if p.K > 0 else torch.zeros((p.M, 0), device="cuda")
    B = _to_dev(p.B)[:, : p.N]
    if C_init is None:
        C_init = p.C0 if p.C0 is not None else np.full((p.M, p.N), np.nan, np.float32)
    Cbuf = _to_dev(C_init)
    C = Cbuf[:, : p.N]
    handle.set_algo(algo)
    handle.set_schedule(schedule)
    handle.gemm(A, B, C, p.alpha, p.beta)
    torch.cuda.synchronize()
    handle.set_schedule(0)
    assert handle.device_error() == 0
    return Cbuf.cpu().numpy()


def _assert_close(got, ref):
    err = np.abs(got.astype(np.float64) - ref)
    tol = fp32_tolerance(ref)
    bad = ~(err <= tol)
    assert not bad.any(), (f"{int(bad.sum())} entries out of tolerance; worst ratio "
                           f"{float(np.nanmax(err / tol)):.3g}")
    return float(np.max(err / tol)) if err.size else 0.0


def _ref(p, threads=0):
    return oracle.sgemm_ref(p.M, p.N, p.K, p.alpha, p.A, p.B, p.beta, p.C0, threads=threads)


FULL = ["sgemm_128", "sgemm_1024", "sgemm_4096", "sgemm_4095x4097x1023"]


@pytest.mark.parametrize("name", FULL)
def test_workload_uniform_full(sg, handle, name):
    w = inputs.WORKLOADS[name]
    p = inputs.workload_problem(w, "uniform")
    got = _gpu(sg, handle, p)[:, : p.N]
    ratio = _assert_close(got, _ref(p))
    assert ratio < 0.5


@pytest.mark.parametrize("name", FULL)
def test_workload_integer_twin_bit_exact(sg, handle, name):
    w = inputs.WORKLOADS[name]
    p = inputs.workload_problem(w, "integer")
    got = _gpu(sg, handle, p)[:, : p.N]
    np.testing.assert_array_equal(got.astype(np.float64), _ref(p))


def _sampled_8192(sg, handle, kind):
    w = inputs.WORKLOADS["sgemm_8192"]
    p = inputs.workload_problem(w, kind)
    A = _to_dev(p.A)
    B = _to_dev(p.B)
    C = torch.empty((w.M, w.N), dtype=torch.float32, device="cuda")
    handle.set_algo(0)
    handle.gemm(A, B, C, w.alpha, w.beta)
    rows, cols = inputs.sample_entries(w.M, w.N, w.samples, w.seed)
    got = C[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().numpy()
    assert handle.device_error() == 0
    ref = oracle.sgemm_ref_entries(w.K, w.alpha, p.A, p.B, rows, cols, w.beta, p.C0)
    return got, ref


def test_workload_8192_sampled_uniform(sg, handle):
    got, ref = _sampled_8192(sg, handle, "uniform")
    _assert_close(got, ref)


def test_workload_8192_sampled_integer_bit_exact(sg, handle):
    got, ref = _sampled_8192(sg, handle, "integer")
    np.testing.assert_array_equal(got.astype(np.float64), ref)


@pytest.mark.parametrize("algo", [10, 16, 17, 18, 19, 20, 21, 23, 24, 27, 28, 29, 30])
@pytest.mark.parametrize("shape", [(1024, 1024, 1024), (300, 517, 263)])
def test_every_tile_configuration(sg, handle, algo, shape):
    M, N, K = shape
    p = inputs.make_problem(M, N, K, seed=40 + algo, alpha=0.5, beta=0.25)
    _assert_close(_gpu(sg, handle, p, algo=algo)[:, :N], _ref(p))
    q = inputs.make_problem(M, N, K, seed=1040 + algo, kind="integer", alpha=0.5, beta=0.25)
    np.testing.assert_array_equal(_gpu(sg, handle, q, algo=algo)[:, :N].astype(np.float64), _ref(q))


def test_tensor_tile_number_in_ffma_mode_is_rejected(sg):
    # 1..3 name the tensor-core tiles of math mode 1; in math mode 0 they
    # name no built configuration, and the product call says so.
    lib = sg.load_library()
    h = sg.Handle()
    h.set_algo(2)
    A = torch.zeros((300, 300), device="cuda")
    C = torch.full((300, 300), 7.0, device="cuda")
    st = lib.sgemmEx(h.ptr, 300, 300, 300, 1.0, A.data_ptr(), 300, A.data_ptr(), 300, 0.0,
                     C.data_ptr(), 300, None)
    assert st == sg.Status.INVALID_VALUE
    torch.cuda.synchronize()
    assert bool((C == 7.0).all())
    h.close()


@pytest.mark.parametrize("schedule", [1, 2])
@pytest.mark.parametrize("algo", [10, 20, 23, 28, 29])
@pytest.mark.parametrize("shape", [(1024, 1024, 1024), (300, 517, 263), (1500, 700, 2000),
                                   (257, 255, 4000)])
def test_schedules(sg, handle, schedule, algo, shape):
    # schedule 1: whole tiles per CTA; schedule 2: stream-K, where tiles are
    # cut between CTAs (here up to ~5 CTAs per tile) and summed in a fixup.
    M, N, K = shape
    p = inputs.make_problem(M, N, K, seed=M + N + K + algo, alpha=0.75, beta=-0.5)
    _assert_close(_gpu(sg, handle, p, algo=algo, schedule=schedule)[:, :N], _ref(p))
    q = inputs.make_problem(M, N, K, seed=M + N + K + algo + 1000, kind="integer",
                            alpha=0.75, beta=-0.5)
    np.testing.assert_array_equal(
        _gpu(sg, handle, q, algo=algo, schedule=schedule)[:, :N].astype(np.float64), _ref(q))


def test_stream_k_chosen_for_uneven_tiles_and_deterministic(sg, handle):
    M = N = K = 4096
    p = inputs.make_problem(512, 512, 512, seed=3)   # content irrelevant for the plan
    A = torch.empty((M, K), device="cuda")
    B = torch.empty((K, N), device="cuda")
    C = torch.empty((M, N), device="cuda")
    handle.set_algo(0)
    handle.set_schedule(0)
    handle._ensure_workspace(handle.workspace_size(M, N, K, A.data_ptr(), K, B.data_ptr(), N))
    plan = handle.plan(A, B, C)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = (M // plan["tile_m"]) * (N // plan["tile_n"])
    assert plan["stream_k"] == (1 if tiles % sms else 0)
    # Stream-K sums the partial tiles in a fixed order: repeated calls agree bitwise.
    M, N, K = 1024, 1024, 1024
    p = inputs.make_problem(M, N, K, seed=21)
    A, B = _to_dev(p.A), _to_dev(p.B)
    handle.set_schedule(2)
    first = torch.empty((M, N), device="cuda")
    handle.gemm(A, B, first)
    C = torch.empty_like(first)
    for _ in range(20):
        handle.gemm(A, B, C)
        assert torch.equal(C.view(torch.int32), first.view(torch.int32))
    handle.set_schedule(0)
    assert handle.device_error() == 0
    _assert_close(first.cpu().numpy(), _ref(p))


_SMALL = [1, 2, 3, 5, 8, 9]
_EDGES = [15, 16, 17, 31, 32, 33, 127, 128, 129]


# algo 0: the automatic choice (the small-product kernel for most of these
# shapes); 29: the 256 x 128 tile of the main kernel pinned.
@pytest.mark.parametrize("algo", [0, 29])
def test_tiny_shapes_integer_exact(sg, handle, algo):
    for M, N, K in itertools.product(_SMALL, _SMALL, _SMALL):
        p = inputs.make_problem(M, N, K, seed=M * 97 + N * 13 + K, kind="integer",
                                alpha=1.0, beta=0.5, with_c=True,
                                lda=K + (M % 3), ldb=N + (K % 2), ldc=N + 1)
        got = _gpu(sg, handle, p, algo=algo)
        np.testing.assert_array_equal(got[:, :N].astype(np.float64), _ref(p),
                                      err_msg=f"shape {(M, N, K)}")
        assert np.isnan(got[:, N:]).all(), "ldc padding was written"


@pytest.mark.parametrize("algo", [0, 29])
def test_edge_shapes_uniform(sg, handle, algo):
    for M, N, K in itertools.product(_EDGES[::2], _EDGES[1::2], _EDGES):
        p = inputs.make_problem(M, N, K, seed=M + 7 * N + 11 * K, alpha=-1.25, beta=0.75)
        _assert_close(_gpu(sg, handle, p, algo=algo)[:, :N], _ref(p))


@pytest.mark.parametrize("M,N,K,lda,ldb,ldc", [
    (255, 257, 129, 132, 260, 264),       # 16-byte pitches, ragged sizes
    (257, 255, 131, 131, 255, 255),       # odd pitches: A and B repacked, scalar C
    (130, 126, 64, 68, 127, 129),         # A in place, B repacked, scalar C
    (129, 131, 513, 515, 132, 136),       # A repacked, B in place, vector C
])
@pytest.mark.parametrize("algo", [0, 29])
def test_leading_dimensions_and_packing(sg, handle, M, N, K, lda, ldb, ldc, algo):
    p = inputs.make_problem(M, N, K, seed=M * N, alpha=1.5, beta=-0.5, lda=lda, ldb=ldb, ldc=ldc)
    got = _gpu(sg, handle, p, algo=algo)
    _assert_close(got[:, :N], _ref(p))
    assert np.isnan(got[:, N:]).all()
    q = inputs.make_problem(M, N, K, seed=M * N + 1, kind="integer", alpha=1.5, beta=-0.5,
                            lda=lda, ldb=ldb, ldc=ldc)
    np.testing.assert_array_equal(_gpu(sg, handle, q, algo=algo)[:, :N].astype(np.float64), _ref(q))


@pytest.mark.parametrize("algo", [0, 29])
def test_unaligned_base_pointers(sg, handle, algo):
    # Views that start one float into their buffers: 4-byte but not 16-byte
    # aligned, so the tile kernel repacks A and B and writes C with scalar
    # stores (the small-product kernel, algo 0, reads them in place).
    M, N, K = 200, 190, 170
    p = inputs.make_problem(M, N, K, seed=77, alpha=1.0, beta=1.0)
    Ab = torch.zeros(M * K + 1, device="cuda")
    Bb = torch.zeros(K * N + 1, device="cuda")
    Cb = torch.zeros(M * N + 1, device="cuda")
    A = Ab[1:].view(M, K); A.copy_(torch.from_numpy(p.A))
    B = Bb[1:].view(K, N); B.copy_(torch.from_numpy(p.B))
    C = Cb[1:].view(M, N); C.copy_(torch.from_numpy(p.C0))
    handle.set_algo(algo)
    plan = handle.plan(A, B, C, 1.0, 1.0)
    if algo:
        assert plan["packs_a"] == 1 and plan["packs_b"] == 1 and plan["vector_epilogue"] == 0
    else:
        assert plan["kind"] == 5
    handle.gemm(A, B, C, 1.0, 1.0)
    handle.set_algo(0)
    _assert_close(C.cpu().numpy(), _ref(p))
    assert float(Cb[0]) == 0.0


def test_beta_zero_never_reads_c(sg, handle):
    p = inputs.make_problem(300, 260, 100, seed=5)
    got = _gpu(sg, handle, p, C_init=np.full((300, 260), np.nan, np.float32))
    assert np.isfinite(got).all()
    _assert_close(got, _ref(p))


def test_alpha_zero_and_k_zero(sg, handle):
    p = inputs.make_problem(70, 90, 30, seed=6, alpha=0.0, beta=-2.0)
    A = torch.full((70, 30), float("nan"), device="cuda")
    B = torch.full((30, 90), float("nan"), device="cuda")
    C = _to_dev(p.C0)
    handle.gemm(A, B, C, 0.0, -2.0)
    np.testing.assert_array_equal(C.cpu().numpy(), -2.0 * p.C0)
    C = _to_dev(p.C0)
    handle.gemm(torch.zeros((70, 0), device="cuda"), torch.zeros((0, 90), device="cuda"), C, 3.0, 0.0)
    np.testing.assert_array_equal(C.cpu().numpy(), np.zeros((70, 90), np.float32))


def test_empty_output_untouched(sg, handle):
    C = torch.full((0, 5), 1.0, device="cuda")
    handle.gemm(torch.zeros((0, 3), device="cuda"), torch.zeros((3, 5), device="cuda"), C)
    C = torch.full((4, 0), 1.0, device="cuda")
    handle.gemm(torch.zeros((4, 3), device="cuda"), torch.zeros((3, 0), device="cuda"), C)
    torch.cuda.synchronize()


@pytest.mark.parametrize("algo", [0, 29])
def test_guard_bands_untouched(sg, handle, algo):
    # C lives inside a larger canary-filled buffer: rows above/below, columns
    # past N (ldc padding) must keep their exact bit patterns.
    M, N, K, ldc = 257, 250, 96, 260
    canary = np.frombuffer(np.uint32(0x7FC0BEEF).tobytes() * ((M + 8) * ldc),
                           dtype=np.float32).reshape(M + 8, ldc).copy()
    p = inputs.make_problem(M, N, K, seed=8, alpha=1.0, beta=0.5, with_c=True)
    canary[4:4 + M, :N] = p.C0[:, :N]
    buf = _to_dev(canary)
    C = buf[4:4 + M, :N]
    handle.set_algo(algo)
    handle.gemm(_to_dev(p.A), _to_dev(p.B), C, 1.0, 0.5)
    handle.set_algo(0)
    out = buf.cpu().numpy()
    mask = np.ones(out.shape, bool)
    mask[4:4 + M, :N] = False
    assert (out.view(np.uint32)[mask] == 0x7FC0BEEF).all()
    _assert_close(out[4:4 + M, :N], _ref(p))


def test_identity_and_permutation_exact(sg, handle):
    n, N = 384, 200
    p = inputs.make_problem(n, N, n, seed=9)
    eye = np.eye(n, dtype=np.float32)
    C = torch.empty((n, N), device="cuda")
    handle.gemm(_to_dev(eye), _to_dev(p.B), C)
    np.testing.assert_array_equal(C.cpu().numpy(), p.B)
    perm = np.random.default_rng(1).permutation(n)
    P = np.zeros((n, n), np.float32)
    P[np.arange(n), perm] = 1.0
    handle.gemm(_to_dev(P), _to_dev(p.B), C)
    np.testing.assert_array_equal(C.cpu().numpy(), p.B[perm])


def test_repeated_calls_bitwise_identical(sg, handle):
    p = inputs.make_problem(1024, 1024, 1024, seed=10)
    A, B = _to_dev(p.A), _to_dev(p.B)
    handle.set_algo(0)
    first = torch.empty((1024, 1024), device="cuda")
    handle.gemm(A, B, first)
    C = torch.empty_like(first)
    for _ in range(30):
        handle.gemm(A, B, C)
        assert torch.equal(C.view(torch.int32), first.view(torch.int32))


def test_non_default_stream(sg, handle):
    p = inputs.make_problem(512, 384, 256, seed=11, beta=1.0)
    s = torch.cuda.Stream()
    A, B, C = _to_dev(p.A), _to_dev(p.B), _to_dev(p.C0)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        handle.gemm(A, B, C, 1.0, 1.0, stream=s)
    s.synchronize()
    _assert_close(C.cpu().numpy(), _ref(p))


def test_default_handle_entry_point(sg):
    p = inputs.make_problem(640, 320, 200, seed=12)
    C = sg.sgemm(_to_dev(p.A), _to_dev(p.B))
    torch.cuda.synchronize()
    _assert_close(C.cpu().numpy(), _ref(p))


def test_workspace_required_without_workspace(sg):
    import ctypes
    lib = sg.load_library()
    h = sg.Handle()
    A = torch.zeros(100 * 33, device="cuda")
    B = torch.zeros(33 * 64, device="cuda")
    C = torch.zeros(100 * 64, device="cuda")
    # The automatic choice runs a product this small in the small-product
    # kernel, which reads A in place and needs no workspace ...
    assert lib.sgemmEx(h.ptr, 100, 64, 33, 1.0, A.data_ptr(), 33, B.data_ptr(), 64, 0.0,
                       C.data_ptr(), 64, None) == 0
    # ... the tile kernel must repack A (a pitch of 33 floats is not TMA-addressable).
    h.set_algo(29)
    st = lib.sgemmEx(h.ptr, 100, 64, 33, 1.0, A.data_ptr(), 33, B.data_ptr(), 64, 0.0,
                     C.data_ptr(), 64, None)
    assert st == sg.Status.WORKSPACE_REQUIRED
    n = ctypes.c_size_t()
    assert lib.sgemmGetWorkspaceSize(h.ptr, 100, 64, 33, A.data_ptr(), 33, B.data_ptr(), 64,
                                     ctypes.byref(n)) == 0
    # Required: room to repack A (pitch 33 -> 36 floats).  The size query
    # may add optional stream-K scratch on top.
    required = (100 * 36 * 4 + 255) // 256 * 256
    assert n.value >= required
    # With exactly the required part the call runs (whole tiles).
    ws = torch.empty(required, dtype=torch.uint8, device="cuda")
    assert lib.sgemmSetWorkspace(h.ptr, ws.data_ptr(), required) == 0
    A.copy_(torch.arange(100 * 33, device="cuda", dtype=torch.float32) % 5 - 2)
    B.copy_(torch.arange(33 * 64, device="cuda", dtype=torch.float32) % 7 - 3)
    assert lib.sgemmEx(h.ptr, 100, 64, 33, 1.0, A.data_ptr(), 33, B.data_ptr(), 64, 0.0,
                       C.data_ptr(), 64, None) == 0
    torch.cuda.synchronize()
    ref = A.view(100, 33).double().cpu().numpy() @ B.view(33, 64).double().cpu().numpy()
    np.testing.assert_array_equal(C.view(100, 64).cpu().numpy().astype(np.float64), ref)
    h.close()


def test_host_buffer_entry_point(sg, handle):
    M, N, K = 1000, 777, 333
    p = inputs.make_problem(M, N, K, seed=13, alpha=0.5, beta=0.25)
    A = torch.from_numpy(p.A).pin_memory()
    B = torch.from_numpy(p.B).pin_memory()
    C = torch.from_numpy(p.C0.copy()).pin_memory()
    ws = torch.empty(sg.host_workspace_size(M, N, K), dtype=torch.uint8, device="cuda")
    sg.sgemm_host(A, B, C, 0.5, 0.25, workspace=ws, handle=handle)
    torch.cuda.synchronize()
    _assert_close(C.numpy(), _ref(p))


@pytest.mark.parametrize("math", [0, 1], ids=["ffma", "tf32x3"])
@pytest.mark.parametrize("M,N,K,alpha,beta", [
    (4099, 515, 257, 0.5, 0.25),     # four row chunks of unequal height
    (2047, 1029, 130, 1.0, 0.0),     # one chunk; C starts as NaN and is never read
    (3072, 96, 1000, -2.0, 1.0),     # three chunks
    (2500, 2100, 300, 0.5, -0.75),   # first row block cut into two column pieces
    (2100, 4500, 100, 1.0, 0.5),     # four column pieces, cuts off the 1125-column grid
])
def test_host_entry_point_chunked_copies(sg, M, N, K, alpha, beta, math):
    h = sg.Handle()
    h.set_math_mode(math)
    try:
        for kind in ("integer", "uniform"):
            p = inputs.make_problem(M, N, K, seed=M + N + K, kind=kind, alpha=alpha, beta=beta,
                                    with_c=True, lda=K + 3, ldb=N + 1, ldc=N + 5)
            A = torch.from_numpy(p.A).pin_memory()
            B = torch.from_numpy(p.B).pin_memory()
            C0 = p.C0.copy()
            if beta == 0.0:
                C0[:, :N] = np.nan
            C = torch.from_numpy(C0).pin_memory()
            ws = torch.empty(sg.host_workspace_size(M, N, K), dtype=torch.uint8, device="cuda")
            stream = torch.cuda.Stream()
            A2 = A[:, :K]
            sg.sgemm_host(A2, B[:, :N], C[:, :N], alpha, beta, workspace=ws, handle=h, stream=stream)
            # Work enqueued on the same stream afterwards is ordered after the
            # copy of C back to the host.
            flag = torch.zeros(1, device="cuda")
            with torch.cuda.stream(stream):
                flag.fill_(1.0)
            stream.synchronize()
            assert flag.item() == 1.0
            assert h.device_error() == 0
            got = C.numpy()
            ref = oracle.sgemm_ref(M, N, K, alpha, p.A, p.B, beta, p.C0)
            if kind == "integer":
                np.testing.assert_array_equal(got[:, :N].astype(np.float64), ref)
            else:
                _assert_close(got[:, :N], ref)
            assert np.isnan(got[:, N:]).all(), "padding columns of C written"
    finally:
        h.close()


def test_bounded_wait_self_test_reports_timeout(sg):
    h = sg.Handle()
    assert h.device_error() == 0
    h.selftest_wait_timeout(50_000_000)          # 50 ms, nothing ever arrives
    code = h.device_error()
    assert code >> 24 == 3
    assert h.device_error() == 0                 # reading cleared it
    # The context is still usable afterwards.
    p = inputs.make_problem(256, 256, 256, seed=14, kind="integer")
    C = torch.empty((256, 256), device="cuda")
    h.gemm(_to_dev(p.A), _to_dev(p.B), C)
    np.testing.assert_array_equal(C.cpu().numpy().astype(np.float64), _ref(p))
    h.close()


def test_kernel_events_bracket_the_main_kernel(sg, handle):
    p = inputs.make_problem(2048, 2048, 2048, seed=31)
    A, B = _to_dev(p.A), _to_dev(p.B)
    C = torch.empty((2048, 2048), device="cuda")
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    e.record()
    torch.cuda.synchronize()
    outer0, outer1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    handle.set_algo(0)
    handle.set_kernel_events(s, e)
    outer0.record()
    handle.gemm(A, B, C)
    outer1.record()
    torch.cuda.synchronize()
    handle.set_kernel_events(None, None)
    k_ms, call_ms = s.elapsed_time(e), outer0.elapsed_time(outer1)
    assert 0.0 < k_ms <= call_ms
    assert k_ms > 0.05            # 17 GFLOP cannot take less than ~0.2 ms on FP32 FMA
    with pytest.raises(sg.SgemmError):
        handle.set_kernel_events(s, None)


@pytest.mark.parametrize("math", [0, 1], ids=["ffma", "tf32x3"])
def test_cuda_graph_capture_and_replay(sg, math):
    # A call enqueues only capturable work (kernel launches and a memset on
    # the given stream), so a product can be captured once and replayed.
    h = sg.Handle()
    h.set_math_mode(math)
    try:
        p = inputs.make_problem(384, 320, 1000, seed=71, kind="integer", alpha=0.5, beta=-1.0)
        A, B = _to_dev(p.A), _to_dev(p.B)
        C = _to_dev(p.C0)
        h.gemm(A, B, C.clone(), p.alpha, p.beta)          # sizes the workspace outside the capture
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                h.gemm(A, B, C, p.alpha, p.beta, stream=s)
        ref = p.C0.astype(np.float64)
        for _ in range(3):
            g.replay()
            torch.cuda.synchronize()
            ref = oracle.sgemm_ref(p.M, p.N, p.K, p.alpha, p.A, p.B, p.beta, ref.astype(np.float32))
            np.testing.assert_array_equal(C.cpu().numpy().astype(np.float64), ref)
        assert h.device_error() == 0
    finally:
        h.close()


@pytest.mark.parametrize("M,N,K", [(33, 4000, 1500), (64, 2048, 777), (48, 1300, 5000),
                                   (4000, 40, 1500), (2500, 64, 999), (1100, 33, 3000),
                                   (24, 16384, 4096), (32, 10000, 2500), (16384, 20, 4096)])
def test_medium_thin_products_take_the_narrow_tiles(sg, handle, M, N, K):
    # 33..64 rows (columns): the 64 x 512 (512 x 64) tile configuration;
    # 17..32 rows (columns), when large: 32 x 1024 (1024 x 32).
    p = inputs.make_problem(M, N, K, seed=M + N + K, alpha=0.5, beta=0.25)
    got = _gpu(sg, handle, p)[:, :N]
    _assert_close(got, _ref(p))
    q = inputs.make_problem(M, N, K, seed=M + N + K + 1000, kind="integer", alpha=0.5, beta=0.25)
    np.testing.assert_array_equal(_gpu(sg, handle, q)[:, :N].astype(np.float64), _ref(q))
    A = _to_dev(p.A)[:, :K]
    B = _to_dev(p.B)[:, :N]
    C = torch.empty((M, N), device="cuda")
    plan = handle.plan(A, B, C)
    small = min(M, N)
    want = (64, 512) if small > 32 else (32, 1024)
    assert plan["kind"] == 1 and (plan["tile_m"], plan["tile_n"]) == (want if M <= N else want[::-1])


@pytest.mark.parametrize("K", [1, 5, 8, 16, 24, 40, 48, 56])
def test_short_k_takes_shallow_slices(sg, handle, K):
    # K <= 64 and not a multiple of 32: 16- or 8-deep K slices; beta == 0
    # with an aligned C also goes through the TMA-store configurations.
    M, N = 1000, 1100
    p = inputs.make_problem(M, N, K, seed=K + 7, kind="integer", alpha=0.5, beta=0.25)
    np.testing.assert_array_equal(_gpu(sg, handle, p)[:, :N].astype(np.float64), _ref(p))
    q = inputs.make_problem(M, N, K, seed=K + 8, alpha=-1.0, beta=0.0)
    _assert_close(_gpu(sg, handle, q)[:, :N], _ref(q))
    A, B, C = _to_dev(q.A)[:, :K], _to_dev(q.B)[:, :N], torch.empty((M, N), device="cuda")
    # beta == 0, aligned C (TMA-stored tiles): the slice depth that divides K.
    assert handle.plan(A, B, C)["tile_k"] == (16 if K % 16 == 0 else 8)
    # C read: 16-deep slices from K = 33 on as well (no TMA store).
    assert handle.plan(A, B, C, 1.0, 0.5)["tile_k"] == (16 if (K % 16 == 0 or K > 32) else 8)


@pytest.mark.parametrize("algo", [23, 24, 27, 28])
@pytest.mark.parametrize("M,N,K,ldc,schedule", [(1024, 1024, 1024, 1024, 0), (300, 520, 263, 520, 0),
                                                (257, 1000, 40, 1012, 0), (70, 36, 8, 40, 0),
                                                (1500, 704, 2000, 708, 2)])
def test_tma_store_epilogue(sg, handle, algo, M, N, K, ldc, schedule):
    # Configurations 22-28 with beta == 0 and a 16-byte aligned C: each warp
    # stages its block in shared memory and TMA stores it, clipped at M and
    # N.  C starts as NaN canaries (never read); the ldc padding and the rows
    # around C must keep them.  Schedule 2 cuts tiles between CTAs (stream-K),
    # so finished tiles also leave through the staging area after the fixup.
    canary = np.frombuffer(np.uint32(0x7FC0BEEF).tobytes() * ((M + 8) * ldc),
                           dtype=np.float32).reshape(M + 8, ldc).copy()
    for kind, alpha in (("uniform", -0.75), ("integer", 0.5)):
        p = inputs.make_problem(M, N, K, seed=M + N + K + algo, kind=kind, alpha=alpha, beta=0.0)
        buf = _to_dev(canary)
        C = buf[4:4 + M, :N]
        A, B = _to_dev(p.A)[:, :K], _to_dev(p.B)[:, :N]
        handle.set_algo(algo)
        handle.set_schedule(schedule)
        plan = handle.plan(A, B, C, alpha, 0.0)
        handle.gemm(A, B, C, alpha, 0.0)
        torch.cuda.synchronize()
        handle.set_schedule(0)
        handle.set_algo(0)
        assert handle.device_error() == 0
        assert plan["vector_epilogue"] == 1 and plan["tile_k"] == {22: 32, 23: 16, 24: 8, 25: 16, 26: 32, 27: 32, 28: 32}[algo]
        out = buf.cpu().numpy()
        mask = np.ones(out.shape, bool)
        mask[4:4 + M, :N] = False
        assert (out.view(np.uint32)[mask] == 0x7FC0BEEF).all()
        if kind == "integer":
            np.testing.assert_array_equal(out[4:4 + M, :N].astype(np.float64), _ref(p))
        else:
            _assert_close(out[4:4 + M, :N], _ref(p))


@pytest.mark.parametrize("algo", [23, 24, 27, 28])
@pytest.mark.parametrize("M,N,K,ldc,beta", [(300, 517, 263, 519, 0.0), (257, 1000, 40, 1001, 0.5),
                                            (70, 36, 8, 37, -1.0), (1500, 707, 2000, 709, 0.25)])
def test_staged_row_run_epilogue(sg, handle, algo, M, N, K, ldc, beta):
    # The same configurations with a C that TMA cannot address (odd ldc): the
    # staged block leaves in row runs of plain stores, reading C first when
    # beta != 0 (NaN canaries when beta == 0: never read).  The ldc padding
    # and the rows around C keep their canaries.
    for kind, alpha in (("uniform", 0.75), ("integer", 2.0)):
        p = inputs.make_problem(M, N, K, seed=M + 3 * N + K + algo, kind=kind, alpha=alpha, beta=beta,
                                with_c=True)
        canary = np.frombuffer(np.uint32(0x7FC0BEEF).tobytes() * ((M + 8) * ldc),
                               dtype=np.float32).reshape(M + 8, ldc).copy()
        if beta != 0.0:
            canary[4:4 + M, :N] = p.C0[:, :N]
        buf = _to_dev(canary)
        C = buf[4:4 + M, :N]
        A, B = _to_dev(p.A)[:, :K], _to_dev(p.B)[:, :N]
        handle.set_algo(algo)
        plan = handle.plan(A, B, C, alpha, beta)
        handle.gemm(A, B, C, alpha, beta)
        torch.cuda.synchronize()
        handle.set_algo(0)
        assert handle.device_error() == 0
        assert plan["vector_epilogue"] == 0 and plan["kind"] == 1
        out = buf.cpu().numpy()
        mask = np.ones(out.shape, bool)
        mask[4:4 + M, :N] = False
        assert (out.view(np.uint32)[mask] == 0x7FC0BEEF).all()
        ref = oracle.sgemm_ref(M, N, K, alpha, p.A, p.B, beta, p.C0 if beta != 0.0 else None)
        if kind == "integer":
            np.testing.assert_array_equal(out[4:4 + M, :N].astype(np.float64), ref)
        else:
            _assert_close(out[4:4 + M, :N], ref)


def test_tma_store_epilogue_batched(sg, handle):
    # Strided batches through configuration 24: the store map's third
    # dimension walks the batch stride (a multiple of 4 elements).
    M, N, K, batch, ldc = 200, 136, 8, 3, 140
    sc = M * ldc + 12
    p = [inputs.make_problem(M, N, K, seed=90 + z, kind="integer", alpha=2.0, beta=0.0) for z in range(batch)]
    A = torch.stack([_to_dev(q.A)[:, :K] for q in p])
    B = torch.stack([_to_dev(q.B)[:, :N] for q in p])
    flat = torch.full((batch * sc + 8,), float("nan"), device="cuda")
    C = torch.as_strided(flat, (batch, M, N), (sc, ldc, 1))
    handle.set_algo(24)
    handle.gemm_batched(A, B, C, 2.0, 0.0)
    torch.cuda.synchronize()
    handle.set_algo(0)
    assert handle.device_error() == 0
    got = C.cpu().numpy()
    for z in range(batch):
        np.testing.assert_array_equal(got[z].astype(np.float64), _ref(p[z]))
    pad = torch.as_strided(flat, (batch, M, ldc - N), (sc, ldc, 1), N)
    assert torch.isnan(pad).all()



# Thin last tile columns (N mod 128 in 1..8, M x K >= 2^21) go to the edge
# job of the preparation launch; the main kernel covers whole tiles.
@pytest.mark.parametrize("M,N,K,lda,ldb,ldc,alpha,beta", [
    (2048, 4096 + 1, 1024, None, None, None, 1.0, 0.0),       # operands read in place
    (2048, 2048 + 3, 1100, 1101, 2051, 2053, 0.5, 0.25),      # both repacked, C read
    (1500, 1024 + 8, 1500, None, 1040, 1036, 1.0, -1.0),      # C 16-byte aligned, read
    (3000, 512 + 5, 800, 801, None, None, 2.0, 0.0),
    (2100, 640 + 7, 1001, 1003, None, None, 1.0, 0.5),        # K mod 4 = 1, products ride on A's repack
    (1500, 1024 + 8, 2048, None, 1040, 1036, 1.0, -1.0),      # K x r too large: full tiles
])
def test_edge_columns_split_off(sg, handle, M, N, K, lda, ldb, ldc, alpha, beta):
    handle.set_algo(0)
    for kind in ("integer", "uniform"):
        p = inputs.make_problem(M, N, K, seed=M + N + K, kind=kind, alpha=alpha, beta=beta,
                                lda=lda, ldb=ldb, ldc=ldc)
        A = _to_dev(p.A)[:, :K]
        B = _to_dev(p.B)[:, :N]
        Cbuf = _to_dev(p.C0 if p.C0 is not None else np.full((M, N), np.nan, np.float32))
        plan = handle.plan(A, B, Cbuf[:, :N], alpha, beta)
        # The edge job stages its K x r values of B in 48 KB of shared memory.
        want = N % plan["tile_n"] if K * (N % plan["tile_n"]) <= 12288 else 0
        assert plan["kind"] == 1 and plan["edge_cols"] == want, plan
        got = _gpu(sg, handle, p)
        if kind == "integer":
            np.testing.assert_array_equal(got[:, :N].astype(np.float64), _ref(p))
        else:
            _assert_close(got[:, :N], _ref(p))
        if p.C0 is not None and p.C0.shape[1] > N:
            np.testing.assert_array_equal(got[:, N:], p.C0[:, N:])   # ldc padding untouched


def test_edge_columns_only_in_the_automatic_setting(sg, handle):
    p = inputs.make_problem(2048, 4097, 1024, seed=9, kind="integer")
    A, B = _to_dev(p.A), _to_dev(p.B)
    C = torch.zeros((2048, 4097), device="cuda")
    handle.set_algo(0)
    assert handle.plan(A, B, C)["edge_cols"] == 1
    handle.set_algo(28)
    plan = handle.plan(A, B, C)
    handle.set_algo(0)
    assert plan["edge_cols"] == 0
    np.testing.assert_array_equal(_gpu(sg, handle, p, algo=28).astype(np.float64), _ref(p))


@pytest.mark.parametrize("M,N,K,want", [
    (4096, 4096, 4096, (256, 128)),
    (300, 300, 4096, (128, 128)),    # 128 x 128 pads 1.64x, the 256-wide tiles 2.18x
    (200, 4096, 512, (128, 256)),    # equal padding, under 256 rows
    (4095, 4097, 1023, (256, 128)),
])
def test_tile_shape_follows_padding(sg, handle, M, N, K, want):
    handle.set_algo(0)
    A = torch.empty((M, K), device="cuda")
    B = torch.empty((K, N), device="cuda")
    C = torch.empty((M, N), device="cuda")
    plan = handle.plan(A, B, C)
    assert plan["kind"] == 1 and (plan["tile_m"], plan["tile_n"]) == want, plan
