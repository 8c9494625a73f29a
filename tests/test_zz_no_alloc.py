"""sgemmNoAlloc: the entry point for callers that cannot allocate device
memory (code running inside an allocator hook or memory pool, under a
framework that owns all device memory, or with a fixed memory budget).

It must give the same products as the regular entry point while using only
the library's static scratch array.  Every call shares that array and it
keeps the previous call's contents, so the checks run two calls in a row.
This file is collected last (its name sorts after the other test files) so
that a stop-at-first-failure run has already run every other test; it also
passes on its own in a fresh process.
"""
import ctypes

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
    m.load_library()
    return m


def _noalloc(lib, A, B, C, alpha, beta):
    M, K = A.shape
    N = B.shape[1]
    st = lib.sgemmNoAlloc(M, N, K, float(alpha), A.data_ptr(), A.stride(0), B.data_ptr(),
                          B.stride(0), float(beta), C.data_ptr(), C.stride(0),
                          torch.cuda.current_stream().cuda_stream or None)
    return st


def _views(p):
    """Device views with the problem's row pitches (odd pitches force repacking)."""
    A = torch.from_numpy(p.A).cuda()[:, : p.K]
    B = torch.from_numpy(p.B).cuda()[:, : p.N]
    return A, B


# 1024^3 leaves most SMs idle with whole tiles, so stream-K scratch is used;
# the odd pitches of the second shape also repack A and B into the array.
SHAPES = [(1024, 1024, 1024, None, None), (1000, 777, 333, 333, 777)]


@pytest.mark.parametrize("M,N,K,lda,ldb", SHAPES)
def test_matches_regular_entry_point_two_calls_in_a_row(sg, M, N, K, lda, ldb):
    lib = sg.load_library()
    h = sg.Handle()
    for call, seed in enumerate((101, 202)):
        p = inputs.make_problem(M, N, K, seed=seed + M, alpha=0.5, beta=0.25, lda=lda, ldb=ldb)
        A, B = _views(p)
        C_init = torch.from_numpy(p.C0).cuda()
        C_ref = C_init.clone()
        h.gemm(A, B, C_ref, 0.5, 0.25)
        C = C_init.clone()
        assert _noalloc(lib, A, B, C, 0.5, 0.25) == sg.Status.SUCCESS, f"call {call}"
        torch.cuda.synchronize()
        got = C.cpu().numpy().astype(np.float64)
        want = C_ref.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - want) <= fp32_tolerance(want)), f"call {call}"
        ref = oracle.sgemm_ref(M, N, K, 0.5, p.A, p.B, 0.25, p.C0)
        assert np.all(np.abs(got - ref) <= fp32_tolerance(ref)), f"call {call} vs oracle"
    assert h.device_error() == 0
    h.close()


def test_integer_inputs_bit_exact_two_calls(sg):
    lib = sg.load_library()
    for seed in (7, 8):
        p = inputs.make_problem(768, 640, 1500, seed=seed, kind="integer")
        A, B = _views(p)
        C = torch.full((768, 640), float("nan"), device="cuda")
        assert _noalloc(lib, A, B, C, 1.0, 0.0) == sg.Status.SUCCESS
        torch.cuda.synchronize()
        np.testing.assert_array_equal(C.cpu().numpy().astype(np.float64),
                                      oracle.sgemm_ref(768, 640, 1500, 1.0, p.A, p.B))


def test_rejects_repacking_beyond_the_static_array(sg):
    lib = sg.load_library()
    # lda = 4095 forces A to be repacked: 4095 x 4096 floats = 64 MiB > 32 MiB.
    A = torch.zeros((4095, 4095), device="cuda")
    B = torch.zeros((4095, 64), device="cuda")
    C = torch.full((4095, 64), 3.0, device="cuda")
    assert _noalloc(lib, A, B, C, 1.0, 0.0) == sg.Status.NOT_SUPPORTED
    torch.cuda.synchronize()
    assert bool((C == 3.0).all()), "nothing may be enqueued on rejection"


def _noalloc_error(lib):
    code = ctypes.c_int(-1)
    st = lib.sgemmNoAllocGetDeviceError(ctypes.byref(code))
    return st, code.value


def test_bounded_wait_expiry_is_reported_and_cleared(sg):
    """A wait that runs out inside this entry point's kernels is recorded in
    the static array's error word, which sgemmNoAllocGetDeviceError reads
    and clears.  The expiry is made by leaving out the stream-K flags (a
    signal nothing then sets; no fault), with a 20 ms limit."""
    lib = sg.load_library()
    M = N = 2048
    K = 512   # 128 tiles of 256 x 128 on 152 SMs: the last wave is split stream-K
    p = inputs.make_problem(M, N, K, seed=31, kind="integer")
    A, B = _views(p)
    C = torch.zeros((M, N), device="cuda")
    assert _noalloc(lib, A, B, C, 1.0, 0.0) == sg.Status.SUCCESS
    assert _noalloc_error(lib) == (sg.Status.SUCCESS, 0)
    assert lib.sgemmNoAllocSetWaitTimeout(20_000_000) == sg.Status.SUCCESS
    assert lib.sgemmNoAllocSetTestWithheldSignal(1) == sg.Status.SUCCESS
    try:
        assert _noalloc(lib, A, B, C, 1.0, 0.0) == sg.Status.SUCCESS
        st, code = _noalloc_error(lib)
    finally:
        lib.sgemmNoAllocSetTestWithheldSignal(0)
        lib.sgemmNoAllocSetWaitTimeout(2_000_000_000)
    assert st == sg.Status.DEVICE_TIMEOUT, (st, code)
    assert code >> 24 == 4, f"expired at site {code >> 24}, expected the stream-K flag wait"
    assert _noalloc_error(lib) == (sg.Status.SUCCESS, 0), "reading the word clears it"
    # The next call is correct again.
    C.fill_(float("nan"))
    assert _noalloc(lib, A, B, C, 1.0, 0.0) == sg.Status.SUCCESS
    torch.cuda.synchronize()
    np.testing.assert_array_equal(C.cpu().numpy().astype(np.float64),
                                  oracle.sgemm_ref(M, N, K, 1.0, p.A, p.B))
    assert _noalloc_error(lib) == (sg.Status.SUCCESS, 0)


def test_settings_checked(sg):
    lib = sg.load_library()
    assert lib.sgemmNoAllocSetWaitTimeout(10) == sg.Status.INVALID_VALUE
    assert lib.sgemmNoAllocSetTestWithheldSignal(7) == sg.Status.INVALID_VALUE
    assert lib.sgemmNoAllocGetDeviceError(None) == sg.Status.INVALID_VALUE


def test_no_device_memory_is_committed_by_later_calls(sg):
    """After the first call on a device, later calls commit no device
    memory, even on shapes that take kernels not launched before (small
    products, skinny products, repacked operands, the scale-only path)."""
    lib = sg.load_library()
    torch.cuda.synchronize()
    cases = []
    for (M, N, K, lda, ldb, alpha, beta) in [
            (96, 80, 72, None, None, 1.0, 0.0),        # small-product kernel
            (8, 4096, 2048, None, None, 1.0, 0.5),     # skinny, TMA-fed
            (5, 777, 301, 301, 777, 1.0, 0.0),         # skinny, plain loads
            (600, 700, 333, 333, 701, 0.5, 0.25),      # both operands repacked
            (300, 200, 100, None, None, 0.0, 2.0),     # scale only
            (1536, 1280, 640, None, None, 1.0, 0.0)]:  # main kernel, stream-K
        p = inputs.make_problem(M, N, K, seed=M + N, kind="integer", alpha=alpha, beta=beta,
                                lda=lda, ldb=ldb)
        A, B = _views(p)
        C = (torch.from_numpy(p.C0).cuda() if p.C0 is not None
             else torch.zeros((M, N), device="cuda"))
        ref = oracle.sgemm_ref(M, N, K, alpha, p.A, p.B, beta, p.C0)
        cases.append((A, B, C, alpha, beta, ref))
    # First call on the device (set-up), if no earlier test made it.
    warm = torch.zeros((64, 64), device="cuda")
    assert _noalloc(lib, warm, warm, warm.clone(), 1.0, 0.0) == sg.Status.SUCCESS
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    reserved_before = torch.cuda.memory_reserved()
    for A, B, C, alpha, beta, _ in cases:
        assert _noalloc(lib, A, B, C, alpha, beta) == sg.Status.SUCCESS
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    assert torch.cuda.memory_reserved() == reserved_before
    assert free_after >= free_before, f"device memory dropped by {free_before - free_after} bytes"
    for A, B, C, alpha, beta, ref in cases:
        np.testing.assert_array_equal(C.cpu().numpy().astype(np.float64), ref)
