"""Failure detection on the GEMM kernels' own bounded waits.

Every wait in the main kernels (the consumers' wait for operand data, the
TMA issuer's wait for a free stage, the finishing CTA's wait for another
CTA's stream-K partial tile) gives up after the handle's limit, records
(site << 24 | CTA) in the handle's error word and lets the kernel return.
These tests make each of those waits run out by having the kernels leave
out the one signal it waits for (a flag nothing sets; no fault, trap or
endless loop), then check the recorded site, and that the same handle and
context still compute a correct product afterwards (the 3xTF32 kernel must
also have released its tensor memory, or the next launch could not
allocate it).
"""
import numpy as np
import pytest

import oracle
from fp32_sgemm_gb300 import inputs

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

LIMIT_NS = 20_000_000          # 20 ms per wait
SITE_DATA, SITE_SLOT, SITE_FLAG = 1, 2, 4
NONE, FLAG, REFILL, RELEASE = 0, 1, 2, 3


@pytest.fixture(scope="module")
def sg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp32_sgemm_gb300 as m
    m.build()
    m.load_library()
    return m


def _operands(M, N, K, seed):
    p = inputs.make_problem(M, N, K, seed=seed, kind="integer")
    return p, torch.from_numpy(p.A).cuda(), torch.from_numpy(p.B).cuda()


def _expire_then_recover(sg, h, M, N, K, which, site, expect_ctas=None, plan_check=None):
    p, A, B = _operands(M, N, K, seed=M + N + K + which)
    C = torch.zeros((M, N), device="cuda")
    h.gemm(A, B, C)            # a normal call first: attaches the workspace the plan depends on
    plan = h.plan(A, B, C)
    if plan_check is not None:
        plan_check(plan)
    if expect_ctas is not None:
        assert plan["ctas"] == expect_ctas, plan
    assert h.device_error() == 0
    h.set_wait_timeout(LIMIT_NS)
    h.set_test_withheld_signal(which)
    try:
        h.gemm(A, B, C)
        code = h.device_error()
    finally:
        h.set_test_withheld_signal(NONE)
        h.set_wait_timeout(2_000_000_000)
    assert code != 0, "the withheld signal's wait did not expire"
    assert code >> 24 == site, f"expired at site {code >> 24}, expected {site} (code {code:#x})"
    assert (code & 0xFFFFFF) < plan["ctas"]
    assert h.device_error() == 0, "reading the error word clears it"
    # The context and the handle still work: a full product, bit exact.
    C2 = torch.full((M, N), float("nan"), device="cuda")
    h.gemm(A, B, C2)
    np.testing.assert_array_equal(C2.cpu().numpy().astype(np.float64),
                                  oracle.sgemm_ref(M, N, K, 1.0, p.A, p.B))
    assert h.device_error() == 0


# FFMA kernel, one CTA (whole tiles, one 256 x 128 tile, 32 K slices on a
# two-stage ring), so the expiry that comes first is certain: the issuer
# starts waiting for a free stage a whole slice before the consumers start
# waiting for the slice it never loads.
@pytest.mark.parametrize("which,site", [(REFILL, SITE_DATA), (RELEASE, SITE_SLOT)])
def test_ffma_pipeline_waits_expire(sg, which, site):
    h = sg.Handle()
    h.set_algo(28)
    h.set_schedule(1)
    _expire_then_recover(sg, h, 256, 128, 1024, which, site, expect_ctas=1)
    h.close()


def test_ffma_stream_k_flag_wait_expires(sg):
    # Four tiles of 16 K slices, one slice per CTA: the CTA holding a tile's
    # first slice waits for the other 15 partial tiles' flags, which never
    # come.
    h = sg.Handle()
    h.set_algo(28)
    h.set_schedule(2)
    _expire_then_recover(sg, h, 512, 256, 512, FLAG, SITE_FLAG, expect_ctas=64,
                         plan_check=lambda pl: pl["stream_k"] == 1 or pytest.fail(str(pl)))
    h.close()


def test_ffma_stream_k_flag_wait_expires_automatic_plan(sg):
    # The default plan of an uneven tile count (the last wave split stream-K).
    h = sg.Handle()
    _expire_then_recover(sg, h, 2048, 2048, 512, FLAG, SITE_FLAG,
                         plan_check=lambda pl: pl["stream_k"] == 1 or pytest.fail(str(pl)))
    h.close()


# Tensor-core kernel: one 128 x 256 tile on one SM (configuration 3), or one
# 256 x 256 tile on an SM pair (configuration 4: both CTAs' copies report to
# the first CTA's barriers, and both must release their shared tensor
# memory allocation).
@pytest.mark.parametrize("config,M,ctas", [(3, 128, 1), (4, 256, 2)])
@pytest.mark.parametrize("which,site", [(REFILL, SITE_DATA), (RELEASE, SITE_SLOT)])
def test_tf32x3_pipeline_waits_expire_and_free_tensor_memory(sg, which, site, config, M, ctas):
    h = sg.Handle()
    h.set_math_mode(1)
    h.set_algo(config)
    h.set_schedule(1)
    _expire_then_recover(sg, h, M, 256, 1024, which, site, expect_ctas=ctas)
    # Several more launches over every SM: each allocates tensor memory.
    p, A, B = _operands(1024, 1024, 512, seed=5)
    C = torch.zeros((1024, 1024), device="cuda")
    for _ in range(3):
        h.gemm(A, B, C)
    np.testing.assert_array_equal(C.cpu().numpy().astype(np.float64),
                                  oracle.sgemm_ref(1024, 1024, 512, 1.0, p.A, p.B))
    assert h.device_error() == 0
    h.close()


@pytest.mark.parametrize("config,M", [(3, 128), (4, 256)])
def test_tf32x3_stream_k_flag_wait_expires(sg, config, M):
    h = sg.Handle()
    h.set_math_mode(1)
    h.set_algo(config)
    h.set_schedule(2)
    _expire_then_recover(sg, h, M, 256, 8192, FLAG, SITE_FLAG,
                         plan_check=lambda pl: pl["stream_k"] == 1 or pytest.fail(str(pl)))
    h.close()


def test_withheld_signal_values_checked(sg):
    h = sg.Handle()
    for bad in (-1, 4, 100):
        with pytest.raises(sg.SgemmError):
            h.set_test_withheld_signal(bad)
    h.close()
