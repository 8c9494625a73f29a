"""The C ABI library without a GPU: it loads, exports every function that
include/*.h declares, and its host-side validation answers before any CUDA
call is made."""
import ctypes
import glob
import os
import re

import pytest

import fp32_sgemm_gb300 as sg
from fp32_sgemm_gb300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    sg.build()
    return sg.load_library()


def _declared_functions():
    names = set()
    for path in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(path).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(sgemm\w*)\s*\(", text):
            names.add(m.group(1))
    return names


def test_header_declares_the_entry_points():
    names = _declared_functions()
    assert {"sgemm", "sgemmEx", "sgemmCreate", "sgemmDestroy", "sgemmGetWorkspaceSize",
            "sgemmSetWorkspace", "sgemmGetDeviceError", "sgemmGetStatusString"} <= names


def test_library_exports_every_declared_function(lib):
    for name in sorted(_declared_functions()):
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_binding_signatures_cover_the_header():
    assert set(_binding.SIGNATURES) == _declared_functions()


def test_header_is_plain_c(tmp_path):
    # The boundary is a C ABI: the header must compile as C99 on its own
    # (no C++ types), and call the library through a C translation unit.
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_header.c"
    src.write_text('#include "sgemm_gb300.h"\n'
                   "int main(void) {\n"
                   "    sgemmPlan_t plan;\n"
                   "    int v = 0;\n"
                   "    (void)plan;\n"
                   "    return sgemmGetVersion(&v) == SGEMM_STATUS_SUCCESS ? 0 : 1;\n"
                   "}\n")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        "-I", cuda_inc, "-c", str(src), "-o", str(tmp_path / "use_header.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_status_strings(lib):
    for st in _binding.Status:
        assert sg.status_string(st) == "SGEMM_STATUS_" + st.name
    assert sg.status_string(99) == "SGEMM_STATUS_UNKNOWN"
    assert sg.version() == 10000


F = 0x10000  # a fake, 256-byte aligned "device" address: never dereferenced


def _call(lib, M, N, K, A=F, lda=None, B=F, ldb=None, C=F, ldc=None, alpha=1.0, beta=0.0):
    lda = max(K, 1) if lda is None else lda
    ldb = max(N, 1) if ldb is None else ldb
    ldc = max(N, 1) if ldc is None else ldc
    return lib.sgemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, None)


@pytest.mark.parametrize("args", [
    dict(M=-1, N=4, K=4), dict(M=4, N=-1, K=4), dict(M=4, N=4, K=-2),
    dict(M=4, N=4, K=8, lda=7), dict(M=4, N=8, K=4, ldb=7), dict(M=4, N=8, K=4, ldc=7),
    dict(M=4, N=4, K=4, C=None), dict(M=4, N=4, K=4, A=None), dict(M=4, N=4, K=4, B=None),
    dict(M=4, N=4, K=0, lda=0),
])
def test_invalid_arguments_rejected_on_host(lib, args):
    assert _call(lib, **args) == _binding.Status.INVALID_VALUE


@pytest.mark.parametrize("args", [
    dict(M=4, N=4, K=4, A=F + 2), dict(M=4, N=4, K=4, B=F + 1), dict(M=4, N=4, K=4, C=F + 3),
])
def test_misaligned_pointers_rejected_on_host(lib, args):
    assert _call(lib, **args) == _binding.Status.MISALIGNED


def test_sizes_beyond_32_bit_indexing_not_supported(lib):
    assert _call(lib, 2 ** 31, 4, 4) == _binding.Status.NOT_SUPPORTED
    assert _call(lib, 4, 4, 2 ** 31, lda=2 ** 31) == _binding.Status.NOT_SUPPORTED


def test_empty_output_is_a_no_op_without_touching_cuda(lib):
    # M == 0 or N == 0 returns before any device query (this host has no GPU).
    assert _call(lib, 0, 5, 5, A=None, B=None, C=None) == 0
    assert _call(lib, 5, 0, 5, A=None, B=None, C=None) == 0


def test_alpha_zero_does_not_need_a_or_b(lib):
    # With alpha == 0, A and B may be NULL; validation passes and the call
    # then needs the device (absent here), so it fails only at that point.
    st = _call(lib, 4, 4, 4, A=None, B=None, alpha=0.0)
    assert st != _binding.Status.INVALID_VALUE


def test_host_workspace_size(lib):
    n = sg.host_workspace_size(4095, 4097, 1023)
    def a256(x):
        return (x + 255) // 256 * 256
    want = a256(4095 * 1024 * 4) + a256(1023 * 4100 * 4) + a256(4095 * 4100 * 4)
    assert n == want


def test_null_handle_rejected(lib):
    assert lib.sgemmEx(None, 4, 4, 4, 1.0, F, 4, F, 4, 0.0, F, 4, None) == _binding.Status.INVALID_VALUE
    assert lib.sgemmSetAlgo(None, 1) == _binding.Status.INVALID_VALUE
    code = ctypes.c_int()
    assert lib.sgemmGetDeviceError(None, ctypes.byref(code)) == _binding.Status.INVALID_VALUE
    assert lib.sgemmSetTestWithheldSignal(None, 1) == _binding.Status.INVALID_VALUE
    assert lib.sgemmDestroy(None) == 0


def test_configurations_not_built_are_rejected(lib):
    # Numbers of tile configurations that are not built (measured slower)
    # are refused before the handle is touched (a fake pointer here).
    for algo in (5, 9, 11, 15, 22, 25, 26, 31, -1):
        assert lib.sgemmSetAlgo(F, algo) == _binding.Status.INVALID_VALUE


def test_no_alloc_settings_validated_on_host(lib):
    # Rejected before any CUDA call (this machine may have no GPU).
    assert lib.sgemmNoAllocSetWaitTimeout(999_999) == _binding.Status.INVALID_VALUE
    assert lib.sgemmNoAllocSetTestWithheldSignal(-1) == _binding.Status.INVALID_VALUE
    assert lib.sgemmNoAllocSetTestWithheldSignal(4) == _binding.Status.INVALID_VALUE
    assert lib.sgemmNoAllocGetDeviceError(None) == _binding.Status.INVALID_VALUE


def _batched(lib, opA=0, opB=0, M=4, N=4, K=4, lda=None, ldb=None, ldc=None, sa=0, sb=0, sc=0,
             batch=2, A=F, B=F, C=F):
    # The handle is a fake pointer: only use with arguments that fail
    # validation or describe an empty product (both return before using it).
    lda = (K if opA == 0 else M) if lda is None else lda
    ldb = (N if opB == 0 else K) if ldb is None else ldb
    ldc = N if ldc is None else ldc
    return lib.sgemmStridedBatched(F, opA, opB, M, N, K, 1.0, A, lda, sa, B, ldb, sb, 0.0, C, ldc,
                                   sc, batch, None)


@pytest.mark.parametrize("args", [
    dict(opA=2), dict(opB=-1), dict(batch=-1), dict(sa=-4), dict(sc=-1),
    dict(opA=1, M=8, K=4, lda=7),      # A stored K x M needs lda >= M
    dict(opB=1, N=8, K=6, ldb=5),      # B stored N x K needs ldb >= K
    dict(opA=0, M=8, K=6, lda=5),
])
def test_batched_invalid_arguments(lib, args):
    assert _batched(lib, **args) == _binding.Status.INVALID_VALUE


def test_batched_empty_is_a_no_op(lib):
    assert _batched(lib, batch=0, A=None, B=None, C=None) == 0
    assert _batched(lib, M=0, A=None, B=None, C=None) == 0
