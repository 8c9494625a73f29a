"""ctypes binding of the C ABI in include/sgemm_gb300.h.

Argument marshalling only: every step of the product runs in the CUDA
library.  torch supplies device memory (operands, workspace) and streams.
If the library has not been built, or cannot be loaded, every call raises;
there is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import enum
import os
import threading

from . import _build

_i64 = ctypes.c_int64
_f32 = ctypes.c_float
_vp = ctypes.c_void_p
_st = ctypes.c_int


class Status(enum.IntEnum):
    SUCCESS = 0
    INVALID_VALUE = 1
    MISALIGNED = 2
    ARCH_MISMATCH = 3
    WORKSPACE_REQUIRED = 4
    LAUNCH_FAILED = 5
    DEVICE_TIMEOUT = 6
    NOT_SUPPORTED = 7
    INTERNAL_ERROR = 8


class SgemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = Status(status) if status in Status._value2member_map_ else status
        super().__init__(f"{where}: {getattr(self.status, 'name', status)}")


class Plan(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int), ("tile_m", ctypes.c_int), ("tile_n", ctypes.c_int),
                ("tile_k", ctypes.c_int), ("stages", ctypes.c_int), ("ctas", ctypes.c_int),
                ("packs_a", ctypes.c_int), ("packs_b", ctypes.c_int),
                ("vector_epilogue", ctypes.c_int), ("kind", ctypes.c_int),
                ("stream_k", ctypes.c_int), ("raster_group", ctypes.c_int),
                ("edge_cols", ctypes.c_int)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


# name -> (restype, argtypes); must list every function of include/sgemm_gb300.h
SIGNATURES = {
    "sgemmGetStatusString": (ctypes.c_char_p, [_st]),
    "sgemmGetVersion": (_st, [ctypes.POINTER(ctypes.c_int)]),
    "sgemmCreate": (_st, [ctypes.POINTER(_vp)]),
    "sgemmDestroy": (_st, [_vp]),
    "sgemmGetDefaultHandle": (_st, [ctypes.POINTER(_vp)]),
    "sgemmGetWorkspaceSize": (_st, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64,
                                    ctypes.POINTER(ctypes.c_size_t)]),
    "sgemmSetWorkspace": (_st, [_vp, _vp, ctypes.c_size_t]),
    "sgemmEx": (_st, [_vp, _i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64, _vp]),
    "sgemm": (_st, [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64, _vp]),
    "sgemmHostWorkspaceSize": (_st, [_i64, _i64, _i64, ctypes.POINTER(ctypes.c_size_t)]),
    "sgemmHostEx": (_st, [_vp, _i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64,
                          _vp, ctypes.c_size_t, _vp]),
    "sgemmQueryPlan": (_st, [_vp, _i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64,
                             ctypes.POINTER(Plan)]),
    "sgemmSetAlgo": (_st, [_vp, ctypes.c_int]),
    "sgemmStridedBatched": (_st, [_vp, ctypes.c_int, ctypes.c_int, _i64, _i64, _i64, _f32, _vp, _i64,
                                  _i64, _vp, _i64, _i64, _f32, _vp, _i64, _i64, _i64, _vp]),
    "sgemmStridedBatchedWorkspaceSize": (_st, [_vp, ctypes.c_int, ctypes.c_int, _i64, _i64, _i64,
                                               _vp, _i64, _i64, _vp, _i64, _i64, _i64,
                                               ctypes.POINTER(ctypes.c_size_t)]),
    "sgemmSetSchedule": (_st, [_vp, ctypes.c_int]),
    "sgemmSetMathMode": (_st, [_vp, ctypes.c_int]),
    "sgemmSetKernelEvents": (_st, [_vp, _vp, _vp]),
    "sgemmSetWaitTimeout": (_st, [_vp, ctypes.c_uint64]),
    "sgemmGetDeviceError": (_st, [_vp, ctypes.POINTER(ctypes.c_int)]),
    "sgemmSelfTestWaitTimeout": (_st, [_vp, ctypes.c_uint64, _vp]),
    "sgemmNoAlloc": (_st, [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64, _vp]),
    "sgemmNoAllocGetDeviceError": (_st, [ctypes.POINTER(ctypes.c_int)]),
    "sgemmNoAllocSetWaitTimeout": (_st, [ctypes.c_uint64]),
    "sgemmNoAllocSetTestWithheldSignal": (_st, [ctypes.c_int]),
    "sgemmSetTestWithheldSignal": (_st, [_vp, ctypes.c_int]),
}

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load_library(build_if_missing: bool = False):
    """The loaded CUDA library (ctypes.CDLL).  Raises if it is not built."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                if not build_if_missing:
                    raise RuntimeError(
                        f"CUDA library {path} is not built; run fp32_sgemm_gb300.build()")
                _build.build()
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _check(status: int, where: str):
    if status != 0:
        raise SgemmError(status, where)


def status_string(status: int) -> str:
    return load_library().sgemmGetStatusString(int(status)).decode()


def version() -> int:
    v = ctypes.c_int()
    _check(load_library().sgemmGetVersion(ctypes.byref(v)), "sgemmGetVersion")
    return v.value


# ---------------------------------------------------------------- torch side

def _torch():
    import torch
    return torch


def _stream_ptr(stream, device_index: int | None = None) -> int | None:
    """cudaStream_t of `stream` (None: torch's current stream on the given
    device, else on the current device)."""
    torch = _torch()
    if stream is None:
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            # The raw-handle query skips building a torch.cuda.Stream object
            # (a few microseconds per call, as much as a small product takes).
            idx = torch.cuda.current_device() if device_index is None else device_index
            return raw(idx) or None
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _matrix(t, name: str, rows: int | None = None, cols: int | None = None):
    """(ptr, ld) of a row-major fp32 CUDA matrix view (stride(1) == 1)."""
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype is not torch.float32:
        raise TypeError(f"{name} must be float32, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    shape = t.shape
    if len(shape) != 2:
        raise ValueError(f"{name} must be 2-D")
    r, c = shape
    stride = t.stride()
    if r > 1 and c > 0 and stride[1] != 1:
        raise ValueError(f"{name} must be row major (stride(1) == 1)")
    ld = stride[0] if r > 1 else max(c, 1)
    if rows is not None and r != rows or cols is not None and c != cols:
        raise ValueError(f"{name} has shape {tuple(shape)}, expected ({rows}, {cols})")
    return t.data_ptr(), max(ld, c, 1)


class Handle:
    """A library handle on one device, with a torch-allocated workspace that
    grows on demand (the C library itself never allocates on the compute
    path)."""

    def __init__(self, device=None):
        torch = _torch()
        self._lib = load_library()
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None
                                   else torch.device(device).index)
        self._h = _vp()
        with torch.cuda.device(self.device):
            _check(self._lib.sgemmCreate(ctypes.byref(self._h)), "sgemmCreate")
        self._ws = None
        # Workspace sizes already asked for, by shape, pitches and operand
        # alignment; the handle's settings enter the size, so their setters
        # clear it.
        self._ws_sizes = {}

    @property
    def ptr(self):
        return self._h

    def close(self):
        if self._h:
            self._lib.sgemmDestroy(self._h)
            self._h = _vp()
            self._ws = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_algo(self, algo: int):
        _check(self._lib.sgemmSetAlgo(self._h, int(algo)), "sgemmSetAlgo")
        self._ws_sizes.clear()

    def set_kernel_events(self, start, stop):
        """Record torch.cuda.Event objects around the main kernel of later
        calls (None, None turns it off).  The events must already have been
        recorded once so that torch has created them."""
        sp = start.cuda_event if start is not None else None
        ep = stop.cuda_event if stop is not None else None
        _check(self._lib.sgemmSetKernelEvents(self._h, sp, ep), "sgemmSetKernelEvents")

    def set_math_mode(self, mode: int):
        """0 FP32 FFMA (default), 1 error-compensated 3xTF32 on the tensor cores."""
        _check(self._lib.sgemmSetMathMode(self._h, int(mode)), "sgemmSetMathMode")
        self._ws_sizes.clear()

    def set_schedule(self, schedule: int):
        """0 automatic, 1 whole tiles per CTA, 2 stream-K when it applies."""
        _check(self._lib.sgemmSetSchedule(self._h, int(schedule)), "sgemmSetSchedule")
        self._ws_sizes.clear()

    def set_wait_timeout(self, ns: int):
        _check(self._lib.sgemmSetWaitTimeout(self._h, int(ns)), "sgemmSetWaitTimeout")

    def set_test_withheld_signal(self, which: int):
        """Test hook: 0 none, 1 stream-K flag, 2 ring refill, 3 stage release
        (the bounded wait for the withheld signal then runs out)."""
        _check(self._lib.sgemmSetTestWithheldSignal(self._h, int(which)), "sgemmSetTestWithheldSignal")

    def device_error(self) -> int:
        code = ctypes.c_int()
        st = self._lib.sgemmGetDeviceError(self._h, ctypes.byref(code))
        if st not in (Status.SUCCESS, Status.DEVICE_TIMEOUT):
            _check(st, "sgemmGetDeviceError")
        return code.value

    def selftest_wait_timeout(self, ns: int, stream=None):
        _check(self._lib.sgemmSelfTestWaitTimeout(self._h, int(ns), _stream_ptr(stream)),
               "sgemmSelfTestWaitTimeout")

    def workspace_size(self, M, N, K, A_ptr, lda, B_ptr, ldb) -> int:
        n = ctypes.c_size_t()
        _check(self._lib.sgemmGetWorkspaceSize(self._h, M, N, K, A_ptr, lda, B_ptr, ldb,
                                               ctypes.byref(n)), "sgemmGetWorkspaceSize")
        return n.value

    def _ensure_workspace(self, nbytes: int):
        torch = _torch()
        if nbytes == 0:
            return
        if self._ws is None or self._ws.numel() < nbytes:
            # Work already enqueued may still use the old buffer: let torch's
            # caching allocator keep it alive until the current stream passes.
            if self._ws is not None:
                self._ws.record_stream(torch.cuda.current_stream(self.device))
            self._ws = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
            _check(self._lib.sgemmSetWorkspace(self._h, self._ws.data_ptr(), self._ws.numel()),
                   "sgemmSetWorkspace")

    def plan(self, A, B, C, alpha=1.0, beta=0.0) -> dict:
        M, K = A.shape
        N = B.shape[1]
        a, lda = _matrix(A, "A")
        b, ldb = _matrix(B, "B")
        c, ldc = _matrix(C, "C")
        p = Plan()
        _check(self._lib.sgemmQueryPlan(self._h, M, N, K, float(alpha), a, lda, b, ldb,
                                        float(beta), c, ldc, ctypes.byref(p)), "sgemmQueryPlan")
        return p.as_dict()

    def gemm_batched(self, A, B, C, alpha: float = 1.0, beta: float = 0.0, trans_a: bool = False,
                     trans_b: bool = False, stream=None):
        """C[z] = alpha * op(A[z]) @ op(B[z]) + beta * C[z] for every z.

        A, B, C: float32 CUDA tensors of shape [batch, rows, cols] (or 2-D for
        batch 1) as stored, row major (stride(-1) == 1); op(X) = X^T when
        trans_x.  Batch strides come from stride(0) (0 broadcasts one matrix).
        """
        def mat3(t, name):
            if t.dim() == 2:
                t = t.unsqueeze(0)
            if t.dim() != 3:
                raise ValueError(f"{name} must be 2-D or 3-D")
            ptr, ld = _matrix(t[0], name)
            return t, ptr, ld, (t.stride(0) if t.shape[0] > 1 else 0)
        A3, a, lda, sa = mat3(A, "A")
        B3, b, ldb, sb = mat3(B, "B")
        C3, c, ldc, sc = mat3(C, "C")
        batch = C3.shape[0]
        M, N = C3.shape[1], C3.shape[2]
        K = A3.shape[1] if trans_a else A3.shape[2]
        if (A3.shape[2] if trans_a else A3.shape[1]) != M or \
                (B3.shape[2] if trans_b else B3.shape[1]) != K or \
                (B3.shape[1] if trans_b else B3.shape[2]) != N:
            raise ValueError("operand shapes do not match")
        if A3.shape[0] not in (1, batch) or B3.shape[0] not in (1, batch):
            raise ValueError("batch sizes do not match")
        oa, ob = int(bool(trans_a)), int(bool(trans_b))
        if M and N and K and batch and alpha != 0.0:
            key = ("batched", oa, ob, M, N, K, lda, sa, ldb, sb, batch, a & 15, b & 15)
            need = self._ws_sizes.get(key)
            if need is None:
                n = ctypes.c_size_t()
                _check(self._lib.sgemmStridedBatchedWorkspaceSize(
                    self._h, oa, ob, M, N, K, a, lda, sa, b, ldb, sb, batch, ctypes.byref(n)),
                    "sgemmStridedBatchedWorkspaceSize")
                if len(self._ws_sizes) > 256:
                    self._ws_sizes.clear()
                need = self._ws_sizes[key] = n.value
            self._ensure_workspace(need)
        _check(self._lib.sgemmStridedBatched(self._h, oa, ob, M, N, K, float(alpha), a, lda, sa, b,
                                             ldb, sb, float(beta), c, ldc, sc, batch,
                                             _stream_ptr(stream, self.device.index)), "sgemmStridedBatched")
        return C

    def gemm(self, A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None):
        """C = alpha*A@B + beta*C in place (C: [M, N] row-major view)."""
        M, K = A.shape
        K2, N = B.shape
        if K2 != K:
            raise ValueError(f"inner dimensions differ: A {tuple(A.shape)}, B {tuple(B.shape)}")
        a, lda = _matrix(A, "A")
        b, ldb = _matrix(B, "B")
        c, ldc = _matrix(C, "C", M, N)
        if M and N and K and alpha != 0.0:
            key = (M, N, K, lda, ldb, a & 15, b & 15)
            need = self._ws_sizes.get(key)
            if need is None:
                if len(self._ws_sizes) > 256:
                    self._ws_sizes.clear()
                need = self._ws_sizes[key] = self.workspace_size(M, N, K, a, lda, b, ldb)
            self._ensure_workspace(need)
        _check(self._lib.sgemmEx(self._h, M, N, K, float(alpha), a, lda, b, ldb, float(beta),
                                 c, ldc, _stream_ptr(stream, self.device.index)), "sgemmEx")
        return C


_default_handles: dict[int, Handle] = {}


def default_handle(device=None) -> Handle:
    torch = _torch()
    idx = torch.cuda.current_device() if device is None else torch.device(device).index
    h = _default_handles.get(idx)
    if h is None:
        h = _default_handles[idx] = Handle(idx)
    return h


def sgemm(A, B, C=None, alpha: float = 1.0, beta: float = 0.0, *, handle: Handle | None = None,
          stream=None):
    """C = alpha * A @ B + beta * C on the GPU; returns C.

    A [M, K], B [K, N], C [M, N]: float32 CUDA tensors, row major with any
    row pitch (stride(0)), stride(1) == 1.  With C None a new tensor is made
    (beta must then be 0).
    """
    torch = _torch()
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C")
        C = torch.empty((A.shape[0], B.shape[1]), dtype=torch.float32, device=A.device)
    h = handle or default_handle(A.device)
    return h.gemm(A, B, C, alpha, beta, stream)


def host_workspace_size(M: int, N: int, K: int) -> int:
    n = ctypes.c_size_t()
    _check(load_library().sgemmHostWorkspaceSize(M, N, K, ctypes.byref(n)),
           "sgemmHostWorkspaceSize")
    return n.value


def sgemm_host(A, B, C, alpha: float = 1.0, beta: float = 0.0, *, workspace, handle=None,
               stream=None):
    """sgemmHostEx on host tensors (pinned CPU float32, row major): copies in,
    multiplies on the GPU, copies the result into C.  Enqueued on `stream`;
    synchronise before reading C."""
    torch = _torch()
    for name, t in (("A", A), ("B", B), ("C", C)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or t.is_cuda or t.dim() != 2:
            raise TypeError(f"{name} must be a 2-D float32 CPU tensor")
        if t.shape[0] > 1 and t.shape[1] > 0 and t.stride(1) != 1:
            raise ValueError(f"{name} must be row major")
    M, K = A.shape
    N = B.shape[1]
    h = handle or default_handle(workspace.device)
    # The device copies are 256-byte aligned with pitches padded to 4 floats;
    # the handle's own workspace must cover the product on them.
    pad4 = lambda n: (max(n, 1) + 3) // 4 * 4
    h._ensure_workspace(h.workspace_size(M, N, K, 256, pad4(K), 256, pad4(N)))
    lib = load_library()
    _check(lib.sgemmHostEx(h.ptr, M, N, K, float(alpha), A.data_ptr(), max(A.stride(0), K, 1),
                           B.data_ptr(), max(B.stride(0), N, 1), float(beta), C.data_ptr(),
                           max(C.stride(0), N, 1), workspace.data_ptr(),
                           workspace.numel() * workspace.element_size(), _stream_ptr(stream)),
           "sgemmHostEx")
    return C
