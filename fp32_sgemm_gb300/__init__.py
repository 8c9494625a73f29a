"""GB300-native FP32 SGEMM: C = alpha * A @ B + beta * C on row-major FP32
matrices, computed by hand-written sm_103a CUDA kernels behind a C ABI
(include/sgemm_gb300.h).  This package holds that library's sources
(csrc/), its in-tree build step and a thin ctypes binding; the seeded input
generator lives in ``inputs``.

The binding is imported lazily so that ``fp32_sgemm_gb300.inputs`` works on
machines without torch's CUDA runtime or the built library.
"""

_BINDING_NAMES = {
    "Handle", "Plan", "SgemmError", "Status", "default_handle", "host_workspace_size",
    "library_path", "load_library", "sgemm", "sgemm_host", "status_string", "version",
    "SIGNATURES",
}


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA library for sm_103a (in tree); returns the .so path."""
    from . import _build
    return _build.build(force=force, verbose=verbose)


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import _binding
        return getattr(_binding, name)
    raise AttributeError(name)
