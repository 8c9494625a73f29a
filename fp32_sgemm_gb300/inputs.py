"""Seeded synthetic inputs for the FP32 GEMM C = alpha*A*B + beta*C.

This module only draws numbers; it holds none of the GEMM arithmetic, so both
the fp64 oracle (under ``oracle/``) and the CUDA path are fed from it without
sharing any code with each other.

Generator (self-defined, counter based).  Output number i (i = 1, 2, ...) of
the stream for seed s is SplitMix64 (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; constants as in Vigna's public
splitmix64) evaluated at state ``s + i * 0x9E3779B97F4A7C15`` (mod 2**64):

    z = state
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
    z = (z ^ (z >> 27)) * 0x94D049BB133111EB
    u = z ^ (z >> 31)

One stream per problem: the logical entries of A (row major, M*K of them)
come first, then B (K*N), then the initial C (M*N).  Padding columns beyond
the logical width (lda > K and so on) are not drawn from the stream.

Value maps
  uniform:  ((u >> 40) * 2**-23) - 1, a multiple of 2**-23 in [-1, 1); every
            such value is exact in fp32.
  integer:  (((u >> 32) * 9) >> 32) - 4, an integer in {-4, ..., 4}; the
            products and all partial sums of a K <= 2**17 dot product are
            exact in fp32, so any summation order gives the same bits.

The problem recipes of the workloads (shapes, alpha, beta, seeds) are in
``WORKLOADS``; the integer twin of a workload uses seed + 1000.
"""

from __future__ import annotations

import dataclasses

import numpy as np

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

INTEGER_TWIN_SEED_OFFSET = 1000


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Outputs start+1 .. start+count of the SplitMix64 stream for ``seed``."""
    out = np.empty(count, dtype=np.uint64)
    s = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
    with np.errstate(over="ignore"):
        for lo in range(0, count, _CHUNK):
            hi = min(count, lo + _CHUNK)
            idx = np.arange(start + lo + 1, start + hi + 1, dtype=np.uint64)
            z = s + idx * GOLDEN_GAMMA
            z = (z ^ (z >> np.uint64(30))) * _MIX1
            z = (z ^ (z >> np.uint64(27))) * _MIX2
            out[lo:hi] = z ^ (z >> np.uint64(31))
    return out


def _to_uniform(u: np.ndarray) -> np.ndarray:
    # (u >> 40) < 2**24 is exact in fp32; the scale and the shift are exact too.
    return ((u >> np.uint64(40)).astype(np.float32) * np.float32(2.0 ** -23)
            - np.float32(1.0))


def _to_integer(u: np.ndarray) -> np.ndarray:
    v = ((u >> np.uint64(32)) * np.uint64(9)) >> np.uint64(32)
    return v.astype(np.float32) - np.float32(4.0)


def draw(seed: int, start: int, count: int, kind: str) -> np.ndarray:
    """``count`` fp32 values, stream positions start+1 .. start+count."""
    u = splitmix64(seed, start, count)
    if kind == "uniform":
        return _to_uniform(u)
    if kind == "integer":
        return _to_integer(u)
    raise ValueError(f"unknown value kind {kind!r}")


def embed(values: np.ndarray, rows: int, cols: int, ld: int,
          fill: float = np.nan) -> np.ndarray:
    """Place a rows x cols row-major matrix into a flat buffer with row pitch
    ``ld``; the padding columns get ``fill``.  Returns a 2-D view [rows, ld]."""
    if ld < cols:
        raise ValueError("ld must be >= cols")
    buf = np.full((rows, ld), fill, dtype=np.float32)
    buf[:, :cols] = values.reshape(rows, cols)
    return buf


@dataclasses.dataclass(frozen=True)
class Problem:
    """One synthetic GEMM instance.  A, B, C0 are [rows, ld] float32 arrays
    whose first K / N / N columns hold the logical matrix."""
    M: int
    N: int
    K: int
    alpha: float
    beta: float
    A: np.ndarray
    B: np.ndarray
    C0: np.ndarray | None

    @property
    def lda(self) -> int:
        return self.A.shape[1]

    @property
    def ldb(self) -> int:
        return self.B.shape[1]

    @property
    def ldc(self) -> int:
        return self.C0.shape[1] if self.C0 is not None else self.N

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


def make_problem(M: int, N: int, K: int, seed: int, *, kind: str = "uniform",
                 alpha: float = 1.0, beta: float = 0.0, with_c: bool | None = None,
                 lda: int | None = None, ldb: int | None = None,
                 ldc: int | None = None, pad_fill: float = np.nan) -> Problem:
    """Draw A, B (and C0 when ``with_c`` or beta != 0) from one stream."""
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    if with_c is None:
        with_c = beta != 0.0
    a = draw(seed, 0, M * K, kind)
    b = draw(seed, M * K, K * N, kind)
    A = embed(a, M, K, max(lda, 1), pad_fill)
    B = embed(b, K, N, max(ldb, 1), pad_fill)
    C0 = None
    if with_c:
        c = draw(seed, M * K + K * N, M * N, kind)
        C0 = embed(c, M, N, max(ldc, 1), pad_fill)
    return Problem(M, N, K, float(alpha), float(beta), A, B, C0)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    alpha: float
    beta: float
    seed: int
    full_check: bool          # False: check sampled entries only
    samples: int = 0


# The five workloads of the FP32 SGEMM study: square 128^3 / 1024^3 / 4096^3
# (the headline size of every page) and 8192^3, plus one non-aligned shape
# with alpha, beta != {1, 0} that exercises edge tiles and the read of C.
WORKLOADS = {
    "sgemm_128": Workload("sgemm_128", 128, 128, 128, 1.0, 0.0, 0, True),
    "sgemm_1024": Workload("sgemm_1024", 1024, 1024, 1024, 1.0, 0.0, 1, True),
    "sgemm_4096": Workload("sgemm_4096", 4096, 4096, 4096, 1.0, 0.0, 2, True),
    "sgemm_4095x4097x1023": Workload("sgemm_4095x4097x1023", 4095, 4097, 1023,
                                     0.5, 0.25, 3, True),
    "sgemm_8192": Workload("sgemm_8192", 8192, 8192, 8192, 1.0, 0.0, 4, False,
                           samples=65536),
}

# Skinny shapes beyond the five workloads: bound by HBM, not by the FMA pipes
# (few rows or few columns of C; intensity about min(M, N) / 2 FLOP/byte).
EXTRA_WORKLOADS = {
    "skinny_m1": Workload("skinny_m1", 1, 16384, 16384, 1.0, 0.0, 11, True),
    "skinny_m8": Workload("skinny_m8", 8, 16384, 16384, 1.0, 0.0, 12, True),
    "skinny_n8": Workload("skinny_n8", 16384, 8, 16384, 1.0, 0.0, 13, True),
    # Short K at large M and N: writing C (1 GiB) bounds these.
    "shortk_k8": Workload("shortk_k8", 16384, 16384, 8, 1.0, 0.0, 14, False),
    "shortk_k16": Workload("shortk_k16", 16384, 16384, 16, 1.0, 0.0, 15, False),
}

def pattern(rows, cols, seed: int = 0):
    """Closed-form integer-valued operand entries, ((7 r + 13 c + 5 seed) mod 9)
    - 4 in {-4..4}, for operands of several GB that the stream would take too
    long to draw.  `rows` and `cols` are integer arrays (numpy or torch, any
    broadcastable shapes); returns float32 of the broadcast shape, computed
    the same way by either library, so the device copy of an operand and the
    oracle's copy of the entries it needs agree exactly."""
    v = (rows * 7 + cols * 13 + seed * 5) % 9 - 4
    return v.astype("float32") if hasattr(v, "astype") else v.float()


SAMPLE_SEED_XOR = 0x5A4D


def sample_entries(M: int, N: int, count: int, seed: int) -> tuple[np.ndarray, np.ndarray]:
    """``count`` seeded (row, col) pairs of an M x N output, drawn from the
    stream of ``seed ^ 0x5A4D`` (row from the high half of each draw, column
    from the low half, each reduced by multiply-high)."""
    u = splitmix64(seed ^ SAMPLE_SEED_XOR, 0, count)
    hi = u >> np.uint64(32)
    lo = u & np.uint64(0xFFFFFFFF)
    rows = ((hi * np.uint64(M)) >> np.uint64(32)).astype(np.int64)
    cols = ((lo * np.uint64(N)) >> np.uint64(32)).astype(np.int64)
    return rows, cols


def workload_problem(w: Workload, kind: str = "uniform") -> Problem:
    seed = w.seed if kind == "uniform" else w.seed + INTEGER_TWIN_SEED_OFFSET
    return make_problem(w.M, w.N, w.K, seed, kind=kind, alpha=w.alpha,
                        beta=w.beta)
