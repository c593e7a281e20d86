"""Seeded synthetic inputs for single-precision GEMM (no GEMM arithmetic here).

Both the CUDA path's tests/benchmark and the CPU oracle are fed from this
module, and it is the only thing they share.  It draws matrices, defines the
named workloads, and picks sample points; it never multiplies anything.

Generator: numpy's counter-based Philox bit generator seeded with the
workload's seed, drawn in stored order: A (its stored shape), then B, then C
(only when beta != 0, since C is not read otherwise).  Uniform[-1, 1] is
2*u - 1 with u a float32 draw from [0, 1) (exact in fp32); N(mu, s^2) is a
float32 standard normal times s.
"""
from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    """One GEMM problem: logical sizes, layouts, scalars and input recipe."""
    name: str
    M: int
    N: int
    K: int
    transA: str = "N"
    transB: str = "N"
    alpha: float = 1.0
    beta: float = 0.0
    dist: str = "uniform"      # "uniform" on [-1, 1] or "normal"
    std: float = 1.0           # standard deviation for "normal"
    seed: int = 0

    @property
    def flops(self) -> int:
        """Algorithmic flop count, 2*M*N*K."""
        return 2 * self.M * self.N * self.K

    def stored_shapes(self):
        """(rows, cols) of the stored A, B and C arrays, row-major."""
        a = (self.M, self.K) if self.transA.upper() == "N" else (self.K, self.M)
        b = (self.K, self.N) if self.transB.upper() == "N" else (self.N, self.K)
        return a, b, (self.M, self.N)

    def compulsory_bytes(self) -> int:
        """Bytes that must cross HBM once: A, B read, C written (+read if beta)."""
        c_passes = 2 if self.beta != 0 else 1
        return 4 * (self.M * self.K + self.K * self.N + c_passes * self.M * self.N)


def _w(name, M, N, K, transA="N", transB="N", **kw):
    return Workload(name=name, M=M, N=N, K=K, transA=transA, transB=transB, **kw)


# The measured problem set: square sizes from 256 to 8192, a non-tile-multiple
# shape in all four layouts, and a skinny memory-heavy NT shape.
WORKLOADS = {w.name: w for w in [
    _w("sq256_nn", 256, 256, 256, seed=0),
    _w("sq1024_nn", 1024, 1024, 1024, seed=1),
    _w("sq2048_nn_ab", 2048, 2048, 2048, alpha=1.5, beta=0.5,
       dist="normal", std=1.0, seed=2),
    _w("ragged_nn", 4095, 3073, 1537, "N", "N", beta=1.0, seed=3),
    _w("ragged_nt", 4095, 3073, 1537, "N", "T", beta=1.0, seed=3),
    _w("ragged_tn", 4095, 3073, 1537, "T", "N", beta=1.0, seed=3),
    _w("ragged_tt", 4095, 3073, 1537, "T", "T", beta=1.0, seed=3),
    _w("sq4096_nn", 4096, 4096, 4096, seed=3),
    # N(0, 1/sqrt(K)) read as variance 1/sqrt(K): std = K**-0.25
    _w("sq8192_nn", 8192, 8192, 8192, dist="normal",
       std=8192 ** -0.25, seed=4),
    _w("skinny_nt", 16384, 64, 8192, "N", "T", seed=5),
    # thin problems: decode's M = 1 to a few dozen ("Matmul II", section 8),
    # up to a batch of 128, and their mirror, a few columns of C; a 512 MB
    # operand streamed once
    _w("decode_m1_nt", 1, 16384, 8192, "N", "T", seed=6),
    _w("decode_m16_nn", 16, 16384, 8192, "N", "N", seed=7),
    _w("decode_m128_nn", 128, 16384, 8192, "N", "N", seed=10),
    _w("matvec_n1_nn", 16384, 1, 8192, "N", "N", beta=1.0, seed=8),
    _w("matvec_n8_tn", 16384, 8, 8192, "T", "N", seed=9),
]}

HEADLINE = "sq4096_nn"


def draw(rng: np.random.Generator, shape, dist="uniform", std=1.0) -> np.ndarray:
    """One fp32 array of the given shape from the workload's distribution."""
    n = int(np.prod(shape)) if len(shape) else 1
    if dist == "uniform":
        x = rng.random(n, dtype=np.float32)
        x *= np.float32(2.0)
        x -= np.float32(1.0)
    elif dist == "normal":
        x = rng.standard_normal(n, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return x.reshape(shape)


def make_inputs(w: Workload):
    """Stored (A, B, C) fp32 arrays of workload w, packed leading dimensions.

    C is None when beta == 0 (the product is written, never read).
    """
    rng = np.random.Generator(np.random.Philox(w.seed))
    sa, sb, sc = w.stored_shapes()
    A = draw(rng, sa, w.dist, w.std)
    B = draw(rng, sb, w.dist, w.std)
    C = draw(rng, sc, w.dist, w.std) if w.beta != 0 else None
    return A, B, C


def random_matrix(seed: int, rows: int, cols: int, ld: int | None = None,
                  dist="uniform", fill=np.nan) -> np.ndarray:
    """A (rows x ld) fp32 array whose first ``cols`` columns are random and
    whose padding columns hold ``fill`` (NaN by default, so a kernel that
    reads or writes the leading-dimension gap is caught)."""
    ld = cols if ld is None else ld
    rng = np.random.Generator(np.random.Philox(seed))
    out = np.full((rows, ld), fill, dtype=np.float32)
    out[:, :cols] = draw(rng, (rows, cols), dist)
    return out


def small_ints(seed: int, shape, lo=-8, hi=8) -> np.ndarray:
    """Integers in [lo, hi] stored as fp32 (exact)."""
    rng = np.random.Generator(np.random.Philox(seed))
    return rng.integers(lo, hi + 1, size=shape).astype(np.float32)


def sample_points(M: int, N: int, count: int, seed: int):
    """(rows, cols) int64 arrays: the four corners, the whole last row and
    last column (up to ``count``), then seeded uniform points; duplicates
    removed, order fixed."""
    if M == 0 or N == 0:
        return np.zeros(0, np.int64), np.zeros(0, np.int64)
    pts = [(0, 0), (0, N - 1), (M - 1, 0), (M - 1, N - 1)]
    step_r = max(1, M // 256)
    step_c = max(1, N // 256)
    pts += [(i, N - 1) for i in range(0, M, step_r)]
    pts += [(M - 1, j) for j in range(0, N, step_c)]
    rng = np.random.Generator(np.random.Philox(seed ^ 0x5EED))
    need = max(0, count - len(pts))
    r = rng.integers(0, M, size=need)
    c = rng.integers(0, N, size=need)
    pts += list(zip(r.tolist(), c.tolist()))
    seen, rows, cols = set(), [], []
    for p in pts:
        if p not in seen:
            seen.add(p)
            rows.append(p[0])
            cols.append(p[1])
    return np.asarray(rows, np.int64), np.asarray(cols, np.int64)


def workload_by_name(name: str) -> Workload:
    return WORKLOADS[name]


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def std_for(K: int) -> float:
    """Standard deviation of the N(0, 1/sqrt(K)) recipe (variance reading)."""
    return K ** -0.25 if K > 0 else 1.0


__all__ = ["Workload", "WORKLOADS", "HEADLINE", "draw", "make_inputs",
           "random_matrix", "small_ints", "sample_points", "workload_by_name",
           "ceil_div", "std_for"]
