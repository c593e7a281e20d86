"""CPU oracle for single-precision GEMM (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg import this package.  The CUDA library never imports, links or
calls it, and it imports nothing from the CUDA library.

The arithmetic lives in ``oracle.c`` (plain C, fp64 accumulation, ascending
k): the GEMM definition C = alpha*op(A)*op(B) + beta*C of "Optimising fp32
GEMM on A100" (section "What is GEMM?") with the alpha/beta epilogue of
"CuTe-ly writing an SM86 SGEMM" (section "epilogue").  This module only
marshals numpy arrays into it and compares a candidate result with what it
returns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, OpenMP if present).

    -ffp-contract=off keeps gcc from fusing a*b+c anywhere but the explicit
    fmaf calls; no fast-math, so no reassociation.
    """
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off",
            "-fPIC", "-shared", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, f32 = ctypes.c_int64, ctypes.c_float
            vp = ctypes.c_void_p
            common = [ctypes.c_char, ctypes.c_char, i64, i64, i64,
                      f32, vp, i64, vp, i64, f32, vp, i64, vp, vp, i64]
            lib.oracle_gemm_f64.argtypes = common + [vp, vp]
            lib.oracle_gemm_f64.restype = ctypes.c_int
            lib.oracle_gemm_f32_seq.argtypes = common + [vp]
            lib.oracle_gemm_f32_seq.restype = ctypes.c_int
            lib.oracle_gemm_epilogue_f64.argtypes = (
                common[:13] + [vp, vp, ctypes.c_int] + common[13:] + [vp, vp])
            lib.oracle_gemm_epilogue_f64.restype = ctypes.c_int
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
            lib.oracle_set_num_threads.restype = None
            _lib = lib
    return _lib


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use."""
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Sets the threads of the oracle's OpenMP loops (results are unchanged:
    every entry is computed by one thread in a fixed order)."""
    _load().oracle_set_num_threads(int(n))


def _ptr(a):
    return None if a is None else a.ctypes.data


def _prep(A, B, C):
    A = None if A is None else np.ascontiguousarray(A, dtype=np.float32).reshape(-1)
    B = None if B is None else np.ascontiguousarray(B, dtype=np.float32).reshape(-1)
    C = None if C is None else np.ascontiguousarray(C, dtype=np.float32).reshape(-1)
    return A, B, C


def _points(points):
    if points is None:
        return None, None, 0
    rows = np.ascontiguousarray(points[0], dtype=np.int64)
    cols = np.ascontiguousarray(points[1], dtype=np.int64)
    assert rows.shape == cols.shape
    return rows, cols, rows.size


class OracleArgError(ValueError):
    """Raised when the oracle rejects an argument (BLAS-style position)."""


def gemm_f64(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
             points=None):
    """Reference result and error bound, both float64.

    A, B, C are the stored fp32 arrays (row-major, flattened with their
    leading dimensions).  ``points=(rows, cols)`` restricts the output to
    those entries; otherwise the result has shape (M, N).
    Returns (ref, bound).
    """
    A, B, C = _prep(A, B, C)
    rows, cols, npts = _points(points)
    n_out = npts if points is not None else M * N
    ref = np.empty(max(n_out, 1), dtype=np.float64)
    bound = np.empty(max(n_out, 1), dtype=np.float64)
    st = _load().oracle_gemm_f64(
        transA.encode(), transB.encode(), M, N, K, float(alpha), _ptr(A), lda,
        _ptr(B), ldb, float(beta), _ptr(C), ldc, _ptr(rows), _ptr(cols), npts,
        ref.ctypes.data, bound.ctypes.data)
    if st != 0:
        raise OracleArgError(f"oracle rejected argument {-st}")
    ref, bound = ref[:n_out], bound[:n_out]
    if points is None:
        ref, bound = ref.reshape(M, N), bound.reshape(M, N)
    return ref, bound


def gemm_f32_seq(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                 points=None):
    """fp32 result in the naive ascending-k FMA order (float32 array)."""
    A, B, C = _prep(A, B, C)
    rows, cols, npts = _points(points)
    n_out = npts if points is not None else M * N
    out = np.empty(max(n_out, 1), dtype=np.float32)
    st = _load().oracle_gemm_f32_seq(
        transA.encode(), transB.encode(), M, N, K, float(alpha), _ptr(A), lda,
        _ptr(B), ldb, float(beta), _ptr(C), ldc, _ptr(rows), _ptr(cols), npts,
        out.ctypes.data)
    if st != 0:
        raise OracleArgError(f"oracle rejected argument {-st}")
    out = out[:n_out]
    return out.reshape(M, N) if points is None else out


def gemm_epilogue_f64(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                      row_scale=None, bias=None, act=0, points=None):
    """Reference and bound of the fused-epilogue GEMM
    D = act(alpha * diag(row_scale) * op(A) op(B) + beta * C + bias[None, :])
    (oracle.c, oracle_gemm_epilogue_f64).  row_scale: M fp32 values or None
    (all ones); bias: N fp32 values or None (zero); act: 0 identity, 1 ReLU.
    Returns (ref, bound) like gemm_f64."""
    A, B, C = _prep(A, B, C)
    rs = None if row_scale is None else np.ascontiguousarray(row_scale, dtype=np.float32)
    bs = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    rows, cols, npts = _points(points)
    n_out = npts if points is not None else M * N
    ref = np.empty(max(n_out, 1), dtype=np.float64)
    bound = np.empty(max(n_out, 1), dtype=np.float64)
    st = _load().oracle_gemm_epilogue_f64(
        transA.encode(), transB.encode(), M, N, K, float(alpha), _ptr(A), lda,
        _ptr(B), ldb, float(beta), _ptr(C), ldc, _ptr(rs), _ptr(bs), int(act),
        _ptr(rows), _ptr(cols), npts, ref.ctypes.data, bound.ctypes.data)
    if st != 0:
        raise OracleArgError(f"oracle rejected argument {-st}")
    ref, bound = ref[:n_out], bound[:n_out]
    if points is None:
        ref, bound = ref.reshape(M, N), bound.reshape(M, N)
    return ref, bound


def compare_bound(candidate, ref, bound):
    """Elementwise |cand - ref| <= bound everywhere (no exact special case:
    the fused-epilogue bound already carries the epilogue's own roundings).
    Same report fields as compare()."""
    cand = np.asarray(candidate, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bound = np.asarray(bound, dtype=np.float64)
    err = np.abs(cand - ref)
    ok = bool(np.all(np.isfinite(cand))) and bool(np.all(err <= bound))
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(bound > 0, err / np.where(bound > 0, bound, 1.0),
                     np.where(err > 0, np.inf, 0.0))
    worst = float(q.max()) if q.size else 0.0
    nz = np.abs(ref) > 2.0 ** -60
    max_rel = float((err[nz] / np.abs(ref[nz])).max()) if nz.any() else 0.0
    return {"pass": ok, "max_err_over_bound": worst, "max_rel": max_rel,
            "n_bad": int(np.count_nonzero(~(err <= bound))), "n": int(cand.size)}


def compare_ieee(candidate, ref, bound):
    """Elementwise check for inputs that may hold infinities or NaN.

    Where the fp64 reference is not finite the candidate must be the same:
    NaN, or an infinity of the same sign.  IEEE arithmetic gives that class
    in fp32 as in fp64 (inf * finite = inf with the product's sign, inf * 0
    and inf - inf = NaN, NaN propagates) as long as no finite partial sum
    overflows fp32.  Elsewhere |cand - ref| <= bound, as in compare().
    """
    cand = np.asarray(candidate, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bound = np.asarray(bound, dtype=np.float64)
    fin = np.isfinite(ref)
    same_class = np.where(np.isnan(ref), np.isnan(cand), cand == ref)
    with np.errstate(invalid="ignore"):
        within = np.abs(cand - ref) <= bound
    good = np.where(fin, within, same_class)
    return {"pass": bool(good.all()), "n_bad": int(np.count_nonzero(~good)),
            "n_nonfinite": int(np.count_nonzero(~fin)), "n": int(cand.size)}


def compare(candidate, ref, bound, K, alpha):
    """Elementwise check of a candidate fp32 result against (ref, bound).

    Pass rule: |cand - ref| <= bound for every entry, the tolerance
    4*K*2^-24*(|alpha|*(|A||B|)_ij + |beta|*|C_ij|).  When no product term
    exists (K == 0 or alpha == 0) the exact result is the single product
    beta*c (or 0), whose correctly rounded fp32 value is the only right
    answer, so the rule becomes cand == fp32(ref).
    Returns a dict with the pass flag, the worst |err|/bound, the max
    relative error over entries with |ref| > 2^-60 and the normwise error.
    """
    cand = np.asarray(candidate, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bound = np.asarray(bound, dtype=np.float64)
    err = np.abs(cand - ref)
    finite = bool(np.all(np.isfinite(cand)))
    if K == 0 or alpha == 0:
        ok = finite and bool(np.all(cand == ref.astype(np.float32).astype(np.float64)))
        worst = 0.0 if ok else float("inf")
    else:
        ok = finite and bool(np.all(err <= bound))
        with np.errstate(divide="ignore", invalid="ignore"):
            q = np.where(bound > 0, err / np.where(bound > 0, bound, 1.0),
                         np.where(err > 0, np.inf, 0.0))
        worst = float(q.max()) if q.size else 0.0
    nz = np.abs(ref) > 2.0 ** -60
    max_rel = float((err[nz] / np.abs(ref[nz])).max()) if nz.any() else 0.0
    rn = float(np.linalg.norm(ref))
    normwise = float(np.linalg.norm(cand - ref) / rn) if rn > 0 else float(np.linalg.norm(cand - ref))
    n_bad = int(np.count_nonzero(~(err <= bound))) if not (K == 0 or alpha == 0) else int(not ok)
    return {"pass": ok, "max_err_over_bound": worst, "max_rel": max_rel,
            "normwise_rel": normwise, "n_bad": n_bad, "n": int(cand.size)}
