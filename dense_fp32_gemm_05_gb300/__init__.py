"""Python binding of the GB300 single-precision GEMM C library.

A thin ctypes layer over libsgemm_gb300.so (include/sgemm_gb300.h): the same
entry points under the same names, argument marshalling only.  Every step of
the computation runs in the library's CUDA kernels; there is no fallback, and
a missing library raises at the first call.  PyTorch, when used, supplies
device memory and the current stream (``gemm`` below), nothing else.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "SGEMM_OK", "SGEMM_ERR_CUDA", "SGEMM_ERR_TIMEOUT", "SGEMM_ERR_NOMEM",
    "SGEMM_ERR_UNSUPPORTED", "SGEMM_ERR_ARG", "SGEMM_ERR_SCRATCH", "PATH_AUTO", "PATH_FFMA",
    "PATH_3XTF32", "PATH_TF32", "PATH_GEMV", "ACT_NONE", "ACT_RELU", "sgemm_epilogue", "SgemmError", "library_path", "load",
    "sgemm", "sgemm_ex", "sgemm_host", "sgemm_plan", "sgemm_plan_detail", "sgemm_status_string",
    "sgemm_device_error", "sgemm_set_wait_limit", "sgemm_release_workspace",
    "sgemm_version", "sgemm_ffma_static_scratch", "sgemm_timing_enable",
    "sgemm_timing_read", "sgemm_launch_count", "sgemm_probe_tf32_rate", "gemm",
    "exported_symbols",
]

SGEMM_OK = 0
SGEMM_ERR_CUDA = 1
SGEMM_ERR_TIMEOUT = 2
SGEMM_ERR_NOMEM = 3
SGEMM_ERR_UNSUPPORTED = 4
SGEMM_ERR_ARG = 5
SGEMM_ERR_SCRATCH = 6

PATH_AUTO = 0
PATH_FFMA = 1
PATH_3XTF32 = 2
PATH_TF32 = 3
PATH_GEMV = 4
ACT_NONE = 0
ACT_RELU = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libsgemm_gb300.so"
_lock = threading.Lock()
_lib = None


class SgemmError(RuntimeError):
    """A non-zero status returned by the library."""

    def __init__(self, status: int, where: str = "sgemm"):
        self.status = status
        super().__init__(f"{where}: status {status} ({sgemm_status_string(status)})")


class PlanInfo(ctypes.Structure):
    """sgemm_plan_info of the C header, field for field."""
    _fields_ = [(n, ctypes.c_int) for n in (
        "path", "tile_m", "tile_n", "vector", "ctas", "split", "dp_tiles", "pair", "fuse_a",
        "fuse_b", "wide", "accumulators", "k_block", "tail_nsplit", "sk_ctas", "sk_tail",
        "pre_transpose")]


def library_path() -> str:
    return os.path.join(_HERE, _LIB_NAME)


def _declare(lib):
    c, i64, f32, vp, i32 = ctypes.c_char, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int
    gemm_args = [c, c, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, vp]
    lib.sgemm.argtypes = gemm_args
    lib.sgemm.restype = i32
    lib.sgemm_ex.argtypes = gemm_args + [i32, i32]
    lib.sgemm_ex.restype = i32
    lib.sgemm_epilogue.argtypes = gemm_args[:13] + [vp, vp, i32, vp, i32, i32]
    lib.sgemm_epilogue.restype = i32
    lib.sgemm_host.argtypes = gemm_args
    lib.sgemm_host.restype = i32
    ip = ctypes.POINTER(ctypes.c_int)
    lib.sgemm_plan.argtypes = [c, c, i64, i64, i64, i64, i64, i64, i32, i32, i32, i32, i32, i32,
                               ip, ip, ip, ip, ip, ip]
    lib.sgemm_plan.restype = i32
    lib.sgemm_plan_detail.argtypes = [c, c, i64, i64, i64, i64, i64, i64, i32, i32, i32, i32, i32,
                                      i32, ctypes.POINTER(PlanInfo)]
    lib.sgemm_plan_detail.restype = i32
    lib.sgemm_status_string.argtypes = [i32]
    lib.sgemm_status_string.restype = ctypes.c_char_p
    lib.sgemm_device_error.argtypes = [vp]
    lib.sgemm_device_error.restype = i32
    lib.sgemm_set_wait_limit.argtypes = [ctypes.c_uint64]
    lib.sgemm_set_wait_limit.restype = i32
    lib.sgemm_release_workspace.argtypes = []
    lib.sgemm_release_workspace.restype = i32
    lib.sgemm_version.argtypes = []
    lib.sgemm_version.restype = i32
    lib.sgemm_timing_enable.argtypes = [i32]
    lib.sgemm_timing_enable.restype = i32
    lib.sgemm_timing_read.argtypes = [ctypes.POINTER(ctypes.c_float), i32]
    lib.sgemm_timing_read.restype = i32
    lib.sgemm_probe_tf32_rate.argtypes = [i32, ctypes.POINTER(ctypes.c_double)]
    lib.sgemm_probe_tf32_rate.restype = i32
    lib.sgemm_launch_count.argtypes = []
    lib.sgemm_launch_count.restype = i64
    lib.sgemm_ffma_static_scratch.argtypes = gemm_args + [i32]
    lib.sgemm_ffma_static_scratch.restype = i32


def load():
    """Loads the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with "
                    "`python -m dense_fp32_gemm_05_gb300.build` (needs nvcc)")
            lib = ctypes.CDLL(path)
            _declare(lib)
            _lib = lib
    return _lib


def exported_symbols(lib=None):
    """Names of the entry points this binding declares, for export checks."""
    return ["sgemm", "sgemm_ex", "sgemm_epilogue", "sgemm_host", "sgemm_plan", "sgemm_plan_detail",
            "sgemm_status_string", "sgemm_device_error",
            "sgemm_set_wait_limit", "sgemm_release_workspace", "sgemm_version",
            "sgemm_ffma_static_scratch", "sgemm_timing_enable", "sgemm_timing_read",
            "sgemm_launch_count", "sgemm_probe_tf32_rate"]


def _b(t: str) -> bytes:
    return t.encode() if isinstance(t, str) else bytes(t)


def _stream(stream) -> int | None:
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return int(getattr(stream, "cuda_stream", stream))


def sgemm(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> int:
    """C = alpha*op(A)*op(B) + beta*C; A, B, C are device addresses (int)."""
    return load().sgemm(_b(transA), _b(transB), M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                        _stream(stream))


def sgemm_ex(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None,
             path=PATH_AUTO, split=0) -> int:
    """sgemm with the path and the FFMA split-K factor forced."""
    return load().sgemm_ex(_b(transA), _b(transB), M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                           _stream(stream), path, split)


def sgemm_epilogue(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, row_scale=0,
                   bias=0, activation=ACT_NONE, stream=None, path=PATH_AUTO, split=0) -> int:
    """GEMM with the fused epilogue C = act(alpha * s_i * AB + beta * C + bias_j);
    row_scale / bias are device addresses (0 = none)."""
    return load().sgemm_epilogue(_b(transA), _b(transB), M, N, K, alpha, A, lda, B, ldb, beta,
                                 C, ldc, row_scale or None, bias or None, activation,
                                 _stream(stream), path, split)


def sgemm_host(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> int:
    """sgemm on HOST buffers (addresses as int), copies pipelined with the
    computation; asynchronous on `stream` (page-locked buffers overlap)."""
    return load().sgemm_host(_b(transA), _b(transB), M, N, K, alpha, A, lda, B, ldb, beta, C,
                             ldc, _stream(stream))


def sgemm_plan(transA, transB, M, N, K, lda, ldb, ldc, a_aligned=True, b_aligned=True,
               c_aligned=True, path=PATH_AUTO, split=0, num_sms=152):
    """The selector's decision, without a GPU: (status, dict)."""
    outs = [ctypes.c_int(0) for _ in range(6)]
    st = load().sgemm_plan(_b(transA), _b(transB), M, N, K, lda, ldb, ldc, int(a_aligned),
                           int(b_aligned), int(c_aligned), path, split, num_sms,
                           *[ctypes.byref(o) for o in outs])
    keys = ("path", "split", "tile_m", "tile_n", "vector", "ctas")
    return st, {k: o.value for k, o in zip(keys, outs)}


def sgemm_plan_detail(transA, transB, M, N, K, lda, ldb, ldc, a_aligned=True, b_aligned=True,
                      c_aligned=True, path=PATH_AUTO, split=0, num_sms=152):
    """The selector's decision down to the kernel variant, without a GPU:
    (status, dict of sgemm_plan_info's fields)."""
    info = PlanInfo()
    st = load().sgemm_plan_detail(_b(transA), _b(transB), M, N, K, lda, ldb, ldc, int(a_aligned),
                                  int(b_aligned), int(c_aligned), path, split, num_sms,
                                  ctypes.byref(info))
    return st, {name: getattr(info, name) for name, _ in PlanInfo._fields_}


def sgemm_status_string(status: int) -> str:
    return load().sgemm_status_string(status).decode()


def sgemm_device_error(stream=None) -> int:
    return load().sgemm_device_error(_stream(stream))


def sgemm_set_wait_limit(nanoseconds: int) -> int:
    return load().sgemm_set_wait_limit(nanoseconds)


def sgemm_release_workspace() -> int:
    return load().sgemm_release_workspace()


def sgemm_version() -> int:
    return load().sgemm_version()


def sgemm_timing_enable(n: int) -> int:
    """Record event pairs around the main kernel of the next n launches."""
    return load().sgemm_timing_enable(n)


def sgemm_probe_tf32_rate(reps: int = 4096):
    """Measured tcgen05 kind::tf32 rate: (status, multiply-adds per clock per SM)."""
    v = ctypes.c_double(0.0)
    st = load().sgemm_probe_tf32_rate(reps, ctypes.byref(v))
    return st, v.value


def sgemm_launch_count() -> int:
    """Kernels the library has launched in this process (all paths)."""
    return int(load().sgemm_launch_count())


def sgemm_timing_read(capacity: int = 4096):
    """Durations (ms) of the recorded main-kernel launches, oldest first."""
    buf = (ctypes.c_float * max(capacity, 1))()
    n = load().sgemm_timing_read(buf, capacity)
    if n < 0:
        raise SgemmError(-n, "sgemm_timing_read")
    return [float(buf[i]) for i in range(n)]


def sgemm_ffma_static_scratch(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                              stream=None, split=0) -> int:
    """The FFMA path with its split-K scratch in the library's static device
    array: allocates nothing (for callers that may not allocate device
    memory).  Overlapping calls on one device race on that array."""
    return load().sgemm_ffma_static_scratch(_b(transA), _b(transB), M, N, K, alpha, A, lda, B,
                                            ldb, beta, C, ldc, _stream(stream), split)


def gemm(A, B, C, transA="N", transB="N", alpha=1.0, beta=0.0, path=PATH_AUTO, split=0,
         stream=None):
    """Runs the library on torch CUDA tensors (marshalling only).

    A, B, C are 2-D float32 CUDA tensors holding the STORED row-major arrays
    (unit stride along the last dimension; stride(0) is the leading
    dimension).  C is updated in place.  Raises SgemmError on any non-zero
    status.  The call is asynchronous on ``stream`` (default: torch's current
    stream on C's device).
    """
    import torch  # local: only needed for this convenience wrapper

    for name, t in (("A", A), ("B", B), ("C", C)):
        if t.dtype != torch.float32 or not t.is_cuda or t.dim() != 2:
            raise ValueError(f"{name} must be a 2-D float32 CUDA tensor")
        if t.size(1) > 1 and t.stride(1) != 1:
            raise ValueError(f"{name} must have unit stride along its last dimension")
    M, N = C.shape
    K = A.shape[1] if transA.upper() == "N" else A.shape[0]
    if stream is None:
        stream = torch.cuda.current_stream(C.device)
    st = sgemm_ex(transA, transB, M, N, K, alpha, A.data_ptr(), max(A.stride(0), 1),
                  B.data_ptr(), max(B.stride(0), 1), beta, C.data_ptr(), max(C.stride(0), 1),
                  stream, path, split)
    if st != SGEMM_OK:
        raise SgemmError(st)
    return C
