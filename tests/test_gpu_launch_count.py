"""The library's launch counter (sgemm_launch_count) against the kernels each
path launches: the benchmark reports its gpu_launches from it.  Results are
not checked here (the parity tests do that); only the counts."""
import pytest

import dense_fp32_gemm_05_gb300 as sg

pytestmark = pytest.mark.gpu


def _launches(ta, tb, M, N, K, path=sg.PATH_AUTO, split=0, alpha=1.0, beta=0.0):
    import torch
    A = torch.rand((M, K) if ta == "N" else (K, M), device="cuda")
    B = torch.rand((K, N) if tb == "N" else (N, K), device="cuda")
    C = torch.rand(max(M, 1), max(N, 1), device="cuda")
    s = torch.cuda.current_stream()
    c0 = sg.sgemm_launch_count()
    st = sg.sgemm_ex(ta, tb, M, N, K, alpha, A.data_ptr(), max(A.shape[1], 1), B.data_ptr(),
                     max(B.shape[1], 1), beta, C.data_ptr(), max(N, 1), s, path, split)
    torch.cuda.synchronize()
    assert st == 0 and sg.sgemm_device_error(s) == 0
    return sg.sgemm_launch_count() - c0


def test_ffma_counts():
    # whole tiles: one kernel; shared K ranges: the kernel and its fixup
    assert _launches("N", "N", 256, 256, 256, sg.PATH_FFMA, 1) == 1
    assert _launches("N", "N", 256, 256, 256, sg.PATH_FFMA, 4) == 2
    # a K-contiguous operand of a large grid: the transpose pre-pass, then the kernel
    assert _launches("N", "N", 300, 2100, 260, sg.PATH_FFMA, 1) == 2


def test_tensor_core_counts():
    # 4096^3 NN: split pre-pass, SM-pair kernel, fixup of the shared last wave
    st, p = sg.sgemm_plan("N", "N", 4096, 4096, 4096, 4096, 4096, 4096, num_sms=152)
    assert st == 0 and p["path"] == sg.PATH_3XTF32 and p["split"] == 3
    assert _launches("N", "N", 4096, 4096, 4096) == 3
    # forced whole tiles (no stream-K): pre-pass and main kernel
    assert _launches("N", "N", 1024, 1024, 1024, sg.PATH_3XTF32, 1) == 2
    # A split inside the kernel and B split in shared memory: one kernel
    assert _launches("N", "T", 512, 512, 512, sg.PATH_3XTF32, 1) == 1


def test_quick_returns_and_thin_problems():
    assert _launches("N", "N", 64, 64, 0, beta=0.5) == 1     # C = beta*C
    assert _launches("N", "N", 64, 64, 64, alpha=0.0) == 1   # C = beta*C
    assert _launches("N", "N", 0, 64, 64) == 0               # nothing to do
    # thin: one pass over the large operand, plus the K-split sum when K is cut
    assert _launches("N", "T", 1, 4096, 4096) == 1
    n = _launches("N", "N", 8, 16384, 8192)
    assert n in (1, 2)
    # S = 16 on the tensor cores: the split of the small operand and the kernel
    assert _launches("N", "N", 16, 16384, 8192) == 2
    # and S = 32, 64 and 128 the same way
    assert _launches("N", "N", 32, 16384, 8192) == 2
    assert _launches("N", "N", 64, 16384, 8192) == 2
    assert _launches("N", "N", 128, 16384, 8192) == 2
