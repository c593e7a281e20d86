"""sgemm_host: the GEMM on host buffers with the copies pipelined against the
computation in K-chunks and row blocks.  Checked against the oracle (within
the fp32 bound) for every layout, beta != 0, odd leading dimensions,
page-locked and pageable buffers, shapes that make one, several and ragged
row blocks, K long enough for 2 to 4 chunks (each chunk after the first
adds into C with beta = 1; the last chunk may be shorter), and the two-phase
form (beta = 0 and M >= 4096: the top rows of C computed and sent home while
the bottom rows' operands still arrive)."""
import numpy as np
import pytest

import dense_fp32_gemm_05_gb300 as sg
import gemm_inputs as gi

pytestmark = pytest.mark.gpu

LAYOUTS = [("N", "N"), ("N", "T"), ("T", "N"), ("T", "T")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from dense_fp32_gemm_05_gb300 import build
    build.build()
    sg.load()


def stored(op_mat, trans, pad):
    base = op_mat if trans == "N" else op_mat.T
    out = np.full((base.shape[0], base.shape[1] + pad), np.nan, np.float32)
    out[:, : base.shape[1]] = base
    return out


@pytest.mark.parametrize("ta,tb", LAYOUTS)
@pytest.mark.parametrize("M,N,K,alpha,beta,pad,pinned", [
    (300, 260, 200, 1.0, 0.0, 0, True),          # one row block, small: FFMA
    (2100, 520, 700, 1.5, 0.5, 3, True),         # four ragged row blocks, 3xTF32
    (1537, 1025, 333, -1.0, 1.0, 1, False),      # pageable buffers
    # K in chunks, each chunk's GEMM adding into C (beta = 1 after the first):
    (2100, 520, 2050, 1.0, 0.5, 3, True),        # 4 chunks of 544, 544, 544, 418
    (1537, 1025, 1500, -1.0, 1.0, 1, False),     # 2 chunks (768, 732), pageable
    (700, 300, 1024, 1.0, 0.0, 0, True),         # 2 equal chunks, beta = 0 over NaN
    # two row phases (beta = 0, M >= 4096): top rows, then bottom rows in
    # 2 chunks whose last runs in 2 row blocks
    (4100, 130, 1100, -1.0, 0.0, 2, True),       # first phase 2 chunks (544, 544 + 12)
    (4097, 64, 2050, 1.0, 0.0, 0, False),        # 4 chunks then 2, pageable
])
def test_host_api_matches_oracle(oracle_mod, ta, tb, M, N, K, alpha, beta, pad, pinned):
    import torch

    opA = gi.random_matrix(61, M, K)
    opB = gi.random_matrix(62, K, N)
    C0 = gi.random_matrix(63, M, N)
    A, B = stored(opA, ta, pad), stored(opB, tb, pad)
    ldc = N + pad
    Cs = np.full((M, ldc), np.nan, np.float32)
    Cs[:, :N] = C0 if beta != 0 else np.nan
    if pinned:
        tA = torch.from_numpy(A).pin_memory()
        tB = torch.from_numpy(B).pin_memory()
        tC = torch.from_numpy(Cs).pin_memory()
        pa, pb, pc = tA.data_ptr(), tB.data_ptr(), tC.data_ptr()
        read = lambda: tC.numpy()
    else:
        pa, pb, pc = A.ctypes.data, B.ctypes.data, Cs.ctypes.data
        read = lambda: Cs
    s = torch.cuda.current_stream()
    st = sg.sgemm_host(ta, tb, M, N, K, alpha, pa, A.shape[1], pb, B.shape[1], beta, pc, ldc, s)
    assert st == 0, sg.sgemm_status_string(st)
    torch.cuda.synchronize()
    out = read()
    assert np.all(np.isnan(out[:, N:])), "the ld gap of C was written"
    Ap = A[:, : (K if ta == "N" else M)].copy()
    Bp = B[:, : (N if tb == "N" else K)].copy()
    ref, bound = oracle_mod.gemm_f64(ta, tb, M, N, K, alpha, Ap, Ap.shape[1], Bp, Bp.shape[1],
                                     beta, C0, N)
    rep = oracle_mod.compare(out[:, :N], ref, bound, K, alpha)
    assert rep["pass"], rep


def test_host_api_quick_returns(oracle_mod):
    import torch
    M, N, K = 700, 300, 50
    C0 = gi.random_matrix(64, M, N)
    # alpha == 0: C = beta * C, A and B never read (null host pointers)
    Cs = C0.copy()
    st = sg.sgemm_host("N", "N", M, N, K, 0.0, 0, K, 0, N, 0.5, Cs.ctypes.data, N,
                       torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert st == 0 and np.array_equal(Cs, np.float32(0.5) * C0)
    # M == 0: nothing
    assert sg.sgemm_host("N", "N", 0, N, K, 1.0, 0, K, 0, N, 0.0, 0, N, None) == 0
    # argument errors as sgemm
    assert sg.sgemm_host("X", "N", M, N, K, 1.0, 8, K, 8, N, 0.0, 8, N, None) == -1
