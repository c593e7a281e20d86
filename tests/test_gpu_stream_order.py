"""Back-to-back calls on one stream with no synchronisation in between, each
reading what the previous call wrote: its C as the next call's A, or the
same C accumulated again with beta = 1.  A call's later kernels (the main
kernel after the split pre-pass, the stream-K fixup, the K-split sum) are
launched as programmatic dependents and wait for their predecessor inside
the kernel; these tests check that every call still sees all of the
previous call's output, its fixup included.  Each result is checked against
the oracle applied to the GPU's own input for that step."""
import numpy as np
import pytest

import dense_fp32_gemm_05_gb300 as sg
import gemm_inputs as gi

pytestmark = pytest.mark.gpu

# (id, path, split, transA, transB, M, n): X_{i+1} = op(X_i) W, X_i stored M x n
# (n x n when transA = 'T'), W n x n
CHAINS = [
    # split pre-pass of both operands, main kernel, stream-K fixup
    ("3xtf32_prepass_fixup", sg.PATH_3XTF32, 4, "T", "N", 512, 512),
    # both operands split inside the kernel, stream-K fixup
    ("3xtf32_fused_fixup", sg.PATH_3XTF32, 4, "N", "T", 512, 512),
    # the selector's own plan for a mid-size square
    ("auto", sg.PATH_AUTO, 0, "N", "N", 1024, 1024),
    # FFMA tiles shared across CTAs, fixup
    ("ffma_fixup", sg.PATH_FFMA, 4, "N", "N", 256, 256),
    # thin: axpy form with the K-split sum
    ("gemv_ksplit", sg.PATH_AUTO, 0, "N", "N", 16, 4096),
]
STEPS = 5


@pytest.mark.parametrize("cid,path,split,ta,tb,M,n", CHAINS, ids=[c[0] for c in CHAINS])
def test_chained_calls_see_previous_output(oracle_mod, cid, path, split, ta, tb, M, n):
    import torch
    if ta == "T":
        assert M == n
    x0 = gi.random_matrix(11, M, n)
    # U[-1, 1] * sqrt(3 / n): unit variance in, unit variance out
    w = (gi.random_matrix(12, n, n) * np.float32(np.sqrt(3.0 / n))).astype(np.float32)
    if tb == "T":
        w = np.ascontiguousarray(w.T)
    s = torch.cuda.current_stream()
    dW = torch.from_numpy(w).cuda()
    xs = [torch.from_numpy(x0).cuda()] + [torch.full((M, n), float("nan"), device="cuda")
                                           for _ in range(STEPS)]
    torch.cuda.synchronize()
    for i in range(STEPS):
        st = sg.sgemm_ex(ta, tb, M, n, n, 1.0, xs[i].data_ptr(), n, dW.data_ptr(), n, 0.0,
                         xs[i + 1].data_ptr(), n, s, path, split)
        assert st == 0, (cid, i, st)
    torch.cuda.synchronize()
    assert sg.sgemm_device_error(s) == 0
    host = [x.cpu().numpy() for x in xs]
    for i in range(STEPS):
        ref, bound = oracle_mod.gemm_f64(ta, tb, M, n, n, 1.0, host[i], n, w, n, 0.0, None, n)
        rep = oracle_mod.compare(host[i + 1], ref, bound, n, 1.0)
        assert rep["pass"], (cid, i, rep)


ACCUM = [
    ("3xtf32_fixup", sg.PATH_3XTF32, 4, 512, 384, 640),
    ("ffma_fixup", sg.PATH_FFMA, 4, 256, 256, 512),
    ("auto_sq1024", sg.PATH_AUTO, 0, 1024, 1024, 1024),
]


@pytest.mark.parametrize("cid,path,split,M,N,K", ACCUM, ids=[c[0] for c in ACCUM])
def test_repeated_accumulation_into_one_c(oracle_mod, cid, path, split, M, N, K):
    """C <- A B + C five times on the same C, back to back: every call's
    epilogue reads the C that the previous call's last kernel wrote.  Each of
    the 5 calls adds at most 4K 2^-24 (|A||B| + |C_i|) with
    |C_i| <= |C_0| + i |A||B|, in all at most 5 times the single-call bound
    of alpha = 5, beta = 1.  A stale read would be off by a whole |AB|."""
    import torch
    A = gi.random_matrix(21, M, K)
    B = gi.random_matrix(22, K, N)
    C0 = gi.random_matrix(23, M, N)
    s = torch.cuda.current_stream()
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (A, B, C0))
    torch.cuda.synchronize()
    for i in range(5):
        st = sg.sgemm_ex("N", "N", M, N, K, 1.0, dA.data_ptr(), K, dB.data_ptr(), N, 1.0,
                         dC.data_ptr(), N, s, path, split)
        assert st == 0, (cid, i, st)
    torch.cuda.synchronize()
    assert sg.sgemm_device_error(s) == 0
    ref, bound = oracle_mod.gemm_f64("N", "N", M, N, K, 5.0, A, K, B, N, 1.0, C0, N)
    err = np.abs(dC.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= 5.0 * bound), (cid, float((err / np.maximum(bound, 1e-300)).max()))
