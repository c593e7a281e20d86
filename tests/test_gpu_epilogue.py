"""Parity of the fused epilogue (sgemm_epilogue) with the oracle on every
path and kernel variant:

  C(i,j) = act(alpha * s_i * (op(A) op(B))(i,j) + beta * C(i,j) + bias_j)

FFMA (whole tiles, stream-K with its fixup, and after the transpose
pre-pass), 3xTF32 (operands split in
the kernel, pre-split operands, SM pairs), the thin-problem kernels (both
forms), and the K == 0 / alpha == 0 quick return; exact on small integers,
within the epilogue oracle's bound on random inputs, and bit for bit the
plain call when no epilogue is asked for."""
import zlib

import numpy as np
import pytest

import dense_fp32_gemm_05_gb300 as sg
import gemm_inputs as gi

pytestmark = pytest.mark.gpu

# (name, path, split, transA, transB, M, N, K): each reaches one kernel variant
CASES = [
    ("ffma_small", sg.PATH_FFMA, 1, "N", "N", 300, 260, 200),
    ("ffma_whole", sg.PATH_FFMA, 1, "N", "T", 300, 260, 700),
    ("ffma_stream_k", sg.PATH_FFMA, 0, "T", "N", 256, 256, 1024),
    ("ffma_pre_transpose", sg.PATH_FFMA, 1, "N", "T", 300, 2100, 260),
    ("tc_fused_nn", sg.PATH_3XTF32, 0, "N", "N", 300, 260, 200),
    ("tc_fused_nt", sg.PATH_3XTF32, 0, "N", "T", 200, 136, 300),
    ("tc_pair_tn", sg.PATH_3XTF32, 0, "T", "N", 300, 260, 200),
    ("tc_narrow_tt", sg.PATH_3XTF32, 0, "T", "T", 257, 64, 129),
    ("gemv_dot", sg.PATH_GEMV, 0, "N", "T", 3, 700, 500),
    ("gemv_axpy", sg.PATH_GEMV, 0, "T", "N", 900, 5, 400),
    ("gemv_tensor_core", sg.PATH_GEMV, 0, "N", "N", 16, 1000, 500),
    ("gemv_tensor_core_s24", sg.PATH_AUTO, 0, "T", "N", 24, 4100, 600),
]

EPILOGUES = [
    ("scale", True, False, sg.ACT_NONE),
    ("bias", False, True, sg.ACT_NONE),
    ("relu", False, False, sg.ACT_RELU),
    ("all", True, True, sg.ACT_RELU),
]


def stored(op_mat, trans):
    return np.ascontiguousarray(op_mat if trans == "N" else op_mat.T)


def run_epi(ta, tb, M, N, K, alpha, A, B, beta, C, s, bias, act, path, split):
    import torch
    dev = "cuda"
    dA = torch.from_numpy(A).to(dev) if A is not None else torch.zeros(1, device=dev)
    dB = torch.from_numpy(B).to(dev) if B is not None else torch.zeros(1, device=dev)
    dC = (torch.from_numpy(C).to(dev) if C is not None
          else torch.full((M, N), float("nan"), device=dev))
    ds = torch.from_numpy(s).to(dev) if s is not None else None
    db = torch.from_numpy(bias).to(dev) if bias is not None else None
    lda = A.shape[1] if A is not None else max(1, K if ta == "N" else M)
    ldb = B.shape[1] if B is not None else max(1, N if tb == "N" else K)
    st = sg.sgemm_epilogue(ta, tb, M, N, K, alpha, dA.data_ptr(), lda, dB.data_ptr(), ldb, beta,
                           dC.data_ptr(), N, ds.data_ptr() if ds is not None else 0,
                           db.data_ptr() if db is not None else 0, act,
                           torch.cuda.current_stream(), path, split)
    torch.cuda.synchronize()
    return st, dC.cpu().numpy()


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("epi", EPILOGUES, ids=[e[0] for e in EPILOGUES])
@pytest.mark.parametrize("beta", [0.0, 0.75])
def test_epilogue_within_bound(oracle_mod, case, epi, beta):
    name, path, split, ta, tb, M, N, K = case
    _, use_s, use_b, act = epi
    t = zlib.crc32(f"{name}/{epi[0]}/{beta}".encode()) % 1000
    opA = gi.random_matrix(900 + t, M, K)
    opB = gi.random_matrix(901 + t, K, N)
    C = gi.random_matrix(902 + t, M, N) if beta else None
    rng = np.random.default_rng(t)
    s = rng.uniform(-2, 2, M).astype(np.float32) if use_s else None
    bias = rng.uniform(-3, 3, N).astype(np.float32) if use_b else None
    A, B = stored(opA, ta), stored(opB, tb)
    st, out = run_epi(ta, tb, M, N, K, 1.25, A, B, beta, C, s, bias, act, path, split)
    assert st == 0
    ref, bound = oracle_mod.gemm_epilogue_f64(ta, tb, M, N, K, 1.25, A, A.shape[1], B,
                                              B.shape[1], beta, C, N, row_scale=s, bias=bias,
                                              act=act)
    rep = oracle_mod.compare_bound(out, ref, bound)
    assert rep["pass"], (name, epi[0], rep)
    if act == sg.ACT_RELU:
        assert np.all(out >= 0)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_epilogue_small_integers_exact(case):
    # integers small enough that every path's sum, scaling and bias are exact
    name, path, split, ta, tb, M, N, K = case
    opA = gi.small_ints(21, (M, K))
    opB = gi.small_ints(22, (K, N))
    C = gi.small_ints(23, (M, N))
    rng = np.random.default_rng(24)
    s = rng.integers(-3, 4, M).astype(np.float32)
    bias = rng.integers(-40, 41, N).astype(np.float32)
    want = (2 * s.astype(np.int64)[:, None] * (opA.astype(np.int64) @ opB.astype(np.int64))
            - C.astype(np.int64) + bias.astype(np.int64)[None, :])
    want = np.maximum(want, 0)
    st, out = run_epi(ta, tb, M, N, K, 2.0, stored(opA, ta), stored(opB, tb), -1.0, C, s, bias,
                      sg.ACT_RELU, path, split)
    assert st == 0
    assert np.array_equal(out.astype(np.float64), want.astype(np.float64)), name


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_plain_epilogue_is_sgemm_ex_bit_for_bit(case):
    import torch
    name, path, split, ta, tb, M, N, K = case
    A = stored(gi.random_matrix(31, M, K), ta)
    B = stored(gi.random_matrix(32, K, N), tb)
    C = gi.random_matrix(33, M, N)
    st, out1 = run_epi(ta, tb, M, N, K, -0.5, A, B, 0.5, C, None, None, sg.ACT_NONE, path, split)
    assert st == 0
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (A, B, C))
    st = sg.sgemm_ex(ta, tb, M, N, K, -0.5, dA.data_ptr(), A.shape[1], dB.data_ptr(),
                     B.shape[1], 0.5, dC.data_ptr(), N, torch.cuda.current_stream(), path, split)
    torch.cuda.synchronize()
    assert st == 0
    assert np.array_equal(out1.view(np.uint32), dC.cpu().numpy().view(np.uint32)), name


@pytest.mark.parametrize("beta", [0.0, 0.5, 1.0])
@pytest.mark.parametrize("which", ["k0", "alpha0"])
def test_epilogue_without_a_product_term(beta, which):
    # C = act(fl(beta * C) + bias) exactly (C not read when beta == 0)
    M, N = 37, 45
    C = gi.random_matrix(41, M, N)
    bias = np.linspace(-1, 1, N).astype(np.float32)
    K, alpha = (0, 1.0) if which == "k0" else (13, 0.0)
    A = gi.random_matrix(42, M, max(K, 1)) if K else None
    B = gi.random_matrix(43, max(K, 1), N) if K else None
    st, out = run_epi("N", "N", M, N, K, alpha, A, B, beta, C if beta else None,
                      np.full(M, 3.0, np.float32), bias, sg.ACT_RELU, sg.PATH_AUTO, 0)
    assert st == 0
    bc = (np.float32(beta) * C) if beta else np.zeros((M, N), np.float32)
    want = np.maximum((bc + bias[None, :]).astype(np.float32), np.float32(0))
    assert np.array_equal(out, want)


def test_epilogue_rejects_an_unknown_activation():
    import torch
    x = torch.zeros(16, device="cuda")
    st = sg.sgemm_epilogue("N", "N", 4, 4, 4, 1.0, x.data_ptr(), 4, x.data_ptr(), 4, 0.0,
                           x.data_ptr(), 4, 0, 0, 7, torch.cuda.current_stream())
    assert st == -16
