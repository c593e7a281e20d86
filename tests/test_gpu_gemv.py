"""Parity of the thin-problem path (SGEMM_PATH_GEMV, min(M, N) <= 16) with the
oracle: exact on small integers, within the fp32 bound on random inputs over
both forms of the kernel (the large operand contiguous along K, or along
the long dimension), both thin sides (few rows of C, few columns), ragged K
and ragged long dimensions, padded leading dimensions and misaligned base
pointers, and the K split across CTAs with its ordered reduction."""
import itertools

import numpy as np
import pytest

import dense_fp32_gemm_05_gb300 as sg
import gemm_inputs as gi
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu

LAYOUTS = [("N", "N"), ("N", "T"), ("T", "N"), ("T", "T")]


def stored(op_mat, trans):
    return np.ascontiguousarray(op_mat if trans == "N" else op_mat.T)


def embed_ld(arr, pad):
    out = np.full((arr.shape[0], arr.shape[1] + pad), np.nan, np.float32)
    out[:, : arr.shape[1]] = arr
    return out


@pytest.mark.parametrize("ta,tb", LAYOUTS)
@pytest.mark.parametrize("thin", ["rows", "cols"])
@pytest.mark.parametrize("S", [1, 3, 16])
@pytest.mark.parametrize("misalign", [False, True])
def test_gemv_small_integers_exact(ta, tb, thin, S, misalign):
    # |partial sums| < 2^24: every summation order gives the exact integer
    P, K = 517, 1031
    M, N = (S, P) if thin == "rows" else (P, S)
    opA = gi.small_ints(11, (M, K))
    opB = gi.small_ints(12, (K, N))
    C = gi.small_ints(13, (M, N))
    want = 2.0 * (opA.astype(np.int64) @ opB.astype(np.int64)) - 1.0 * C.astype(np.int64)
    A, B = stored(opA, ta), stored(opB, tb)
    off = (1, 3, 1) if misalign else (0, 0, 0)
    st, out = gh.run(ta, tb, M, N, K, 2.0, A, A.shape[1], B, B.shape[1], -1.0, C, N,
                     path=sg.PATH_GEMV, offsets=off)
    assert st == 0
    assert np.array_equal(out.astype(np.float64), want.astype(np.float64))


def _cases():
    rng = np.random.default_rng(23)
    S_vals = [1, 2, 5, 8, 9, 15, 16]
    P_vals = [1, 7, 129, 1000, 4097]
    K_vals = [1, 3, 64, 300, 2049, 20000]
    combos = list(itertools.product(S_vals, P_vals, K_vals))
    picks = rng.choice(len(combos), size=36, replace=False)
    out = []
    for t, i in enumerate(picks):
        S, P, K = combos[i]
        ta, tb = LAYOUTS[t % 4]
        thin = "rows" if (t // 4) % 2 == 0 else "cols"
        out.append((t, S, P, K, ta, tb, thin))
    # the K split across CTAs (long K, few blocks of the long dimension)
    out.append((99, 4, 300, 40000, "N", "N", "rows"))
    out.append((98, 2, 200, 30000, "T", "N", "cols"))
    return out


@pytest.mark.parametrize("t,S,P,K,ta,tb,thin", _cases())
def test_gemv_random_within_bound(oracle_mod, t, S, P, K, ta, tb, thin):
    M, N = (S, P) if thin == "rows" else (P, S)
    opA = gi.random_matrix(600 + t, M, K)
    opB = gi.random_matrix(700 + t, K, N)
    C = gi.random_matrix(800 + t, M, N)
    alpha, beta = [(1.0, 0.0), (-1.5, 0.5), (0.75, 1.0), (2.0, -1.0)][t % 4]
    A, B = stored(opA, ta), stored(opB, tb)
    pad = (t % 3, (t + 1) % 3)
    A, B = embed_ld(A, pad[0]), embed_ld(B, pad[1])
    ldc = N + t % 2
    Cpad = embed_ld(C, ldc - N)
    st, out = gh.run(ta, tb, M, N, K, alpha, A, A.shape[1], B, B.shape[1], beta,
                     C if beta else None, ldc, path=sg.PATH_GEMV,
                     offsets=(t % 2, (t // 2) % 2, 0))
    assert st == 0, (M, N, K)
    ref, bound = oracle_mod.gemm_f64(ta, tb, M, N, K, alpha, A, A.shape[1], B, B.shape[1],
                                     beta, Cpad if beta else None, ldc)
    rep = oracle_mod.compare(out, ref, bound, K, alpha)
    assert rep["pass"], rep


@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_gemv_is_the_selectors_choice(ta, tb):
    # min(M, N) <= 4: sgemm() (AUTO) runs this path in every layout, bit for
    # bit (from 5 up, a K-contiguous large operand goes to the tensor cores)
    M, N, K = 4, 3000, 777
    A = stored(gi.random_matrix(31, M, K), ta)
    B = stored(gi.random_matrix(32, K, N), tb)
    st1, out1 = gh.run(ta, tb, M, N, K, 1.0, A, A.shape[1], B, B.shape[1], 0.0, None, N,
                       path=sg.PATH_GEMV)
    st2, out2 = gh.run(ta, tb, M, N, K, 1.0, A, A.shape[1], B, B.shape[1], 0.0, None, N,
                       path=sg.PATH_AUTO)
    assert st1 == 0 and st2 == 0
    assert np.array_equal(out1.view(np.uint32), out2.view(np.uint32))


def test_gemv_special_cases(oracle_mod):
    # beta = 0 never reads C (NaN stays out); K = 0 and alpha = 0 scale C
    M, N, K = 1, 900, 500
    A = gi.random_matrix(41, M, K)
    B = gi.random_matrix(42, K, N)
    st, out = gh.run("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, None, N, path=sg.PATH_GEMV)
    assert st == 0 and np.all(np.isfinite(out))
    C = gi.random_matrix(43, M, N)
    st, out = gh.run("N", "N", M, N, 0, 1.0, None, 1, None, N, 0.5, C, N, path=sg.PATH_GEMV)
    assert st == 0 and np.array_equal(out, (np.float32(0.5) * C).astype(np.float32))
    st, out = gh.run("N", "N", M, N, K, 0.0, A, K, B, N, -2.0, C, N, path=sg.PATH_GEMV)
    assert st == 0 and np.array_equal(out, (np.float32(-2.0) * C).astype(np.float32))


def test_gemv_forced_on_a_wide_problem_is_refused():
    import torch
    x = torch.zeros(129 * 129, device="cuda")
    st = sg.sgemm_ex("N", "N", 129, 129, 129, 1.0, x.data_ptr(), 129, x.data_ptr(), 129, 0.0,
                     x.data_ptr(), 129, torch.cuda.current_stream(), sg.PATH_GEMV, 0)
    assert st == sg.SGEMM_ERR_UNSUPPORTED


@pytest.mark.parametrize("M", [8, 16])
def test_staged_timeout_reports_and_recovers(oracle_mod, M):
    """The thin-problem kernels that stage the large operand (K x N
    row-major) through shared memory with TMA: on the CUDA cores at S = 8, on
    the tensor cores at S = 16.  A 1 ns wait limit makes their bounded waits
    run out; the call raises SGEMM_ERR_TIMEOUT through the device error word
    and the next call computes the right result.  The limit is a suspend hint
    of mbarrier.try_wait, so the waits must meet real memory latency: the
    large operand (256 MB) is larger than L2, and L2 is flushed before the
    call (with the operand resident in L2 every copy could land in time)."""
    import torch
    N, K = 8192, 8192
    A = gi.random_matrix(61, M, K)
    B = gi.random_matrix(62, K, N)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.zeros((M, N), device="cuda")
    s = torch.cuda.current_stream()
    assert sg.sgemm_device_error(s) == 0
    flush = torch.empty(64 << 20, device="cuda")
    flush.fill_(1.0)
    assert sg.sgemm_set_wait_limit(1) == 0
    try:
        st = sg.sgemm_ex("N", "N", M, N, K, 1.0, dA.data_ptr(), K, dB.data_ptr(), N, 0.0,
                         dC.data_ptr(), N, s, sg.PATH_GEMV, 0)
        assert st == 0
        assert sg.sgemm_device_error(s) == sg.SGEMM_ERR_TIMEOUT
        assert sg.sgemm_device_error(s) == 0          # read-and-clear
    finally:
        sg.sgemm_set_wait_limit(0)
    st = sg.sgemm_ex("N", "N", M, N, K, 1.0, dA.data_ptr(), K, dB.data_ptr(), N, 0.0,
                     dC.data_ptr(), N, s, sg.PATH_GEMV, 0)
    assert st == 0 and sg.sgemm_device_error(s) == 0
    ref, bound = oracle_mod.gemm_f64("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, None, N)
    assert oracle_mod.compare(dC.cpu().numpy(), ref, bound, K, 1.0)["pass"]


# The tensor-core form of the thin path (S >= 12 and the large operand's rows
# along the long dimension, 16-byte aligned): 3xTF32 on tcgen05, K split into
# ranges of multiples of 32 with the partial sums added by the sum kernel.
TC_THIN = [
    # (S, P, K, thin side, alpha, beta); P % 4 == 0: the large operand's rows
    # (P floats) start 16-byte aligned, as the tensor-core form needs
    (12, 1000, 777, "rows", 1.0, 0.0),
    (13, 132, 31, "cols", -1.5, 0.5),        # ragged P tile, K below one block
    (16, 16384, 2049, "rows", 0.75, 1.0),
    (16, 300, 40000, "rows", 1.0, 0.0),      # K split across 50 CTAs
    (15, 4100, 9000, "cols", 2.0, -1.0),
    # 16 < S <= 128: the same kernel, Small's hi and lo filling a 64-, 128- or
    # 256-row operand
    (17, 1000, 777, "rows", 1.0, 0.0),
    (24, 4100, 3000, "cols", -0.5, 0.25),     # ragged P tile
    (32, 2048, 20000, "rows", 1.0, 1.0),      # K split across CTAs
    (29, 16384, 33, "rows", 1.5, 0.0),        # K one block and a bit
    (33, 1000, 777, "rows", 1.0, 0.0),
    (48, 4100, 3000, "cols", -0.5, 0.25),     # ragged P tile
    (64, 2048, 20000, "rows", 1.0, 1.0),      # K split across CTAs
    (65, 1000, 777, "rows", 1.0, 0.0),
    (100, 4100, 3000, "cols", -0.5, 0.25),    # ragged P tile
    (128, 2048, 20000, "rows", 1.0, 1.0),     # K split across CTAs
]


@pytest.mark.parametrize("S,P,K,thin,alpha,beta", TC_THIN)
def test_thin_tensor_core_within_bound(oracle_mod, S, P, K, thin, alpha, beta):
    import torch
    M, N = (S, P) if thin == "rows" else (P, S)
    ta, tb = ("N", "N") if thin == "rows" else ("T", "N")   # the large operand along P
    opA = gi.random_matrix(900 + S, M, K, dist="normal")
    opB = gi.random_matrix(901 + S, K, N, dist="normal")
    C = gi.random_matrix(902 + S, M, N)
    A, B = stored(opA, ta), stored(opB, tb)
    c0 = sg.sgemm_launch_count()
    st, out = gh.run(ta, tb, M, N, K, alpha, A, A.shape[1], B, B.shape[1], beta,
                     C if beta else None, N, path=sg.PATH_AUTO)
    assert st == 0
    # the split of the small operand, the tensor-core kernel, and the sum when K is split
    assert sg.sgemm_launch_count() - c0 in (2, 3)
    lda, ldb = A.shape[1], B.shape[1]
    st, d = sg.sgemm_plan_detail(ta, tb, M, N, K, lda, ldb, N)
    assert st == 0 and d["path"] == sg.PATH_GEMV and d["tile_n"] == 128 and d["accumulators"] == 8
    ref, bound = oracle_mod.gemm_f64(ta, tb, M, N, K, alpha, A, A.shape[1], B, B.shape[1], beta,
                                     C if beta else None, N)
    rep = oracle_mod.compare(out, ref, bound, K, alpha)
    assert rep["pass"], rep
    # 3xTF32, not single-pass TF32: well inside the fp32 bound at this K
    assert rep["max_err_over_bound"] < 0.05, rep
