"""Parity of the CUDA paths with the CPU oracle, through the C-ABI.

Floating-point rule (the tolerance of the method): every entry must satisfy
|C - C_ref| <= 4*K*2^-24*(|alpha|*(|A||B|)_ij + |beta|*|C_ij|), with C_ref and
the bound from the fp64 oracle.  Exact cases (all-ones, identity,
permutation, small integers) must match exactly, and the FFMA path without
split-K must equal the oracle's fp32 ascending-k FMA evaluation bit for bit.
Every run is guard-banded (tests/gpu_harness.py): nothing outside C's M x N
window may change.
"""
import itertools

import numpy as np
import pytest

import dense_fp32_gemm_05_gb300 as sg
import gemm_inputs as gi
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu

LAYOUTS = [("N", "N"), ("N", "T"), ("T", "N"), ("T", "T")]
ACCURATE_PATHS = [sg.PATH_FFMA, sg.PATH_3XTF32]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from dense_fp32_gemm_05_gb300 import build
    build.build()
    sg.load()


def stored(op_mat, trans):
    return np.ascontiguousarray(op_mat if trans == "N" else op_mat.T)


def ld_of(arr, pad=0):
    return max(arr.shape[1] + pad, 1)


def oracle_check(orc, ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C, out, points=None):
    ref, bound = orc.gemm_f64(ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C, N, points=points)
    cand = out if points is None else out[points]
    rep = orc.compare(cand, ref, bound, K, alpha)
    assert rep["pass"], rep
    return rep


def pad_cols(arr, ld):
    out = np.full((arr.shape[0], ld), np.nan, np.float32)
    out[:, : arr.shape[1]] = arr
    return out


# ------------------------------------------------------------ exact pins
@pytest.mark.parametrize("path", ACCURATE_PATHS)
@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_all_ones_exact(path, ta, tb):
    M, N, K = 300, 260, 1000
    A = np.ones((M, K) if ta == "N" else (K, M), np.float32)
    B = np.ones((K, N) if tb == "N" else (N, K), np.float32)
    st, out = gh.run(ta, tb, M, N, K, 1.0, A, ld_of(A), B, ld_of(B), 0.0, None, N, path=path)
    assert st == 0
    assert np.all(out == np.float32(K))
    C = np.full((M, N), 3.0, np.float32)
    st, out = gh.run(ta, tb, M, N, K, 2.0, A, ld_of(A), B, ld_of(B), -0.5, C, N, path=path)
    assert st == 0 and np.all(out == np.float32(2 * K - 1.5))


def same_or_split_exact(out, want, path):
    """FFMA: bit-exact.  3xTF32: x*1 is computed as hi(x) + lo(x), which drops
    the part of x below the 22nd significant bit: |out - x| <= 2^-22 |x|."""
    if path == sg.PATH_FFMA:
        return np.array_equal(out, want)
    return bool(np.all(np.abs(out.astype(np.float64) - want) <= 2.0 ** -22 * np.abs(want)))


@pytest.mark.parametrize("path", ACCURATE_PATHS)
@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_identity_and_permutation_exact(path, ta, tb):
    rng = np.random.default_rng(5)
    M, N = 200, 136
    X = gi.random_matrix(7, M, N)
    eye = np.eye(M, dtype=np.float32)
    st, out = gh.run(ta, tb, M, N, M, 1.0, stored(eye, ta), M, stored(X, tb), ld_of(stored(X, tb)),
                     0.0, None, N, path=path)
    assert st == 0 and same_or_split_exact(out, X, path)
    perm = rng.permutation(M)
    P = np.zeros((M, M), np.float32)
    P[np.arange(M), perm] = 1.0
    st, out = gh.run(ta, tb, M, N, M, 1.0, stored(P, ta), M, stored(X, tb), ld_of(stored(X, tb)),
                     0.0, None, N, path=path)
    assert st == 0 and same_or_split_exact(out, X[perm], path)
    sigma = rng.permutation(N)
    Q = np.zeros((N, N), np.float32)
    Q[sigma, np.arange(N)] = 1.0
    st, out = gh.run(ta, tb, M, N, N, 1.0, stored(X, ta), ld_of(stored(X, ta)), stored(Q, tb), N,
                     0.0, None, N, path=path)
    assert st == 0 and same_or_split_exact(out, X[:, sigma], path)


RANK1_SHAPES = [(300, 260, 200), (1000, 900, 700)]   # small-problem kernel / tile kernels


@pytest.mark.parametrize("path", ACCURATE_PATHS)
@pytest.mark.parametrize("ta,tb", LAYOUTS)
@pytest.mark.parametrize("M,N,K", RANK1_SHAPES)
def test_rank_one_closed_form_exact(path, ta, tb, M, N, K):
    """A(i, k) = u_i, B(k, j) = v_j with small integers: C(i, j) = K u_i v_j,
    exact in fp32 (every partial sum is an integer below 2^24) and in TF32
    (integers below 2^11 have no lo part)."""
    rng = np.random.default_rng(17)
    u = rng.integers(-8, 9, M).astype(np.float32)
    v = rng.integers(-8, 9, N).astype(np.float32)
    opA = np.repeat(u[:, None], K, axis=1)
    opB = np.repeat(v[None, :], K, axis=0)
    st, out = gh.run(ta, tb, M, N, K, 1.0, stored(opA, ta), ld_of(stored(opA, ta)), stored(opB, tb),
                     ld_of(stored(opB, tb)), 0.0, None, N, path=path)
    assert st == 0
    want = (K * np.outer(u.astype(np.int64), v.astype(np.int64))).astype(np.float64)
    assert np.array_equal(out.astype(np.float64), want)


FLIP = {"N": "T", "T": "N"}


@pytest.mark.parametrize("path,split", [(sg.PATH_FFMA, 1), (sg.PATH_3XTF32, 0)])
@pytest.mark.parametrize("ta,tb", LAYOUTS)
@pytest.mark.parametrize("M,N,K", [(300, 260, 200), (1000, 900, 700)])
def test_transpose_symmetry(oracle_mod, path, split, ta, tb, M, N, K):
    """(op(A) op(B))^T = op(B)^T op(A)^T: the same stored arrays through the
    swapped, flag-flipped call give C^T.  FFMA without a split sums every
    output in ascending k on both sides (and a*b = b*a), so the two agree bit
    for bit; 3xTF32 runs other tiles on the swapped problem and is held to
    the bound."""
    opA = gi.random_matrix(41, M, K, dist="normal")
    opB = gi.random_matrix(42, K, N, dist="normal")
    A, B = stored(opA, ta), stored(opB, tb)
    st, c1 = gh.run(ta, tb, M, N, K, 1.0, A, ld_of(A), B, ld_of(B), 0.0, None, N, path=path,
                    split=split)
    assert st == 0
    # op(B)^T is B read with the flipped flag, and likewise A
    st, c2 = gh.run(FLIP[tb], FLIP[ta], N, M, K, 1.0, B, ld_of(B), A, ld_of(A), 0.0, None, M,
                    path=path, split=split)
    assert st == 0
    if path == sg.PATH_FFMA:
        assert np.array_equal(c2.T.view(np.uint32), c1.view(np.uint32))
    else:
        oracle_check(oracle_mod, FLIP[tb], FLIP[ta], N, M, K, 1.0, B, ld_of(B), A, ld_of(A), 0.0,
                     None, c2)


@pytest.mark.parametrize("path", ACCURATE_PATHS)
@pytest.mark.parametrize("ta,tb", LAYOUTS)
@pytest.mark.parametrize("misalign", [False, True])
def test_small_integers_exact(path, ta, tb, misalign):
    M, N, K = 257, 129, 145
    opA = gi.small_ints(1, (M, K))
    opB = gi.small_ints(2, (K, N))
    C = gi.small_ints(3, (M, N))
    want = 2.0 * (opA.astype(np.int64) @ opB.astype(np.int64)) - 1.0 * C.astype(np.int64)
    A, B = stored(opA, ta), stored(opB, tb)
    off = (1, 3, 1) if misalign else (0, 0, 0)
    st, out = gh.run(ta, tb, M, N, K, 2.0, A, ld_of(A), B, ld_of(B), -1.0, C, N, path=path,
                     offsets=off)
    assert st == 0
    assert np.array_equal(out.astype(np.float64), want.astype(np.float64))


# ------------------------------------------------------------ bitwise (FFMA)
@pytest.mark.parametrize("ta,tb", LAYOUTS)
@pytest.mark.parametrize("M,N,K,alpha,beta,pad,off", [
    (300, 260, 200, 1.0, 0.0, (0, 0, 0), (0, 0, 0)),
    (129, 131, 1000, -1.5, 0.5, (3, 1, 2), (0, 0, 0)),
    (256, 128, 64, 1.0, 1.0, (0, 0, 0), (0, 0, 0)),
    (77, 300, 33, 0.75, -2.0, (1, 0, 5), (1, 2, 3)),
    (520, 300, 700, 1.0, 0.5, (2, 3, 1), (3, 1, 2)),
])
def test_ffma_bitwise_equals_sequential_oracle(oracle_mod, ta, tb, M, N, K, alpha, beta, pad, off):
    opA = gi.random_matrix(11, M, K, dist="normal")
    opB = gi.random_matrix(12, K, N, dist="normal")
    C = gi.random_matrix(13, M, N)
    A, B = stored(opA, ta), stored(opB, tb)
    lda, ldb, ldc = ld_of(A, pad[0]), ld_of(B, pad[1]), N + pad[2]
    st, out = gh.run(ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C if beta else None, ldc,
                     path=sg.PATH_FFMA, split=1, offsets=off)
    assert st == 0
    want = oracle_mod.gemm_f32_seq(ta, tb, M, N, K, alpha, pad_cols(A, lda), lda,
                                   pad_cols(B, ldb), ldb, beta, C, N)
    assert np.array_equal(out.view(np.uint32), want.view(np.uint32))
    oracle_check(oracle_mod, ta, tb, M, N, K, alpha, A, A.shape[1], B, B.shape[1], beta, C, out)


def test_ffma_hand_worked_order_cases():
    """The hand-worked fp32 cases of the oracle pins, on the GPU: ascending
    k with fused multiply-adds (row [1, 2^24, -2^24] sums to 0, not 1)."""
    a = np.array([[1.0, 2.0 ** 24, -(2.0 ** 24)]], np.float32)
    b = np.ones((3, 1), np.float32)
    st, out = gh.run("N", "N", 1, 1, 3, 1.0, a, 3, b, 1, 0.0, None, 1, split=1)
    assert st == 0 and out[0, 0] == 0.0
    x = np.float32(1.0 + 2.0 ** -12)
    a = np.array([[-1.0, x]], np.float32)
    b = np.array([[1.0], [x]], np.float32)
    st, out = gh.run("N", "N", 1, 1, 2, 1.0, a, 2, b, 1, 0.0, None, 1, split=1)
    assert st == 0 and out[0, 0] == np.float32(2.0 ** -11 + 2.0 ** -24)


# ------------------------------------------------------------ within the bound
@pytest.mark.parametrize("ta,tb", LAYOUTS)
@pytest.mark.parametrize("split", [0, 2, 3, 7])
def test_split_k_within_bound(oracle_mod, ta, tb, split):
    M, N, K = 200, 330, 1500
    opA = gi.random_matrix(21, M, K)
    opB = gi.random_matrix(22, K, N)
    C = gi.random_matrix(23, M, N)
    A, B = stored(opA, ta), stored(opB, tb)
    st, out = gh.run(ta, tb, M, N, K, 1.0, A, ld_of(A), B, ld_of(B), 0.5, C, N,
                     path=sg.PATH_FFMA, split=split)
    assert st == 0
    oracle_check(oracle_mod, ta, tb, M, N, K, 1.0, A, A.shape[1], B, B.shape[1], 0.5, C, out)


SIZES = [1, 2, 3, 7, 8, 9, 15, 16, 17, 31, 33, 127, 128, 129]


@pytest.mark.parametrize("path", ACCURATE_PATHS)
@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_brute_force_tiny_shapes(oracle_mod, path, ta, tb):
    rng = np.random.default_rng(17)
    combos = list(itertools.product(SIZES, SIZES, SIZES))
    for t, i in enumerate(rng.choice(len(combos), size=24, replace=False)):
        M, N, K = combos[i]
        opA = gi.random_matrix(300 + t, M, K)
        opB = gi.random_matrix(400 + t, K, N)
        C = gi.random_matrix(500 + t, M, N)
        alpha, beta = [(1.0, 0.0), (-1.0, 0.5), (1.5, 1.0), (0.5, -1.0)][t % 4]
        A, B = stored(opA, ta), stored(opB, tb)
        pad = (t % 3, (t + 1) % 3, t % 2)
        lda, ldb, ldc = ld_of(A, pad[0]), ld_of(B, pad[1]), N + pad[2]
        st, out = gh.run(ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C if beta else None, ldc,
                         path=path, offsets=(t % 2, 0, (t // 2) % 2))
        assert st == 0, (M, N, K)
        if path == sg.PATH_3XTF32 and K < 16:
            # the dropped lo*lo and residual terms (~3*2^-22 |ab| per product)
            # can exceed 4*K*2^-24 for K < 3; the selector never sends K < 16
            # here, a forced call is held to 4*16*2^-24 instead
            ref, bound = oracle_mod.gemm_f64(ta, tb, M, N, K, alpha, A, A.shape[1], B,
                                             B.shape[1], beta, C, N)
            assert np.all(np.abs(out - ref) <= bound * 16.0 / K), (M, N, K)
        else:
            oracle_check(oracle_mod, ta, tb, M, N, K, alpha, A, A.shape[1], B, B.shape[1], beta,
                         C, out)


# ------------------------------------------------------------ BLAS special cases
@pytest.mark.parametrize("path", [sg.PATH_AUTO] + ACCURATE_PATHS)
def test_special_cases(path):
    M, N, K = 70, 50, 40
    C = gi.random_matrix(31, M, N)
    A = gi.random_matrix(32, M, K)
    B = gi.random_matrix(33, K, N)
    # alpha == 0: C = beta*C, A and B not read (null pointers)
    st, out = gh.run("N", "N", M, N, K, 0.0, None, K, None, N, 0.5, C, N, path=path)
    assert st == 0 and np.array_equal(out, np.float32(0.5) * C)
    # K == 0
    st, out = gh.run("N", "N", M, N, 0, 1.0, None, 1, None, N, -2.0, C, N, path=path)
    assert st == 0 and np.array_equal(out, np.float32(-2.0) * C)
    # alpha == 0 and beta == 0 over NaN: zeros, C not read
    st, out = gh.run("N", "N", M, N, K, 0.0, None, K, None, N, 0.0, None, N, path=path)
    assert st == 0 and np.all(out == 0)
    # beta == 0 over NaN C: finite
    st, out = gh.run("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, None, N, path=path)
    assert st == 0 and np.all(np.isfinite(out))
    # beta == 1 with K == 0: C unchanged
    st, out = gh.run("N", "N", M, N, 0, 1.0, None, 1, None, N, 1.0, C, N, path=path)
    assert st == 0 and np.array_equal(out, C)
    # empty
    st, _ = gh.run("N", "N", 0, N, K, 1.0, None, K, B, N, 0.0, None, N, path=path)
    assert st == 0


# ------------------------------------------------------------ full-size configs
# Workloads up to this many flop are compared on every output entry (the
# oracle runs at ~10 GFLOP/s on the GPU host's cores); larger ones on seeded
# sample points.
FULL_COMPARE_FLOPS = 4.0e10


@pytest.mark.parametrize("name", list(gi.WORKLOADS))
def test_workload_full_size(oracle_mod, name):
    """Every measured workload at full size through sgemm() (the call the
    benchmark times) and, where every entry is compared, through the forced
    FFMA path too; against the fp64 oracle within the bound.  Workloads up to
    FULL_COMPARE_FLOPS are compared on every entry of C, larger ones on
    seeded sample points (corners, last row and column, uniform points)."""
    import torch

    w = gi.WORKLOADS[name]
    A, B, C = gi.make_inputs(w)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    full = w.flops <= FULL_COMPARE_FLOPS
    points = None if full else gi.sample_points(w.M, w.N, 4096, seed=w.seed)
    ref, bound = oracle_mod.gemm_f64(w.transA, w.transB, w.M, w.N, w.K, w.alpha, A, A.shape[1],
                                     B, B.shape[1], w.beta, C, w.N, points=points)
    for path in ((sg.PATH_AUTO, sg.PATH_FFMA) if full else (sg.PATH_AUTO,)):
        dC = (torch.from_numpy(C).cuda() if C is not None
              else torch.full((w.M, w.N), float("nan"), device="cuda"))
        st = sg.sgemm_ex(w.transA, w.transB, w.M, w.N, w.K, w.alpha, dA.data_ptr(), A.shape[1],
                         dB.data_ptr(), B.shape[1], w.beta, dC.data_ptr(), w.N,
                         torch.cuda.current_stream(), path, 0)
        torch.cuda.synchronize()
        assert st == 0
        out = dC.cpu().numpy()
        assert np.all(np.isfinite(out))
        rep = oracle_mod.compare(out if full else out[points], ref, bound, w.K, w.alpha)
        assert rep["pass"], (path, rep)
        del dC


@pytest.mark.parametrize("name", ["sq4096_nn", "ragged_tn", "skinny_nt", "sq1024_nn"])
def test_ffma_full_size_sampled(oracle_mod, name):
    """The FFMA path at full size with the selector's stream-K decomposition
    (shares crossing tile boundaries, fixup of shared tiles), sampled against
    the fp64 oracle within the bound; and forced whole tiles (split = 1)
    bit-identical to the oracle's ascending-k FMA evaluation on the samples."""
    import torch

    w = gi.WORKLOADS[name]
    A, B, C = gi.make_inputs(w)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    rows, cols = gi.sample_points(w.M, w.N, 2048, seed=w.seed + 7)
    ref, bound = oracle_mod.gemm_f64(w.transA, w.transB, w.M, w.N, w.K, w.alpha, A, A.shape[1],
                                     B, B.shape[1], w.beta, C, w.N, points=(rows, cols))
    seq = oracle_mod.gemm_f32_seq(w.transA, w.transB, w.M, w.N, w.K, w.alpha, A, A.shape[1],
                                  B, B.shape[1], w.beta, C, w.N, points=(rows, cols))
    for split in (0, 1):
        dC = (torch.from_numpy(C).cuda() if C is not None
              else torch.full((w.M, w.N), float("nan"), device="cuda"))
        st = sg.sgemm_ex(w.transA, w.transB, w.M, w.N, w.K, w.alpha, dA.data_ptr(), A.shape[1],
                         dB.data_ptr(), B.shape[1], w.beta, dC.data_ptr(), w.N,
                         torch.cuda.current_stream(), sg.PATH_FFMA, split)
        torch.cuda.synchronize()
        assert st == 0
        out = dC.cpu().numpy()[rows, cols]
        rep = oracle_mod.compare(out, ref, bound, w.K, w.alpha)
        assert rep["pass"], (split, rep)
        if split == 1:
            assert np.array_equal(out.view(np.uint32), seq.view(np.uint32))
