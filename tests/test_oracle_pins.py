"""Pins for the CPU oracle: closed forms, invariants, exact integer cases,
library cross-checks and hand-worked rounding cases.

The oracle is the GEMM definition C = alpha*op(A)*op(B) + beta*C of
"Optimising fp32 GEMM on A100" (section "What is GEMM?").  Each pin below
fixes its output by something other than the oracle itself, so that a dropped
term, a flipped sign, a wrong index or a transposed operand fails at least one
of them.
"""
import itertools

import numpy as np
import pytest

import gemm_inputs as gi

LAYOUTS = [("N", "N"), ("N", "T"), ("T", "N"), ("T", "T")]
U = 2.0 ** -24


def stored(op_mat, trans, ld_pad=0, fill=np.nan):
    """Stored fp32 array (with ld padding) whose op() is op_mat."""
    base = op_mat if trans == "N" else op_mat.T
    rows, cols = base.shape
    ld = max(cols + ld_pad, 1)
    out = np.full((rows, ld), fill, dtype=np.float32)
    out[:, :cols] = base
    return out, ld


def run_f64(orc, ta, tb, opA, opB, alpha, beta, C=None, pad=(0, 0, 0)):
    M, K = opA.shape
    N = opB.shape[1]
    A, lda = stored(opA, ta, pad[0])
    B, ldb = stored(opB, tb, pad[1])
    ldc = max(N + pad[2], 1)
    Cs = None
    if C is not None:
        Cs = np.full((M, ldc), np.nan, dtype=np.float32)
        Cs[:, :N] = C
    return orc.gemm_f64(ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, Cs, ldc)


def run_f32(orc, ta, tb, opA, opB, alpha, beta, C=None):
    M, K = opA.shape
    N = opB.shape[1]
    A, lda = stored(opA, ta)
    B, ldb = stored(opB, tb)
    return orc.gemm_f32_seq(ta, tb, M, N, K, alpha, A, lda, B, ldb, beta,
                            C, max(N, 1))


# ---------------------------------------------------------------- P1 ones
@pytest.mark.parametrize("ta,tb", LAYOUTS)
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (5, 7, 3), (33, 17, 3001)])
def test_all_ones(oracle_mod, ta, tb, M, N, K):
    opA = np.ones((M, K), np.float32)
    opB = np.ones((K, N), np.float32)
    ref, bound = run_f64(oracle_mod, ta, tb, opA, opB, 1.0, 0.0)
    assert np.all(ref == K)
    assert np.allclose(bound, 4 * K * U * K, rtol=0, atol=0)
    # with beta: alpha*K + beta*c, every term exact in double
    C = np.full((M, N), 3.0, np.float32)
    ref, bound = run_f64(oracle_mod, ta, tb, opA, opB, 2.0, -0.5, C)
    assert np.all(ref == 2.0 * K - 1.5)
    assert np.all(bound == 4 * K * U * (2.0 * K + 0.5 * 3.0))
    # fp32 sequential order: K < 2^24 so every partial sum is exact
    out = run_f32(oracle_mod, ta, tb, opA, opB, 1.0, 0.0)
    assert np.all(out == np.float32(K))


# ---------------------------------------------------------------- P2 identity
@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_identity_left_and_right(oracle_mod, ta, tb):
    M, N = 19, 23
    X = gi.random_matrix(11, M, N)          # any values
    # op(A) = I_M  =>  C = op(B)
    ref, _ = run_f64(oracle_mod, ta, tb, np.eye(M, dtype=np.float32), X, 1.0, 0.0)
    assert np.array_equal(ref, X.astype(np.float64))
    # op(B) = I_N  =>  C = op(A)
    ref, _ = run_f64(oracle_mod, ta, tb, X, np.eye(N, dtype=np.float32), 1.0, 0.0)
    assert np.array_equal(ref, X.astype(np.float64))
    # alpha, beta with identity: 1.5*x + 0.25*c is one double rounding of
    # two exact products, i.e. the correctly rounded value of the real result
    C = gi.random_matrix(12, M, N)
    ref, _ = run_f64(oracle_mod, ta, tb, np.eye(M, dtype=np.float32), X, 1.5, 0.25, C)
    exact = 1.5 * X.astype(np.float64) + 0.25 * C.astype(np.float64)
    assert np.array_equal(ref, exact)


# ---------------------------------------------------------------- P3 permutation
@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_permutation(oracle_mod, ta, tb):
    rng = np.random.default_rng(3)
    M, K, N = 13, 13, 29
    perm = rng.permutation(K)
    P = np.zeros((M, K), np.float32)
    P[np.arange(M), perm] = 1.0              # row i of P picks k = perm[i]
    X = gi.random_matrix(21, K, N)
    ref, _ = run_f64(oracle_mod, ta, tb, P, X, 1.0, 0.0)
    assert np.array_equal(ref, X[perm].astype(np.float64))
    # right permutation: column j of Q picks row sigma[j] of op(B)=Q
    N2 = 17
    sigma = rng.permutation(N2)
    Q = np.zeros((N2, N2), np.float32)
    Q[sigma, np.arange(N2)] = 1.0
    Y = gi.random_matrix(22, 9, N2)
    ref, _ = run_f64(oracle_mod, ta, tb, Y, Q, 1.0, 0.0)
    assert np.array_equal(ref, Y[:, sigma].astype(np.float64))


# ---------------------------------------------------------------- P4 rank one
@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_rank_one_closed_forms(oracle_mod, ta, tb):
    M, N, K = 11, 14, 37
    u = (np.arange(M) - 5).astype(np.float32)            # small integers
    v = (2.0 ** -np.arange(N)).astype(np.float32)         # powers of two
    opA = np.repeat(u[:, None], K, axis=1)                # A_ik = u_i
    opB = np.repeat(v[None, :], K, axis=0)                # B_kj = v_j
    ref, _ = run_f64(oracle_mod, ta, tb, opA, opB, 1.0, 0.0)
    assert np.array_equal(ref, K * np.outer(u, v).astype(np.float64))
    # A = u e0^T, B = e0 v^T  =>  C = u v^T
    a = np.zeros((M, K), np.float32); a[:, 0] = u
    b = np.zeros((K, N), np.float32); b[0, :] = v
    ref, _ = run_f64(oracle_mod, ta, tb, a, b, -1.0, 0.0)
    assert np.array_equal(ref, -np.outer(u, v).astype(np.float64))


# ---------------------------------------------------------------- P5 integers
@pytest.mark.parametrize("ta,tb", LAYOUTS)
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (-1.0, 1.0), (2.0, -1.0), (0.5, 2.0)])
def test_small_integers_exact(oracle_mod, ta, tb, alpha, beta):
    M, N, K = 31, 45, 129
    Ai = gi.small_ints(1, (M, K))
    Bi = gi.small_ints(2, (K, N))
    Ci = gi.small_ints(3, (M, N))
    exact = Ai.astype(np.int64) @ Bi.astype(np.int64)      # library integer matmul
    want = alpha * exact.astype(np.float64) + (beta * Ci.astype(np.float64) if beta else 0.0)
    ref, _ = run_f64(oracle_mod, ta, tb, Ai, Bi, alpha, beta, Ci if beta else None)
    assert np.array_equal(ref, want)
    # fp32 sequential: all partial sums are integers < 2^24, exact too
    out = run_f32(oracle_mod, ta, tb, Ai, Bi, alpha, beta, Ci if beta else None)
    assert np.array_equal(out.astype(np.float64), want)


# ---------------------------------------------------------------- P6 library
SHAPES = [1, 2, 3, 7, 8, 9, 16, 17, 33]


@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_brute_force_vs_numpy(oracle_mod, ta, tb):
    rng = np.random.default_rng(7)
    combos = list(itertools.product(SHAPES, SHAPES, SHAPES))
    idx = rng.choice(len(combos), size=40, replace=False)
    for t, i in enumerate(idx):
        M, N, K = combos[i]
        opA = gi.random_matrix(100 + t, M, K)
        opB = gi.random_matrix(200 + t, K, N)
        C = gi.random_matrix(300 + t, M, N)
        alpha, beta = [(1.0, 0.0), (-1.0, 0.5), (1.5, 1.0), (0.0, 0.5)][t % 4]
        ref, bound = run_f64(oracle_mod, ta, tb, opA, opB, alpha, beta, C,
                             pad=(t % 3, (t + 1) % 3, t % 2))
        A64, B64, C64 = (x.astype(np.float64) for x in (opA, opB, C))
        lib = alpha * np.matmul(A64, B64) + (beta * C64 if beta else 0.0)
        mag = abs(alpha) * np.matmul(np.abs(A64), np.abs(B64)) + abs(beta) * np.abs(C64)
        assert np.all(np.abs(ref - lib) <= 1e-13 * mag + 1e-300)
        assert np.allclose(bound, 4 * K * U * mag, rtol=1e-13, atol=0)


@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_f32_sequential_within_bound(oracle_mod, ta, tb):
    """The fp32 evaluation obeys the fp32 error bound of the definition."""
    for t, (M, N, K) in enumerate([(5, 6, 7), (17, 9, 300), (3, 40, 1025)]):
        opA = gi.random_matrix(400 + t, M, K, dist="normal")
        opB = gi.random_matrix(500 + t, K, N, dist="normal")
        C = gi.random_matrix(600 + t, M, N)
        out = run_f32(oracle_mod, ta, tb, opA, opB, 1.25, -0.75, C)
        ref, bound = run_f64(oracle_mod, ta, tb, opA, opB, 1.25, -0.75, C)
        rep = oracle_mod.compare(out, ref, bound, K, 1.25)
        assert rep["pass"], rep
        assert rep["max_err_over_bound"] < 0.25


# ---------------------------------------------------------------- P7 special
@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_special_cases(oracle_mod, ta, tb):
    M, N, K = 6, 5, 4
    C = gi.random_matrix(31, M, N)
    # alpha == 0: C = beta*C and A, B are never read (null pointers accepted)
    ref, bound = oracle_mod.gemm_f64(ta, tb, M, N, K, 0.0, None, max(K if ta == "N" else M, 1),
                                     None, max(N if tb == "N" else K, 1), 0.5, C, N)
    assert np.array_equal(ref, 0.5 * C.astype(np.float64))
    out = oracle_mod.gemm_f32_seq(ta, tb, M, N, K, 0.0, None, max(K if ta == "N" else M, 1),
                                  None, max(N if tb == "N" else K, 1), 0.5, C, N)
    assert np.array_equal(out, np.float32(0.5) * C)
    # K == 0: no product term, bound 0
    ref, bound = oracle_mod.gemm_f64(ta, tb, M, N, 0, 1.0, None, max(1 if ta == "N" else M, 1),
                                     None, max(N if tb == "N" else 1, 1), -2.0, C, N)
    assert np.array_equal(ref, -2.0 * C.astype(np.float64)) and np.all(bound == 0)
    # beta == 0 with NaN in C: C is not read
    Cnan = np.full((M, N), np.nan, np.float32)
    opA = gi.random_matrix(32, M, K)
    opB = gi.random_matrix(33, K, N)
    ref, _ = run_f64(oracle_mod, ta, tb, opA, opB, 1.0, 0.0, Cnan)
    assert np.all(np.isfinite(ref))
    # alpha == 0 and beta == 0: zero, even over NaN C
    ref, _ = run_f64(oracle_mod, ta, tb, opA, opB, 0.0, 0.0, Cnan)
    assert np.all(ref == 0)
    # empty outputs
    r0, b0 = oracle_mod.gemm_f64(ta, tb, 0, N, K, 1.0, None, max(K if ta == "N" else 1, 1),
                                 opB, max(N if tb == "N" else K, 1), 0.0, None, N)
    assert r0.shape == (0, N)


def test_argument_errors(oracle_mod):
    A = np.zeros(64, np.float32)
    with pytest.raises(oracle_mod.OracleArgError, match="argument 1"):
        oracle_mod.gemm_f64("X", "N", 2, 2, 2, 1.0, A, 2, A, 2, 0.0, None, 2)
    with pytest.raises(oracle_mod.OracleArgError, match="argument 2"):
        oracle_mod.gemm_f64("N", "Q", 2, 2, 2, 1.0, A, 2, A, 2, 0.0, None, 2)
    with pytest.raises(oracle_mod.OracleArgError, match="argument 3"):
        oracle_mod.gemm_f64("N", "N", -1, 2, 2, 1.0, A, 2, A, 2, 0.0, None, 2)
    with pytest.raises(oracle_mod.OracleArgError, match="argument 8"):
        oracle_mod.gemm_f64("N", "N", 2, 2, 3, 1.0, A, 2, A, 2, 0.0, None, 2)
    with pytest.raises(oracle_mod.OracleArgError, match="argument 10"):
        oracle_mod.gemm_f64("N", "T", 2, 2, 3, 1.0, A, 3, A, 2, 0.0, None, 2)
    with pytest.raises(oracle_mod.OracleArgError, match="argument 13"):
        oracle_mod.gemm_f64("N", "N", 2, 5, 3, 1.0, A, 3, A, 5, 0.0, None, 4)


# ---------------------------------------------------------------- P8 order
def test_f32_sequential_order_hand_worked(oracle_mod):
    """Hand-worked fp32 cases that fix the summation order and the FMA.

    Row [1, 2^24, -2^24] times a column of ones, k ascending:
      fma(1,1,0) = 1;  fma(2^24,1,1) = 2^24+1 -> tie, rounds to even 2^24;
      fma(-2^24,1,2^24) = 0.   Exact (fp64) answer: 1.  Descending order: 1.
    So the ascending fp32 loop must give exactly 0.
    """
    a = np.array([[1.0, 2.0 ** 24, -(2.0 ** 24)]], np.float32)
    b = np.ones((3, 1), np.float32)
    out = run_f32(oracle_mod, "N", "N", a, b, 1.0, 0.0)
    assert out[0, 0] == 0.0
    ref, _ = run_f64(oracle_mod, "N", "N", a, b, 1.0, 0.0)
    assert ref[0, 0] == 1.0
    # reversed k order gives the exact value 1: the order is what decides
    out_rev = run_f32(oracle_mod, "N", "N", a[:, ::-1].copy(), b, 1.0, 0.0)
    assert out_rev[0, 0] == 1.0

    # Fused multiply-add, not multiply then add:
    # x = 1 + 2^-12, x*x = 1 + 2^-11 + 2^-24.  fma(x, x, -1) keeps the
    # 2^-24 (result 2^-11 + 2^-24, exact in fp32); a rounded multiply would
    # tie-round x*x to 1 + 2^-11 and give 2^-11.
    x = np.float32(1.0 + 2.0 ** -12)
    a = np.array([[-1.0, x]], np.float32)
    b = np.array([[1.0], [x]], np.float32)
    out = run_f32(oracle_mod, "N", "N", a, b, 1.0, 0.0)
    assert out[0, 0] == np.float32(2.0 ** -11 + 2.0 ** -24)

    # epilogue fmaf(alpha, acc, beta*c): alpha = x, acc = x, beta*c = -1
    a = np.array([[x]], np.float32)
    b = np.array([[1.0]], np.float32)
    c = np.array([[-1.0]], np.float32)
    out = run_f32(oracle_mod, "N", "N", a, b, float(x), 1.0, c)
    assert out[0, 0] == np.float32(2.0 ** -11 + 2.0 ** -24)
    # beta == 0: plain rounded product alpha*acc = fl(x*x) = 1 + 2^-11
    out = run_f32(oracle_mod, "N", "N", a, b, float(x), 0.0, None)
    assert out[0, 0] == np.float32(1.0 + 2.0 ** -11)


# ---------------------------------------------------------------- invariants
@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_transpose_symmetry(oracle_mod, ta, tb):
    """(op(A) op(B))^T = op(B)^T op(A)^T via the swapped, flag-flipped call."""
    M, N, K = 12, 9, 21
    opA = gi.random_matrix(41, M, K)
    opB = gi.random_matrix(42, K, N)
    A, lda = stored(opA, ta)
    B, ldb = stored(opB, tb)
    ref, _ = oracle_mod.gemm_f64(ta, tb, M, N, K, 1.0, A, lda, B, ldb, 0.0, None, N)
    flip = {"N": "T", "T": "N"}
    refT, _ = oracle_mod.gemm_f64(flip[tb], flip[ta], N, M, K, 1.0, B, ldb, A, lda,
                                  0.0, None, M)
    assert np.array_equal(ref, refT.T)


@pytest.mark.parametrize("ta,tb", LAYOUTS)
def test_leading_dimension_gaps(oracle_mod, ta, tb):
    """NaN in every gap element changes nothing (gaps are never read)."""
    M, N, K = 10, 7, 13
    opA = gi.random_matrix(51, M, K)
    opB = gi.random_matrix(52, K, N)
    C = gi.random_matrix(53, M, N)
    r0, b0 = run_f64(oracle_mod, ta, tb, opA, opB, 1.0, 1.0, C)
    r1, b1 = run_f64(oracle_mod, ta, tb, opA, opB, 1.0, 1.0, C, pad=(3, 5, 2))
    assert np.array_equal(r0, r1) and np.array_equal(b0, b1)


def test_sampled_points_match_full(oracle_mod):
    M, N, K = 40, 33, 50
    opA = gi.random_matrix(61, M, K)
    opB = gi.random_matrix(62, K, N)
    C = gi.random_matrix(63, M, N)
    full, fb = oracle_mod.gemm_f64("N", "T", M, N, K, 1.0, opA, K, opB.T.copy(), K, 0.5, C, N)
    rows, cols = gi.sample_points(M, N, 200, seed=9)
    s, sb = oracle_mod.gemm_f64("N", "T", M, N, K, 1.0, opA, K, opB.T.copy(), K, 0.5, C, N,
                                points=(rows, cols))
    assert np.array_equal(s, full[rows, cols]) and np.array_equal(sb, fb[rows, cols])
    f32 = oracle_mod.gemm_f32_seq("N", "T", M, N, K, 1.0, opA, K, opB.T.copy(), K, 0.5, C, N)
    f32s = oracle_mod.gemm_f32_seq("N", "T", M, N, K, 1.0, opA, K, opB.T.copy(), K, 0.5, C, N,
                                   points=(rows, cols))
    assert np.array_equal(f32s, f32[rows, cols])


def test_compare_detects_errors(oracle_mod):
    """The comparison flags an off-by-one-ulp-of-bound error and NaN."""
    M, N, K = 8, 8, 16
    opA = gi.random_matrix(71, M, K)
    opB = gi.random_matrix(72, K, N)
    ref, bound = run_f64(oracle_mod, "N", "N", opA, opB, 1.0, 0.0)
    good = ref.astype(np.float32)
    assert oracle_mod.compare(good, ref, bound, K, 1.0)["pass"]
    bad = good.copy()
    bad[3, 4] = np.float32(ref[3, 4] + 2 * bound[3, 4])
    rep = oracle_mod.compare(bad, ref, bound, K, 1.0)
    assert not rep["pass"] and rep["n_bad"] == 1
    bad = good.copy()
    bad[0, 0] = np.nan
    assert not oracle_mod.compare(bad, ref, bound, K, 1.0)["pass"]


# ------------------------------------------------------------ non-finite inputs
def test_nonfinite_hand_worked(oracle_mod):
    """IEEE classes by hand: an infinity times a positive value keeps its
    sign, times a negative one flips it, times zero is NaN; +inf and -inf in
    one sum give NaN; NaN propagates; a value near FLT_MAX times a small one
    stays finite.  Both oracle functions, every layout."""
    inf, big = np.float32(np.inf), np.float32(3.4e38)
    rows = [
        ([inf, 1.0], [1.0, 1.0], np.inf),
        ([inf, 2.0], [-1.0, 1.0], -np.inf),
        ([inf, -inf], [1.0, 1.0], np.nan),
        ([inf, 1.0], [0.0, 1.0], np.nan),
        ([np.nan, 1.0], [1.0, 1.0], np.nan),
        ([big, 1.0], [2.0 ** -100, 2.0], float(big) * 2.0 ** -100 + 2.0),
    ]
    for a, b, want in rows:
        opA = np.array([a], np.float32)
        opB = np.array(b, np.float32).reshape(2, 1)
        for ta, tb in LAYOUTS:
            ref, bound = run_f64(oracle_mod, ta, tb, opA, opB, 1.0, 0.0)
            f32 = run_f32(oracle_mod, ta, tb, opA, opB, 1.0, 0.0)
            if np.isnan(want):
                assert np.isnan(ref[0, 0]) and np.isnan(f32[0, 0])
            elif np.isinf(want):
                assert ref[0, 0] == want and f32[0, 0] == want
            else:
                assert abs(ref[0, 0] - want) <= 2.0 ** -52 * abs(want)
                assert abs(f32[0, 0] - want) <= bound[0, 0]


def test_compare_ieee_classes(oracle_mod):
    """compare_ieee: non-finite reference entries need the same class,
    finite ones the bound; a wrong sign, NaN for inf, a finite value for inf
    and an error beyond the bound each fail."""
    ref = np.array([np.inf, -np.inf, np.nan, 1.0])
    bound = np.array([np.inf, np.inf, np.nan, 1e-6])
    good = np.array([np.inf, -np.inf, np.nan, 1.0], np.float32)
    assert oracle_mod.compare_ieee(good, ref, bound)["pass"]
    for i, v in [(0, -np.inf), (0, np.nan), (1, 3.0), (2, np.inf), (3, 1.1), (3, np.nan)]:
        bad = good.copy()
        bad[i] = v
        rep = oracle_mod.compare_ieee(bad, ref, bound)
        assert not rep["pass"] and rep["n_bad"] == 1, (i, v)


# ------------------------------------------------------------ fused epilogue
# D = act(alpha * s_i * (op(A) op(B))_ij + beta * C_ij + bias_j): each term
# pinned against something other than the epilogue oracle itself.

def _epi_inputs(seed, M, N, K):
    rng = np.random.default_rng(seed)
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    C = rng.uniform(-1, 1, (M, N)).astype(np.float32)
    return A, B, C


def test_epilogue_reduces_to_the_plain_definition(oracle_mod):
    M, N, K = 7, 9, 13
    A, B, C = _epi_inputs(1, M, N, K)
    for beta, Cin in ((0.0, None), (0.5, C)):
        r0, _ = oracle_mod.gemm_f64("N", "N", M, N, K, 1.5, A, K, B, N, beta, Cin, N)
        r1, _ = oracle_mod.gemm_epilogue_f64("N", "N", M, N, K, 1.5, A, K, B, N, beta, Cin, N)
        assert np.array_equal(r0, r1)


def test_epilogue_row_scale_scales_rows(oracle_mod):
    # powers of two: exact in fp64, so row i is exactly s_i times the plain row
    M, N, K = 6, 5, 11
    A, B, _ = _epi_inputs(2, M, N, K)
    s = np.array([2.0 ** (i % 5 - 2) * (-1) ** i for i in range(M)], np.float32)
    r0, _ = oracle_mod.gemm_f64("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, None, N)
    r1, _ = oracle_mod.gemm_epilogue_f64("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, None, N,
                                         row_scale=s)
    assert np.array_equal(r1, s.astype(np.float64)[:, None] * r0)


def test_epilogue_bias_is_per_column(oracle_mod):
    # alpha = beta = 0: only the bias is left, the same in every row; A, B, C unread
    M, N = 4, 6
    bias = np.arange(N, dtype=np.float32) - 2.5
    r, b = oracle_mod.gemm_epilogue_f64("N", "N", M, N, 3, 0.0, None, 3, None, N, 0.0, None, N,
                                        bias=bias)
    assert np.array_equal(r, np.tile(bias.astype(np.float64), (M, 1)))
    assert np.array_equal(b, (4 * 3 + 3) * 2.0 ** -24 * np.abs(np.tile(bias, (M, 1))).astype(np.float64))


def test_epilogue_relu_clamps_the_identity_result(oracle_mod):
    M, N, K = 8, 8, 17
    A, B, C = _epi_inputs(3, M, N, K)
    bias = np.linspace(-1, 1, N).astype(np.float32)
    r_id, b_id = oracle_mod.gemm_epilogue_f64("T", "N", M, N, K, 1.0, np.ascontiguousarray(A.T), M,
                                              B, N, 0.5, C, N, bias=bias, act=0)
    r_re, b_re = oracle_mod.gemm_epilogue_f64("T", "N", M, N, K, 1.0, np.ascontiguousarray(A.T), M,
                                              B, N, 0.5, C, N, bias=bias, act=1)
    assert np.array_equal(r_re, np.maximum(r_id, 0.0))
    assert np.array_equal(b_re, b_id)
    assert (r_id < 0).any() and (r_id > 0).any()


def test_epilogue_small_integers_exact(oracle_mod):
    # every term an integer: the int64 computation is the exact answer
    rng = np.random.default_rng(4)
    M, N, K = 9, 7, 23
    A = rng.integers(-8, 9, (M, K)).astype(np.float32)
    B = rng.integers(-8, 9, (N, K)).astype(np.float32)          # stored N x K ('T')
    C = rng.integers(-8, 9, (M, N)).astype(np.float32)
    s = rng.integers(-3, 4, M).astype(np.float32)
    bias = rng.integers(-50, 51, N).astype(np.float32)
    want = (2 * s.astype(np.int64)[:, None] * (A.astype(np.int64) @ B.astype(np.int64).T)
            - 1 * C.astype(np.int64) + bias.astype(np.int64)[None, :])
    for act in (0, 1):
        r, _ = oracle_mod.gemm_epilogue_f64("N", "T", M, N, K, 2.0, A, K, B, K, -1.0, C, N,
                                            row_scale=s, bias=bias, act=act)
        w = want if act == 0 else np.maximum(want, 0)
        assert np.array_equal(r, w.astype(np.float64))


def test_epilogue_bound_closed_form(oracle_mod):
    # all ones, alpha = 2, s_i = 3, beta = -1 (c = 1), bias = 5:
    # bound = (4K + 3) 2^-24 (6 K + 1 + 5)
    M, N, K = 3, 4, 10
    A = np.ones((M, K), np.float32)
    B = np.ones((K, N), np.float32)
    C = np.ones((M, N), np.float32)
    r, b = oracle_mod.gemm_epilogue_f64("N", "N", M, N, K, 2.0, A, K, B, N, -1.0, C, N,
                                        row_scale=np.full(M, 3.0, np.float32),
                                        bias=np.full(N, 5.0, np.float32))
    assert np.all(r == 6.0 * K - 1.0 + 5.0)
    assert np.allclose(b, (4 * K + 3) * 2.0 ** -24 * (6.0 * K + 1.0 + 5.0), rtol=0, atol=0)


def test_epilogue_rejects_unknown_activation(oracle_mod):
    with pytest.raises(oracle_mod.OracleArgError):
        oracle_mod.gemm_epilogue_f64("N", "N", 2, 2, 2, 1.0, np.ones((2, 2), np.float32), 2,
                                     np.ones((2, 2), np.float32), 2, 0.0, None, 2, act=7)


def test_thread_count_does_not_change_results(oracle_mod):
    """Every entry is summed by one thread in a fixed order: one thread and
    all threads give the same bits."""
    M, N, K = 37, 29, 301
    A = gi.random_matrix(81, M, K)
    B = gi.random_matrix(82, K, N)
    n = oracle_mod.num_threads()
    try:
        oracle_mod.set_num_threads(1)
        assert oracle_mod.num_threads() == 1
        r1, b1 = oracle_mod.gemm_f64("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, None, N)
        f1 = oracle_mod.gemm_f32_seq("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, None, N)
    finally:
        oracle_mod.set_num_threads(n)
    r2, b2 = oracle_mod.gemm_f64("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, None, N)
    f2 = oracle_mod.gemm_f32_seq("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, None, N)
    assert np.array_equal(r1, r2) and np.array_equal(b1, b2)
    assert np.array_equal(f1.view(np.uint32), f2.view(np.uint32))
