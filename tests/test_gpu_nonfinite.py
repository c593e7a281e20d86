"""Infinite, NaN and near-FLT_MAX inputs on every GPU path.

The fp32 result of a sum that meets an infinite input is what IEEE
arithmetic gives: an infinity times a nonzero value keeps the product's
sign, an infinity times zero and +inf plus -inf are NaN, and NaN
propagates.  The fp64 oracle gives the same class as long as no finite
partial sum overflows fp32, so every entry is checked with
oracle.compare_ieee: the same class where the reference is not finite,
the fp32 bound elsewhere.  The FFMA path without split-K must also equal the
oracle's fp32 ascending-k evaluation bit for bit (NaN for NaN).

On the tensor cores the TF32 parts of an infinity (and of a finite value
above (2 - 2^-11) 2^127, which rounds to an infinite TF32 part) turn the sums
they enter into NaN; the library recomputes such outputs in fp32, and these
cases make it do so: partners whose low part is zero (1.0, 0.5), zeros, both
signs, +inf and -inf in one sum, and FLT_MAX and -3.4025e38 against small
partners (finite results).  Whole tiles are fixed in the main kernel, shared
(stream-K) tiles in the fixup kernel, and the SM-pair kernel's tiles by each
CTA for its rows.
"""
import numpy as np
import pytest

import dense_fp32_gemm_05_gb300 as sg
import gemm_inputs as gi

pytestmark = pytest.mark.gpu

FLT_MAX = np.float32(np.finfo(np.float32).max)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from dense_fp32_gemm_05_gb300 import build
    build.build()
    sg.load()


def planted(M, N, K, seed):
    """op(A) (M x K) and op(B) (K x N), uniform [-1, 1], with infinities,
    zeros, exact partners and values near FLT_MAX planted."""
    A = gi.random_matrix(seed, M, K)
    B = gi.random_matrix(seed + 1, K, N)
    inf = np.float32(np.inf)
    i0, i1, k0, k1, k2 = 1, M - 2, 3, K // 2, K - 4
    A[i0, k0] = inf                       # row i0: sign of B[k0, j], NaN where B[k0, j] = 0
    B[k0, :8] = [0.0, 1.0, -1.0, 0.5, -2.0, 0.0, 3.0, -0.25]
    A[i1, k1] = inf                       # row i1: +inf and -inf meet
    A[i1, k2] = -inf
    B[k1, 0], B[k2, 0] = 1.0, 1.0         # (i1, 0): inf - inf = NaN
    j0 = N - 3
    B[k2 + 1, j0] = -inf                  # column j0: -inf times op(A)[:, k2 + 1]
    A[: M // 2, k2 + 1] = 1.0             # exact partners (low part zero)
    A[M // 2, k2 + 1] = 0.0               # NaN at (M // 2, j0)
    A[M - 1, 5] = np.nan                  # a NaN input: row M - 1 all NaN
    # near FLT_MAX, against small partners: finite products
    r0, r1, kb0, kb1 = M // 4, M // 4 + 1, 7, 9
    A[r0, kb0] = FLT_MAX
    A[r1, kb1] = np.float32(-3.4025e38)   # TF32 round-to-nearest would overflow
    B[kb0, :] *= np.float32(2.0 ** -110)
    B[kb1, :] *= np.float32(2.0 ** -110)
    A[:, kb0] = np.where(np.arange(M) == r0, A[:, kb0], A[:, kb0] * np.float32(2.0 ** -110))
    A[:, kb1] = np.where(np.arange(M) == r1, A[:, kb1], A[:, kb1] * np.float32(2.0 ** -110))
    c0 = N // 2
    kb2 = 11
    B[kb2, c0] = FLT_MAX                  # FLT_MAX on the B side too
    A[:, kb2] *= np.float32(2.0 ** -110)
    return A, B


def stored(op_mat, trans):
    return np.ascontiguousarray(op_mat if trans == "N" else op_mat.T)


def run(ta, tb, M, N, K, A, B, alpha, beta, C, path, split):
    import torch
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = (torch.from_numpy(C).cuda() if C is not None
          else torch.full((M, N), float("nan"), device="cuda"))
    s = torch.cuda.current_stream()
    st = sg.sgemm_ex(ta, tb, M, N, K, alpha, dA.data_ptr(), A.shape[1], dB.data_ptr(), B.shape[1],
                     beta, dC.data_ptr(), N, s, path, split)
    assert st == sg.SGEMM_OK, sg.sgemm_status_string(st)
    assert sg.sgemm_device_error(s) == sg.SGEMM_OK
    return dC.cpu().numpy()


# layout, M, N, K, path, split, what it reaches
CASES = [
    ("T", "N", 300, 260, 700, sg.PATH_3XTF32, 1, "SM pairs, both operands pre-split"),
    ("N", "T", 300, 260, 700, sg.PATH_3XTF32, 1, "A in tensor memory, B split in shared memory"),
    ("N", "N", 300, 100, 700, sg.PATH_3XTF32, 0, "WIDE tiles (A_hi in TMEM, A_lo in SMEM)"),
    ("T", "N", 513, 64, 2000, sg.PATH_3XTF32, 0, "three accumulators, stream-K + fixup"),
    ("N", "N", 1024, 1024, 1024, sg.PATH_3XTF32, 0, "A in TMEM, stream-K + fixup"),
    ("T", "T", 300, 260, 700, sg.PATH_TF32, 0, "single-pass TF32"),
    ("N", "N", 300, 260, 700, sg.PATH_FFMA, 1, "FFMA, whole tiles"),
    ("T", "T", 100, 77, 300, sg.PATH_AUTO, 0, "FFMA, small-problem kernel"),
    ("T", "N", 300, 260, 700, sg.PATH_FFMA, 3, "FFMA, split-K"),
    ("N", "T", 300, 2100, 700, sg.PATH_FFMA, 1, "FFMA, A copied transposed first"),
    ("T", "T", 2100, 130, 700, sg.PATH_FFMA, 1, "FFMA, B copied transposed first"),
    ("N", "T", 8, 700, 500, sg.PATH_GEMV, 0, "thin problem, dot form"),
    ("N", "N", 16, 700, 500, sg.PATH_GEMV, 0, "thin problem on the tensor cores"),
    ("N", "N", 32, 4100, 600, sg.PATH_AUTO, 0, "thin problem on the tensor cores, S = 32"),
    ("T", "N", 64, 4100, 600, sg.PATH_AUTO, 0, "thin problem on the tensor cores, S = 64"),
    ("N", "N", 128, 4100, 600, sg.PATH_AUTO, 0, "thin problem on the tensor cores, S = 128"),
    ("T", "N", 700, 8, 500, sg.PATH_GEMV, 0, "thin problem, axpy form"),
]


@pytest.mark.parametrize("ta,tb,M,N,K,path,split,what", CASES, ids=[c[-1] for c in CASES])
@pytest.mark.parametrize("beta", [0.0, 0.5])
def test_nonfinite_inputs_follow_ieee(oracle_mod, ta, tb, M, N, K, path, split, what, beta):
    opA, opB = planted(M, N, K, 77)
    A, B = stored(opA, ta), stored(opB, tb)
    C = gi.random_matrix(79, M, N) if beta else None
    out = run(ta, tb, M, N, K, A, B, 1.0, beta, C, path, split)
    ref, bound = oracle_mod.gemm_f64(ta, tb, M, N, K, 1.0, A, A.shape[1], B, B.shape[1], beta, C, N)
    assert (~np.isfinite(ref)).sum() > M, "the planted values must reach many outputs"
    if path == sg.PATH_TF32:
        # single-pass TF32: its own bound on finite entries, IEEE classes elsewhere
        mag = bound / (4 * K * 2.0 ** -24)
        bound = (2.0 ** -10 + 4 * K * 2.0 ** -24) * mag
    rep = oracle_mod.compare_ieee(out, ref, bound)
    assert rep["pass"], (what, rep)
    # the near-FLT_MAX values dominate finite entries of their rows (and of
    # column N // 2), which compare_ieee held to the bound above
    for r in (M // 4, M // 4 + 1):
        fin = np.isfinite(ref[r])
        assert fin.any() and np.abs(ref[r][fin]).max() > 1e4, what
    if path == sg.PATH_FFMA and split == 1:
        seq = oracle_mod.gemm_f32_seq(ta, tb, M, N, K, 1.0, A, A.shape[1], B, B.shape[1], beta,
                                      C, N)
        nan = np.isnan(seq)
        assert np.array_equal(nan, np.isnan(out))
        assert np.array_equal(out[~nan].view(np.uint32), seq[~nan].view(np.uint32))


def test_clean_call_after_nonfinite_call(oracle_mod):
    """A call without infinities right after one with them is correct, on
    the same stream and shapes (nothing of the first call's recomputation
    carries over)."""
    M, N, K = 1024, 1024, 1024
    opA, opB = planted(M, N, K, 91)
    run("N", "N", M, N, K, opA, opB, 1.0, 0.0, None, sg.PATH_3XTF32, 0)
    A = gi.random_matrix(92, M, K)
    B = gi.random_matrix(93, K, N)
    out = run("N", "N", M, N, K, A, B, 1.0, 0.0, None, sg.PATH_3XTF32, 0)
    ref, bound = oracle_mod.gemm_f64("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, None, N)
    assert oracle_mod.compare(out, ref, bound, K, 1.0)["pass"]


def test_nonfinite_pair_last_wave_stream_k(oracle_mod):
    """4096 x 4096 x 2048 runs on SM pairs with the last wave's tiles shared
    in k (their partial sums added by the fixup kernel).  The planted rows
    and columns cross both whole and shared tiles; they are checked in full,
    with seeded points elsewhere."""
    import torch
    M, N, K = 4096, 4096, 2048
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, d = sg.sgemm_plan_detail("N", "N", M, N, K, K, N, N, path=sg.PATH_3XTF32, num_sms=sms)
    assert st == 0 and d["pair"] == 1 and d["sk_tail"] == 1, d
    A, B = planted(M, N, K, 81)
    out = run("N", "N", M, N, K, A, B, 1.0, 0.0, None, sg.PATH_3XTF32, 0)
    rows = [1, M - 2, M // 2, M - 1, M // 4, M // 4 + 1]
    cols = [N - 3, N // 2] + list(range(8))
    r = np.concatenate([np.repeat(rows, N), np.tile(np.arange(M), len(cols))])
    c = np.concatenate([np.tile(np.arange(N), len(rows)), np.repeat(cols, M)])
    rs, cs = gi.sample_points(M, N, 4096, seed=83)
    r, c = np.concatenate([r, rs]), np.concatenate([c, cs])
    ref, bound = oracle_mod.gemm_f64("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, None, N,
                                     points=(r, c))
    assert (~np.isfinite(ref)).sum() > M
    rep = oracle_mod.compare_ieee(out[r, c], ref, bound)
    assert rep["pass"], rep
