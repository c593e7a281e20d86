"""The FFMA tile path's transpose pre-pass.  On a large grid, a K-contiguous
operand (A 'N', B 'T') is first copied transposed, and the kernel then reads
it as an M- or N-contiguous one.  The per-output FMA order does not change:
whole tiles still equal the oracle's fp32 sequential evaluation bit for bit.
That holds in every layout, with misaligned bases and padded leading
dimensions (the copy itself is aligned), and shared tiles (stream-K) stay
within the bound.  Each case first asserts, through sgemm_plan_detail, which
operands the pre-pass copies."""
import numpy as np
import pytest

import dense_fp32_gemm_05_gb300 as sg
import gemm_inputs as gi
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from dense_fp32_gemm_05_gb300 import build
    build.build()
    sg.load()


def stored(op_mat, trans):
    return np.ascontiguousarray(op_mat if trans == "N" else op_mat.T)


def pad_cols(arr, ld):
    out = np.full((arr.shape[0], ld), np.nan, np.float32)
    out[:, : arr.shape[1]] = arr
    return out


# (transA, transB, M, N, K, alpha, beta, pads of lda/ldb/ldc, element offsets
# of A/B/C, pre_transpose bits: 1 op(A), 2 op(B))
SHAPES = [
    ("N", "N", 300, 2100, 260, 1.0, 0.0, (0, 0, 0), (0, 0, 0), 1),
    ("N", "T", 2050, 2049, 257, -1.5, 0.5, (3, 1, 2), (1, 2, 3), 3),
    ("T", "T", 2049, 130, 300, 0.75, 1.0, (0, 5, 0), (0, 1, 0), 2),
    ("N", "T", 2051, 300, 1000, 1.0, -1.0, (1, 0, 0), (3, 0, 0), 2),
]


def _plan(ta, tb, M, N, K, lda, ldb, ldc, split):
    st, info = sg.sgemm_plan_detail(ta, tb, M, N, K, lda, ldb, ldc, 1, 1, 1, sg.PATH_FFMA, split,
                                    152)
    assert st == 0 and info["path"] == sg.PATH_FFMA
    return info


@pytest.mark.parametrize("ta,tb,M,N,K,alpha,beta,pad,off,bits", SHAPES)
def test_whole_tiles_bitwise_equal_sequential_oracle(oracle_mod, ta, tb, M, N, K, alpha, beta, pad,
                                                     off, bits):
    opA = gi.random_matrix(51, M, K, dist="normal")
    opB = gi.random_matrix(52, K, N, dist="normal")
    C = gi.random_matrix(53, M, N)
    A, B = stored(opA, ta), stored(opB, tb)
    lda, ldb, ldc = A.shape[1] + pad[0], B.shape[1] + pad[1], N + pad[2]
    info = _plan(ta, tb, M, N, K, lda, ldb, ldc, 1)
    assert info["pre_transpose"] == bits and info["tile_n"] == 128, info
    st, out = gh.run(ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C if beta else None, ldc,
                     path=sg.PATH_FFMA, split=1, offsets=off)
    assert st == 0
    want = oracle_mod.gemm_f32_seq(ta, tb, M, N, K, alpha, pad_cols(A, lda), lda,
                                   pad_cols(B, ldb), ldb, beta, C, N)
    assert np.array_equal(out.view(np.uint32), want.view(np.uint32)), (ta, tb, M, N, K)


def test_shared_tiles_within_bound(oracle_mod):
    # a grid under one wave: every tile's k range shared (stream-K + fixup)
    ta, tb, M, N, K = "N", "T", 2050, 2049, 1000
    opA = gi.random_matrix(61, M, K)
    opB = gi.random_matrix(62, K, N)
    C = gi.random_matrix(63, M, N)
    A, B = stored(opA, ta), stored(opB, tb)
    info = _plan(ta, tb, M, N, K, K, K, N, 0)
    assert info["pre_transpose"] == 3 and info["ctas"] > info["dp_tiles"], info
    st, out = gh.run(ta, tb, M, N, K, 1.5, A, K, B, K, 0.5, C, N, path=sg.PATH_FFMA, split=0)
    assert st == 0
    rng = np.random.default_rng(64)
    rows = rng.integers(0, M, 4096)
    cols = rng.integers(0, N, 4096)
    ref, bound = oracle_mod.gemm_f64(ta, tb, M, N, K, 1.5, A, K, B, K, 0.5, C, N,
                                     points=(rows, cols))
    rep = oracle_mod.compare(out[rows, cols], ref, bound, K, 1.5)
    assert rep["pass"], rep


def test_below_the_threshold_nothing_is_copied():
    # the other side shorter than 2048, or a short K, or an M- / N-contiguous operand
    for ta, tb, M, N, K in [("N", "N", 4096, 2047, 4096), ("N", "T", 2047, 2047, 4096),
                            ("N", "N", 4096, 4096, 255), ("T", "N", 4096, 4096, 4096)]:
        lda = K if ta == "N" else M
        ldb = N if tb == "N" else K
        assert _plan(ta, tb, M, N, K, lda, ldb, N, 0)["pre_transpose"] == 0, (ta, tb, M, N, K)
