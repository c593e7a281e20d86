"""The one-launch small-problem FFMA kernel (16 x 16 tiles, k in chunks of
128): every output is the ascending-k fused multiply-add sum, so it must
equal the oracle's fp32 sequential evaluation bit for bit, in every layout,
at ragged sizes, with padded leading dimensions and misaligned base
pointers, and around its chunk and selector boundaries.  Each case first
asserts (through sgemm_plan_detail) that the selector really sends it to
this kernel."""
import numpy as np
import pytest

import dense_fp32_gemm_05_gb300 as sg
import gemm_inputs as gi
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu

LAYOUTS = [("N", "N"), ("N", "T"), ("T", "N"), ("T", "T")]


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


def plan_of(ta, tb, M, N, K, lda, ldb, ldc, path):
    st, info = sg.sgemm_plan_detail(ta, tb, M, N, K, lda, ldb, ldc, 1, 1, 1, path, 0, 152)
    assert st == 0
    return info


# (M, N, K, alpha, beta, pads of lda/ldb/ldc, element offsets of A/B/C)
SHAPES = [
    (256, 256, 256, 1.0, 0.0, (0, 0, 0), (0, 0, 0)),      # config c0's shape
    (17, 17, 1, 1.0, 0.0, (0, 0, 0), (0, 0, 0)),          # one k, ragged tiles
    (100, 77, 127, -1.5, 0.5, (3, 1, 2), (1, 2, 3)),      # one partial chunk
    (33, 200, 128, 0.75, -2.0, (0, 5, 0), (3, 0, 1)),     # exactly one chunk
    (130, 31, 129, 1.0, 1.0, (1, 1, 1), (0, 0, 0)),       # a chunk and one k
    (48, 48, 512, 2.0, 0.25, (0, 0, 0), (2, 2, 2)),       # the longest K taken
    (2048, 32, 500, 1.0, 0.0, (0, 0, 0), (0, 0, 0)),      # tall, 256 tiles
]


@pytest.mark.parametrize("ta,tb", LAYOUTS)
@pytest.mark.parametrize("M,N,K,alpha,beta,pad,off", SHAPES)
def test_small_kernel_bitwise_equals_sequential_oracle(oracle_mod, ta, tb, M, N, K, alpha, beta,
                                                       pad, off):
    opA = gi.random_matrix(21, M, K, dist="normal")
    opB = gi.random_matrix(22, K, N, dist="normal")
    C = gi.random_matrix(23, M, N)
    A, B = stored(opA, ta), stored(opB, tb)
    lda, ldb, ldc = A.shape[1] + pad[0], B.shape[1] + pad[1], N + pad[2]
    for path in (sg.PATH_AUTO, sg.PATH_FFMA):
        info = plan_of(ta, tb, M, N, K, lda, ldb, ldc, path)
        assert info["path"] == sg.PATH_FFMA and info["tile_m"] == info["tile_n"] == 16, info
        assert info["ctas"] == ((M + 15) // 16) * ((N + 15) // 16) and info["k_block"] == 128
        st, out = gh.run(ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C if beta else None, ldc,
                         path=path, split=0, offsets=off)
        assert st == 0
        want = oracle_mod.gemm_f32_seq(ta, tb, M, N, K, alpha, pad_cols(A, lda), lda,
                                       pad_cols(B, ldb), ldb, beta, C, N)
        assert np.array_equal(out.view(np.uint32), want.view(np.uint32)), (path, ta, tb)
    ref, bound = oracle_mod.gemm_f64(ta, tb, M, N, K, alpha, A, A.shape[1], B, B.shape[1], beta,
                                     C, N)
    assert oracle_mod.compare(out, ref, bound, K, alpha)["pass"]


def test_small_kernel_next_to_tile_kernel(oracle_mod):
    """Either side of the K edge (512 small, 513 tile kernel, split 1): both
    equal the sequential oracle, so the two FFMA kernels agree bit for bit on
    the common prefix of work."""
    for K in (512, 513):
        M, N = 64, 96
        opA = gi.random_matrix(31, M, K, dist="normal")
        opB = gi.random_matrix(32, K, N, dist="normal")
        st, out = gh.run("N", "N", M, N, K, 1.0, opA, K, opB, N, 0.0, None, N,
                         path=sg.PATH_FFMA, split=1)
        assert st == 0
        want = oracle_mod.gemm_f32_seq("N", "N", M, N, K, 1.0, opA, K, opB, N, 0.0, None, N)
        assert np.array_equal(out.view(np.uint32), want.view(np.uint32)), K
