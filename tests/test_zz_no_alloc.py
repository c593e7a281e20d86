"""The allocation-free FFMA entry point, sgemm_ffma_static_scratch.

Some callers of this library may not allocate device memory: a host
framework that owns the whole device memory pool, or a latency-critical loop
that must not enter the allocator.  For them the library offers a variant of
the FFMA split-K launch whose partial sums live in a fixed 16 MiB static
device array instead of the allocated workspace.  This test calls it through
the C ABI several times in a row, on different problems that all need split-K
scratch, and checks each result bit for bit against sgemm_ex's FFMA path with
the same decomposition (the same k-tiles shared by the same CTAs and added in
the same order), and against the oracle within the fp32 tolerance the other
parity tests use (|d| <= 4*K*2^-24*(|alpha||A||B| + |beta||C|)).  One call
leaves the split to the selector, whose choice needs more scratch than the
array holds, so the call shares the work among fewer CTAs.  It also checks
that a forced split needing more scratch than the array holds is refused
before any launch.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest

import dense_fp32_gemm_05_gb300 as sg
import gemm_inputs as gi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from dense_fp32_gemm_05_gb300 import build
    build.build()
    sg.load()


def _case(ta, tb, M, N, K, alpha, beta, seed):
    a_shape = (M, K) if ta == "N" else (K, M)
    b_shape = (K, N) if tb == "N" else (N, K)
    A = gi.random_matrix(seed, *a_shape)
    B = gi.random_matrix(seed + 1, *b_shape)
    C = gi.random_matrix(seed + 2, M, N)
    return A, B, C


def test_static_scratch_matches_sgemm_ex_on_two_calls_in_a_row(oracle_mod):
    import torch

    s = torch.cuda.current_stream()
    cases = [
        # layout, M, N, K, alpha, beta, split for the static call, split of
        # the sgemm_ex call with the same decomposition, seed:
        # 4 tiles x 8 slices, then 6 tiles x 3 slices of the same static array
        ("N", "N", 256, 256, 4096, 1.0, 0.0, 8, 8, 101),
        ("T", "T", 300, 200, 1000, 1.5, 0.5, 3, 3, 202),
        # the selector's own choice (split 0) would share 1024^3's 64 tiles x
        # 64 k-tiles among 304 CTAs, more than the array holds: the static
        # call shares them among 128 CTAs, as sgemm_ex does with split 2
        ("N", "N", 1024, 1024, 1024, 1.0, 0.0, 0, 2, 303),
    ]
    for ta, tb, M, N, K, alpha, beta, split, split_ex, seed in cases:
        A, B, C = _case(ta, tb, M, N, K, alpha, beta, seed)
        dA = torch.from_numpy(A).cuda()
        dB = torch.from_numpy(B).cuda()
        c_new = torch.from_numpy(C).cuda()
        c_old = torch.from_numpy(C).cuda()
        st = sg.sgemm_ffma_static_scratch(ta, tb, M, N, K, alpha, dA.data_ptr(), A.shape[1],
                                          dB.data_ptr(), B.shape[1], beta, c_new.data_ptr(), N,
                                          s, split)
        assert st == sg.SGEMM_OK, sg.sgemm_status_string(st)
        st = sg.sgemm_ex(ta, tb, M, N, K, alpha, dA.data_ptr(), A.shape[1], dB.data_ptr(),
                         B.shape[1], beta, c_old.data_ptr(), N, s, sg.PATH_FFMA, split_ex)
        assert st == sg.SGEMM_OK
        torch.cuda.synchronize()
        new, old = c_new.cpu().numpy(), c_old.cpu().numpy()
        # the same decomposition and the same summation order: bit for bit
        assert np.array_equal(new.view(np.uint32), old.view(np.uint32)), (M, N, K, split)
        ref, bound = oracle_mod.gemm_f64(ta, tb, M, N, K, alpha, A, A.shape[1], B, B.shape[1],
                                         beta, C, N)
        rep = oracle_mod.compare(new, ref, bound, K, alpha)
        assert rep["pass"], rep


def test_static_scratch_refuses_plans_beyond_its_size():
    # 4096 x 4096 has 1024 tiles; split 2 on every tile needs 2048 partial
    # tiles, far beyond the 256 the array holds: refused, nothing launched
    # (the pointers are never dereferenced).
    fake = 1 << 20
    st = sg.sgemm_ffma_static_scratch("N", "N", 4096, 4096, 4096, 1.0, fake, 4096, fake, 4096,
                                      0.0, fake, 4096, None, 2)
    assert st == sg.SGEMM_ERR_SCRATCH
