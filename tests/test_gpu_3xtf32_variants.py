"""3xTF32 accuracy pinned on every tensor-core kernel variant.

At large K the fp32 bound 4*K*2^-24 per unit of sum|a||b| is loose enough
for single-pass TF32 to pass it, so a variant that lost its hi*lo or lo*hi
products would still pass the ordinary parity tests.  This file closes that
gap with a pin that only the three-product split meets:

  op(A) = S, a selection matrix (one 1 per row, at column sigma(i)), and
  op(B) = X, full-mantissa fp32 values, give C(i, j) = X(sigma(i), j) exactly
  in real arithmetic.  3xTF32 computes each such entry as hi(x) + lo(x), which
  misses x by at most 2^-22 |x|; TF32 alone computes hi(x), which misses by
  up to 2^-11 |x|.  The same with X on the A side (op(B) a selection matrix)
  pins the split of A.

Each shape below first asserts, through sgemm_plan_detail, the kernel
variant it reaches (SM pairs, tensor-memory A, shared-memory B, WIDE tiles,
three accumulators, last-wave slices, stream-K), so that a change of the
selector cannot silently empty the test.  The selection product is the
permutation pin of the GEMM definition ("Optimising fp32 GEMM on A100",
section "What is GEMM?") with a non-square selection in place of the
permutation.
"""
import numpy as np
import pytest

import dense_fp32_gemm_05_gb300 as sg
import gemm_inputs as gi

pytestmark = pytest.mark.gpu

PIN = 2.0 ** -22           # 3xTF32: |out - x| <= 2^-22 |x|
TF32_PIN = 2.0 ** -11      # single-pass TF32: |out - x| <= 2^-11 |x|

# name, layout, M, N, K, forced split, the plan fields the shape must reach
VARIANTS = [
    ("pair_tail_slices", "N", "N", 4096, 4096, 256, 0,
     dict(pair=1, tail_nsplit=2, sk_tail=0, sk_ctas=0)),
    ("pair_sk_tail", "N", "N", 4096, 4096, 2048, 0, dict(pair=1, sk_tail=1)),
    ("pair_whole", "T", "N", 2048, 2048, 1024, 0,
     dict(pair=1, tail_nsplit=1, sk_tail=0, sk_ctas=0)),
    ("pair_bn128_slices", "T", "N", 1024, 128, 512, 0, dict(pair=1, tile_n=128, tail_nsplit=2)),
    ("pair_bn64", "T", "N", 2048, 64, 512, 1, dict(pair=1, tile_n=64, accumulators=1)),
    ("single_presplit_slices", "N", "N", 128, 4096, 512, 0,
     dict(pair=0, fuse_a=0, fuse_b=0, tile_n=256, tail_nsplit=4)),
    ("tmem_a_whole", "N", "N", 2048, 2048, 2048, 0,
     dict(fuse_a=1, fuse_b=0, wide=0, sk_ctas=0, tail_nsplit=1)),
    ("tmem_a_slices", "N", "N", 4096, 256, 512, 1, dict(fuse_a=1, wide=0, tail_nsplit=4)),
    ("tmem_a_sk", "N", "N", 1024, 1024, 1024, 0, dict(fuse_a=1, fuse_b=0, wide=0, sk_ctas=128)),
    ("tmem_a_smem_b_sk", "N", "T", 1024, 1024, 1024, 0, dict(fuse_a=1, fuse_b=1, sk_ctas=128)),
    ("tmem_a_smem_b_slices", "N", "T", 1024, 1024, 1024, 1,
     dict(fuse_a=1, fuse_b=1, tail_nsplit=4)),
    ("smem_b_slices", "T", "T", 1024, 2048, 512, 0, dict(fuse_a=0, fuse_b=1, tail_nsplit=2)),
    ("smem_b_bn64_sk", "T", "T", 512, 64, 1024, 0,
     dict(fuse_b=1, tile_n=64, accumulators=3, sk_ctas=32)),
    ("presplit_sk", "T", "N", 1024, 1024, 1024, 0, dict(fuse_a=0, fuse_b=0, sk_ctas=128)),
    ("bn64_three_acc_sk", "T", "N", 513, 64, 2000, 0,
     dict(tile_n=64, accumulators=3, wide=0, pair=0, sk_ctas=75)),
    ("bn64_three_acc_sk_tail", "T", "N", 128, 64, 2000, 0,
     dict(tile_n=64, accumulators=3, pair=0, sk_tail=1)),
    ("bn128_single_sk", "T", "N", 513, 128, 2000, 0,
     dict(tile_n=128, pair=0, wide=0, fuse_a=0, accumulators=1, sk_ctas=75)),
    ("bn128_single_slices", "T", "N", 128, 128, 512, 1,
     dict(tile_n=128, pair=0, wide=0, tail_nsplit=2)),
    ("smem_b_bn128_sk", "T", "T", 1024, 128, 1024, 0,
     dict(tile_n=128, fuse_b=1, wide=0, sk_ctas=64)),
    ("wide128_slices", "N", "T", 20480, 128, 256, 0, dict(wide=1, tile_n=128, tail_nsplit=2)),
    ("wide64_whole", "N", "T", 20480, 64, 256, 0, dict(wide=1, tile_n=64, sk_ctas=0)),
    ("wide64_sk", "N", "N", 513, 64, 2000, 0, dict(wide=1, tile_n=64, sk_ctas=35)),
    ("wide128_sk", "N", "T", 4096, 128, 2048, 0, dict(wide=1, tile_n=128, sk_ctas=128)),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from dense_fp32_gemm_05_gb300 import build
    build.build()
    sg.load()


def stored(op_mat, trans):
    return np.ascontiguousarray(op_mat if trans == "N" else op_mat.T)


def selection(rows, cols, seed):
    """rows x cols with a single 1 per row, at a seeded column, and the columns."""
    pick = np.random.default_rng(seed).integers(0, cols, rows)
    S = np.zeros((rows, cols), np.float32)
    S[np.arange(rows), pick] = 1.0
    return S, pick


def full_mantissa(seed, rows, cols):
    """Uniform [-1, 1] values, checked to carry bits below TF32's 11: a value
    rounded to TF32 alone misses them by more than 2^-20 of its size."""
    X = gi.random_matrix(seed, rows, cols)
    bits = X.view(np.uint32)
    hi = ((bits + np.uint32(0x1000)) & np.uint32(0xFFFFE000)).view(np.float32)
    rel = np.abs(X.astype(np.float64) - hi) / np.maximum(np.abs(X), 1e-30)
    assert rel.max() > 2.0 ** -20
    return X


def run(ta, tb, M, N, K, A, B, path, split):
    import torch
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.full((M, N), float("nan"), device="cuda")
    s = torch.cuda.current_stream()
    st = sg.sgemm_ex(ta, tb, M, N, K, 1.0, dA.data_ptr(), A.shape[1], dB.data_ptr(), B.shape[1],
                     0.0, dC.data_ptr(), N, s, path, split)
    assert st == sg.SGEMM_OK, sg.sgemm_status_string(st)
    assert sg.sgemm_device_error(s) == sg.SGEMM_OK
    return dC.cpu().numpy()


def worst_rel(out, want):
    err = np.abs(out.astype(np.float64) - want)
    return float((err / np.maximum(np.abs(want.astype(np.float64)), 1e-30)).max())


def check_plan(ta, tb, M, N, K, split, want, path=sg.PATH_3XTF32):
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    lda = K if ta == "N" else M
    ldb = N if tb == "N" else K
    st, d = sg.sgemm_plan_detail(ta, tb, M, N, K, lda, ldb, N, path=path, split=split,
                                 num_sms=sms)
    assert st == sg.SGEMM_OK
    got = {k: d[k] for k in want}
    assert got == want, f"plan {d} does not reach the variant {want}"


@pytest.mark.parametrize("name,ta,tb,M,N,K,split,want", VARIANTS, ids=[v[0] for v in VARIANTS])
def test_3xtf32_split_pin_per_variant(name, ta, tb, M, N, K, split, want):
    check_plan(ta, tb, M, N, K, split, dict(want, path=sg.PATH_3XTF32))
    # X on the B side: C(i, j) = X(sigma(i), j)
    S, sigma = selection(M, K, 1000 + M + K)
    X = full_mantissa(2000 + N, K, N)
    out = run(ta, tb, M, N, K, stored(S, ta), stored(X, tb), sg.PATH_3XTF32, split)
    assert worst_rel(out, X[sigma]) <= PIN, (name, "B side")
    # X on the A side: C(i, j) = X(i, tau(j))
    T, tau = selection(N, K, 3000 + N + K)
    Y = full_mantissa(4000 + M, M, K)
    out = run(ta, tb, M, N, K, stored(Y, ta), stored(np.ascontiguousarray(T.T), tb),
              sg.PATH_3XTF32, split)
    assert worst_rel(out, Y[:, tau]) <= PIN, (name, "A side")


@pytest.mark.parametrize("name", ["pair_sk_tail", "tmem_a_sk", "wide64_sk"])
def test_tf32_fails_the_split_pin(name):
    """The pin tells the modes apart on the GPU: single-pass TF32 on the same
    shapes misses 2^-22 but stays within its own 2^-11."""
    _, ta, tb, M, N, K, split, _ = next(v for v in VARIANTS if v[0] == name)
    S, sigma = selection(M, K, 1000 + M + K)
    X = full_mantissa(2000 + N, K, N)
    out = run(ta, tb, M, N, K, stored(S, ta), stored(X, tb), sg.PATH_TF32, split)
    rel = worst_rel(out, X[sigma])
    assert PIN < rel <= TF32_PIN, rel
