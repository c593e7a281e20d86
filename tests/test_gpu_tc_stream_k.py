"""Stream-K on the tensor-core paths: the tiles x k-blocks iterations shared
in equal contiguous ranges by the CTAs, partial sums of shared tiles added in
k order by the fixup kernel.  Forced splits on every layout (operands split
in the kernel or by the pre-pass), 256-, 128- and 64-wide tiles, both
tensor-core modes, the fused epilogue, and a shape the selector sends to
stream-K by itself, each against the oracle."""
import zlib

import numpy as np
import pytest

import dense_fp32_gemm_05_gb300 as sg
import gemm_inputs as gi
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu

LAYOUTS = [("N", "N"), ("N", "T"), ("T", "N"), ("T", "T")]
# (M, N, K): 256-, 128- and 64-wide tiles; ragged in every dimension
SHAPES = [(300, 260, 1000), (257, 100, 700), (513, 64, 2000)]


def stored(op_mat, trans):
    return np.ascontiguousarray(op_mat if trans == "N" else op_mat.T)


def seed_of(*parts):
    return zlib.crc32("/".join(map(str, parts)).encode()) % 100000


@pytest.mark.parametrize("ta,tb", LAYOUTS)
@pytest.mark.parametrize("shape", SHAPES, ids=["bn256", "bn128", "bn64"])
@pytest.mark.parametrize("split", [2, 5])
def test_3xtf32_stream_k_within_bound(oracle_mod, ta, tb, shape, split):
    M, N, K = shape
    t = seed_of(ta, tb, shape, split)
    opA, opB = gi.random_matrix(t, M, K), gi.random_matrix(t + 1, K, N)
    C = gi.random_matrix(t + 2, M, N)
    A, B = stored(opA, ta), stored(opB, tb)
    st, p = sg.sgemm_plan(ta, tb, M, N, K, A.shape[1], B.shape[1], N, path=sg.PATH_3XTF32,
                          split=split)
    assert st == 0 and p["tile_m"] == 128 and p["split"] >= 1 and p["ctas"] > 0
    st, out = gh.run(ta, tb, M, N, K, 1.25, A, A.shape[1], B, B.shape[1], -0.5, C, N,
                     path=sg.PATH_3XTF32, split=split)
    assert st == 0
    ref, bound = oracle_mod.gemm_f64(ta, tb, M, N, K, 1.25, A, A.shape[1], B, B.shape[1], -0.5,
                                     C, N)
    rep = oracle_mod.compare(out, ref, bound, K, 1.25)
    assert rep["pass"], rep


@pytest.mark.parametrize("ta,tb", LAYOUTS)
@pytest.mark.parametrize("path", [sg.PATH_3XTF32, sg.PATH_TF32])
@pytest.mark.parametrize("shape", SHAPES, ids=["bn256", "bn128", "bn64"])
def test_stream_k_small_integers_exact(ta, tb, path, shape):
    # integers are exact in TF32 and every partial sum stays below 2^24
    M, N, K = shape
    opA, opB = gi.small_ints(51, (M, K)), gi.small_ints(52, (K, N))
    C = gi.small_ints(53, (M, N))
    want = 2 * (opA.astype(np.int64) @ opB.astype(np.int64)) - C.astype(np.int64)
    st, out = gh.run(ta, tb, M, N, K, 2.0, stored(opA, ta), stored(opA, ta).shape[1],
                     stored(opB, tb), stored(opB, tb).shape[1], -1.0, C, N, path=path, split=3)
    assert st == 0
    assert np.array_equal(out.astype(np.int64), want)


@pytest.mark.parametrize("ta,tb", [("N", "T"), ("T", "N")])
def test_stream_k_is_deterministic(ta, tb):
    M, N, K = 300, 260, 1000
    A = stored(gi.random_matrix(61, M, K), ta)
    B = stored(gi.random_matrix(62, K, N), tb)
    outs = []
    for _ in range(2):
        st, out = gh.run(ta, tb, M, N, K, 1.0, A, A.shape[1], B, B.shape[1], 0.0, None, N,
                         path=sg.PATH_3XTF32, split=4)
        assert st == 0
        outs.append(out.view(np.uint32).copy())
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("shape", SHAPES, ids=["bn256", "bn128", "bn64"])
def test_stream_k_fused_epilogue(oracle_mod, shape):
    import torch
    M, N, K = shape
    A = gi.random_matrix(71, M, K)
    B = gi.random_matrix(72, N, K)          # NT
    C = gi.random_matrix(73, M, N)
    rng = np.random.default_rng(74)
    s = rng.uniform(-2, 2, M).astype(np.float32)
    bias = rng.uniform(-3, 3, N).astype(np.float32)
    dA, dB, dC, ds, db = (torch.from_numpy(x).cuda() for x in (A, B, C, s, bias))
    st = sg.sgemm_epilogue("N", "T", M, N, K, 0.75, dA.data_ptr(), K, dB.data_ptr(), K, 0.5,
                           dC.data_ptr(), N, ds.data_ptr(), db.data_ptr(), sg.ACT_RELU,
                           torch.cuda.current_stream(), sg.PATH_3XTF32, 3)
    torch.cuda.synchronize()
    assert st == 0
    ref, bound = oracle_mod.gemm_epilogue_f64("N", "T", M, N, K, 0.75, A, K, B, K, 0.5, C, N,
                                              row_scale=s, bias=bias, act=1)
    rep = oracle_mod.compare_bound(dC.cpu().numpy(), ref, bound)
    assert rep["pass"], rep


def test_selector_takes_stream_k_for_few_tiles_and_long_k(oracle_mod):
    """2048 x 64 x 8192 NT: 16 tiles of 128 x 64 for 152 SMs.  The selector
    shares the iterations among 9 CTAs per tile (144, every range inside one
    tile); the whole result is checked."""
    import torch
    M, N, K = 2048, 64, 8192
    st, p = sg.sgemm_plan("N", "T", M, N, K, K, K, N, num_sms=152)
    assert st == 0 and p["path"] == sg.PATH_3XTF32 and p["ctas"] == 144 and p["split"] == 9
    A = gi.random_matrix(81, M, K)
    B = gi.random_matrix(82, N, K)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.full((M, N), float("nan"), device="cuda")
    st = sg.sgemm("N", "T", M, N, K, 1.0, dA.data_ptr(), K, dB.data_ptr(), K, 0.0, dC.data_ptr(),
                  N, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert st == 0 and sg.sgemm_device_error(torch.cuda.current_stream()) == 0
    ref, bound = oracle_mod.gemm_f64("N", "T", M, N, K, 1.0, A, K, B, K, 0.0, None, N)
    rep = oracle_mod.compare(dC.cpu().numpy(), ref, bound, K, 1.0)
    assert rep["pass"], rep


def test_stream_k_one_k_block_per_cta(oracle_mod):
    # more CTAs than k-blocks per tile: every tile shared by several CTAs,
    # some CTAs holding a single k-block
    M, N, K = 256, 256, 96
    A = gi.random_matrix(91, M, K)
    B = gi.random_matrix(92, K, N)
    st, p = sg.sgemm_plan("N", "N", M, N, K, K, N, N, path=sg.PATH_3XTF32, split=8)
    assert st == 0 and p["ctas"] > 0
    st, out = gh.run("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, None, N, path=sg.PATH_3XTF32,
                     split=8)
    assert st == 0
    ref, bound = oracle_mod.gemm_f64("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, None, N)
    assert oracle_mod.compare(out, ref, bound, K, 1.0)["pass"]


@pytest.mark.parametrize("shape,pair", [((4096, 4096, 256), True), ((2560, 2048, 256), False)],
                         ids=["pair_half_units", "single_sm_tmem_a_units"])
def test_last_wave_slices_sampled(oracle_mod, shape, pair):
    """The tiles after the last full wave run as narrower column slices
    (checked through the plan), every other tile whole; seeded samples over
    the whole result, the last rows and columns included, against the oracle."""
    import torch
    M, N, K = shape
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, p = sg.sgemm_plan("N", "N", M, N, K, K, N, N, num_sms=sms)
    assert st == 0 and p["split"] > 1 and (p["tile_m"] == 256) == pair
    A = gi.random_matrix(101, M, K)
    B = gi.random_matrix(102, K, N)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.full((M, N), float("nan"), device="cuda")
    st = sg.sgemm("N", "N", M, N, K, 1.0, dA.data_ptr(), K, dB.data_ptr(), N, 0.0, dC.data_ptr(), N,
                  torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert st == 0
    out = dC.cpu().numpy()
    assert np.all(np.isfinite(out))
    rows, cols = gi.sample_points(M, N, 12000, seed=103)
    ref, bound = oracle_mod.gemm_f64("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, None, N,
                                     points=(rows, cols))
    rep = oracle_mod.compare(out[rows, cols], ref, bound, K, 1.0)
    assert rep["pass"], rep


@pytest.mark.parametrize("ta,tb", [("N", "N"), ("T", "T")])
def test_last_wave_stream_k_on_pairs_sampled(oracle_mod, ta, tb):
    """4096 x 4096 x 2048 on SM pairs: three waves of whole 256 x 256 tiles,
    then the k-blocks of the last 28 tiles shared by all pairs, each pair's
    CTAs writing their 128 rows of a partial tile; the fixup adds them in k
    order.  Seeded samples over the whole result against the oracle."""
    import torch
    M = N = 4096
    K = 2048
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    lda = K if ta == "N" else M
    ldb = N if tb == "N" else K
    st, p = sg.sgemm_plan(ta, tb, M, N, K, lda, ldb, N, num_sms=sms)
    assert st == 0 and p["tile_m"] == 256 and p["split"] > 1
    opA = gi.random_matrix(111, M, K)
    opB = gi.random_matrix(112, K, N)
    A, B = stored(opA, ta), stored(opB, tb)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.full((M, N), float("nan"), device="cuda")
    st = sg.sgemm(ta, tb, M, N, K, 1.0, dA.data_ptr(), lda, dB.data_ptr(), ldb, 0.0, dC.data_ptr(), N,
                  torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert st == 0 and sg.sgemm_device_error(torch.cuda.current_stream()) == 0
    out = dC.cpu().numpy()
    assert np.all(np.isfinite(out))
    # the last wave's tiles are the last in raster order: sample them densely
    rows, cols = gi.sample_points(M, N, 12000, seed=113)
    ref, bound = oracle_mod.gemm_f64(ta, tb, M, N, K, 1.0, A, lda, B, ldb, 0.0, None, N,
                                     points=(rows, cols))
    rep = oracle_mod.compare(out[rows, cols], ref, bound, K, 1.0)
    assert rep["pass"], rep
    # and the whole result matches a run with every tile whole (same sums up
    # to the order of the partial-sum additions: inside the fp32 bound)
    dC2 = torch.full((M, N), float("nan"), device="cuda")
    st = sg.sgemm_ex(ta, tb, M, N, K, 1.0, dA.data_ptr(), lda, dB.data_ptr(), ldb, 0.0, dC2.data_ptr(),
                     N, torch.cuda.current_stream(), sg.PATH_3XTF32, 1)
    torch.cuda.synchronize()
    assert st == 0
    diff = np.abs(out - dC2.cpu().numpy())
    assert np.all(diff <= 2 * 4 * K * 2.0 ** -24 * np.abs(opA).max() * np.abs(opB).max() * K)


@pytest.mark.parametrize("ta,tb,N", [("N", "N", 128), ("N", "T", 128), ("N", "T", 96)])
def test_narrow_tile_last_wave_slices_sampled(oracle_mod, ta, tb, N):
    """20480 x N x 256 with A split in the kernel: 160 tiles of 128 x 128 (A_hi in
    TMEM, A_lo in shared memory, one N = 2 x width MMA over [B_hi | B_lo]); the
    8 after the full wave run as 64-wide units, whose hi*lo products land at
    column 128 + 64 of the accumulator.  N = 96 also cuts the last unit's
    columns short.  Seeded samples, the last rows and columns included."""
    import torch
    M, K = 20480, 256
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ldb = N if tb == "N" else K
    st, p = sg.sgemm_plan(ta, tb, M, N, K, K, ldb, N, num_sms=sms)
    assert st == 0 and p["tile_n"] == 128 and (sms != 152 or p["split"] == 2)
    opA = gi.random_matrix(121, M, K)
    opB = gi.random_matrix(122, K, N)
    A, B = stored(opA, ta), stored(opB, tb)
    C = gi.random_matrix(123, M, N)
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (A, B, C))
    st = sg.sgemm(ta, tb, M, N, K, 1.5, dA.data_ptr(), K, dB.data_ptr(), ldb, -0.5, dC.data_ptr(), N,
                  torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert st == 0 and sg.sgemm_device_error(torch.cuda.current_stream()) == 0
    out = dC.cpu().numpy()
    rows, cols = gi.sample_points(M, N, 16000, seed=124)
    # and every column of the last 1024 rows (the last tiles in raster order)
    tail_r = np.repeat(np.arange(M - 1024, M), N)
    tail_c = np.tile(np.arange(N), 1024)
    rows, cols = np.concatenate([rows, tail_r]), np.concatenate([cols, tail_c])
    ref, bound = oracle_mod.gemm_f64(ta, tb, M, N, K, 1.5, A, K, B, ldb, -0.5, C, N,
                                     points=(rows, cols))
    rep = oracle_mod.compare(out[rows, cols], ref, bound, K, 1.5)
    assert rep["pass"], rep
