"""Host-side checks of the C-ABI library that need no GPU: it builds, loads,
exports every entry point the header declares, validates arguments BLAS-style
before touching the device, and its selector makes the documented choices."""
import ctypes
import os
import re
import subprocess

import pytest

import dense_fp32_gemm_05_gb300 as sg
from dense_fp32_gemm_05_gb300 import build as sgbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    sgbuild.build()
    return sg.load()


def header_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(sgemm\w*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_entry_points():
    names = header_functions()
    assert {"sgemm", "sgemm_ex", "sgemm_plan", "sgemm_status_string"} <= set(names)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", sg.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(\w+)$", out, flags=re.M))
    for name in header_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None
    for name in sg.exported_symbols():
        assert name in exported


def test_version_and_status_strings(lib):
    assert sg.sgemm_version() >= 100
    for st in (0, 1, 2, 3, 4, 5):
        assert sg.sgemm_status_string(st)
    assert "argument" in sg.sgemm_status_string(-3)


FAKE = 1 << 20   # never dereferenced: every case below fails validation first


@pytest.mark.parametrize("args,want", [
    (("X", "N", 4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4), -1),
    (("N", "Z", 4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4), -2),
    (("N", "N", -1, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4), -3),
    (("N", "N", 4, -2, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4), -4),
    (("N", "N", 4, 4, -5, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4), -5),
    (("N", "N", 4, 4, 4, 1.0, 0, 4, FAKE, 4, 0.0, FAKE, 4), -7),
    (("N", "N", 4, 4, 8, 1.0, FAKE, 7, FAKE, 4, 0.0, FAKE, 4), -8),
    (("T", "N", 9, 4, 8, 1.0, FAKE, 8, FAKE, 4, 0.0, FAKE, 4), -8),
    (("N", "N", 4, 4, 4, 1.0, FAKE, 4, 0, 4, 0.0, FAKE, 4), -9),
    (("N", "N", 4, 6, 4, 1.0, FAKE, 4, FAKE, 5, 0.0, FAKE, 6), -10),
    (("N", "T", 4, 6, 9, 1.0, FAKE, 9, FAKE, 8, 0.0, FAKE, 6), -10),
    (("N", "N", 4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, 0, 4), -12),
    (("N", "N", 4, 6, 4, 1.0, FAKE, 4, FAKE, 6, 0.0, FAKE, 5), -13),
    (("N", "N", 2 ** 31, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4), -3),
])
def test_argument_validation_without_gpu(lib, args, want):
    assert sg.sgemm(*args) == want
    assert sg.sgemm_ex(*args, path=sg.PATH_FFMA, split=1) == want


def test_epilogue_argument_validation_without_gpu(lib):
    # checked before any CUDA call: unknown activation, then the GEMM arguments
    assert sg.sgemm_epilogue("N", "N", 4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4,
                             activation=3) == -16
    assert sg.sgemm_epilogue("Q", "N", 4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4,
                             bias=FAKE, activation=sg.ACT_RELU) == -1
    assert sg.sgemm_epilogue("N", "N", 4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 3,
                             row_scale=FAKE) == -13
    assert sg.sgemm_epilogue("N", "N", 0, 4, 4, 1.0, 0, 4, 0, 4, 0.0, 0, 4,
                             bias=FAKE, activation=sg.ACT_RELU) == sg.SGEMM_OK


def test_quick_return_touches_nothing(lib):
    # M == 0 / N == 0: nothing to do, valid with null pointers, no CUDA call
    assert sg.sgemm("N", "N", 0, 5, 7, 1.0, 0, 7, 0, 5, 0.0, 0, 5) == sg.SGEMM_OK
    assert sg.sgemm("T", "T", 5, 0, 7, 1.0, 0, 5, 0, 7, 1.0, 0, 1) == sg.SGEMM_OK


def test_aux_argument_errors(lib):
    assert sg.sgemm_ex("N", "N", 4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4,
                       path=9) == sg.SGEMM_ERR_ARG
    assert sg.sgemm_ex("N", "N", 4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4,
                       split=-1) == sg.SGEMM_ERR_ARG
    st, _ = sg.sgemm_plan("N", "N", 8, 8, 8, 8, 8, 8, num_sms=0)
    assert st == sg.SGEMM_ERR_ARG


def test_plan_vector_and_edge_path(lib):
    F = sg.PATH_FFMA
    st, p = sg.sgemm_plan("N", "N", 4096, 4096, 4096, 4096, 4096, 4096, path=F)
    assert st == 0 and p["vector"] == 1 and p["path"] == F
    assert (p["tile_m"], p["tile_n"]) == (128, 128)
    # odd leading dimensions: 16-byte loads are illegal, the 4-byte path runs
    st, p = sg.sgemm_plan("N", "T", 4095, 3073, 1537, 1537, 1537, 3073, path=F)
    assert st == 0 and p["vector"] == 0
    # misaligned base pointer
    st, p = sg.sgemm_plan("N", "N", 512, 512, 512, 512, 512, 512, a_aligned=False, path=F)
    assert st == 0 and p["vector"] == 0


def test_plan_auto_path_choice(lib):
    # large problems go to the tensor cores (3xTF32), with N-sized MMA tiles
    st, p = sg.sgemm_plan("N", "N", 4096, 4096, 4096, 4096, 4096, 4096)
    assert st == 0 and p["path"] == sg.PATH_3XTF32 and p["tile_n"] == 256
    st, p = sg.sgemm_plan("N", "T", 16384, 64, 8192, 8192, 8192, 64)
    assert st == 0 and p["path"] == sg.PATH_3XTF32 and p["tile_n"] == 64
    # odd leading dimensions do not matter to the tensor-core path (pre-pass)
    st, p = sg.sgemm_plan("T", "T", 4095, 3073, 1537, 4095, 1537, 3073)
    assert st == 0 and p["path"] == sg.PATH_3XTF32
    # small problems run the one-launch 16 x 16 FFMA kernel ...
    for shp in [(256, 256, 256), (128, 128, 128), (17, 17, 32), (384, 384, 384), (2048, 32, 512)]:
        st, p = sg.sgemm_plan("N", "N", *shp, shp[2], shp[1], shp[1])
        assert st == 0 and p["path"] == sg.PATH_FFMA and p["tile_m"] == p["tile_n"] == 16, shp
        assert p["split"] == 1 and p["ctas"] == ((shp[0] + 15) // 16) * ((shp[1] + 15) // 16)
    # ... but long K, many tiles or more flops go to the tensor cores when K >= 32
    for shp in [(128, 128, 2048), (256, 256, 1024), (1024, 1024, 32), (448, 448, 448)]:
        st, p = sg.sgemm_plan("N", "N", *shp, shp[2], shp[1], shp[1])
        assert st == 0 and p["path"] == sg.PATH_3XTF32, shp
    # short K stays on the CUDA cores
    for shp in [(8192, 8192, 16), (256, 256, 31), (17, 17, 1)]:
        st, p = sg.sgemm_plan("N", "N", *shp, shp[2], shp[1], shp[1])
        assert st == 0 and p["path"] == sg.PATH_FFMA, shp
    # TF32 is never chosen automatically
    for shp in [(4096, 4096, 4096), (1024, 1024, 1024), (300, 300, 40)]:
        st, p = sg.sgemm_plan("N", "N", *shp, shp[2], shp[1], shp[1])
        assert p["path"] != sg.PATH_TF32


def test_plan_sm_pair_tiles(lib):
    # both operands through the split pre-pass and M > 128: 256-row tiles on SM pairs
    st, p = sg.sgemm_plan("N", "N", 4096, 4096, 4096, 4096, 4096, 4096)
    assert st == 0 and p["tile_m"] == 256 and p["ctas"] % 2 == 0
    st, p = sg.sgemm_plan("T", "N", 4096, 3000, 1000, 4096, 3000, 3000, path=sg.PATH_3XTF32)
    assert st == 0 and p["tile_m"] == 256
    # an operand split in shared memory (K-contiguous, small other side): single SMs
    st, p = sg.sgemm_plan("N", "N", 2048, 2048, 2048, 2048, 2048, 2048)
    assert st == 0 and p["tile_m"] == 128
    st, p = sg.sgemm_plan("N", "T", 16384, 64, 8192, 8192, 8192, 64)
    assert st == 0 and p["tile_m"] == 128
    # M fits one 128-row tile
    st, p = sg.sgemm_plan("T", "N", 128, 4096, 4096, 128, 4096, 4096, path=sg.PATH_3XTF32)
    assert st == 0 and p["tile_m"] == 128


def test_plan_tensor_core_stream_k(lib):
    # 16384 x 64 x 8192 skinny: 128 tiles for 152 SMs, 256 k-blocks each ->
    # the iterations are shared by one CTA per SM
    st, p = sg.sgemm_plan("N", "T", 16384, 64, 8192, 8192, 8192, 64, num_sms=152)
    assert st == 0 and p["path"] == sg.PATH_3XTF32 and p["ctas"] == 152 and p["split"] == 2
    # 16 tiles: 9 CTAs per tile (144) keep every range inside one tile
    st, p = sg.sgemm_plan("N", "T", 2048, 64, 8192, 8192, 8192, 64, num_sms=152)
    assert st == 0 and p["ctas"] == 144 and p["split"] == 9
    # 1024^3: 32 tiles of 128 x 256, 4 CTAs each
    st, p = sg.sgemm_plan("N", "N", 1024, 1024, 1024, 1024, 1024, 1024, num_sms=152)
    assert st == 0 and p["ctas"] == 128 and p["split"] == 4
    # deep K on a few tiles
    st, p = sg.sgemm_plan("N", "N", 512, 512, 16384, 16384, 512, 512, num_sms=152)
    assert st == 0 and p["path"] == sg.PATH_3XTF32 and p["ctas"] == 152
    # 2048^3: the partial tiles' traffic outweighs the 128/152 fill
    st, p = sg.sgemm_plan("N", "N", 2048, 2048, 2048, 2048, 2048, 2048, num_sms=152)
    assert st == 0 and p["ctas"] == 128 and p["split"] == 1
    # a full wave or more: never over every tile (4096^3 stays on SM pairs;
    # its last wave of 28 tiles is shared by the 76 pairs: 3 per tile)
    st, p = sg.sgemm_plan("N", "N", 4096, 4096, 4096, 4096, 4096, 4096, num_sms=152)
    assert st == 0 and p["tile_m"] == 256 and p["split"] == 3 and p["ctas"] == 152
    # forced: split = 1 keeps tiles whole; split = s shares among s x tiles CTAs
    st, p = sg.sgemm_plan("N", "T", 16384, 64, 8192, 8192, 8192, 64, num_sms=152, split=1)
    assert st == 0 and p["ctas"] == 128 and p["split"] == 1
    st, p = sg.sgemm_plan("T", "N", 300, 260, 1000, 300, 260, 260, num_sms=152,
                          path=sg.PATH_3XTF32, split=3)
    assert st == 0 and p["tile_m"] == 128 and p["ctas"] == 18 and p["split"] == 3
    # capped at 8 CTAs per SM and at one k-block per CTA
    st, p = sg.sgemm_plan("N", "N", 4096, 4096, 4096, 4096, 4096, 4096, num_sms=152,
                          path=sg.PATH_3XTF32, split=64)
    assert st == 0 and p["ctas"] == 8 * 152
    st, p = sg.sgemm_plan("N", "N", 256, 256, 96, 96, 256, 256, path=sg.PATH_3XTF32, split=8)
    assert st == 0 and p["ctas"] == 12


def test_plan_tensor_core_last_wave_slices(lib):
    # 4096 x 4096 x 256 on SM pairs: 256 tiles = 3 waves of 76 + 28; with K this
    # short a shared last wave costs more in partial sums than it saves, and
    # the 28 run as 56 half-width units (a half unit measured ~0.9 of a tile)
    st, p = sg.sgemm_plan("N", "N", 4096, 4096, 256, 256, 4096, 4096, num_sms=152)
    assert st == 0 and p["tile_m"] == 256 and p["split"] == 2
    # 4096^3 and 8192^3: the last wave shared by all pairs instead (stream-K)
    for n in (4096, 8192):
        st, p = sg.sgemm_plan("N", "N", n, n, n, n, n, n, num_sms=152)
        assert st == 0 and p["tile_m"] == 256 and p["split"] > 1 and p["ctas"] == 152
    # 4095 x 3073 x 1537: 208 tiles = 2 waves + 56; narrow units would cost
    # more rounds than one more wave of whole tiles (1.43x measured)
    st, p = sg.sgemm_plan("N", "N", 4095, 3073, 1537, 1537, 3073, 3073, num_sms=152)
    assert st == 0 and p["tile_m"] == 256 and p["split"] == 1
    # single SMs with A split into TMEM: 160 tiles = 152 + 8 -> the 8 as narrower units
    st, p = sg.sgemm_plan("N", "N", 2560, 2048, 256, 256, 2048, 2048, num_sms=152)
    assert st == 0 and p["tile_m"] == 128 and p["split"] in (2, 4)


def test_plan_ffma_stream_k_tail(lib):
    # 4096^3: 1024 tiles = 3 full waves of 304 + 112; the 112 are shared by 304 CTAs
    st, p = sg.sgemm_plan("N", "N", 4096, 4096, 4096, 4096, 4096, 4096, num_sms=152,
                          path=sg.PATH_FFMA)
    assert st == 0 and p["split"] > 1 and p["ctas"] == 912 + 304
    # exactly 4 waves (4096 x 4864): nothing left over, every tile whole
    st, p = sg.sgemm_plan("N", "N", 4096, 4864, 4096, 4096, 4864, 4864, num_sms=152,
                          path=sg.PATH_FFMA)
    assert st == 0 and p["split"] == 1 and p["ctas"] == 1216
    # a short K leaves too few k-tiles to share: the tail stays whole
    st, p = sg.sgemm_plan("N", "N", 4096, 4096, 64, 64, 4096, 4096, num_sms=152,
                          path=sg.PATH_FFMA)
    assert st == 0 and p["split"] == 1


def test_plan_split_k_for_small_grids(lib):
    F = sg.PATH_FFMA
    # 256 x 256 x 2048: 4 tiles for 304 CTA slots -> the K loop is split
    st, p = sg.sgemm_plan("N", "N", 256, 256, 2048, 2048, 256, 256, num_sms=152, path=F)
    assert st == 0 and p["split"] > 1 and p["tile_m"] == 128
    # 256^3 forced to FFMA without a split: the one-launch small kernel
    st, p = sg.sgemm_plan("N", "N", 256, 256, 256, 256, 256, 256, num_sms=152, path=F)
    assert st == 0 and p["split"] == 1 and p["tile_m"] == p["tile_n"] == 16
    # 16384 x 64 x 8192 skinny on the FFMA path: 128 tiles, long K -> split
    st, p = sg.sgemm_plan("N", "T", 16384, 64, 8192, 8192, 8192, 64, num_sms=152,
                          path=sg.PATH_FFMA)
    assert st == 0 and p["split"] > 1
    # forced split is honoured, forced 1 disables it
    st, p = sg.sgemm_plan("N", "N", 256, 256, 256, 256, 256, 256, split=1, path=F)
    assert p["split"] == 1
    st, p = sg.sgemm_plan("N", "N", 256, 256, 256, 256, 256, 256, split=3, path=F)
    assert p["split"] == 3


def test_plan_thin_problems_take_the_gemv_path(lib):
    # min(M, N) <= 16 ("Matmul II", section 8: decode's M = 1 to a few dozen)
    for (ta, tb, M, N, K) in [("N", "T", 1, 16384, 8192), ("N", "T", 4, 4096, 4096),
                              ("N", "N", 16, 4096, 4096), ("T", "N", 16384, 8, 8192),
                              ("N", "T", 5, 5, 5), ("N", "T", 16, 4096, 16)]:
        lda = K if ta == "N" else M
        ldb = N if tb == "N" else K
        st, p = sg.sgemm_plan(ta, tb, M, N, K, lda, ldb, N)
        assert st == 0 and p["path"] == sg.PATH_GEMV, (ta, tb, M, N, K)
        assert p["tile_m"] == min(M, N)
    # large operand K-contiguous (weights stored [N][K]) and S > 4: the
    # tensor cores are ahead there
    for (ta, tb, M, N, K) in [("N", "T", 16, 16384, 8192), ("N", "T", 8, 4096, 4096),
                              ("N", "N", 16384, 8, 8192), ("N", "T", 5, 4096, 1024)]:
        lda = K if ta == "N" else M
        ldb = N if tb == "N" else K
        st, p = sg.sgemm_plan(ta, tb, M, N, K, lda, ldb, N)
        assert st == 0 and p["path"] == sg.PATH_3XTF32, (ta, tb, M, N, K)
    # forced, the thin path still takes them
    st, p = sg.sgemm_plan("N", "T", 16, 16384, 8192, 8192, 8192, 16384, path=sg.PATH_GEMV)
    assert st == 0 and p["path"] == sg.PATH_GEMV
    # a large operand the tensor-core kernel cannot split itself stays thin
    st, p = sg.sgemm_plan("N", "T", 16, 16384, 8191, 8191, 8191, 16384)
    assert st == 0 and p["path"] == sg.PATH_GEMV
    st, p = sg.sgemm_plan("N", "T", 16, 16384, 8192, 8192, 8192, 16384, True, False, True)
    assert st == 0 and p["path"] == sg.PATH_GEMV
    # 17 to 128 with the large operand's rows along the long side (aligned):
    # the thin path's tensor-core form; otherwise, and from 129, the tile paths
    for (ta, tb, M, N, K) in [("N", "N", 17, 4096, 4096), ("N", "N", 32, 16384, 8192),
                              ("T", "T", 16384, 24, 8192), ("N", "N", 33, 4096, 4096),
                              ("N", "N", 64, 16384, 8192), ("T", "T", 16384, 48, 8192),
                              ("N", "N", 65, 16384, 8192), ("N", "N", 128, 16384, 8192)]:
        lda = K if ta == "N" else M
        ldb = N if tb == "N" else K
        st, d = sg.sgemm_plan_detail(ta, tb, M, N, K, lda, ldb, N)
        assert st == 0 and d["path"] == sg.PATH_GEMV and d["tile_n"] == 128, (ta, tb, M, N, K)
    for args in [("N", "N", 129, 4096, 4096, 4096, 4096, 4096),      # S = 129
                 ("N", "T", 24, 4096, 4096, 4096, 4096, 4096),       # large operand K-contiguous
                 ("N", "N", 24, 4094, 4096, 4096, 4094, 4094),       # its ld not a multiple of 4
                 ("N", "N", 24, 4096, 16, 16, 4096, 4096)]:          # K < 32
        st, p = sg.sgemm_plan(*args)
        assert st == 0 and p["path"] != sg.PATH_GEMV, args
    # forced: 17..32 only where the tensor-core form applies
    st, p = sg.sgemm_plan("N", "N", 24, 4096, 16, 16, 4096, 4096, path=sg.PATH_GEMV)
    assert st == 0 and p["path"] == sg.PATH_GEMV
    st, _ = sg.sgemm_plan("N", "T", 24, 4096, 4096, 4096, 4096, 4096, path=sg.PATH_GEMV)
    assert st == sg.SGEMM_ERR_UNSUPPORTED
    # forced on a wide problem: refused
    st, _ = sg.sgemm_plan("N", "N", 129, 129, 129, 129, 129, 129, path=sg.PATH_GEMV)
    assert st == sg.SGEMM_ERR_UNSUPPORTED
    st, _ = sg.sgemm_plan("N", "N", 64, 64, 64, 64, 64, 64, path=5)
    assert st == sg.SGEMM_ERR_ARG


def test_plan_forced_tensor_core_path(lib):
    st, p = sg.sgemm_plan("N", "N", 1024, 1024, 1024, 1024, 1024, 1024, path=sg.PATH_3XTF32)
    assert st == 0 and p["path"] == sg.PATH_3XTF32


def test_plan_detail_agrees_with_plan(lib):
    """sgemm_plan_detail repeats sgemm_plan's fields and spells out the
    tensor-core variant; NULL output is rejected."""
    shapes = [("N", "N", 4096, 4096, 4096), ("T", "N", 513, 64, 2000), ("N", "T", 16384, 64, 8192),
              ("N", "N", 300, 200, 16), ("N", "T", 4, 5000, 300), ("T", "T", 4095, 3073, 1537)]
    for ta, tb, M, N, K in shapes:
        lda = K if ta == "N" else M
        ldb = N if tb == "N" else K
        st, p = sg.sgemm_plan(ta, tb, M, N, K, lda, ldb, N)
        st2, d = sg.sgemm_plan_detail(ta, tb, M, N, K, lda, ldb, N)
        assert st == st2 == 0
        for k in p:
            assert d[k] == p[k], (ta, tb, M, N, K, k)
        if d["path"] in (sg.PATH_3XTF32, sg.PATH_TF32):
            assert d["k_block"] in (16, 32) and d["accumulators"] in (1, 2, 3)
            assert not (d["pair"] and (d["fuse_a"] or d["fuse_b"]))
            assert not (d["wide"] and not d["fuse_a"])
        else:
            assert d["pair"] == d["fuse_a"] == d["fuse_b"] == d["wide"] == 0
    assert lib.sgemm_plan_detail(b"N", b"N", 8, 8, 8, 8, 8, 8, 1, 1, 1, 0, 0, 152, None) == -15


def test_plan_detail_reaches_every_pinned_variant(lib):
    """The shapes of the GPU 3xTF32 variant pins reach the variants they are
    named for (152 SMs), so a selector change cannot empty those pins."""
    from tests.test_gpu_3xtf32_variants import VARIANTS
    seen = set()
    for name, ta, tb, M, N, K, split, want in VARIANTS:
        lda = K if ta == "N" else M
        ldb = N if tb == "N" else K
        st, d = sg.sgemm_plan_detail(ta, tb, M, N, K, lda, ldb, N, path=sg.PATH_3XTF32,
                                     split=split, num_sms=152)
        assert st == 0
        assert {k: d[k] for k in want} == want, (name, d)
        seen.add((d["tile_n"], d["pair"], d["fuse_a"], d["fuse_b"], d["wide"],
                  d["sk_ctas"] > 0, d["sk_tail"], d["tail_nsplit"] > 1))
    # every kernel template of the 3xTF32 path is among them
    templates = {(t, p, w) for t, p, _, _, w, _, _, _ in seen}
    assert templates >= {(256, 1, 0), (128, 1, 0), (64, 1, 0), (256, 0, 0), (128, 0, 0),
                         (64, 0, 0), (128, 0, 1), (64, 0, 1)}


def test_tf32_rate_probe_argument_errors(lib):
    """The rate probe rejects its arguments before touching a device."""
    v = ctypes.c_double(0.0)
    assert lib.sgemm_probe_tf32_rate(10, ctypes.byref(v)) == -1
    assert lib.sgemm_probe_tf32_rate(1 << 21, ctypes.byref(v)) == -1
    assert lib.sgemm_probe_tf32_rate(4096, None) == -2


def test_small_kernel_selector_boundaries(lib):
    """The rule's edges, on the CPU side of the plan: 2MNK <= 1.2e8, K <= 512
    and at most 1024 tiles of 16 x 16 take the small kernel; a forced split
    or any edge crossed takes the tile kernels."""
    def small(M, N, K, path=sg.PATH_AUTO, split=0):
        st, info = sg.sgemm_plan_detail("N", "N", M, N, K, K, N, N, 1, 1, 1, path, split, 152)
        assert st == 0
        return info["tile_m"] == 16
    assert small(48, 48, 512) and not small(48, 48, 513)
    assert small(512, 512, 64) and not small(512, 528, 64)        # 1024 / 1056 tiles
    assert small(384, 384, 384) and not small(400, 400, 400)      # 1.13e8 / 1.28e8 flops
    assert small(256, 256, 256, sg.PATH_FFMA, 1)
    assert not small(256, 256, 256, sg.PATH_FFMA, 2)              # forced split-K
    assert not small(256, 256, 256, sg.PATH_3XTF32)               # forced tensor cores
    assert not small(8, 256, 256)                                 # thin: GEMV


def test_plan_detail_thin_problems_on_the_tensor_cores(lib):
    """S >= 12 with the large operand's rows along the long dimension (16-byte
    aligned, leading dimension a multiple of 4): the thin path's tensor-core
    form, 128 columns per CTA; otherwise the CUDA-core forms (tile_n 0)."""
    def detail(ta, tb, M, N, K, lda, ldb, a_al=1, b_al=1):
        st, info = sg.sgemm_plan_detail(ta, tb, M, N, K, lda, ldb, N, a_al, b_al, 1, 0, 0, 152)
        assert st == 0 and info["path"] == sg.PATH_GEMV
        return info
    i = detail("N", "N", 16, 16384, 8192, 8192, 16384)
    assert (i["tile_n"], i["ctas"], i["split"], i["k_block"], i["accumulators"]) == (128, 128, 1, 32, 8)
    i = detail("T", "N", 16384, 12, 8192, 16384, 12)          # N small: A ('T') is the large operand
    assert i["tile_n"] == 128 and i["ctas"] == 128
    i = detail("N", "N", 16, 300, 40000, 40000, 300)          # few columns, long K: split over CTAs
    assert i["tile_n"] == 128 and i["split"] == 50 and i["ctas"] == 150
    for args in [("N", "N", 11, 16384, 8192, 8192, 16384),     # S below 12
                 ("N", "N", 16, 1001, 500, 500, 1001),         # ldb not a multiple of 4
                 ("N", "N", 16, 16384, 8192, 8192, 16384, 1, 0),   # B not 16-byte aligned
                 ("N", "T", 16, 4096, 4096, 4096, 4096)]:      # rows along K (dot form)
        st, info = sg.sgemm_plan_detail(*args[:7], args[3], *(args[7:] or (1, 1)), 1, 4, 0, 152)
        assert st == 0 and info["tile_n"] == 0, args


def test_ffma_pre_transpose_selector():
    """The FFMA tile path copies a K-contiguous operand transposed when the
    grid is large (M, N >= 128, K >= 256) and the problem's other side is at
    least 2048: bit 0 op(A) (A 'N'), bit 1 op(B) (B 'T')."""
    cases = [("N", "N", 4096, 4096, 4096, 1), ("N", "T", 4096, 4096, 4096, 3),
             ("T", "N", 4096, 4096, 4096, 0), ("T", "T", 4096, 4096, 4096, 2),
             ("N", "N", 4096, 2047, 4096, 0), ("N", "T", 2047, 4096, 4096, 1),
             ("N", "N", 4096, 4096, 255, 0), ("N", "N", 127, 4096, 4096, 0)]
    for ta, tb, M, N, K, want in cases:
        lda = K if ta == "N" else M
        ldb = N if tb == "N" else K
        st, info = sg.sgemm_plan_detail(ta, tb, M, N, K, lda, ldb, N, path=sg.PATH_FFMA)
        assert st == 0 and info["path"] == sg.PATH_FFMA, (ta, tb, M, N, K)
        assert info["pre_transpose"] == want, (ta, tb, M, N, K, info)
    # the small-problem kernel, the tensor cores and the thin path never copy
    for args, path in [(("N", "N", 256, 256, 256, 256, 256, 256), sg.PATH_FFMA),
                       (("N", "N", 4096, 4096, 4096, 4096, 4096, 4096), sg.PATH_AUTO),
                       (("N", "T", 4, 4096, 4096, 4096, 4096, 4096), sg.PATH_AUTO)]:
        st, info = sg.sgemm_plan_detail(*args, path=path)
        assert st == 0 and info["pre_transpose"] == 0, (args, info)


def test_b_split_in_the_kernel_only_for_short_m_or_narrow_n():
    """B (K-contiguous) is split in shared memory inside the tensor-core
    kernel only up to M = 1024, or up to M = 2048 for a narrow B (N <= 128)
    or a problem under a GFLOP; wider problems take the pre-pass (measured
    faster from M = 1536 on)."""
    cases = [(("N", "T", 1024, 1024, 1024, 1024, 1024, 1024), 1, 1),
             (("N", "T", 2048, 2048, 2048, 2048, 2048, 2048), 1, 0),
             (("N", "T", 1536, 4096, 1536, 1536, 1536, 4096), 0, 0),
             (("N", "T", 2048, 64, 8192, 8192, 8192, 64), 1, 1),
             (("N", "T", 16384, 64, 8192, 8192, 8192, 64), 1, 0),
             (("T", "T", 2048, 1024, 2048, 2048, 2048, 1024), 0, 0),
             # under a GFLOP the pre-pass launch costs more than the split
             (("N", "T", 1536, 256, 256, 256, 256, 256), 1, 1)]
    for args, fa, fb in cases:
        st, d = sg.sgemm_plan_detail(*args, path=sg.PATH_3XTF32)
        assert st == 0 and (d["fuse_a"], d["fuse_b"]) == (fa, fb), (args, d)
    # both operands pre-split and enough rows: the SM-pair kernel
    st, d = sg.sgemm_plan_detail("T", "T", 2048, 1024, 2048, 2048, 2048, 1024)
    assert st == 0 and d["pair"] == 1


def test_stream_k_over_every_tile_only_when_it_pays():
    """Stream-K over every tile (single SMs), or whole tiles: whole tiles only
    where they already fill >= 60 % of the SMs, the operand panels that tiles
    share do not fit in L2, and the tile grid is at least as tall as wide
    with 4 columns or more (the measured cases of the selector's comment)."""
    cases = [(("N", "N"), (2048, 2048, 8192), 0), (("N", "N"), (3072, 1280, 8192), 0),
             (("N", "N"), (4096, 1024, 8192), 0), (("T", "T"), (768, 4096, 8192), 152),
             (("N", "T"), (1024, 4096, 8192), 152), (("N", "N"), (8192, 512, 8192), 152),
             (("N", "N"), (1280, 2048, 8192), 152), (("N", "N"), (1280, 2048, 4096), 152),
             (("N", "T"), (16384, 64, 8192), 152), (("N", "N"), (1024, 1024, 1024), 128)]
    for (ta, tb), (M, N, K), sk in cases:
        lda = K if ta == "N" else M
        ldb = N if tb == "N" else K
        st, d = sg.sgemm_plan_detail(ta, tb, M, N, K, lda, ldb, N)
        assert st == 0 and d["sk_ctas"] == sk, ((ta, tb, M, N, K), d)
    # a forced split still shares the k-blocks
    st, d = sg.sgemm_plan_detail("N", "N", 2048, 2048, 8192, 8192, 2048, 2048, split=2)
    assert st == 0 and d["sk_ctas"] > 0


def test_plan_invariants_over_random_shapes():
    """The selector's decisions over 3000 seeded random problems (sizes
    around every threshold, all layouts, padded leading dimensions,
    misaligned bases, forced paths and splits): sgemm_plan and
    sgemm_plan_detail agree field for field, forced paths are honoured, and
    each plan is one the launchers accept (pairs never split an operand in
    the kernel, an operand is split in the kernel only when TMA may read it
    raw, the thin path stays within its range, the FFMA pre-pass only copies
    K-contiguous operands)."""
    import random
    rng = random.Random(1234)
    dims = [1, 2, 3, 5, 8, 12, 16, 17, 24, 31, 32, 33, 63, 64, 65, 100, 127, 128, 129, 200, 255,
            256, 257, 500, 511, 512, 513, 1000, 1023, 1024, 1500, 2047, 2048, 2049, 3000, 4095,
            4096, 6000, 8192, 16384, 65536]
    for _ in range(3000):
        M, N, K = rng.choice(dims), rng.choice(dims), rng.choice(dims)
        ta, tb = rng.choice("NT"), rng.choice("NT")
        lda = (K if ta == "N" else M) + rng.choice([0, 0, 1, 3, 4])
        ldb = (N if tb == "N" else K) + rng.choice([0, 0, 1, 4])
        ldc = N + rng.choice([0, 1])
        al = [rng.random() < 0.85 for _ in range(3)]
        path = rng.choice([0, 0, 0, 1, 2, 3, 4])
        split = rng.choice([0, 0, 1, 2, 5])
        key = (ta, tb, M, N, K, lda, ldb, ldc, al, path, split)
        st, d = sg.sgemm_plan_detail(ta, tb, M, N, K, lda, ldb, ldc, *al, path, split, 152)
        st2, p = sg.sgemm_plan(ta, tb, M, N, K, lda, ldb, ldc, *al, path, split, 152)
        assert st == st2, key
        if st != 0:
            assert path == sg.PATH_GEMV and st == sg.SGEMM_ERR_UNSUPPORTED, key
            continue
        for f in ("path", "tile_m", "tile_n", "ctas", "split", "vector"):
            assert d[f] == p[f], (f, key, d, p)
        assert d["path"] in (1, 2, 3, 4) and d["ctas"] >= 1 and d["split"] >= 1, (key, d)
        if path:
            assert d["path"] == path, (key, d)
        if d["path"] == sg.PATH_GEMV:
            assert min(M, N) <= 128 and d["tile_m"] == min(M, N), (key, d)
            if d["tile_n"] == 128:
                # the tensor-core form: 128 columns of the long side per CTA,
                # split = CTAs along K (at least 32 k each), 8 accumulators
                P = max(M, N)
                assert d["ctas"] == (P + 127) // 128 * d["split"], (key, d)
                assert d["split"] <= max(1, K // 32) and d["accumulators"] == 8, (key, d)
            else:
                assert min(M, N) <= 16 and d["tile_n"] == 0, (key, d)
        if d["path"] in (sg.PATH_3XTF32, sg.PATH_TF32):
            assert d["tile_n"] in (64, 128, 256) and d["k_block"] in (16, 32), (key, d)
            assert d["pair"] == (d["tile_m"] == 256), (key, d)
            assert not (d["pair"] and (d["fuse_a"] or d["fuse_b"])), (key, d)
            assert d["sk_ctas"] <= 8 * 152 and d["pre_transpose"] == 0, (key, d)
            if d["fuse_a"]:
                assert ta == "N" and al[0] and lda % 4 == 0, (key, d)
            if d["fuse_b"]:
                assert tb == "T" and al[1] and ldb % 4 == 0, (key, d)
        if d["path"] == sg.PATH_FFMA:
            assert not (d["tile_n"] == 16 and d["pre_transpose"]), (key, d)
            assert not (d["pre_transpose"] & 1 and ta != "N"), (key, d)
            assert not (d["pre_transpose"] & 2 and tb != "T"), (key, d)
