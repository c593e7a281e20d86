// Host-side argument checks and the per-shape selector.  Pure C++: no CUDA
// calls, so the same logic is reachable through sgemm_plan() on a machine
// without a GPU.
#pragma once

#include <algorithm>
#include <cstdint>

#include "../../include/sgemm_gb300.h"

namespace sgemm_gb300 {

inline bool is_notrans(char t) { return t == 'N' || t == 'n'; }
inline bool is_trans(char t) { return t == 'T' || t == 't' || t == 'C' || t == 'c'; }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// BLAS-style validation; returns 0 or -(1-based index of the bad argument).
// Sizes must fit in 31 bits (the kernels index tiles with int).
inline int check_args(char ta, char tb, int64_t M, int64_t N, int64_t K, float alpha,
                      const float *A, int64_t lda, const float *B, int64_t ldb, float beta,
                      const float *C, int64_t ldc, bool pointers_checked = true) {
    (void)beta;
    const int64_t lim = INT32_MAX;
    if (!is_notrans(ta) && !is_trans(ta)) return -1;
    if (!is_notrans(tb) && !is_trans(tb)) return -2;
    if (M < 0 || M > lim) return -3;
    if (N < 0 || N > lim) return -4;
    if (K < 0 || K > lim) return -5;
    const int64_t a_row = is_notrans(ta) ? K : M;
    const int64_t b_row = is_notrans(tb) ? N : K;
    if (lda < std::max<int64_t>(1, a_row)) return -8;
    if (ldb < std::max<int64_t>(1, b_row)) return -10;
    if (ldc < std::max<int64_t>(1, N)) return -13;
    if (pointers_checked) {
        const bool need_ab = M > 0 && N > 0 && K > 0 && alpha != 0.0f;
        if (need_ab && A == nullptr) return -7;
        if (need_ab && B == nullptr) return -9;
        if (M > 0 && N > 0 && C == nullptr) return -12;
    }
    return 0;
}

struct Plan {
    int path = SGEMM_PATH_FFMA;
    int split = 1;      // FFMA: CTAs per shared tile, rounded up (1 = every tile whole)
    int ctas = 0;       // FFMA: CTAs sharing the iterations of the tiles after dp_tiles
    int dp_tiles = 0;   // tiles computed whole (tensor cores: at full width)
    int tile_m = 128, tile_n = 128;
    int vector = 1;     // 16-byte operand loads (else 4-byte edge path)
    int c_vector = 1;   // 16-byte C accesses
    int group_m = 8;    // rasterisation group height (tiles)
    int tail_nsplit = 1;  // tensor cores: column slices of the last-wave tiles
    int fuse_a = 1;       // tensor cores: split A in shared memory when its layout allows
    int fuse_b = 1;       // tensor cores: same for B
    int pair = 0;         // tensor cores: 256-row tiles on a pair of SMs (cta_group::2)
    int tc_sk = 0;        // tensor cores: stream-K CTAs sharing all k-block iterations (0: off)
    int tc_sk_tail = 0;   // tensor cores: the tiles after the last full wave shared by all CTAs
    int small = 0;        // FFMA: the one-launch small-problem kernel (16 x 16 tiles)
    int t_a = 0;          // FFMA: op(A) (K-contiguous) copied M-contiguous by a pre-pass
    int t_b = 0;          // FFMA: op(B) (K-contiguous) copied N-contiguous by a pre-pass
};

// The small-problem FFMA kernel takes problems of at most kSmallFlops
// (2 M N K), K <= kSmallMaxK and at most kSmallMaxTiles tiles of 16 x 16
// when the path is chosen automatically, or forced to FFMA without a split.
// Measured on GB300 (per call, L2 flushed; small kernel against the
// tensor-core path): 128^3 8.9 / 13.0 us, 256^3 10.9 / 17.1, 384^3 19.1 /
// 21.2, 448^3 27.3 / 23.2; 512 x 512 x 128 15.0 / 15.0.  Long K or many
// tiles lose (one CTA per tile, each 128-k chunk waits for its copies):
// 256 x 256 x 1024 29.3 / 21.2, 128 x 128 x 2048 49.8 / 21.2, 1024 x 1024 x
// 32 23.3 / 11.9.
constexpr double kSmallFlops = 1.2e8;
// The FFMA tile path copies a K-contiguous operand transposed first when the
// other side of the problem is at least this long (see make_plan).
constexpr int64_t kFfmaTransposeMin = 2048;
// Stream-K over every tensor-core tile stays open at any grid fill while the
// operands, as the kernel reads them, fit in this much of L2 (see make_plan).
constexpr double kStreamKL2Bytes = 96e6;
constexpr int64_t kSmallMaxK = 512;
constexpr int64_t kSmallMaxTiles = 1024;

// Chooses path, tile, split and vectorisation.  `path`/`split` 0 = auto.
inline int make_plan(char ta, char tb, int64_t M, int64_t N, int64_t K, int64_t lda,
                     int64_t ldb, int64_t ldc, bool a_al, bool b_al, bool c_al, int path,
                     int split, int sms, Plan *out) {
    Plan pl;
    // Thin problems (min(M, N) <= 16, "Matmul II", section 8: decode's
    // M = 1 to a few dozen) stream their large operand once on the CUDA
    // cores; the tile paths would compute mostly padding.  Except when the
    // large operand's rows run along K (the dot form: weights stored [N][K])
    // and more than 4 outputs share each of its elements: there the
    // tensor-core path, which splits both operands inside its kernel, is
    // ahead despite the padding (measured on GB300, S x 16384 x 8192 NT:
    // S = 8 279 -> 165 us, S = 16 418 -> 166 us; S = 4 stays at 124 us).
    // The large operand must also allow the in-kernel split (16-byte base,
    // leading dimension a multiple of 4); otherwise the pre-pass would copy it
    // twice over and the thin path stays ahead.
    const int64_t thin = std::min(M, N);
    const bool big_kcontig = M <= N ? !is_notrans(tb) : is_notrans(ta);
    const bool big_al = M <= N ? (b_al && ldb % 4 == 0) : (a_al && lda % 4 == 0);
    const bool thin_on_tc = thin > 4 && big_kcontig && big_al && K >= 32;
    // 16 < S <= 128 with the large operand's rows along the long side,
    // aligned: the thin path's tensor-core form (its MMAs cost about the same
    // up to S = 128), where the tile path would compute padding and pre-split
    // the whole large operand.  K >= 32 as for the tensor cores in general.
    const bool tc_form = thin >= 12 && thin <= 128 && !big_kcontig && big_al;   // as run_gemv's
    const bool small = 2.0 * (double)M * (double)N * (double)K <= kSmallFlops && K <= kSmallMaxK &&
                       ((M + 15) / 16) * ((N + 15) / 16) <= kSmallMaxTiles;
    // (problems small enough for the one-launch FFMA kernel stay there, and
    // the other side must be long: the form's CTAs are 128 of its columns)
    const bool thin_tc_wide = thin > 16 && tc_form && K >= 32 && !small && std::max(M, N) >= 8 * thin;
    if (path == SGEMM_PATH_GEMV ||
        (path == SGEMM_PATH_AUTO && ((thin <= 16 && !thin_on_tc) || thin_tc_wide))) {
        if (thin > 16 && !tc_form) return SGEMM_ERR_UNSUPPORTED;
        pl.path = SGEMM_PATH_GEMV;
        pl.tile_m = (int)std::min(M, N);
        pl.tile_n = 0;
        pl.split = 1;
        pl.vector = (a_al && b_al && lda % 4 == 0 && ldb % 4 == 0) ? 1 : 0;
        *out = pl;
        return 0;
    }
    if ((path == SGEMM_PATH_AUTO || path == SGEMM_PATH_FFMA) && small && split <= 1) {
        // One launch of 16 x 16 tiles, every output summed in ascending k
        // (ffma_small.cuh): below the crossover the fixed costs of the
        // tile kernels (their launches, fill and, on the tensor cores, the
        // split pre-pass and the fixup) outweigh their throughput.
        pl.path = SGEMM_PATH_FFMA;
        pl.small = 1;
        pl.tile_m = pl.tile_n = 16;
        pl.split = 1;
        pl.dp_tiles = (int)(((M + 15) / 16) * ((N + 15) / 16));
        pl.ctas = 0;
        pl.vector = 0;
        pl.c_vector = 0;
        *out = pl;
        return 0;
    }
    if (path == SGEMM_PATH_AUTO) {
        // 3xTF32 runs the tensor cores at 3 MMAs per product and beats the
        // CUDA-core path by 2x (1024^3) to 5x (8192^3) on GB300.  Small
        // problems are bound by fixed costs on either path, and there too
        // the tensor-core path is ahead (128^3: 13.3 against 16.5 us;
        // 384^3: 21.5 against 21.5; 128 x 128 x 2048: 19.6 against 32.8).
        // K < 32 stays on FFMA: there the dropped split terms are not small
        // against the fp32 bound 4*K*2^-24.
        pl.path = K >= 32 ? SGEMM_PATH_3XTF32 : SGEMM_PATH_FFMA;
    } else {
        pl.path = path;
    }
    pl.vector = (a_al && lda % 4 == 0 && b_al && ldb % 4 == 0) ? 1 : 0;
    pl.c_vector = (c_al && ldc % 4 == 0) ? 1 : 0;
    if (pl.path == SGEMM_PATH_FFMA) {
        // A grid of at least one full wave (2 CTAs per SM) runs its full waves
        // as whole tiles; the k-tile iterations of the tiles of a partly
        // filled last wave are shared equally by one wave of CTAs ("stream-K",
        // each share at least 8 k-tiles, else the tail stays whole too):
        // 4096^3 on GB300 0.758 -> 0.787 of the FFMA peak.  A grid smaller than
        // one wave has all its iterations shared by up to a wave of CTAs (at
        // least 2 k-tiles, 32 of K, each, at most 32 CTAs per tile): 1024^3
        // runs 1.7x faster that way, 256^3 (4 tiles, 32 CTAs) 1.4x faster
        // than with 8 k-tiles per CTA.  Forced split s: every tile cut into s K
        // slices; s = 1 keeps every tile whole, bit-identical to the naive loop.
        const int64_t tiles = ((M + 127) / 128) * ((N + 127) / 128);
        const int64_t kt = std::max<int64_t>((K + 15) / 16, 1);
        const int64_t slots = 2LL * sms;
        int64_t dp, sk;
        if (split == 1) {
            dp = tiles;
            sk = 0;
        } else if (split > 1) {
            dp = 0;
            sk = tiles * std::min<int64_t>(split, kt);
        } else if (tiles >= slots) {
            const int64_t rem = tiles % slots;
            if (rem > 0 && rem * kt >= 8 * slots) {
                dp = tiles - rem;
                sk = slots;
            } else {
                dp = tiles;
                sk = 0;
            }
        } else {
            dp = 0;
            sk = std::max<int64_t>(1, std::min<int64_t>(std::min<int64_t>(slots, (tiles * kt + 1) / 2),
                                                        32 * tiles));
        }
        pl.dp_tiles = (int)dp;
        pl.ctas = (int)std::min<int64_t>(sk, INT32_MAX);
        // An operand whose rows run along K is staged through registers and
        // stored transposed in every k-tile; one whose rows run along M or N
        // is copied as it is (cp.async).  The layout with both copied (TN)
        // is the fastest: 4096^3 on GB300 64.7 TFLOP/s against NN 62.7, TT
        // 62.6, NT 59.3.  A transpose pre-pass costs the operand's bytes
        // twice at the HBM rate, ~41/N (A) or ~41/M (B) of the kernel's time,
        // so it is taken for large grids whose other side is at least
        // kFfmaTransposeMin.
        const bool big = M >= 128 && N >= 128 && K >= 256;
        pl.t_a = big && is_notrans(ta) && N >= kFfmaTransposeMin ? 1 : 0;
        pl.t_b = big && is_trans(tb) && M >= kFfmaTransposeMin ? 1 : 0;
        const int64_t rem = tiles - dp;
        pl.split = (sk == 0 || rem == 0) ? 1 : (int)((sk + rem - 1) / rem);
    } else {
        // tensor-core path: 128-row tiles (256 on SM pairs), N of the MMA from
        // the problem's N, one CTA (pair) per SM.  Tiles after the last full
        // wave may run as 2 or 4 narrower units, or all tiles x k-blocks
        // iterations may be shared by the CTAs (stream-K), when a model of
        // their cost says so (below).
        pl.tile_m = 128;
        pl.tile_n = N > 128 ? 256 : (N > 64 ? 128 : 64);
        pl.split = 1;
        // Splitting an operand in the kernel saves its pre-pass (12 bytes of
        // HBM traffic per element) but slows the main loop; the pre-pass of A
        // costs ~285/N of the tensor work (at the measured HBM and TF32
        // rates), so A is split in the kernel (into TMEM) when N <= 2048, and
        // only when the operand is K-contiguous and 16-byte aligned (TMA reads
        // it raw).  B's split lands in shared memory, beside the MMAs' own
        // operand reads, and the split warps then carry both operands: on
        // wide tiles it pays only up to M = 1024 (measured on GB300, split in
        // the kernel against the pre-pass: 2048^3 NT 101.0 against 78.5 us, TT
        // 104.1 against 84.6, 1536 x 4096 x 1536 NT 127.6 against 93.8;
        // 1024^3 and below equal or slightly ahead; 2048 x 512 x 8192 NT
        // 100.5 against 85.7).  A narrow B (N <= 128: 64 or 128 rows per
        // stage), or a problem under a GFLOP, whose pre-pass launch would
        // cost more than the split (1536 x 256 x 256 NT 17.1 against 19.1),
        // stays split in the kernel up to M = 2048.
        pl.fuse_a = N <= 2048 && is_notrans(ta) && a_al && lda % 4 == 0;
        pl.fuse_b = (M <= 1024 || N <= 128 || 2.0 * (double)M * (double)N * (double)K < 1e9) &&
                    M <= 2048 && is_trans(tb) && b_al && ldb % 4 == 0;
        // 256-row tiles on an SM pair when both operands come pre-split and
        // M fills them: each SM holds half of B, a third less shared-memory
        // traffic per flop (+6 % at 4096^3 and 8192^3 on GB300).  With an
        // operand split in shared memory the pair measured 2-4 % slower.
        pl.pair = (M > 128 && !pl.fuse_a && !pl.fuse_b) ? 1 : 0;
        pl.tile_m = pl.pair ? 256 : 128;
        const int64_t tiles = ((M + pl.tile_m - 1) / pl.tile_m) * ((N + pl.tile_n - 1) / pl.tile_n);
        const int64_t slots = pl.pair ? std::max(sms / 2, 1) : sms;
        const int64_t full = (tiles / slots) * slots;
        const int64_t tail = tiles - full;
        double best = (double)((tiles + slots - 1) / slots);
        pl.dp_tiles = (int)tiles;
        pl.tail_nsplit = 1;
        const bool three = pl.path == SGEMM_PATH_3XTF32;
        // Time of a unit 1/ns as wide as a tile, in tile-times, measured on
        // GB300: narrow units are bound by the stage ring's round trip and the
        // per-stage TMA issue (SM pairs, shared-memory operands), or by MMAs
        // reading A from TMEM at a cost nearly independent of N (A split in
        // the kernel), not by their share of the flops.  (4095 x 3073 x 1537
        // ran 1.43x faster with whole tiles than with quarter units.)
        const bool tmem_a = !pl.pair && pl.fuse_a;
        auto unit_cost = [&](int ns) {
            if (!tmem_a) return ns == 2 ? 0.90 : 0.76;
            if (three) return ns == 2 ? 0.97 : 0.96;
            return ns == 2 ? 0.90 : 0.87;
        };
        for (int ns = 2; ns <= 4 && pl.tile_n / ns >= 64; ns *= 2) {
            if (tail == 0) break;
            const double waves = (double)((tail * ns + slots - 1) / slots);
            const double c = (double)(full / slots) + waves * unit_cost(ns);
            if (c < best * 0.995) {
                best = c;
                pl.dp_tiles = (int)full;
                pl.tail_nsplit = ns;
            }
        }
        const int64_t kp = (K + 31) / 32 * 32;
        const double tile_us = 128.0 * pl.tile_n * (double)kp * (three ? 3 : 1) /
                               (2047.0 * 1900.0 * (pl.tile_n >= 128 ? 0.75 : 0.45));
        double cur_us = best * tile_us;
        // Stream-K over the last wave (persistent CTAs: both operands come
        // pre-split): the whole waves first, then the k-blocks of the
        // remaining tiles shared equally by all CTAs (pairs), instead of
        // narrower units.  Charged one partial epilogue per CTA (4.5 us for
        // 128 x 256 rows per SM) and the fixup (3 us plus the partial tiles'
        // traffic at 6 TB/s); taken when 2 % faster.
        if (split == 0 && tail > 0 && !pl.fuse_a && !pl.fuse_b) {
            const double t_sk = (double)(full / slots) * tile_us + (double)tail / slots * tile_us +
                                4.5 * (pl.tile_m / 128) * pl.tile_n / 256.0 + 3.0 +
                                (double)(slots + tail) * pl.tile_m * pl.tile_n * 8.0 / 6.0e6;
            if (t_sk < 0.98 * cur_us) {
                cur_us = t_sk;
                pl.dp_tiles = (int)full;
                pl.tail_nsplit = 1;
                pl.tc_sk_tail = 1;
                pl.split = (int)((slots + tail - 1) / tail);
            }
        }
        // Stream-K on single SMs: with fewer 128-row tiles than SMs, the
        // tiles x k-blocks iterations are shared in equal contiguous ranges
        // by up to one CTA per SM (at least 8 k-blocks each), so all CTAs
        // end together; tiles that several CTAs share leave partial sums for
        // a fixup pass.  Modelled in microseconds: a tile's main loop at the
        // measured MMA rate (2047 MAC per clock per SM at ~1.9 GHz; 0.75 of
        // it reached on 128- and 256-wide tiles, 0.45 on 64-wide ones), one
        // or two partial-tile epilogues per CTA (4.5 us for 128 x 256), and the
        // fixup as 3 us plus its partial-tile traffic at 6 TB/s; taken when
        // 5 % faster than the choice above.  A forced split s > 1 runs
        // stream-K with min(s x tiles, 8 x SMs, iterations) CTAs; split = 1
        // never does.
        const int64_t nkb = kp / ((three && !(pl.tile_n <= 128 && pl.fuse_a)) ? 16 : 32);
        const int64_t tm1 = (M + 127) / 128, tn1 = (N + pl.tile_n - 1) / pl.tile_n;
        const int64_t tiles1 = tm1 * tn1;
        // Whole tiles instead of stream-K over every tile, an empirical rule:
        // ranges that start at scattered k positions share no operand panel
        // with their neighbours in L2.  Whole tiles won where they already
        // fill >= 60 % of the SMs, the panels that tiles share (A's across a
        // tile row, B's down a tile column, as the kernel reads them) do not
        // fit in L2, and the grid has at least as many tile rows as columns,
        // and 4 columns or more.  Measured on GB300, whole tiles against
        // stream-K, us (NN unless noted):
        //   * won: 2048 x 2048 x 8192 286 / 393; 3072 x 1280 x 8192 270 /
        //     320; 1536 x 2048 x 8192 286 / 309; 4096 x 1024 x 8192 265 /
        //     276;
        //   * lost: TT 768 x 4096 x 8192 345 / 257; NT 1024 x 4096 x 8192
        //     349 / 328; 8192 x 512 x 8192 264 / 249; 1280 x 2048 x 8192
        //     (80 tiles) 286 / 270; 1280 x 2048 x 4096 (operands in L2) 150 /
        //     118;
        //   * even: 2048 x 1536 x 8192 274 / 270.
        const double shared_operand_bytes =
            (tn1 > 1 ? (double)M * kp * (pl.fuse_a ? 4 : (three ? 8 : 4)) : 0.0) +
            (tm1 > 1 ? (double)N * kp * (pl.fuse_b ? 4 : (three ? 8 : 4)) : 0.0);
        const bool whole_fills = 5 * tiles1 >= 3 * sms && shared_operand_bytes > kStreamKL2Bytes &&
                                 tm1 >= tn1 && tn1 >= 4;
        const int64_t iters = tiles1 * nkb;
        int64_t g_sk = 0;
        if (split > 1) {
            g_sk = std::min<int64_t>(std::min<int64_t>(tiles1 * split, 8LL * sms), iters);
        } else if (split == 0 && tiles1 < sms && !whole_fills) {
            // g CTAs: most ranges straddle two tiles (two partial epilogues,
            // back to back where A is split into TMEM); a multiple of the
            // tile count keeps every range inside one tile (one epilogue)
            const int64_t g1 = std::min<int64_t>(sms, iters / 8);
            const int64_t g2 = tiles1 * (g1 / tiles1);
            double t_best = 0.95 * cur_us;
            for (int pass = 0; pass < 2; ++pass) {
                const int64_t g = pass == 0 ? g1 : g2;
                if (g <= tiles1 || (pass == 1 && g2 == g1)) continue;
                const double epi = (pass == 0 && g1 % tiles1 != 0 ? 2.0 : 1.0) * 4.5 * pl.tile_n / 256.0;
                const double fix = 3.0 + (double)(g + tiles1) * 128.0 * pl.tile_n * 8.0 / 6.0e6;
                const double t_sk = (double)iters / (double)g / (double)nkb * tile_us + epi + fix;
                if (t_sk < t_best) {
                    t_best = t_sk;
                    g_sk = g;
                }
            }
        }
        if (g_sk > 0) {
            pl.pair = 0;
            pl.tile_m = 128;
            pl.dp_tiles = (int)tiles1;
            pl.tail_nsplit = 1;
            pl.tc_sk_tail = 0;
            pl.tc_sk = (int)g_sk;
            pl.split = (int)((g_sk + tiles1 - 1) / tiles1);
        }
    }
    *out = pl;
    return 0;
}

// The tensor-core kernel variant a plan runs (run_tc launches exactly this).
struct TcVariant {
    bool fuse_a = false;   // A split in the kernel (into tensor memory)
    bool fuse_b = false;   // B split in the kernel (in shared memory)
    bool sk = false;       // stream-K over every tile, single SMs
    bool pair = false;     // 256-row tiles on SM pairs (cta_group::2)
    bool sk_tail = false;  // the tiles after the last full wave shared by all CTAs
    bool wide = false;     // 3xTF32 with 32-wide k-blocks, A_hi in TMEM and A_lo in shared memory
    int nacc = 1;          // accumulators per tile, summed by the epilogue
    int bk = 32;           // k-block width in floats
};

inline TcVariant tc_variant(const Plan &pl) {
    TcVariant v;
    const bool three = pl.path == SGEMM_PATH_3XTF32;
    v.fuse_a = pl.fuse_a != 0;
    v.fuse_b = pl.fuse_b != 0;
    v.sk = pl.tc_sk > 0;
    // the pair kernel takes pre-split operands only; stream-K over every
    // tile runs on single SMs, stream-K over the last wave on either
    v.pair = pl.pair != 0 && !v.fuse_a && !v.fuse_b && !v.sk;
    v.sk_tail = !v.sk && pl.tc_sk_tail != 0 && !v.fuse_a && !v.fuse_b;
    v.wide = three && pl.tile_n <= 128 && v.fuse_a && !v.pair;
    v.nacc = (pl.tile_n == 64 && !v.pair) ? (three ? 3 : 2) : (v.wide ? 3 : 1);
    v.bk = (v.wide || !three) ? 32 : 16;
    return v;
}

}  // namespace sgemm_gb300
