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
    int split = 1;      // FFMA: K slices of the tail tiles (1 = none)
    int dp_tiles = 0;   // FFMA: tiles computed whole
    int tile_m = 128, tile_n = 128;
    int vector = 1;     // 16-byte operand loads (else 4-byte edge path)
    int c_vector = 1;   // 16-byte C accesses
    int group_m = 8;    // rasterisation group height (tiles)
    int tail_nsplit = 1;  // tensor cores: column slices of the last-wave tiles
};

// Cost model of the FFMA path in units of one k-tile step of one CTA
// (about 2 us at 2 CTAs per SM).  CTAs run in waves of `slots`; a whole
// tile takes kt steps, a slice ceil(kt / split).  `dp` (0 or a multiple of
// `slots`) whole tiles run first, then the sliced tail units.  Each partial
// block costs ~0.01 step of HBM traffic in the reduction, which also adds a
// fixed ~2 steps (a second launch).
inline double ffma_cost(int64_t tiles, int64_t kt, int64_t dp, int64_t split, int64_t slots) {
    if (split == 1) return (double)((tiles + slots - 1) / slots) * (double)kt;
    const int64_t units = (tiles - dp) * split;
    const int64_t slice = (kt + split - 1) / split;
    const int64_t slice_waves = (units + slots - 1) / slots;
    return (double)(dp / slots) * (double)kt + (double)slice_waves * (double)slice +
           0.01 * (double)units + 2.0;
}

// Chooses path, tile, split and vectorisation.  `path`/`split` 0 = auto.
inline int make_plan(char ta, char tb, int64_t M, int64_t N, int64_t K, int64_t lda,
                     int64_t ldb, int64_t ldc, bool a_al, bool b_al, bool c_al, int path,
                     int split, int sms, Plan *out) {
    (void)ta; (void)tb;
    Plan pl;
    if (path == SGEMM_PATH_AUTO) {
        // 3xTF32 runs the tensor cores at 3 MMAs per product and beats the
        // CUDA-core path by 1.5x (1024^3) to 5x (8192^3) on GB300, but it
        // carries a split pre-pass and a launch more: small problems stay on
        // FFMA, and so does K < 32, where the dropped split terms are not
        // small against the fp32 bound 4*K*2^-24.
        const bool big = (double)M * (double)N * (double)K >= (double)(1 << 27);
        pl.path = (big && K >= 32) ? SGEMM_PATH_3XTF32 : SGEMM_PATH_FFMA;
    } else {
        pl.path = path;
    }
    pl.vector = (a_al && lda % 4 == 0 && b_al && ldb % 4 == 0) ? 1 : 0;
    pl.c_vector = (c_al && ldc % 4 == 0) ? 1 : 0;
    if (pl.path == SGEMM_PATH_FFMA) {
        const int64_t tiles = ((M + 127) / 128) * ((N + 127) / 128);
        const int64_t kt = (K + 15) / 16;
        const int64_t slots = 2LL * sms;        // two 256-thread CTAs per SM
        if (split > 0) {
            pl.split = (int)std::min<int64_t>(split, std::max<int64_t>(kt, 1));
            pl.dp_tiles = pl.split == 1 ? (int)tiles : 0;
        } else {
            // try "all tiles whole" and, for each split s, "whole waves of
            // whole tiles + the rest sliced in s"; keep the cheapest
            double best = ffma_cost(tiles, kt, tiles, 1, slots);
            pl.split = 1;
            pl.dp_tiles = (int)tiles;
            const int64_t max_split = std::min<int64_t>(16, kt / 4);   // slices >= 64 of K
            for (int64_t s = 2; s <= max_split; ++s) {
                const int64_t dp = (tiles / slots) * slots;            // whole waves
                for (int64_t d : {dp, (int64_t)0}) {
                    if (d == tiles) continue;
                    const double c = ffma_cost(tiles, kt, d, s, slots);
                    if (c < best * 0.97) {                              // must win clearly
                        best = c;
                        pl.split = (int)s;
                        pl.dp_tiles = (int)d;
                    }
                }
            }
        }
        if (pl.split == 1) pl.dp_tiles = (int)tiles;
    } else {
        // tensor-core path: 128-row tiles, N of the MMA from the problem's N,
        // one CTA per SM.  Tiles after the last full wave may run as 2 or 4
        // narrower CTAs (MMA N = tile_n / slices, at least 64) so the last
        // wave is short; a narrower tile is charged ~5 % per halving for its
        // higher shared-memory traffic per flop.
        pl.tile_m = 128;
        pl.tile_n = N > 128 ? 256 : (N > 64 ? 128 : 64);
        pl.split = 1;
        const int64_t tiles = ((M + 127) / 128) * ((N + pl.tile_n - 1) / pl.tile_n);
        const int64_t slots = sms;
        const int64_t full = (tiles / slots) * slots;
        const int64_t tail = tiles - full;
        double best = (double)((tiles + slots - 1) / slots);
        pl.dp_tiles = (int)tiles;
        pl.tail_nsplit = 1;
        for (int ns = 2; ns <= 4 && pl.tile_n / ns >= 64; ns *= 2) {
            if (tail == 0) break;
            const double waves = (double)((tail * ns + slots - 1) / slots);
            const double c = (double)(full / slots) + waves / ns * (ns == 2 ? 1.05 : 1.10);
            if (c < best * 0.97) {
                best = c;
                pl.dp_tiles = (int)full;
                pl.tail_nsplit = ns;
            }
        }
    }
    *out = pl;
    return 0;
}

}  // namespace sgemm_gb300
