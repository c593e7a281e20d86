// CUDA-core (FFMA) single-precision GEMM kernel for sm_103a.
//
// Structure (the nest of tiles of "Matmul II: register blocking, warp tiling,
// tensor cores", sections 1-5, re-derived for this GPU):
//   * block tile 128 x 128 of C per CTA, 128 threads, k-tiles of BK = 16;
//   * warp tile 64 x 64: 4 warps as 2 x 2, a square warp tile so that a
//     warp's shared-memory reads per k are its perimeter, not its area
//     (section 5, "v7: warp tiling", whose 64 x 64 warp tile this is);
//   * thread tile 8 x 16: a lane owns rows am + {0..3}, am + 32 + {0..3} and
//     columns bn + 16 g + {0..3}, g = 0..3.  One k-step is 6 sixteen-byte
//     shared loads (2 of A, 4 of B) feeding 128 FMAs, issued as 64 packed
//     fma.rn.f32x2 (two independent round-to-nearest FMAs each).  The 8 x 16
//     tile is what keeps shared-memory delivery (128 bytes per clock per SM)
//     below the FMA rate: 24 loaded floats per 128 FMAs instead of the 16 per
//     64 of an 8 x 8 tile (section 4 counts the same ratio at one level less).
//     The lanes of each quad hold a 2 x 2 block of row and column groups, so
//     every 16-byte shared load costs 2 wavefronts instead of 4;
//   * both operand tiles sit in shared memory k-major ([k][m] and [k][n]).
//     An operand whose rows run along K in global memory (A with 'N', B with
//     'T') is loaded as float4 along K into registers and stored transposed
//     (section 4, "transposed tile"), in two halves per k-tile so that only
//     8 staging registers are live; one whose rows run along M or N is copied
//     with cp.async as-is ("CuTe-ly writing an SM86 SGEMM", section
//     "host-side setup": 16-byte cp.async.cg);
//   * an XOR swizzle of each shared row (bits 3-4 of the column flipped by
//     bits 2-3 of k) keeps the transposing stores and the 16-byte loads free
//     of bank conflicts ("CuTe-ly writing an SM86 SGEMM", section "swizzles &
//     shared memory");
//   * three shared-memory stages: the cp.async copies of k-tiles t+1 and t+2
//     are in flight while k-tile t is multiplied (a register-staged operand
//     runs one k-tile ahead); "Matmul II", section 7, t3's double buffer with
//     one stage more (measured on GB300, 4096^3: NN 62.2 -> 62.7, TN 64.2 ->
//     64.6 TFLOP/s, bit-identical);
//   * fused alpha/beta epilogue with 16-byte stores where C allows.
//
// Work decomposition (data-parallel tiles + "stream-K" remainder): tiles are
// numbered in grouped raster order.  The first dp_tiles are computed whole,
// one CTA each, wave after wave (neighbouring CTAs share A and B panels in
// L2).  The k-tile iterations of the remaining tiles are cut into sk_ctas
// contiguous, equal shares, one per further CTA: a share that covers a whole
// tile writes C; a share that starts or ends inside a tile leaves a partial
// sum in the workspace, and sk_fixup_kernel adds a shared tile's partials in
// ascending k order (deterministic) and writes C.  So the last, partly
// filled wave of whole tiles becomes one short wave that keeps every SM busy,
// and a grid with fewer tiles than CTA slots is spread over all of them;
// with dp_tiles = 0 and sk_ctas = s * tiles every tile is cut into s
// contiguous K slices (split-K, "Matmul II", section 8).
//
// Every output is summed in ascending k with one fused multiply-add per
// term, starting from +0; a k-tile past K is zero-filled and adds exactly 0.
// So a tile computed whole equals, bit for bit, the naive loop
// acc = fmaf(a, b, acc) followed by alpha*acc or fmaf(alpha, acc, beta*c)
// ("How to get a matmul kernel into the top percentile (worklog)",
// "Optimization 1": same ascending order, identical fp32 result).
#pragma once

#include <cstdint>
#include <type_traits>
#include <cuda_runtime.h>

#include "epilogue.cuh"
#include "ptx_util.cuh"

namespace sgemm_gb300 {
namespace ffma {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK = 16;
constexpr int THREADS = 128;
constexpr int CHUNKS = (BM * BK / 4) / THREADS;    // float4 chunks per thread per operand tile

struct Params {
    const float *A;
    const float *B;
    float *C;
    float *partial;        // [2 * sk_ctas][BM * BN]: slot 2c = share c's first tile, 2c+1 its last
    int64_t lda, ldb, ldc;
    int M, N, K;
    float alpha, beta;
    int tiles_m, tiles_n;
    int group_m;           // CTA rasterisation: tile rows per group
    int kt;                // k-tiles per tile, ceil(K / BK)
    int dp_tiles;          // tiles computed whole (CTAs 0 .. dp_tiles-1)
    int sk_ctas;           // CTAs sharing the remaining tiles' iterations
    int64_t sk_iters;      // (tiles - dp_tiles) * kt, counted from tile dp_tiles
    int c_vec;             // C base 16-byte aligned and ldc % 4 == 0
    const float *row_scale;   // fused epilogue: M row scales or null
    const float *bias;        // N column biases or null
    int act;                  // SGEMM_ACT_*
};

// First remaining-tile iteration of share c.
__host__ __device__ __forceinline__ int64_t share_begin(int64_t iters, int ctas, int c) {
    return iters * c / ctas;
}

// The share containing remaining-tile iteration x (largest c with begin <= x).
__host__ __device__ __forceinline__ int share_owner(int64_t iters, int ctas, int64_t x) {
    return (int)(((x + 1) * ctas - 1) / iters);
}

// Workspace slot of share c's partial sum of remaining tile u: its first tile or its last.
__host__ __device__ __forceinline__ int partial_slot(const Params &p, int c, int u) {
    return (share_begin(p.sk_iters, p.sk_ctas, c) / p.kt == u) ? 2 * c : 2 * c + 1;
}

// Tile index -> (tile row, tile column), grouped rasterisation: consecutive
// tiles walk down a group of group_m tile rows before moving one tile column
// right, so CTAs working on neighbouring tiles share the group's A panels and
// a few B panels in L2 ("Optimising fp32 GEMM on A100", "Kernel 5 (grid
// swizzling)").
__host__ __device__ __forceinline__ void raster(int t, int tiles_m, int tiles_n, int group_m,
                                                int &tm, int &tn) {
    const int per_group = group_m * tiles_n;
    const int g = t / per_group;
    const int first_m = g * group_m;
    const int gm = min(tiles_m - first_m, group_m);
    const int r = t - g * per_group;
    tm = first_m + r % gm;
    tn = r / gm;
}

// Column swizzle of the k-major shared tiles: XOR bits 3-4 of the column with
// bits 2-3 of k.  Bits 0-1 are untouched, so aligned float4 groups stay whole.
__device__ __forceinline__ int swz(int k, int col) { return col ^ (((k >> 2) & 3) << 3); }

// Register staging for an operand whose global rows run along K: the 128 x 16
// tile is 512 float4 chunks, CHUNKS per thread; chunk c covers row c / 4 and
// k = 4*(c % 4) .. +3.  A warp covers 8 whole 64-byte row pieces.  Chunks
// H0 and H0 + 1 of this thread are loaded into r.
template <bool VEC, int H0>
__device__ __forceinline__ void kmajor_load(const float *__restrict__ X, int64_t ldx,
                                            int rows_total, int K, int row0, int k0,
                                            int tid, float (&r)[2][4]) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int c = tid + (H0 + hh) * THREADS;
        const int gr = row0 + (c >> 2);
        const int gk = k0 + (c & 3) * 4;
        const float *src = X + (int64_t)gr * ldx + gk;
        if (VEC && gr < rows_total && gk + 3 < K) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(src));
            r[hh][0] = v.x; r[hh][1] = v.y; r[hh][2] = v.z; r[hh][3] = v.w;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                r[hh][j] = (gr < rows_total && gk + j < K) ? __ldg(src + j) : 0.0f;
        }
    }
}

// Transposing store of the staged chunks H0, H0 + 1 into the k-major tile.
// For a fixed j the 32 lanes of a warp hit 32 different banks: the low three
// bits of the row come from the lane, bits 3-4 from (warp ^ k-quad).
template <int H0>
__device__ __forceinline__ void kmajor_store(float *__restrict__ s, int tid,
                                             const float (&r)[2][4]) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int c = tid + (H0 + hh) * THREADS;
        const int row = c >> 2;
        const int kq = c & 3;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int k = kq * 4 + j;
            s[k * BM + swz(k, row)] = r[hh][j];
        }
    }
}

// cp.async for an operand whose global rows run along K's partner (M or N):
// the 16 x 128 tile is 16 rows of 32 float4 chunks; a warp copies one whole
// 512-byte row.  Out-of-range bytes are zero-filled by the copy itself.
template <bool VEC>
__device__ __forceinline__ void mnmajor_async(const float *__restrict__ X, int64_t ldx,
                                              int cols_total, int K, int col0, int k0,
                                              int tid, float *__restrict__ s) {
#pragma unroll
    for (int h = 0; h < CHUNKS; ++h) {
        const int c = tid + h * THREADS;
        const int k = c >> 5;
        const int cc = (c & 31) * 4;
        const int gk = k0 + k;
        const int gc = col0 + cc;
        const uint32_t dst = smem_u32(s + k * BN + swz(k, cc));
        if (VEC) {
            int bytes = 0;
            if (gk < K) {
                const int left = cols_total - gc;
                bytes = left >= 4 ? 16 : (left > 0 ? left * 4 : 0);
            }
            const float *src = bytes ? X + (int64_t)gk * ldx + gc : X;
            cp_async_16(dst, src, bytes);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool ok = gk < K && gc + j < cols_total;
                const float *src = ok ? X + (int64_t)gk * ldx + gc + j : X;
                cp_async_4(dst + 4 * j, src, ok ? 4 : 0);
            }
        }
    }
}

// alpha/beta epilogue of one element (beta == 0 is handled by the caller:
// C is then not read).
__device__ __forceinline__ float axpby(float alpha, float acc, float beta, float c) {
    return __fmaf_rn(alpha, acc, __fmul_rn(beta, c));
}

// One output quad (4 consecutive columns of one row) into C.
__device__ __forceinline__ void store_quad(const Params &p, int row, int col, float4 v) {
    if (row >= p.M || col >= p.N) return;
    float *dst = p.C + (int64_t)row * p.ldc + col;
    // alpha * s_row with a row scale (fused epilogue), else alpha
    const float alpha = epi_alpha(p.alpha, p.row_scale, row), beta = p.beta;
    const bool tail = p.bias || p.act != SGEMM_ACT_NONE;
    if (p.c_vec && col + 3 < p.N) {
        float4 o;
        if (beta == 0.0f) {
            o = make_float4(__fmul_rn(alpha, v.x), __fmul_rn(alpha, v.y),
                            __fmul_rn(alpha, v.z), __fmul_rn(alpha, v.w));
        } else {
            const float4 c = *reinterpret_cast<const float4 *>(dst);
            o = make_float4(axpby(alpha, v.x, beta, c.x), axpby(alpha, v.y, beta, c.y),
                            axpby(alpha, v.z, beta, c.z), axpby(alpha, v.w, beta, c.w));
        }
        if (tail) {
            o.x = epi_tail(o.x, p.bias, col, p.act);
            o.y = epi_tail(o.y, p.bias, col + 1, p.act);
            o.z = epi_tail(o.z, p.bias, col + 2, p.act);
            o.w = epi_tail(o.w, p.bias, col + 3, p.act);
        }
        *reinterpret_cast<float4 *>(dst) = o;
    } else {
        const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (col + j < p.N) {
                float t = (beta == 0.0f) ? __fmul_rn(alpha, vv[j])
                                         : axpby(alpha, vv[j], beta, dst[j]);
                if (tail) t = epi_tail(t, p.bias, col + j, p.act);
                dst[j] = t;
            }
        }
    }
}

// k-tiles [j0, j1) of tile t; a whole tile goes to C, a part to partial[slot].
template <bool A_KMAJOR, bool B_KMAJOR, bool VEC>
__device__ __forceinline__ void run_share(const Params &p, float (*sA)[BK * BM],
                                          float (*sB)[BK * BN], int t, int j0, int j1, int slot) {
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    int tm, tn;
    raster(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
    const int m0 = tm * BM;
    const int n0 = tn * BN;
    const int nkt = j1 - j0;

    // thread -> outputs: 4 warps as 2 x 2 of 64 x 64; a lane has row group
    // lr (8 per warp) and column group lc (4 per warp).  Each quad of lanes
    // (4i .. 4i+3) is a 2 x 2 block of (lr, lc): a 16-byte shared load is
    // served per lane quad, so a quad that asks for 2 distinct A (or B) chunks
    // costs half the wavefronts of one that asks for 4 (measured on GB300:
    // 12 instead of 20 wavefronts per warp k-step).
    const int wm = warp & 1;
    const int wn = warp >> 1;
    const int lr = ((lane >> 3) << 1) | ((lane >> 1) & 1);   // 0..7
    const int lc = (((lane >> 2) & 1) << 1) | (lane & 1);    // 0..3
    const int am = wm * 64 + lr * 4;    // rows am + {0..3}, am + 32 + {0..3}
    const int bn = wn * 64 + lc * 4;    // columns bn + 16 g + {0..3}

    float2 acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = make_float2(0.0f, 0.0f);

    float ra[2][4], rb[2][4];
    using H_0 = std::integral_constant<int, 0>;
    using H_2 = std::integral_constant<int, 2>;
    // K-contiguous operands are staged through registers in two halves:
    // chunks 0-1 are loaded at the start of a k-tile and parked in shared
    // memory half way through it, chunks 2-3 are loaded then and parked at its
    // end; MN-contiguous operands are copied with cp.async.
    auto issue_async = [&](int kt, int stage) {
        const int k0 = kt * BK;
        if (!A_KMAJOR) mnmajor_async<VEC>(p.A, p.lda, p.M, p.K, m0, k0, tid, sA[stage]);
        if (!B_KMAJOR) mnmajor_async<VEC>(p.B, p.ldb, p.N, p.K, n0, k0, tid, sB[stage]);
        cp_async_commit();
    };
    auto load_half = [&](int kt, auto h0) {
        constexpr int H0 = decltype(h0)::value;
        const int k0 = kt * BK;
        if (A_KMAJOR) kmajor_load<VEC, H0>(p.A, p.lda, p.M, p.K, m0, k0, tid, ra);
        if (B_KMAJOR) kmajor_load<VEC, H0>(p.B, p.ldb, p.N, p.K, n0, k0, tid, rb);
    };
    auto park_half = [&](int stage, auto h0) {
        constexpr int H0 = decltype(h0)::value;
        if (A_KMAJOR) kmajor_store<H0>(sA[stage], tid, ra);
        if (B_KMAJOR) kmajor_store<H0>(sB[stage], tid, rb);
    };

    issue_async(j0, 0);
    if (nkt > 1) issue_async(j0 + 1, 1);
    else cp_async_commit();
    load_half(j0, H_0{});
    park_half(0, H_0{});
    load_half(j0, H_2{});
    park_half(0, H_2{});
    cp_async_wait_group<1>();
    __syncthreads();

    int stage = 0;
    for (int it = 0; it < nkt; ++it) {
        const int nxt = stage == 2 ? 0 : stage + 1;
        const int nxt2 = nxt == 2 ? 0 : nxt + 1;
        const bool has_next = it + 1 < nkt;
        // the stage two ahead was last read in the previous k-tile (barrier passed)
        if (it + 2 < nkt) issue_async(j0 + it + 2, nxt2);
        else cp_async_commit();
        if (has_next) load_half(j0 + it + 1, H_0{});
        const float *As = sA[stage];
        const float *Bs = sB[stage];
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            if (k == BK / 2 && has_next) {
                park_half(nxt, H_0{});
                load_half(j0 + it + 1, H_2{});
            }
            const int s = ((k >> 2) & 3) << 3;
            const float4 a0 = *reinterpret_cast<const float4 *>(As + k * BM + (am ^ s));
            const float4 a1 = *reinterpret_cast<const float4 *>(As + k * BM + ((am + 32) ^ s));
            float2 b[8];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const float4 bg =
                    *reinterpret_cast<const float4 *>(Bs + k * BN + ((bn + 16 * g) ^ s));
                b[2 * g] = make_float2(bg.x, bg.y);
                b[2 * g + 1] = make_float2(bg.z, bg.w);
            }
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            // Column pair outer (consecutive packed FMAs share their b operand),
            // except with both operands staged through registers by 16-byte
            // loads, where that order makes the compiler spill (measured on
            // GB300: NN 4096^3 +1.6 % for the column order, NT -25 % for it).
            if constexpr (!(A_KMAJOR && B_KMAJOR && VEC)) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        acc[i][j] = __ffma2_rn(make_float2(a[i], a[i]), b[j], acc[i][j]);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 ai = make_float2(a[i], a[i]);
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[i][j] = __ffma2_rn(ai, b[j], acc[i][j]);
                }
            }
        }
        if (has_next) park_half(nxt, H_2{});
        cp_async_wait_group<1>();
        __syncthreads();
        stage = nxt;
    }

    if (nkt != p.kt) {
        // raw partial sums into this share's dense 128 x 128 block
        float *blk = p.partial + (int64_t)slot * (BM * BN);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = am + (i & 3) + (i >> 2) * 32;
#pragma unroll
            for (int g = 0; g < 4; ++g)
                *reinterpret_cast<float4 *>(blk + r * BN + bn + 16 * g) =
                    make_float4(acc[i][2 * g].x, acc[i][2 * g].y, acc[i][2 * g + 1].x,
                                acc[i][2 * g + 1].y);
        }
        return;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = m0 + am + (i & 3) + (i >> 2) * 32;
#pragma unroll
        for (int g = 0; g < 4; ++g)
            store_quad(p, row, n0 + bn + 16 * g,
                       make_float4(acc[i][2 * g].x, acc[i][2 * g].y, acc[i][2 * g + 1].x,
                                   acc[i][2 * g + 1].y));
    }
}

// A_KMAJOR: op(A) rows run along K in memory (transA 'N').
// B_KMAJOR: op(B) columns run along K in memory (transB 'T').
// VEC: A and B base pointers are 16-byte aligned and their leading
//      dimensions are multiples of 4, so 16-byte loads/copies are legal.
template <bool A_KMAJOR, bool B_KMAJOR, bool VEC>
__global__ void __launch_bounds__(THREADS, 2) ffma_gemm_kernel(const Params p) {
    __shared__ __align__(16) float sA[3][BK * BM];
    __shared__ __align__(16) float sB[3][BK * BN];
    pdl_wait();      // after a transpose pre-pass: its copies are complete
    pdl_trigger();   // the stream-K fixup may launch; it waits for this grid
    if ((int)blockIdx.x < p.dp_tiles) {
        run_share<A_KMAJOR, B_KMAJOR, VEC>(p, sA, sB, blockIdx.x, 0, p.kt, 0);
        return;
    }
    const int c = blockIdx.x - p.dp_tiles;
    const int64_t end = share_begin(p.sk_iters, p.sk_ctas, c + 1);
    int64_t it = share_begin(p.sk_iters, p.sk_ctas, c);
    bool first = true;
    while (it < end) {
        const int u = (int)(it / p.kt);
        const int j0 = (int)(it - (int64_t)u * p.kt);
        const int j1 = (int)((int64_t)j0 + (end - it) < (int64_t)p.kt ? j0 + (end - it) : p.kt);
        // the shared tiles are free again: the share's last k-tile ended in a barrier
        run_share<A_KMAJOR, B_KMAJOR, VEC>(p, sA, sB, p.dp_tiles + u, j0, j1,
                                           first ? 2 * c : 2 * c + 1);
        it += j1 - j0;
        first = false;
    }
}

// Grid (remaining tiles, FIX_PARTS): block (u, part) handles rows
// 16*part .. +15 of remaining tile u.  A tile cut between several shares gets
// C = alpha * (sum of its partial blocks, added in ascending k order) + beta*C;
// a tile inside one share was written by it and is skipped.  The shares'
// workspace slots are looked up once per block; threads then walk the rows
// four columns each (coalesced).
constexpr int FIX_PARTS = 8;
constexpr int FIX_MAX_SHARES = 64;

__global__ void __launch_bounds__(256) sk_fixup_kernel(const Params p) {
    __shared__ int slots[FIX_MAX_SHARES];
    __shared__ int nslots;
    pdl_wait();   // the main kernel's partial blocks are complete and visible
    const int u = blockIdx.x;
    const int64_t x0 = (int64_t)u * p.kt;
    const int c_lo = share_owner(p.sk_iters, p.sk_ctas, x0);
    const int c_hi = share_owner(p.sk_iters, p.sk_ctas, x0 + p.kt - 1);
    if (c_lo == c_hi) return;
    if (threadIdx.x == 0) {
        int n = 0;
        for (int c = c_lo; c <= c_hi; ++c) {
            if (share_begin(p.sk_iters, p.sk_ctas, c) == share_begin(p.sk_iters, p.sk_ctas, c + 1))
                continue;                                       // empty share
            if (n < FIX_MAX_SHARES) slots[n] = partial_slot(p, c, u);
            ++n;
        }
        nslots = n;
    }
    __syncthreads();
    // the selector keeps shares per tile <= 32; more would not fit the table
    if (nslots > FIX_MAX_SHARES) return;
    int tm, tn;
    raster(p.dp_tiles + u, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
    const int m0 = tm * BM, n0 = tn * BN;
    const int rows = BM / FIX_PARTS;
    const int n = nslots;
    for (int e = blockIdx.y * rows * BN + threadIdx.x * 4; e < (blockIdx.y + 1) * rows * BN;
         e += blockDim.x * 4) {
        const int r = e / BN, col = e % BN;
        if (m0 + r >= p.M || n0 + col >= p.N) continue;
        float4 s = *reinterpret_cast<const float4 *>(p.partial + (int64_t)slots[0] * (BM * BN) + e);
        for (int q = 1; q < n; ++q) {
            const float4 v = *reinterpret_cast<const float4 *>(
                p.partial + (int64_t)slots[q] * (BM * BN) + e);
            s.x = __fadd_rn(s.x, v.x); s.y = __fadd_rn(s.y, v.y);
            s.z = __fadd_rn(s.z, v.z); s.w = __fadd_rn(s.w, v.w);
        }
        store_quad(p, m0 + r, n0 + col, s);
    }
}

// The FFMA path's pre-pass: a K-contiguous operand copied transposed, so
// that the kernel reads it as it reads an M- or N-contiguous one (cp.async,
// no register staging): dst[c * ldd + r] = src[r * lds + c] for r < rows, c
// < cols.  32 x 32 tiles turned around in shared memory (padded rows: no bank
// conflicts), reads and writes coalesced; job 0 takes CTAs [0, j0.tiles), job
// 1 the rest.
struct TransposeJob {
    const float *src;
    int64_t lds;
    float *dst;
    int64_t ldd;
    int rows, cols;     // of src
    int tiles_c;        // ceil(cols / 32)
    int tiles;          // CTAs of this job
};

__global__ void __launch_bounds__(256) transpose_pair_kernel(const TransposeJob j0,
                                                             const TransposeJob j1) {
    pdl_trigger();   // the GEMM may launch; it waits for this grid's writes
    __shared__ float tile[32][33];
    const bool second = (int)blockIdx.x >= j0.tiles;
    const TransposeJob &j = second ? j1 : j0;
    const int b = second ? (int)blockIdx.x - j0.tiles : (int)blockIdx.x;
    const int r0 = (b / j.tiles_c) * 32, c0 = (b % j.tiles_c) * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = r0 + ty + 8 * i, c = c0 + tx;
        if (r < j.rows && c < j.cols) tile[ty + 8 * i][tx] = __ldg(j.src + (int64_t)r * j.lds + c);
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int c = c0 + ty + 8 * i, r = r0 + tx;
        if (r < j.rows && c < j.cols) j.dst[(int64_t)c * j.ldd + r] = tile[tx][ty + 8 * i];
    }
}

// C = beta * C (C = 0 when beta == 0, without reading C): the K == 0 and
// alpha == 0 quick return; with a fused epilogue's bias and activation
// applied after it (the product term is zero, so a row scale has no effect).
__global__ void scale_c_kernel(int M, int N, float beta, float *__restrict__ C, int64_t ldc,
                               const float *bias, int act) {
    const int64_t total = (int64_t)M * N;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = idx / N, col = idx - row * N;
        float *dst = C + row * ldc + col;
        const float t = (beta == 0.0f) ? 0.0f : __fmul_rn(beta, *dst);
        *dst = epi_tail(t, bias, (int)col, act);
    }
}

}  // namespace ffma
}  // namespace sgemm_gb300
