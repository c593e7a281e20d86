// CUDA-core (FFMA) single-precision GEMM kernel for sm_103a.
//
// Structure (the nest of tiles of "Matmul II: register blocking, warp tiling,
// tensor cores", sections 1-5, re-derived for this GPU):
//   * block tile 128 x 128 of C per CTA, 256 threads, k-tiles of BK = 16;
//   * warp tile 32 (rows) x 64 (cols): 8 warps as 4 x 2, square enough that
//     a warp's shared-memory reads per k are its perimeter, not its area
//     (section 5, "v7: warp tiling");
//   * thread tile 8 x 8 as a 2 x 2 grid of 4 x 4 blocks (rows tr*4 + {0..3}
//     and 16 + tr*4 + {0..3}, columns tc*4 + {0..3} and 32 + tc*4 + {0..3}),
//     so that one k-step is four 16-byte shared loads feeding 64 FMAs
//     (section 4, "v6: wider loads and a transposed tile"), issued as 32
//     packed fma.rn.f32x2 (two independent round-to-nearest FMAs each);
//   * both operand tiles sit in shared memory k-major ([k][m] and [k][n]), so
//     an operand whose rows run along K in global memory (A with 'N', B with
//     'T') is transposed on the way in through registers, and one whose rows
//     run along M or N is copied with cp.async as-is ("CuTe-ly writing an
//     SM86 SGEMM", section "host-side setup": 16-byte cp.async.cg);
//   * an XOR swizzle of each shared row (bits 3-4 of the column flipped by
//     bits 2-3 of k) keeps the transposing stores and the 16-byte loads free
//     of bank conflicts ("CuTe-ly writing an SM86 SGEMM", section "swizzles &
//     shared memory");
//   * two shared-memory stages: the copy of k-tile t+1 is in flight while
//     k-tile t is multiplied ("Matmul II", section 7, t3's double buffer);
//   * fused alpha/beta epilogue with 16-byte stores where C allows.
// Every output is summed in ascending k with one fused multiply-add per
// term, starting from +0; a k-tile past K is zero-filled and adds exactly 0.
// So with one K slice the result equals, bit for bit, the naive loop
// acc = fmaf(a, b, acc) followed by alpha*acc or fmaf(alpha, acc, beta*c)
// ("How to get a matmul kernel into the top percentile (worklog)",
// "Optimization 1": same ascending order, identical fp32 result).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "ptx_util.cuh"

namespace sgemm_gb300 {
namespace ffma {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK = 16;
constexpr int THREADS = 256;

// Work decomposition: tiles are numbered in rasterised order.  The first
// dp_tiles tiles are computed whole by one CTA each (blockIdx.x < dp_tiles);
// every later tile is cut into `split` contiguous K slices, one CTA each,
// whose raw partial sums go to a 128 x 128 block of `partial` and are added
// by splitk_reduce_kernel in ascending slice order.  This evens out the last,
// partly filled wave of CTAs and fills the GPU for problems with few tiles
// ("Matmul II", section 8: split-K when M*N is too small to fill the SMs).
struct Params {
    const float *A;
    const float *B;
    float *C;
    float *partial;        // [(tile - dp_tiles) * split + slice][BM * BN]
    int64_t lda, ldb, ldc;
    int M, N, K;
    float alpha, beta;
    int tiles_m, tiles_n;
    int group_m;           // CTA rasterisation: tile rows per group
    int dp_tiles;          // tiles computed whole
    int split;             // K slices of each remaining tile
    int kt_per_split;      // BK-tiles per K slice
    int c_vec;             // C base 16-byte aligned and ldc % 4 == 0
};

// Tile index -> (tile row, tile column), grouped rasterisation: consecutive
// tiles walk down a group of group_m tile rows before moving one tile column
// right, so co-resident CTAs share the group's A panels and a few B panels in
// L2 ("Optimising fp32 GEMM on A100", "Kernel 5 (grid swizzling)").
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
// tile is 512 float4 chunks, two per thread; chunk c covers row c / 4 and
// k = 4*(c % 4) .. +3.  A warp covers 8 whole 64-byte row pieces.
template <bool VEC>
__device__ __forceinline__ void kmajor_load(const float *__restrict__ X, int64_t ldx,
                                            int rows_total, int K, int row0, int k0,
                                            int tid, float (&r)[2][4]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int c = tid + h * THREADS;
        const int gr = row0 + (c >> 2);
        const int gk = k0 + (c & 3) * 4;
        const float *src = X + (int64_t)gr * ldx + gk;
        if (VEC && gr < rows_total && gk + 3 < K) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(src));
            r[h][0] = v.x; r[h][1] = v.y; r[h][2] = v.z; r[h][3] = v.w;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                r[h][j] = (gr < rows_total && gk + j < K) ? __ldg(src + j) : 0.0f;
        }
    }
}

// Transposing store of the staged chunks into the k-major shared tile.
// For a fixed j the 32 lanes of a warp hit 32 different banks: the low three
// bits of the row come from the lane, bits 3-4 from (warp ^ k-quad).
__device__ __forceinline__ void kmajor_store(float *__restrict__ s, int tid,
                                             const float (&r)[2][4]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int c = tid + h * THREADS;
        const int row = c >> 2;
        const int kq = c & 3;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int k = kq * 4 + j;
            s[k * BM + swz(k, row)] = r[h][j];
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
    for (int h = 0; h < 2; ++h) {
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

// One output quad (4 consecutive columns of one row): alpha/beta epilogue.
__device__ __forceinline__ float axpby(float alpha, float acc, float beta, float c) {
    // beta == 0 is handled by the caller (C is then not read)
    return __fmaf_rn(alpha, acc, __fmul_rn(beta, c));
}

__device__ __forceinline__ void store_quad(const Params &p, int row, int col, float4 v) {
    if (row >= p.M || col >= p.N) return;
    float *dst = p.C + (int64_t)row * p.ldc + col;
    const float alpha = p.alpha, beta = p.beta;
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
        *reinterpret_cast<float4 *>(dst) = o;
    } else {
        const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (col + j < p.N) {
                dst[j] = (beta == 0.0f) ? __fmul_rn(alpha, vv[j])
                                        : axpby(alpha, vv[j], beta, dst[j]);
            }
        }
    }
}

// A_KMAJOR: op(A) rows run along K in memory (transA 'N').
// B_KMAJOR: op(B) columns run along K in memory (transB 'T').
// VEC: A and B base pointers are 16-byte aligned and their leading
//      dimensions are multiples of 4, so 16-byte loads/copies are legal.
template <bool A_KMAJOR, bool B_KMAJOR, bool VEC>
__global__ void __launch_bounds__(THREADS, 2) ffma_gemm_kernel(const Params p) {
    __shared__ __align__(16) float sA[2][BK * BM];
    __shared__ __align__(16) float sB[2][BK * BN];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;

    const int total_kt = (p.K + BK - 1) / BK;
    int tile, unit = -1, kt_begin = 0, kt_end = total_kt;
    if ((int)blockIdx.x < p.dp_tiles) {
        tile = blockIdx.x;
    } else {
        unit = blockIdx.x - p.dp_tiles;                 // partial block index
        tile = p.dp_tiles + unit / p.split;
        kt_begin = (unit % p.split) * p.kt_per_split;
        kt_end = min(kt_begin + p.kt_per_split, total_kt);
    }
    int tm, tn;
    raster(tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
    const int m0 = tm * BM;
    const int n0 = tn * BN;
    const int nkt = kt_end - kt_begin;

    // thread -> outputs
    const int wm = warp & 3;            // warp row   (4 x 32 rows)
    const int wn = warp >> 2;           // warp col   (2 x 64 cols)
    const int tr = lane >> 3;           // 0..3
    const int tc = lane & 7;            // 0..7
    const int am = wm * 32 + tr * 4;    // first of the thread's A rows in the tile
    const int bn = wn * 64 + tc * 4;    // first of the thread's B cols in the tile

    float2 acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.0f, 0.0f);

    float ra[2][4], rb[2][4];

    auto issue = [&](int kt, int stage) {
        const int k0 = kt * BK;
        if (A_KMAJOR) kmajor_load<VEC>(p.A, p.lda, p.M, p.K, m0, k0, tid, ra);
        else mnmajor_async<VEC>(p.A, p.lda, p.M, p.K, m0, k0, tid, sA[stage]);
        if (B_KMAJOR) kmajor_load<VEC>(p.B, p.ldb, p.N, p.K, n0, k0, tid, rb);
        else mnmajor_async<VEC>(p.B, p.ldb, p.N, p.K, n0, k0, tid, sB[stage]);
        cp_async_commit();
    };
    auto park = [&](int stage) {
        if (A_KMAJOR) kmajor_store(sA[stage], tid, ra);
        if (B_KMAJOR) kmajor_store(sB[stage], tid, rb);
    };

    if (nkt > 0) {
        issue(kt_begin, 0);
        park(0);
        cp_async_wait_all();
        __syncthreads();
    }

    for (int it = 0; it < nkt; ++it) {
        const int stage = it & 1;
        const bool has_next = it + 1 < nkt;
        if (has_next) issue(kt_begin + it + 1, stage ^ 1);

        const float *As = sA[stage];
        const float *Bs = sB[stage];
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            const int s = ((k >> 2) & 3) << 3;
            const float4 a0 = *reinterpret_cast<const float4 *>(As + k * BM + (am ^ s));
            const float4 a1 = *reinterpret_cast<const float4 *>(As + k * BM + ((am + 16) ^ s));
            const float4 b0 = *reinterpret_cast<const float4 *>(Bs + k * BN + (bn ^ s));
            const float4 b1 = *reinterpret_cast<const float4 *>(Bs + k * BN + ((bn + 32) ^ s));
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float2 b[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w),
                                 make_float2(b1.x, b1.y), make_float2(b1.z, b1.w)};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float2 ai = make_float2(a[i], a[i]);
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = __ffma2_rn(ai, b[j], acc[i][j]);
            }
        }

        if (has_next) {
            park(stage ^ 1);
            cp_async_wait_all();
        }
        __syncthreads();
    }

    if (unit >= 0) {
        // raw partial sums into this unit's dense 128 x 128 block
        float *blk = p.partial + (int64_t)unit * (BM * BN);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = am + (i & 3) + (i >> 2) * 16;
            *reinterpret_cast<float4 *>(blk + r * BN + bn) =
                make_float4(acc[i][0].x, acc[i][0].y, acc[i][1].x, acc[i][1].y);
            *reinterpret_cast<float4 *>(blk + r * BN + bn + 32) =
                make_float4(acc[i][2].x, acc[i][2].y, acc[i][3].x, acc[i][3].y);
        }
        return;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = m0 + am + (i & 3) + (i >> 2) * 16;
        store_quad(p, row, n0 + bn,
                   make_float4(acc[i][0].x, acc[i][0].y, acc[i][1].x, acc[i][1].y));
        store_quad(p, row, n0 + bn + 32,
                   make_float4(acc[i][2].x, acc[i][2].y, acc[i][3].x, acc[i][3].y));
    }
}

// For each split tile (one CTA per tile): C = alpha * (sum of its K-slice
// partial blocks, added in ascending slice order) + beta * C.  Threads walk
// the 128 x 128 tile row by row, four columns each, so reads of the partial
// blocks and of C are coalesced.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const Params p) {
    const int tile = p.dp_tiles + blockIdx.x;
    int tm, tn;
    raster(tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
    const int m0 = tm * BM, n0 = tn * BN;
    const float *base = p.partial + (int64_t)blockIdx.x * p.split * (BM * BN);
    for (int e = threadIdx.x * 4; e < BM * BN; e += blockDim.x * 4) {
        const int r = e / BN, c = e % BN;
        if (m0 + r >= p.M || n0 + c >= p.N) continue;
        float4 s = *reinterpret_cast<const float4 *>(base + e);
        for (int q = 1; q < p.split; ++q) {
            const float4 t = *reinterpret_cast<const float4 *>(base + q * (BM * BN) + e);
            s.x = __fadd_rn(s.x, t.x); s.y = __fadd_rn(s.y, t.y);
            s.z = __fadd_rn(s.z, t.z); s.w = __fadd_rn(s.w, t.w);
        }
        store_quad(p, m0 + r, n0 + c, s);
    }
}

// C = beta * C (C = 0 when beta == 0, without reading C): the K == 0 and
// alpha == 0 quick return.
__global__ void scale_c_kernel(int M, int N, float beta, float *__restrict__ C, int64_t ldc) {
    const int64_t total = (int64_t)M * N;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = idx / N, col = idx - row * N;
        float *dst = C + row * ldc + col;
        *dst = (beta == 0.0f) ? 0.0f : __fmul_rn(beta, *dst);
    }
}

}  // namespace ffma
}  // namespace sgemm_gb300
