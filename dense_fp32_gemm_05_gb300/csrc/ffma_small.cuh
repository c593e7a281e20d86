// Small problems on the CUDA cores in one launch, every output summed in
// ascending k.
//
// Below a few tens of megaflops a GEMM is bound by fixed costs: launches,
// the first loads' latency, pipeline fill.  The tile kernels pay for their
// throughput with exactly those (the 128 x 128 FFMA tile leaves most SMs idle
// at 256^3; the tensor-core path adds a split pre-pass and a stream-K fixup,
// three launches in all).  This kernel is the plain tiled loop of "Optimising
// fp32 GEMM on A100" (kernel 2, shared-memory tiling) and "Matmul II"
// (section 3, register blocking) at the smallest useful scale:
//   * a 16 x 16 tile of C per CTA of 64 threads, so that even 256^3 has 256
//     CTAs for 152 SMs; each thread owns a 2 x 2 block (rows 2 ty + {0, 1},
//     columns 2 tx + {0, 1}), advanced by two packed fma.rn.f32x2 per k;
//   * k in chunks of 128, double-buffered in shared memory by 4-byte
//     cp.async copies (any layout, any alignment; past the matrix edge the
//     copy zero-fills), stored k-major ([k][m], [k][n]) with an odd row pitch
//     of 17 floats, so that the copies (consecutive k or consecutive m/n
//     across a warp) and the 2 x 2 fragment reads meet no bank conflicts;
//   * the k loop stops at K (no zero-filled terms are added), so every output
//     is acc = fmaf(a_k, b_k, acc) for k = 0, 1, ..., K - 1 from +0: bit for
//     bit the FFMA tile kernel with whole tiles and the naive loop;
//   * the fused alpha/beta epilogue of the other FFMA kernel, element by
//     element.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "epilogue.cuh"
#include "ptx_util.cuh"

namespace sgemm_gb300 {
namespace ffma_small {

constexpr int TM = 16;
constexpr int TN = 16;
constexpr int THREADS = 64;
constexpr int KC = 128;        // k per shared-memory chunk
constexpr int PITCH = 17;      // floats per k row of a chunk (TM or TN, padded odd)

struct Params {
    const float *A;
    const float *B;
    float *C;
    int64_t lda, ldb, ldc;
    int M, N, K;
    float alpha, beta;
    int tiles_n;
    const float *row_scale;    // fused epilogue: M row scales or null
    const float *bias;         // N column biases or null
    int act;                   // SGEMM_ACT_*
};

// Copies chunk [k0, k0 + KC) of this CTA's A rows and B columns into the
// k-major shared tiles.  Consecutive threads take consecutive elements along
// the operand's contiguous direction (k for A 'N' and B 'T', m or n
// otherwise), so each warp reads whole 64- or 128-byte runs.
template <bool A_KMAJOR, bool B_KMAJOR>
__device__ __forceinline__ void copy_chunk(const Params &p, int m0, int n0, int k0, float *as,
                                           float *bs, int tid) {
#pragma unroll 4
    for (int i = 0; i < TM * KC / THREADS; ++i) {
        const int e = tid + i * THREADS;
        const int m = A_KMAJOR ? e / KC : e % TM;
        const int k = A_KMAJOR ? e % KC : e / TM;
        const int gm = m0 + m, gk = k0 + k;
        const bool ok = gm < p.M && gk < p.K;
        const float *src = !ok ? p.A
                               : (A_KMAJOR ? p.A + (int64_t)gm * p.lda + gk
                                           : p.A + (int64_t)gk * p.lda + gm);
        cp_async_4(smem_u32(as + k * PITCH + m), src, ok ? 4 : 0);
    }
#pragma unroll 4
    for (int i = 0; i < TN * KC / THREADS; ++i) {
        const int e = tid + i * THREADS;
        const int n = B_KMAJOR ? e / KC : e % TN;
        const int k = B_KMAJOR ? e % KC : e / TN;
        const int gn = n0 + n, gk = k0 + k;
        const bool ok = gn < p.N && gk < p.K;
        const float *src = !ok ? p.B
                               : (B_KMAJOR ? p.B + (int64_t)gn * p.ldb + gk
                                           : p.B + (int64_t)gk * p.ldb + gn);
        cp_async_4(smem_u32(bs + k * PITCH + n), src, ok ? 4 : 0);
    }
    cp_async_commit();
}

// A_KMAJOR: op(A) rows run along K in memory (transA 'N').
// B_KMAJOR: op(B) columns run along K in memory (transB 'T').
template <bool A_KMAJOR, bool B_KMAJOR>
__global__ void __launch_bounds__(THREADS) ffma_small_kernel(const Params p) {
    __shared__ float As[2][KC * PITCH];
    __shared__ float Bs[2][KC * PITCH];
    const int tid = threadIdx.x;
    const int tx = tid & 7, ty = tid >> 3;
    const int m0 = (int)(blockIdx.x / p.tiles_n) * TM;
    const int n0 = (int)(blockIdx.x % p.tiles_n) * TN;
    const int chunks = (p.K + KC - 1) / KC;

    float2 acc0 = make_float2(0.0f, 0.0f), acc1 = make_float2(0.0f, 0.0f);
    copy_chunk<A_KMAJOR, B_KMAJOR>(p, m0, n0, 0, As[0], Bs[0], tid);
    for (int c = 0; c < chunks; ++c) {
        const int st = c & 1;
        if (c + 1 < chunks) {
            // the other stage was last read before the barrier that ended chunk c - 1
            copy_chunk<A_KMAJOR, B_KMAJOR>(p, m0, n0, (c + 1) * KC, As[st ^ 1], Bs[st ^ 1], tid);
            cp_async_wait_group<1>();
        } else {
            cp_async_wait_group<0>();
        }
        __syncthreads();
        const float *a = As[st] + 2 * ty;
        const float *b = Bs[st] + 2 * tx;
        const int kn = min(KC, p.K - c * KC);
        auto step = [&](int k) {
            const float a0 = a[k * PITCH], a1 = a[k * PITCH + 1];
            const float2 bk = make_float2(b[k * PITCH], b[k * PITCH + 1]);
            acc0 = __ffma2_rn(make_float2(a0, a0), bk, acc0);
            acc1 = __ffma2_rn(make_float2(a1, a1), bk, acc1);
        };
        if (kn == KC) {
#pragma unroll 16
            for (int k = 0; k < KC; ++k) step(k);
        } else {
#pragma unroll 4
            for (int k = 0; k < kn; ++k) step(k);
        }
        __syncthreads();
    }

    const float v[2][2] = {{acc0.x, acc0.y}, {acc1.x, acc1.y}};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int row = m0 + 2 * ty + i;
        if (row >= p.M) continue;
        const float alpha = epi_alpha(p.alpha, p.row_scale, row);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int col = n0 + 2 * tx + j;
            if (col >= p.N) continue;
            float *dst = p.C + (int64_t)row * p.ldc + col;
            const float t = p.beta == 0.0f ? __fmul_rn(alpha, v[i][j])
                                           : __fmaf_rn(alpha, v[i][j], __fmul_rn(p.beta, *dst));
            *dst = epi_tail(t, p.bias, col, p.act);
        }
    }
}

}  // namespace ffma_small
}  // namespace sgemm_gb300
