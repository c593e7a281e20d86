// Thin GEMMs: min(M, N) <= 16, or <= 128 on the tensor cores (SGEMM_PATH_GEMV).
//
// "Matmul II: register blocking, warp tiling, tensor cores", section 8
// ("What cuBLAS does that we do not"): when M is 1 (decode) to a few dozen,
// none of the tile kernels' compute tricks apply; the GEMM is a memory-bound
// GEMV and the only thing that counts is streaming the large operand once.
// So this path has no tiles.  With S = min(M, N) (the small dimension) and P
// the other one:
//
//   out(s, p) = sum_k Small(s, k) * Big(p, k)
//
// M small: s = row of C, p = column; Small = op(A), Big(p, k) = op(B)(k, p).
// N small: s = column of C, p = row;  Small(s, k) = op(B)(k, s), Big = op(A).
// Then C(s, p) = alpha * out + beta * C (C not read when beta == 0), with
// the same epilogue roundings as the other paths.
//
// Two kernels, by how Big lies in memory:
//   * dot form (Big's rows run along K): a warp owns PB rows of Big and
//     streams them with 16-byte loads along K, each lane summing 4 of every
//     128 consecutive k; Small (S x K, a few KB per row) is read through L1.
//     A warp butterfly adds the 32 lane sums of each output.
//   * axpy form (Big's rows run along P): a lane owns 4 consecutive p and
//     reads Big(p .. p+3, k) with one 16-byte load per k; Small(s, k) is the
//     same for the whole warp (a broadcast load).  The 8 warps of a CTA take
//     interleaved k of the CTA's K range and are added through shared
//     memory in warp order; when K is also split across CTAs (to fill the
//     GPU), the CTAs' partial sums are added in K order by a second kernel.
//     For S = 8 and 16, where 16 or 64 accumulators per lane leave few
//     registers for row loads, a variant streams Big through a shared-memory
//     ring with TMA instead (gemv_axpy_tma_kernel).
// Every sum is a fixed order of fp32 FMAs and adds: deterministic, and, as
// any summation order, inside the 4 K 2^-24 bound.
//
// The selector sends dot-form problems with S > 4 and K >= 32 (and a Big
// the tensor-core kernel can split itself) to the 3xTF32 path, which is
// faster there despite its padded tiles; forced, this path still runs them.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "../../include/sgemm_gb300.h"
#include "gemv.h"
#include "plan.h"
#include "ptx_util.cuh"
#include "tc_gemm.h"

namespace sgemm_gb300 {
namespace gemv {

constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;
constexpr int AX_P = 128;              // axpy form: p per CTA (32 lanes x 4)

struct Params {
    const float *big;
    int64_t big_ld;
    const float *small;
    int64_t small_ss, small_sk;        // Small(s, k) = small[s * ss + k * sk]
    float *C;
    int64_t c_s, c_p;                  // C(s, p) = C[s * c_s + p * c_p]
    int S, P, K;
    float alpha, beta;
    float *partial;                    // axpy form, K split: [ksplit][S][P]
    int ksplit, kchunk;                // K range of CTA y: [y * kchunk, min(K, +kchunk))
    int rows_thin;                     // s is the row of C (M small), else its column
    const float *row_scale;            // fused epilogue: M row scales or null
    const float *bias;                 // N column biases or null
    int act;                           // SGEMM_ACT_*
    unsigned long long wait_ns;        // bounded-wait limit of the staged kernel
};

__device__ unsigned int g_error;       // sticky device error word of this path

__device__ __forceinline__ void store_out(const Params &p, int s, int q, float v) {
    float *dst = p.C + (int64_t)s * p.c_s + (int64_t)q * p.c_p;
    const int row = p.rows_thin ? s : q, col = p.rows_thin ? q : s;
    const float a = epi_alpha(p.alpha, p.row_scale, row);
    const float t = p.beta == 0.0f ? __fmul_rn(a, v) : __fmaf_rn(a, v, __fmul_rn(p.beta, *dst));
    *dst = epi_tail(t, p.bias, col, p.act);
}

// ------------------------------------------------------------ dot form
// SM: compile-time bound on S; PB: rows of Big per warp; VEC: Big rows and
// Small rows start 16-byte aligned with K-contiguous Small (16-byte loads).
template <int SM, int PB, bool VEC>
__global__ void __launch_bounds__(THREADS) gemv_dot_kernel(const Params p) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int p0 = (blockIdx.x * WARPS + warp) * PB;
    if (p0 >= p.P) return;
    // acc[s][b]: two partial sums of output (s, p0 + b), k = 4i + {0, 1} and
    // 4i + {2, 3}, advanced together by packed fma.rn.f32x2
    float2 acc[SM][PB];
#pragma unroll
    for (int s = 0; s < SM; ++s)
#pragma unroll
        for (int b = 0; b < PB; ++b) acc[s][b] = make_float2(0.0f, 0.0f);
    const float *rows[PB];
#pragma unroll
    for (int b = 0; b < PB; ++b)
        rows[b] = p.big + (int64_t)min(p0 + b, p.P - 1) * p.big_ld;   // clamped: a row past P is read, never stored
    int k = lane * 4;
    // k-steps unrolled (their row loads issued together).  Measured on GB300,
    // S x 16384 x 8192 NT, unrolled 2 -> this: S = 4 208 -> 124 us and S = 8
    // 563 -> 282 us with 8; S = 16 438 -> 414 us with 4 (8 spills there,
    // 676 us); S <= 2 unchanged at 2.  Two rows per warp instead of four for
    // S > 8 was slower still (1888 us): each warp then reads Small twice as
    // often per byte of Big.
    constexpr int DOT_UNROLL = SM >= 16 ? 4 : SM >= 4 ? 8 : 2;
    if (VEC) {
#pragma unroll DOT_UNROLL
        for (; k + 3 < p.K; k += 128) {
            float4 bv[PB];
#pragma unroll
            for (int b = 0; b < PB; ++b) bv[b] = __ldg(reinterpret_cast<const float4 *>(rows[b] + k));
#pragma unroll
            for (int s = 0; s < SM; ++s) {
                if (s < p.S) {
                    const float4 a = __ldg(reinterpret_cast<const float4 *>(p.small + s * p.small_ss + k));
#pragma unroll
                    for (int b = 0; b < PB; ++b) {
                        acc[s][b] = __ffma2_rn(make_float2(a.x, a.y), make_float2(bv[b].x, bv[b].y), acc[s][b]);
                        acc[s][b] = __ffma2_rn(make_float2(a.z, a.w), make_float2(bv[b].z, bv[b].w), acc[s][b]);
                    }
                }
            }
        }
    }
    // the rest (all of K without 16-byte loads): 4 consecutive k per lane
    for (; k < p.K; k += 128) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (k + j < p.K) {
                float bv[PB];
#pragma unroll
                for (int b = 0; b < PB; ++b) bv[b] = __ldg(rows[b] + k + j);
#pragma unroll
                for (int s = 0; s < SM; ++s) {
                    if (s < p.S) {
                        const float a = __ldg(p.small + s * p.small_ss + (int64_t)(k + j) * p.small_sk);
#pragma unroll
                        for (int b = 0; b < PB; ++b) acc[s][b].x = __fmaf_rn(a, bv[b], acc[s][b].x);
                    }
                }
            }
        }
    }
    // butterfly over the warp, then output (s, b) is stored by lane (s * PB + b) % 32
#pragma unroll
    for (int s = 0; s < SM; ++s) {
#pragma unroll
        for (int b = 0; b < PB; ++b) {
            float v = __fadd_rn(acc[s][b].x, acc[s][b].y);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (s < p.S && p0 + b < p.P && lane == (s * PB + b) % 32) store_out(p, s, p0 + b, v);
        }
    }
}

// ------------------------------------------------------------ axpy form
constexpr int AX_KC = 256;             // k per shared-memory chunk of Small
constexpr int AX_U = 8;                // consecutive k per warp step (row loads in flight)

template <int SM>
constexpr int ax_smem_floats() { return WARPS * SM * AX_P + AX_KC * SM; }

// Small(s, kc .. kc+kn-1) -> smt[k][s] by NT threads (this one is tid),
// reading along Small's contiguous dimension.  Element t = tid + j NT, j <
// PER, sits at (slow, fast) = (t / major, t % major); both advance by NT
// with one carry.  Every load is issued before the first store: a chunk
// costs one L2 round trip, not one per element of the thread.
// As stage_small, with 4-byte cp.async copies straight into shared memory
// (no registers; zero-filled for s >= S); the caller commits and waits.
template <int SM, int NT, int PER>
__device__ __forceinline__ void stage_small_async(const Params &p, float *smt, int kc, int kn,
                                                  int tid) {
    const bool s_fast = p.small_ss == 1;
    const int major = s_fast ? SM : kn;
    const int dq = NT / major, dr = NT % major;
    const int total = kn * SM;
    int q = tid / major, r = tid % major;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int s = s_fast ? r : q, kk = s_fast ? q : r;
        if (tid + j * NT < total) {
            const bool in = s < p.S;
            const float *src = in ? p.small + (int64_t)s * p.small_ss + (int64_t)(kc + kk) * p.small_sk
                                  : p.small;
            cp_async_4(smem_u32(smt + kk * SM + s), src, in ? 4 : 0);
        }
        q += dq;
        r += dr;
        if (r >= major) { r -= major; ++q; }
    }
}

template <int SM, int NT, int PER>
__device__ __forceinline__ void stage_small(const Params &p, float *smt, int kc, int kn,
                                            int tid) {
    const bool s_fast = p.small_ss == 1;               // Small's stored rows run along s
    const int major = s_fast ? SM : kn;
    const int dq = NT / major, dr = NT % major;
    const int total = kn * SM;
    float v[PER];
    int q = tid / major, r = tid % major;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int s = s_fast ? r : q, kk = s_fast ? q : r;
        v[j] = (tid + j * NT < total && s < p.S)
                   ? __ldg(p.small + (int64_t)s * p.small_ss + (int64_t)(kc + kk) * p.small_sk)
                   : 0.0f;
        q += dq;
        r += dr;
        if (r >= major) { r -= major; ++q; }
    }
    q = tid / major;
    r = tid % major;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int s = s_fast ? r : q, kk = s_fast ? q : r;
        if (tid + j * NT < total) smt[kk * SM + s] = v[j];
        q += dq;
        r += dr;
        if (r >= major) { r -= major; ++q; }
    }
}

template <int SM, bool VEC>
__global__ void __launch_bounds__(THREADS, 2) gemv_axpy_kernel(const Params p) {
    pdl_trigger();   // the K-split sum may launch; it waits for this grid
    extern __shared__ __align__(16) float smem_f[];
    float *red = smem_f;                               // [WARPS][SM][AX_P]
    float *smt = smem_f + WARPS * SM * AX_P;           // Small chunk, [AX_KC][SM]
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int pc = blockIdx.x * AX_P + lane * 4;       // this lane's first p
    const int k0 = blockIdx.y * p.kchunk;
    const int k1 = min(p.K, k0 + p.kchunk);
    // acc[s][h] = outputs (s, pc + 2h), (s, pc + 2h + 1): packed fma.rn.f32x2,
    // two independent round-to-nearest FMAs, half the issue slots
    float2 acc[SM][2];
#pragma unroll
    for (int s = 0; s < SM; ++s) acc[s][0] = acc[s][1] = make_float2(0.0f, 0.0f);
    const bool whole = VEC && pc + 3 < p.P;
    constexpr int U = AX_U;
    for (int kc = k0; kc < k1; kc += AX_KC) {
        const int kn = min(AX_KC, k1 - kc);
        __syncthreads();                               // the previous chunk is consumed
        stage_small<SM, THREADS, (AX_KC * SM + THREADS - 1) / THREADS>(p, smt, kc, kn,
                                                                      threadIdx.x);
        __syncthreads();
        // warp w takes U consecutive k at a time (k = kc + (w + 8 i) U ..):
        // all U row loads are issued before the first FMA
        for (int kb = kc + warp * U; kb < kc + kn; kb += WARPS * U) {
            float bv[U][4];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int k = kb + u;
                const float *row = p.big + (int64_t)k * p.big_ld;
                if (k >= kc + kn) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) bv[u][j] = 0.0f;
                } else if (whole) {
                    const float4 v = __ldg(reinterpret_cast<const float4 *>(row + pc));
                    bv[u][0] = v.x; bv[u][1] = v.y; bv[u][2] = v.z; bv[u][3] = v.w;
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) bv[u][j] = pc + j < p.P ? __ldg(row + pc + j) : 0.0f;
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int k = kb + u;
                if (k >= kc + kn) break;                // this chunk's Small ends here
                const float *a = smt + (k - kc) * SM;  // the same address in every lane
                float av[SM];
                if constexpr (SM % 4 == 0) {
#pragma unroll
                    for (int s = 0; s < SM; s += 4) {
                        const float4 v = *reinterpret_cast<const float4 *>(a + s);
                        av[s] = v.x; av[s + 1] = v.y; av[s + 2] = v.z; av[s + 3] = v.w;
                    }
                } else {
#pragma unroll
                    for (int s = 0; s < SM; ++s) av[s] = a[s];
                }
                const float2 b01 = make_float2(bv[u][0], bv[u][1]);
                const float2 b23 = make_float2(bv[u][2], bv[u][3]);
#pragma unroll
                for (int s = 0; s < SM; ++s) {
                    const float2 a2 = make_float2(av[s], av[s]);
                    acc[s][0] = __ffma2_rn(a2, b01, acc[s][0]);
                    acc[s][1] = __ffma2_rn(a2, b23, acc[s][1]);
                }
            }
        }
    }
#pragma unroll
    for (int s = 0; s < SM; ++s)
        *reinterpret_cast<float4 *>(red + (warp * SM + s) * AX_P + lane * 4) =
            make_float4(acc[s][0].x, acc[s][0].y, acc[s][1].x, acc[s][1].y);
    __syncthreads();
    // thread t: outputs (s, q) with s * AX_P + q = t, t + 256, ...; warps added in order
    for (int o = threadIdx.x; o < SM * AX_P; o += THREADS) {
        const int s = o / AX_P, q = o % AX_P;
        const int pp = blockIdx.x * AX_P + q;
        if (s >= p.S || pp >= p.P) continue;
        float v = red[s * AX_P + q];
        for (int w = 1; w < WARPS; ++w) v = __fadd_rn(v, red[(w * SM + s) * AX_P + q]);
        if (p.ksplit == 1) store_out(p, s, pp, v);
        else p.partial[((int64_t)blockIdx.y * p.S + s) * p.P + pp] = v;
    }
}

// ------------------------------------------------------------ axpy form, staged
// For S = 8 and 16 the axpy kernel above holds its row loads in registers
// next to 64 accumulators, too few bytes in flight per SM to stream Big at
// HBM speed.  This variant moves Big through shared memory instead: one
// producer warp streams boxes of TX_KS rows x 128 columns of Big with TMA into
// a ring of TX_ST stages (tensor map over Big: p innermost, row stride
// big_ld), and TX_CW consumer warps read their rows from there.  Small comes
// in chunks of TX_KC k, double-buffered in shared memory by 4-byte cp.async
// copies, so that the next chunk's copies are in flight while this one is
// consumed (measured: 16 x 16384 x 8192 NN 22.6 -> 24.1 TFLOP/s against
// staging each chunk through registers between two barriers; the ring gave
// up its sixth stage to keep 2 CTAs per SM).  Warp w takes
// rows 4w .. 4w+3 of each stage; the sums per output stay in k order within
// a warp and the warps are added in warp order, as in the kernel above.  Eight
// warps per CTA (7 consumers + the producer) keep 2 CTAs per SM at 128
// registers a thread; 9 would put 5 warps on some of the SM's 4 schedulers
// and cap them at 96 (measured: spills on the 16-output kernel).
constexpr int TX_CW = 7;               // consumer warps
constexpr int TX_CT = TX_CW * 32;      // consumer threads
constexpr int TX_KS = 4 * TX_CW;       // rows of Big per stage: 4 per consumer warp
constexpr int TX_KC = 9 * TX_KS;       // rows per Small chunk (9 stages)
constexpr int TX_ST = 5;               // stages in flight
constexpr int TX_THREADS = TX_CT + 32;     // + the producer warp
constexpr int TX_STAGE_FLOATS = TX_KS * AX_P;

template <int SM>
constexpr int tx_smem_bytes() {
    // ring, Small chunk, barriers (the reduction reuses the ring), alignment
    // slack: two CTAs per SM
    return (TX_ST * TX_STAGE_FLOATS + 2 * TX_KC * SM) * 4 + 2 * TX_ST * 8 + 128;
}

__device__ __forceinline__ uint32_t tx_su32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ bool tx_try(uint32_t bar, uint32_t ph) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred q;\n\tmbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}" : "=r"(ok) : "r"(bar), "r"(ph) : "memory");
    return ok != 0;
}
// The same with the suspension bounded by `ns` nanoseconds instead of the
// hardware's own window.
__device__ __forceinline__ bool tx_try_for(uint32_t bar, uint32_t ph, uint32_t ns) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred q;\n\tmbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}" : "=r"(ok) : "r"(bar), "r"(ph), "r"(ns) : "memory");
    return ok != 0;
}
// Bounded wait; on expiry the device error word is raised and false returned.
// A limit below 100 us (only the test hook sets one) is one try_wait whose
// suspension it bounds: %globaltimer does not tick every nanosecond, and
// try_wait on its own suspends a thread for a hardware-chosen while, so such
// a limit could otherwise outlast a wait of a microsecond or two.
__device__ __forceinline__ bool tx_wait(uint32_t bar, uint32_t ph, uint64_t limit_ns) {
    if (limit_ns < 100000u) {
        if (tx_try_for(bar, ph, (uint32_t)limit_ns)) return true;
        atomicExch(&g_error, (unsigned)SGEMM_ERR_TIMEOUT);
        return false;
    }
    if (tx_try(bar, ph)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!tx_try(bar, ph)) {
        if (global_timer_ns() - t0 > limit_ns) {
            atomicExch(&g_error, (unsigned)SGEMM_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

template <int SM>
__global__ void __launch_bounds__(TX_THREADS, 2)
    gemv_axpy_tma_kernel(const __grid_constant__ CUtensorMap big_map, const Params p) {
    static_assert(SM % 4 == 0, "Small is read four values (two pairs) at a time");
    pdl_trigger();   // the K-split sum may launch; it waits for this grid
    extern __shared__ __align__(16) float tx_smem[];
    // the ring on a 128-byte boundary (TMA destination), as an element offset
    // from the shared array so that every access stays a shared-memory one
    float *ring = tx_smem + (((128u - (tx_su32(tx_smem) & 127u)) & 127u) >> 2);
    float *smt0 = ring + TX_ST * TX_STAGE_FLOATS;       // Small chunks, 2 x [TX_KC][SM]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smt0 + 2 * TX_KC * SM);
    const uint32_t bar0 = tx_su32(bars);
    auto full = [&](int st) { return bar0 + 8u * st; };
    auto empty = [&](int st) { return bar0 + 8u * (TX_ST + st); };
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int p0 = blockIdx.x * AX_P;
    const int k0 = blockIdx.y * p.kchunk;
    const int k1 = min(p.K, k0 + p.kchunk);
    const int nst = (k1 - k0 + TX_KS - 1) / TX_KS;      // stages of this CTA
    const uint64_t lim = p.wait_ns;
    __shared__ int gave_up;                             // a consumer's wait ran out
    if (threadIdx.x == 0) {
        gave_up = 0;
        for (int st = 0; st < TX_ST; ++st) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(full(st)) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(empty(st)), "r"(TX_CW) : "memory");
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&big_map)) : "memory");
    }
    __syncthreads();

    if (warp == TX_CW) {
        // ------------------------------------------------ producer
        if (lane == 0) {
            int i = 0;
            for (; i < nst; ++i) {
                const int st = i % TX_ST;
                const uint32_t ph = (uint32_t)(i / TX_ST) & 1u;
                if (!tx_wait(empty(st), ph ^ 1u, lim)) break;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                             :: "r"(full(st)), "r"((uint32_t)(TX_STAGE_FLOATS * 4)) : "memory");
                asm volatile(
                    "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
                    " [%0], [%1, {%3, %4}], [%2];"
                    :: "r"(tx_su32(ring + st * TX_STAGE_FLOATS)),
                       "l"(reinterpret_cast<uint64_t>(&big_map)), "r"(full(st)), "r"(p0),
                       "r"(k0 + i * TX_KS)
                    : "memory");
            }
            // every issued copy has landed before the CTA can leave (a fixed
            // 1 s bound, independent of the settable limit, so that a tiny
            // limit never cuts the drain short)
            for (int q = (i > TX_ST ? i - TX_ST : 0); q < i; ++q)
                tx_wait(full(q % TX_ST), (uint32_t)(q / TX_ST) & 1u, 1000000000ull);
        }
        return;
    }

    // ---------------------------------------------------- consumers (warps 0..TX_CW-1)
    // packed pairs along s: acc[t][e] = (out(2t, p_e), out(2t + 1, p_e)) for the
    // lane's 4 columns p_e, so that Small's pairs come straight from its 16-byte
    // loads and only Big's 4 values are duplicated per k (measured on GB300:
    // ~5 % faster than pairs along p, which duplicated all of Small's values)
    float2 acc[SM / 2][4];
#pragma unroll
    for (int t = 0; t < SM / 2; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[t][e] = make_float2(0.0f, 0.0f);
    // A failed wait stops the compute and the empty-slot arrivals (the
    // producer then times out too), but never a barrier: every consumer
    // thread runs the same sequence of named-barrier syncs.
    bool ok = true;
    int i = 0;                                          // next stage
    constexpr int SPER = (TX_KC * SM + TX_CT - 1) / TX_CT;
    const int nchunks = (k1 - k0 + TX_KC - 1) / TX_KC;
    if (nchunks > 0)
        stage_small_async<SM, TX_CT, SPER>(p, smt0, k0, min(TX_KC, k1 - k0), threadIdx.x);
    cp_async_commit();
    for (int c = 0; c < nchunks; ++c) {
        const int kc = k0 + c * TX_KC;
        const int kn = min(TX_KC, k1 - kc);
        const float *smt = smt0 + (c & 1) * (TX_KC * SM);
        if (c + 1 < nchunks) {
            // the next chunk's copies fly while this one is consumed; its buffer
            // was released by the barrier that ended chunk c - 1
            stage_small_async<SM, TX_CT, SPER>(p, smt0 + ((c + 1) & 1) * (TX_KC * SM), kc + TX_KC,
                                               min(TX_KC, k1 - kc - TX_KC), threadIdx.x);
            cp_async_commit();
            cp_async_wait_group<1>();
        } else {
            cp_async_wait_group<0>();
        }
        asm volatile("bar.sync 1, %0;" :: "r"(TX_CT) : "memory");   // chunk c in shared memory
        // the stages of this chunk (TX_KC is a multiple of TX_KS)
        for (; i < nst && k0 + i * TX_KS < kc + kn; ++i) {
            const int st = i % TX_ST;
            if (ok && !tx_wait(full(st), (uint32_t)(i / TX_ST) & 1u, lim)) ok = false;
            if (!ok) continue;
            const float *rows = ring + st * TX_STAGE_FLOATS;
#pragma unroll
            for (int u = 0; u < TX_KS / TX_CW; ++u) {
                const int r = warp * (TX_KS / TX_CW) + u;
                const int k = k0 + i * TX_KS + r;
                if (k >= k1) break;
                const float4 b = *reinterpret_cast<const float4 *>(rows + r * AX_P + lane * 4);
                const float *a = smt + (k - kc) * SM;  // the same address in every lane
                const float2 bb[4] = {make_float2(b.x, b.x), make_float2(b.y, b.y),
                                      make_float2(b.z, b.z), make_float2(b.w, b.w)};
                // Small four values at a time: few registers beside the accumulators
#pragma unroll
                for (int s = 0; s < SM; s += 4) {
                    const float4 v = *reinterpret_cast<const float4 *>(a + s);
                    const float2 a01 = make_float2(v.x, v.y), a23 = make_float2(v.z, v.w);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        acc[s / 2][e] = __ffma2_rn(a01, bb[e], acc[s / 2][e]);
                        acc[s / 2 + 1][e] = __ffma2_rn(a23, bb[e], acc[s / 2 + 1][e]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(empty(st)) : "memory");
        }
        asm volatile("bar.sync 1, %0;" :: "r"(TX_CT) : "memory");   // chunk c's buffer free
    }
    // all consumers are past the ring before it is reused for the reduction.
    // If any consumer's wait ran out, copies the producer issued may still
    // land in the ring: then no consumer touches it again and nothing is
    // stored (the error word is raised; the producer drains its copies).
    if (!ok) gave_up = 1;
    asm volatile("bar.sync 1, %0;" :: "r"(TX_CT) : "memory");
    if (gave_up) return;
    float *red = ring;                                  // [TX_CW][SM][AX_P]
#pragma unroll
    for (int t = 0; t < SM / 2; ++t) {
        *reinterpret_cast<float4 *>(red + (warp * SM + 2 * t) * AX_P + lane * 4) =
            make_float4(acc[t][0].x, acc[t][1].x, acc[t][2].x, acc[t][3].x);
        *reinterpret_cast<float4 *>(red + (warp * SM + 2 * t + 1) * AX_P + lane * 4) =
            make_float4(acc[t][0].y, acc[t][1].y, acc[t][2].y, acc[t][3].y);
    }
    asm volatile("bar.sync 1, %0;" :: "r"(TX_CT) : "memory");
    for (int o = threadIdx.x; o < SM * AX_P; o += TX_CT) {
        const int s = o / AX_P, q = o % AX_P;
        const int pp = p0 + q;
        if (s >= p.S || pp >= p.P) continue;
        float v = red[s * AX_P + q];
        for (int w = 1; w < TX_CW; ++w) v = __fadd_rn(v, red[(w * SM + s) * AX_P + q]);
        if (p.ksplit == 1) store_out(p, s, pp, v);
        else p.partial[((int64_t)blockIdx.y * p.S + s) * p.P + pp] = v;
    }
}

// The K-split CTAs' partial sums, added in K order, then the epilogue.
__global__ void __launch_bounds__(THREADS) gemv_ksum_kernel(const Params p) {
    pdl_wait();   // the K-split CTAs' partial sums are complete and visible
    const int64_t n = (int64_t)p.S * p.P;
    for (int64_t o = blockIdx.x * (int64_t)THREADS + threadIdx.x; o < n;
         o += (int64_t)gridDim.x * THREADS) {
        float v = p.partial[o];
        for (int y = 1; y < p.ksplit; ++y) v = __fadd_rn(v, p.partial[(int64_t)y * n + o]);
        store_out(p, (int)(o / p.P), (int)(o % p.P), v);
    }
}

}  // namespace gemv

namespace {

template <int SM, int PB, bool VEC>
void launch_dot(const gemv::Params &p, cudaStream_t s) {
    const int rows_per_cta = gemv::WARPS * PB;
    count_launch();
    gemv::gemv_dot_kernel<SM, PB, VEC><<<(p.P + rows_per_cta - 1) / rows_per_cta, gemv::THREADS, 0, s>>>(p);
}

template <int SM, bool VEC>
void launch_dot_pb(const gemv::Params &p, int pb, cudaStream_t s) {
    if (pb == 4) launch_dot<SM, 4, VEC>(p, s);
    else if (pb == 2) launch_dot<SM, 2, VEC>(p, s);
    else launch_dot<SM, 1, VEC>(p, s);
}

template <bool VEC>
void launch_dot_s(const gemv::Params &p, int pb, cudaStream_t s) {
    if (p.S <= 1) launch_dot_pb<1, VEC>(p, pb, s);
    else if (p.S <= 2) launch_dot_pb<2, VEC>(p, pb, s);
    else if (p.S <= 4) launch_dot_pb<4, VEC>(p, pb, s);
    else if (p.S <= 8) launch_dot_pb<8, VEC>(p, pb, s);
    else launch_dot_pb<16, VEC>(p, pb, s);
}

template <int SM, bool VEC>
int launch_axpy(const gemv::Params &p, cudaStream_t s) {
    auto kern = gemv::gemv_axpy_kernel<SM, VEC>;
    const int smem = gemv::ax_smem_floats<SM>() * (int)sizeof(float);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    dim3 grid((p.P + gemv::AX_P - 1) / gemv::AX_P, p.ksplit);
    count_launch();
    kern<<<grid, gemv::THREADS, smem, s>>>(p);
    return SGEMM_OK;
}

template <bool VEC>
int launch_axpy_s(const gemv::Params &p, cudaStream_t s) {
    if (p.S <= 1) return launch_axpy<1, VEC>(p, s);
    if (p.S <= 2) return launch_axpy<2, VEC>(p, s);
    if (p.S <= 4) return launch_axpy<4, VEC>(p, s);
    if (p.S <= 8) return launch_axpy<8, VEC>(p, s);
    return launch_axpy<16, VEC>(p, s);
}

bool al16(const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; }

// The axpy form runs on the tensor cores (tc_thin_kernel) from this S up.
// Measured on GB300 (S x 16384 x 8192 NN, and its TN twin, us per call,
// L2 flushed; FFMA staged kernel / tensor cores): S = 8 105 / 154, S = 12
// 176 / 154, S = 16 179 / 155.  Below it each element of Big feeds too few
// FMAs for the CUDA cores to be the bound.
constexpr int kThinTcMinS = 12;

std::mutex g_gemv_mu;
uint64_t g_gemv_wait_ns = 2000000000ull;   // 2 s, as the tensor-core path

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                              const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                              const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn gemv_encode_fn() {
    static EncodeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(ptr);
    });
    return fn;
}

// The staged axpy kernel (S = 8 or 16, Big 16-byte aligned with a leading
// dimension that is a multiple of 4).  Returns false when it cannot run, so
// that the caller launches the register-staged kernel instead.
template <int SM>
bool launch_axpy_tma(const gemv::Params &p, cudaStream_t s, int *status) {
    EncodeFn enc = gemv_encode_fn();
    if (!enc) return false;
    CUtensorMap map;
    const cuuint64_t dims[2] = {(cuuint64_t)p.P, (cuuint64_t)p.K};
    const cuuint64_t strides[1] = {(cuuint64_t)p.big_ld * sizeof(float)};
    const cuuint32_t box[2] = {(cuuint32_t)gemv::AX_P, (cuuint32_t)gemv::TX_KS};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(p.big), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    auto kern = gemv::gemv_axpy_tma_kernel<SM>;
    const int smem = gemv::tx_smem_bytes<SM>();
    static uint64_t attr_done = 0;   // bit d: the opt-in is set on device d
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { *status = SGEMM_ERR_CUDA; return true; }
    const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0;
    if (!bit || !(__atomic_load_n(&attr_done, __ATOMIC_ACQUIRE) & bit)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        __atomic_fetch_or(&attr_done, bit, __ATOMIC_RELEASE);
    }
    dim3 grid((p.P + gemv::AX_P - 1) / gemv::AX_P, p.ksplit);
    count_launch();
    kern<<<grid, gemv::TX_THREADS, smem, s>>>(map, p);
    *status = SGEMM_OK;
    return true;
}

int last_cuda_status() {
    return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_CUDA;
}

}  // namespace

// The thin path's tensor-core form (tc_thin_kernel) takes kThinTcMinS <= S
// <= kThinTcMaxS with the large operand's rows along the long dimension,
// 16-byte aligned with a leading dimension that is a multiple of 4.
bool thin_on_tensor_cores(char ta, char tb, int64_t M, int64_t N, int64_t lda, int64_t ldb,
                          bool a_al, bool b_al) {
    const bool rows_thin = M <= N;
    const int64_t S = rows_thin ? M : N;
    const bool big_mn = rows_thin ? is_notrans(tb) : !is_notrans(ta);
    const bool big_al = rows_thin ? (b_al && ldb % 4 == 0) : (a_al && lda % 4 == 0);
    return S >= kThinTcMinS && S <= kThinTcMaxS && big_mn && big_al;
}

// Its grid: one CTA per SM and 128 columns p; K split by the same waves x (k
// per CTA + fixed cost) model as the axpy form, the fixed cost of a CTA
// being ~512 k (its pipeline fill) and the ranges multiples of 32.
ThinTc thin_tc_geometry(int64_t P, int64_t K, int sms) {
    const int64_t pblocks = (P + 127) / 128;
    const int64_t slots = std::max(1, sms);
    const int64_t ks_max = std::max<int64_t>(1, std::min<int64_t>(K / 256, 64));
    int64_t ks = 1;
    double best = 1e30;
    for (int64_t c = 1; c <= ks_max; ++c) {
        const double t = (double)((pblocks * c + slots - 1) / slots) * ((double)K / (double)c + 512.0);
        if (t < best * 0.999) {
            best = t;
            ks = c;
        }
    }
    ThinTc g;
    g.kchunk = (int)(((K + ks - 1) / ks + 31) / 32 * 32);
    g.ksplit = (int)((K + g.kchunk - 1) / g.kchunk);
    g.ctas = (int)(pblocks * g.ksplit);
    return g;
}

namespace {

// Launch geometry shared by run_gemv and gemv_ctas.
struct Geometry {
    bool dot;            // the large operand's rows run along K
    int S, P;
    int pb;              // dot form: rows of the large operand per warp
    int kchunk, ksplit;  // axpy form: K range per CTA, CTAs along K
    int ctas;
};

Geometry geometry(char ta, char tb, int64_t M, int64_t N, int64_t K, int sms) {
    Geometry g{};
    const bool rows_thin = M <= N;
    g.S = (int)(rows_thin ? M : N);
    g.P = (int)(rows_thin ? N : M);
    g.dot = rows_thin ? !is_notrans(tb) : is_notrans(ta);
    if (g.dot) {
        // rows per warp: 4, 2 or 1, the largest that still gives 2 CTAs per SM
        g.pb = 1;
        for (int c : {4, 2}) {
            if ((g.P + gemv::WARPS * c - 1) / (gemv::WARPS * c) >= 2 * sms) { g.pb = c; break; }
        }
        g.ctas = (g.P + gemv::WARPS * g.pb - 1) / (gemv::WARPS * g.pb);
        g.ksplit = 1;
        return g;
    }
    // axpy form: split K over CTAs (each keeping at least 256 k, 32 per
    // warp).  The time goes as the waves of 2 CTAs per SM times each CTA's
    // k plus a fixed cost (staging Small, the reduction, the partial sums)
    // of about 256 k, so take the split that minimises that (128 column
    // blocks, K = 8192, 2 x 152 slots: 7 slices fill 2.95 waves, where the 3
    // that first cover one wave leave 1.26).
    const int pblocks = (g.P + gemv::AX_P - 1) / gemv::AX_P;
    const int64_t slots = std::max(1, 2 * sms);
    const int64_t ks_max = std::max<int64_t>(1, std::min<int64_t>(K / 256, 64));
    int64_t ks = 1;
    double best = 1e30;
    for (int64_t c = 1; c <= ks_max; ++c) {
        const double t = (double)((pblocks * c + slots - 1) / slots) * ((double)K / (double)c + 256.0);
        if (t < best * 0.999) {
            best = t;
            ks = c;
        }
    }
    g.kchunk = (int)((K + ks - 1) / ks);
    g.ksplit = (int)((K + g.kchunk - 1) / g.kchunk);
    g.ctas = pblocks * g.ksplit;
    return g;
}

}  // namespace

void gemv_set_wait_limit(uint64_t ns) {
    std::lock_guard<std::mutex> lk(g_gemv_mu);
    g_gemv_wait_ns = ns ? ns : 2000000000ull;
}

int gemv_take_device_error() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, gemv::g_error, sizeof(v)) != cudaSuccess) return SGEMM_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(gemv::g_error, &zero, sizeof(zero)) != cudaSuccess)
        return SGEMM_ERR_CUDA;
    return v == 0 ? SGEMM_OK : (int)v;
}

int gemv_ctas(char ta, char tb, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
              bool a_al, bool b_al, int sms) {
    if (thin_on_tensor_cores(ta, tb, M, N, lda, ldb, a_al, b_al))
        return thin_tc_geometry(std::max(M, N), std::max<int64_t>(K, 1), sms).ctas;
    return geometry(ta, tb, M, N, std::max<int64_t>(K, 1), sms).ctas;
}

int run_gemv(char ta, char tb, int64_t M, int64_t N, int64_t K, float alpha, const float *A,
             int64_t lda, const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
             cudaStream_t s, int sms, const Epilogue &epi) {
    // S above the CUDA-core forms' 16 only on the tensor cores
    const bool tc_form = thin_on_tensor_cores(ta, tb, M, N, lda, ldb, al16(A), al16(B));
    if (std::min(M, N) > (tc_form ? kThinTcMaxS : kGemvMaxSmall)) return SGEMM_ERR_UNSUPPORTED;
    const bool a_n = is_notrans(ta), b_n = is_notrans(tb);
    gemv::Params p{};
    p.K = (int)K;
    p.alpha = alpha;
    p.beta = beta;
    p.C = C;
    p.rows_thin = M <= N;
    p.row_scale = epi.row_scale;
    p.bias = epi.bias;
    p.act = epi.act;
    bool big_kcontig;
    if (M <= N) {
        // s = row i of C, p = column j: Small = op(A) (M x K), Big(j, k) = op(B)(k, j)
        p.S = (int)M;
        p.P = (int)N;
        p.small = A;
        p.small_ss = a_n ? lda : 1;
        p.small_sk = a_n ? 1 : lda;
        p.big = B;
        p.big_ld = ldb;
        big_kcontig = !b_n;                 // B 'T' is stored N x K
        p.c_s = ldc;
        p.c_p = 1;
    } else {
        // s = column j of C, p = row i: Small(j, k) = op(B)(k, j), Big = op(A)
        p.S = (int)N;
        p.P = (int)M;
        p.small = B;
        p.small_ss = b_n ? 1 : ldb;
        p.small_sk = b_n ? ldb : 1;
        p.big = A;
        p.big_ld = lda;
        big_kcontig = a_n;                  // A 'N' is stored M x K
        p.c_s = 1;
        p.c_p = ldc;
    }
    const Geometry g = geometry(ta, tb, M, N, K, sms);
    if (g.dot != big_kcontig) return SGEMM_ERR_UNSUPPORTED;   // the two views agree by construction
    if (big_kcontig) {
        // (with S = 1 Small's row stride is never used)
        const bool vec = al16(p.big) && p.big_ld % 4 == 0 && p.small_sk == 1 && al16(p.small) &&
                         (p.S == 1 || p.small_ss % 4 == 0);
        timing_mark(s, true);
        if (vec) launch_dot_s<true>(p, g.pb, s);
        else launch_dot_s<false>(p, g.pb, s);
        timing_mark(s, false);
        return last_cuda_status();
    }
    if (tc_form && (p.small_sk == 1 || p.small_ss == 1)) {
        const ThinTc tg = thin_tc_geometry(p.P, K, sms);
        ThinCall tcall{};
        tcall.S = p.S; tcall.P = p.P; tcall.K = p.K;
        tcall.kchunk = tg.kchunk;
        tcall.ksplit = tg.ksplit;
        tcall.big = p.big; tcall.big_ld = p.big_ld;
        tcall.small = p.small; tcall.small_ss = p.small_ss; tcall.small_sk = p.small_sk;
        tcall.C = p.C; tcall.c_s = p.c_s; tcall.c_p = p.c_p;
        tcall.rows_thin = p.rows_thin;
        tcall.alpha = p.alpha; tcall.beta = p.beta;
        tcall.row_scale = p.row_scale; tcall.bias = p.bias; tcall.act = p.act;
        if (tcall.ksplit > 1) {
            void *ws = nullptr;
            int st = workspace(s, (size_t)tcall.ksplit * p.S * p.P * sizeof(float), &ws, 2);
            if (st != SGEMM_OK) return st;
            tcall.partial = static_cast<float *>(ws);
        }
        int st = run_tc_thin(tcall, s);
        if (st != SGEMM_ERR_UNSUPPORTED) {
            if (st != SGEMM_OK || tcall.ksplit == 1) return st;
            p.ksplit = tcall.ksplit;
            p.partial = tcall.partial;
            const int64_t n = (int64_t)p.S * p.P;
            const int blocks = (int)std::min<int64_t>((n + gemv::THREADS - 1) / gemv::THREADS, 4 * sms);
            launch_dependent(gemv::gemv_ksum_kernel, dim3(blocks), dim3(gemv::THREADS), 0, s, p);
            return last_cuda_status();
        }
    }
    if (p.S > kGemvMaxSmall) return SGEMM_ERR_UNSUPPORTED;   // the CUDA-core forms take S <= 16
    p.kchunk = g.kchunk;
    p.ksplit = g.ksplit;
    if (p.ksplit > 1) {
        void *ws = nullptr;
        int st = workspace(s, (size_t)p.ksplit * p.S * p.P * sizeof(float), &ws, 2);
        if (st != SGEMM_OK) return st;
        p.partial = static_cast<float *>(ws);
    }
    const bool vec = al16(p.big) && p.big_ld % 4 == 0;
    {
        std::lock_guard<std::mutex> lk(g_gemv_mu);
        p.wait_ns = g_gemv_wait_ns;
    }
    timing_mark(s, true);
    int st = SGEMM_OK;
    bool staged = false;
    if (vec && p.S > 4)
        staged = p.S <= 8 ? launch_axpy_tma<8>(p, s, &st) : launch_axpy_tma<16>(p, s, &st);
    if (!staged) st = vec ? launch_axpy_s<true>(p, s) : launch_axpy_s<false>(p, s);
    timing_mark(s, false);
    if (st != SGEMM_OK) return st;
    if (p.ksplit > 1) {
        const int64_t n = (int64_t)p.S * p.P;
        const int blocks = (int)std::min<int64_t>((n + gemv::THREADS - 1) / gemv::THREADS, 4 * sms);
        launch_dependent(gemv::gemv_ksum_kernel, dim3(blocks), dim3(gemv::THREADS), 0, s, p);
    }
    return last_cuda_status();
}

}  // namespace sgemm_gb300
