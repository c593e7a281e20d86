// Tensor-core path for sm_103a: tcgen05 kind::tf32 MMAs into TMEM, operands
// brought into shared memory by TMA, fp32 accuracy by a 3xTF32 split.
//
// Each fp32 operand x is split into two TF32 numbers: hi = rna_tf32(x),
// lo = rna_tf32(x - hi) (x - hi is exact in fp32).  Then
//   a*b = a_hi*b_hi + a_hi*b_lo + a_lo*b_hi + a_lo*b_lo
// and the last term (~2^-22 |ab|) is dropped: the three TF32 products are
// accumulated in fp32 in TMEM.  Single-pass TF32 keeps only a_hi*b_hi (the
// tensor-core mode of "Optimising fp32 GEMM on A100", kernels 1-7, which
// trade accuracy for speed).  An operand is split either by a pre-pass into
// a K-contiguous workspace, or, when its rows already run along K, inside
// the kernel: A into tensor memory (on 64- and 128-wide tiles only A_hi, with
// A_lo in shared memory), B in shared memory.
//
// Kernel (320 threads; tiles of 128 x BN, or 256 x BN on a pair of SMs):
//   warp 0, one lane : TMA producer - per k-block (16 wide for 3xTF32, 32 for
//                      TF32 and for narrow tiles with A split in TMEM) loads
//                      the hi/lo (or raw) A and B tiles into a ring of
//                      shared stages, completing on the stage's "full"
//                      mbarrier (for a pair: the leader's, counting both);
//   warp 1           : allocates TMEM; one lane of the leader issues the MMAs
//                      (K = 8 per instruction) and commits them to the
//                      stage's "empty" mbarrier, and after a tile's last
//                      k-block to the "accumulator full" one;
//   warps 2..9       : split raw tiles while the main loop runs, then the
//                      epilogue - tcgen05.ld of the accumulator (warp w reads
//                      TMEM lanes 32*(w%4)..+31 = its rows), the fused
//                      alpha/beta (+ row scale, bias, activation) epilogue,
//                      row-contiguous stores.
// CTAs are persistent (one per SM, or per SM pair) when no operand is split
// in the kernel: the stage ring runs on across tiles and two TMEM
// accumulators alternate, so a tile's epilogue overlaps the next main loop.
// Tiles after the last full wave may be shared in k (stream-K, see Params),
// as may every tile of a problem with fewer tiles than SMs.
// The multi-stage ring is the asynchronous copy pipeline of "CuTe-ly
// writing an SM86 SGEMM" (section "mainloop") and "Matmul II" (section 7)
// rebuilt on TMA + mbarriers; the operand and accumulator placement is
// Blackwell's (shared-memory descriptors, TMEM, CTA pairs) and has no
// counterpart on the pages.
// Every mbarrier wait is bounded (%globaltimer): on expiry the thread sets
// the library's device error word, stops its role, drains what it issued
// (also bounded) and the CTA frees its TMEM and exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>
#include <vector>

#include "ptx_util.cuh"
#include "tc_gemm.h"

namespace sgemm_gb300 {
namespace tc {

constexpr int BM = 128;
// k-block width in fp32: 3xTF32 uses 16 (64-byte rows, 64-byte swizzle: six
// MMAs per block and twice the stages); single-pass TF32 uses 32 (128-byte
// rows and swizzle: four MMAs per block, so the per-block barrier round trip
// of the MMA thread stays small against the tensor work).  Cfg's WIDE
// variant gives 3xTF32 32-wide blocks too.
template <bool THREE> struct KBlock { static constexpr int BK = THREE ? 16 : 32; };
constexpr int KPAD = 32;               // K padding of the split operands
constexpr int THREADS = 320;               // 10 warps: TMA, MMA, 8 split/epilogue
constexpr int WORKERS = THREADS - 64;      // split/epilogue threads (warps 2..9)
constexpr int EPI_LD = 33;             // padded row of the epilogue staging tile
constexpr int SMEM_LIMIT = 232448;     // opt-in dynamic shared memory per block
constexpr uint64_t kDefaultWaitNs = 2000000000ull;   // 2 s
// Limit of the teardown waits (copies and MMAs already issued must retire
// before the CTA frees TMEM and exits); independent of the test hook so that
// a tiny role-wait limit never cuts a drain short.
constexpr uint64_t kDrainNs = 1000000000ull;         // 1 s

__device__ unsigned int g_error;        // sticky device error word (per device)

// PAIR: a cluster of two CTAs on two SMs computes a 256 x BN tile with
// tcgen05.mma.cta_group::2 (M = 256): each CTA holds its 128 rows of A and
// half (BN / 2 columns) of B, and its 128 rows of the accumulator.
// WIDE: 3xTF32 with 32-wide k-blocks (128-byte rows): the 64- and 128-wide
// tiles whose raw A streams from HBM (one or two tile columns read each row
// of A), where 64-byte row pieces halve DRAM efficiency.  Their split puts
// A_hi in TMEM and A_lo in shared memory: an MMA reading A from TMEM costs
// about the same at any N, so A_hi x [B_hi | B_lo] is one such MMA of twice
// the width, and A_lo x B_hi a shared-memory MMA.
template <int BN, bool THREE, bool PAIR = false, bool WIDE = false>
struct Cfg {
    static constexpr int BK = WIDE ? 32 : KBlock<THREE>::BK;
    static constexpr int A_BYTES = BM * BK * 4;
    static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * BK * 4;
    static constexpr int PARTS = THREE ? 2 : 1;
    static constexpr int STAGE_BYTES = PARTS * (A_BYTES + B_BYTES);
    static constexpr int EPI_BYTES = (WORKERS / 32) * 32 * EPI_LD * 4;   // a 32 x 33 tile per epilogue warp
    static constexpr int BAR_BYTES = 512;
    static constexpr int FIXED = EPI_BYTES + BAR_BYTES + 1024;
    static constexpr int STAGES_RAW = (SMEM_LIMIT - FIXED) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
    static constexpr int SMEM = STAGES * STAGE_BYTES + FIXED;
    // TMEM: the accumulators from column 0 (two of NACC * BN columns when the
    // CTA walks several tiles); a CTA that splits A in the kernel keeps one
    // accumulator, and the columns after it hold one slot of A per stage (hi,
    // then lo: PARTS * BK columns; WIDE: hi only).
    static constexpr uint32_t TMEM_COLS = 512;
    // N = 64 MMAs are short enough that one dependent chain of them into a
    // single accumulator runs at about half the tensor rate: such tiles keep
    // independent accumulators (3xTF32: one per product; TF32: even and odd
    // k-slices), summed by the epilogue.  WIDE tiles keep one per product too
    // (lo*hi at 0, hi*hi at BN, hi*lo at BN + the unit's width).
    static constexpr int NACC = (BN == 64 && !PAIR) ? (THREE ? 3 : 2) : (WIDE ? 3 : 1);
    static constexpr int NBUF = WIDE ? 1 : 2;
    static constexpr int A_TMEM_COL = WIDE ? NACC * BN : 256;
    static constexpr int A_SLOT_COLS = WIDE ? BK : PARTS * BK;
    static_assert(NBUF * NACC * BN <= 512 && NACC * BN <= A_TMEM_COL, "accumulator columns");
    static_assert(A_TMEM_COL + STAGES * A_SLOT_COLS <= 512, "A slots in TMEM");
    static_assert(STAGES >= 2, "need at least two stages");
    static_assert(BN == 64 || BN == 128 || BN == 256, "N of the MMA");
};

// Work decomposition: tiles (BM x BN) in grouped raster order.  The first
// dp_tiles run as whole tiles; each later tile (the last, partly filled
// wave) runs as tail_nsplit CTAs of BN / tail_nsplit columns each, so the
// last wave finishes in a fraction of a tile's time.
// Stream-K (sk_ctas > 0): the k-block iterations of tiles sk_tile0.. (tile
// after tile, num_kb each) are cut into sk_ctas contiguous ranges of equal
// length, one per CTA (pair).  A range covers the end of one tile, any number
// of whole tiles and the start of another; a tile it covers only in part
// leaves its fp32 partial sum in `partial` (slot 2c for the range's first
// tile, 2c + 1 for its last), and sk_fixup_kernel adds a tile's partials in
// ascending k order and applies the epilogue.  Either every tile is shared
// this way (sk_tile0 = 0, single SMs), or the CTAs first compute the first
// dp_units tiles whole, one wave after another, and share only the rest: the
// last, partly filled wave.
// The caller's operands as given.
struct RawOps {
    const float *A, *B;
    int64_t lda, ldb;
    int ta_n, tb_n;             // transA / transB is 'N'
    int K;
};

struct Params {
    float *C;
    int64_t ldc;
    int M, N, K;
    float alpha, beta;
    int tiles_m, tiles_n, group_m;
    int dp_tiles;               // tiles computed at full width
    int tail_nsplit;            // 1, 2 or 4 column slices for the rest
    int num_kb;                 // k-blocks of BK
    int fuse_a, fuse_b;         // operand loaded raw (fp32) and split in shared memory
    int units;                  // dp_tiles + (tiles - dp_tiles) * tail_nsplit
    unsigned long long wait_ns; // bounded-wait limit
    const float *row_scale;     // fused epilogue: M row scales or null
    const float *bias;          // N column biases or null
    int act;                    // SGEMM_ACT_*
    int dp_units;               // units computed whole before any stream-K range
    int sk_ctas;                // stream-K: CTAs (pairs) sharing the iterations (0: off)
    int sk_tile0;               // stream-K: first shared tile
    long long sk_iters;         // stream-K: shared tiles * num_kb
    float *partial;             // stream-K: 2 * sk_ctas tiles of TM x BN floats
    RawOps raw;                 // the caller's A and B (for the fp32 redo of non-finite sums)
    int three;                  // 3xTF32 (else single-pass TF32)
};

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Non-blocking test of the same (try_wait may suspend the thread for a while;
// a thread that polls two barriers must not sleep on either).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait for the phase of `parity` to complete.  Returns false (and
// raises the device error word) when the limit passes first.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) {
            atomicExch(&g_error, (unsigned)SGEMM_ERR_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand whose rows are
// ROW_BYTES (64 or 128) long and swizzled over that span: 8-row atoms
// 8*ROW_BYTES apart (stride byte offset), descriptor version 1, base offset 0
// (every tile is 1024-byte aligned; each +32-byte step to the next K = 8 slice
// stays inside the row).  Swizzle codes: 4 = 64-byte, 2 = 128-byte.
template <int ROW_BYTES>
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
    static_assert(ROW_BYTES == 64 || ROW_BYTES == 128, "swizzle span");
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFF) >> 4);            // start address
    d |= (uint64_t)1 << 16;                             // leading byte offset (unused here)
    d |= (uint64_t)((8 * ROW_BYTES) >> 4) << 32;        // stride byte offset
    d |= (uint64_t)1 << 46;                             // version
    d |= (uint64_t)(ROW_BYTES == 64 ? 4 : 2) << 61;     // swizzle mode
    return d;
}

// Instruction descriptor of kind::tf32: D fp32, A and B tf32, both K-major,
// N >> 3 at bit 17, M >> 4 at bit 24.
__device__ __forceinline__ uint32_t idesc_tf32(int n) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(bar) : "memory");
}

// ---- two-CTA (cluster pair) forms
__device__ __forceinline__ void umma_tf32_pair(uint32_t d_tmem, uint64_t a, uint64_t b,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}

// Arrives on the barrier at the same offset in both CTAs of the pair once
// this thread's earlier pair MMAs have completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
                 " [%0], %1;" :: "r"(bar), "h"((uint16_t)3) : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The address of a local shared variable in the leader CTA (rank 0) of the pair.
__device__ __forceinline__ uint32_t leader_addr(uint32_t local) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"(local));
    return r;
}

// Arrive with release at cluster scope: the once-per-tile hand-back of an
// accumulator, ordering this warp's TMEM reads before the leader's next MMAs.
// (Such a release stalls the thread for about an L2 round trip, longer than
// a stage's MMAs, so nothing per stage goes through a thread's arrive: the
// peer's TMA loads count their bytes on the leader's barrier directly.)
__device__ __forceinline__ void remote_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];"
                 :: "r"(cluster_addr) : "memory");
}

// TMA load into this CTA's shared memory whose completion (bytes) is counted
// on a barrier of the pair given by its cluster address (the leader's).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map,
                                                 uint32_t bar_cluster, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait on a barrier that the peer CTA also arrives on (cluster scope).
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_cluster(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) {
            atomicExch(&g_error, (unsigned)SGEMM_ERR_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// A operand from tensor memory: M = 128 lanes (rows) x 8 columns (k) of tf32.
__device__ __forceinline__ void umma_tf32_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}

// 32 lanes x 8 columns of 32-bit values from registers into tensor memory.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 :: "r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
                    "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
                    "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                    "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 columns of 32-bit accumulators -> 32 registers per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Round-to-nearest, ties away from zero, of an fp32 value to TF32 (10 stored
// mantissa bits, the low 13 bits cleared), by the conversion instruction.
__device__ __forceinline__ float tf32_round(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// Non-finite inputs.  The split is exact (up to lo's rounding) for every
// finite x whose rounding to TF32 stays finite.  An infinite x (hi = inf,
// lo = inf - inf = NaN), or a finite one that rounds to infinity (|x| above
// (2 - 2^-11) 2^127: lo = x - inf), makes every 3xTF32 sum it enters NaN,
// where fp32 arithmetic gives an infinity, NaN or, in the rounding case, a
// finite value; in single-pass TF32 such a sum is infinite or NaN.  Those
// sums are redone in fp32 after the fact: the epilogue checks its outputs
// (one packed FMA by zero per two outputs finds any NaN or infinity), and a
// block with a NaN sum (3xTF32) or a non-finite one (TF32) has those outputs
// recomputed by the warp straight from A and B.  A sum whose true value is
// infinite or NaN comes out of the redo the same, so the result is the IEEE
// fp32 one on this path too; the split itself pays nothing.
__device__ __forceinline__ float f32_inf() { return __uint_as_float(0x7f800000u); }

template <bool THREE>
__device__ __forceinline__ bool needs_redo(float v) {
    return THREE ? v != v : !(fabsf(v) < f32_inf());
}

// sum_k op(A)(row, k) * op(B)(k, col) in fp32 by the whole warp: lane l adds
// k = l, l + 32, ... with fused multiply-adds, then a butterfly adds the lanes.
// Every lane returns the sum.
__device__ __noinline__ float dot_fp32_warp(const RawOps o, int row, int col, int lane) {
    float acc = 0.0f;
    for (int k = lane; k < o.K; k += 32) {
        const float a = o.ta_n ? o.A[(int64_t)row * o.lda + k] : o.A[(int64_t)k * o.lda + row];
        const float b = o.tb_n ? o.B[(int64_t)k * o.ldb + col] : o.B[(int64_t)col * o.ldb + k];
        acc = __fmaf_rn(a, b, acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
    return acc;
}

// Warp-collective: the 32 x 32 block of sums staged at `stg` (row stride ld;
// lane l's row is row0 + l, columns col0..col0+31) has its NaN (3xTF32) or
// non-finite (TF32) entries inside M x N recomputed with dot_fp32_warp.
template <bool THREE>
__device__ __noinline__ void redo_block(float *stg, int ld, const RawOps o, int M, int N, int row0,
                                        int col0, int lane) {
    uint32_t mask = 0;
    if (row0 + lane < M)
        for (int jj = 0; jj < 32 && col0 + jj < N; ++jj)
            if (needs_redo<THREE>(stg[lane * ld + jj])) mask |= 1u << jj;
    while (true) {
        const uint32_t lanes = __ballot_sync(0xffffffffu, mask != 0);
        if (lanes == 0) break;
        const int src = __ffs(lanes) - 1;
        const int jj = __ffs(__shfl_sync(0xffffffffu, mask, src)) - 1;
        const float v = dot_fp32_warp(o, row0 + src, col0 + jj, lane);
        if (lane == src) {
            stg[lane * ld + jj] = v;
            mask &= ~(1u << jj);
        }
    }
    __syncwarp();
}

// Any NaN or infinity among 32 values (a packed FMA by zero keeps the sum 0
// unless one is).
__device__ __forceinline__ bool any_nonfinite32(const float (&v)[32]) {
    float2 z = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int j = 0; j < 32; j += 2) z = __ffma2_rn(make_float2(v[j], v[j + 1]), make_float2(0.0f, 0.0f), z);
    const float s = __fadd_rn(z.x, z.y);
    return s != s;
}

// In-place split of `n16` 16-byte groups of a shared tile: hi = round(x)
// written over x, lo = round(x - hi) written to the twin tile (THREE only).
// The WORKERS split threads stride through the tile together.
template <bool THREE>
__device__ __forceinline__ void split_tile(uint32_t hi, uint32_t lo, int n16, int ct) {
    for (int i = ct; i < n16; i += WORKERS) {
        float4 v;
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(hi + 16u * i));
        const float4 h = make_float4(tf32_round(v.x), tf32_round(v.y), tf32_round(v.z),
                                     tf32_round(v.w));
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};"
                     :: "r"(hi + 16u * i), "f"(h.x), "f"(h.y), "f"(h.z), "f"(h.w) : "memory");
        if (THREE) {
            const float4 l = make_float4(tf32_round(__fsub_rn(v.x, h.x)),
                                         tf32_round(__fsub_rn(v.y, h.y)),
                                         tf32_round(__fsub_rn(v.z, h.z)),
                                         tf32_round(__fsub_rn(v.w, h.w)));
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};"
                         :: "r"(lo + 16u * i), "f"(l.x), "f"(l.y), "f"(l.z), "f"(l.w) : "memory");
        }
    }
}

// Split of this thread's row of a raw A tile (TMA-swizzled, rows of BK
// floats) into tensor memory: row r = 32 q + lane, k = half * BK/2 .. +BK/2;
// hi = round(x) to columns tslot + k, lo = round(x - hi) to tslot + BK + k
// (THREE only).  TMA's 64-byte swizzle (BK_ = 16) flips the 16-byte chunk
// index by bits 1-2 of the row, its 128-byte swizzle (BK_ = 32) by bits 0-2.
// `taddr` is the warp's lane quarter and column tslot of tensor memory.
template <bool THREE, int BK_>
__device__ __forceinline__ void split_a_to_tmem(uint32_t raw, uint32_t taddr, int q, int half,
                                                int lane) {
    constexpr int KH = BK_ / 2;                       // k values per thread: 8 or 16
    const int r = q * 32 + lane;
    const uint32_t sw = BK_ == 16 ? (uint32_t)((r >> 1) & 3) : (uint32_t)(r & 7);
    const uint32_t row = raw + (uint32_t)(r * BK_ * 4);
#pragma unroll
    for (int g = 0; g < KH / 8; ++g) {                // 8 k values per TMEM store
        float hi[8], lo[8];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const uint32_t chunk = (uint32_t)(half * (KH / 4) + g * 2 + c);
            float4 v;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                         : "r"(row + ((chunk ^ sw) << 4)));
            const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                hi[4 * c + e] = tf32_round(x[e]);
                if (THREE) lo[4 * c + e] = tf32_round(__fsub_rn(x[e], hi[4 * c + e]));
            }
        }
        const uint32_t col = (uint32_t)(half * KH + g * 8);
        tmem_st8(taddr + col, hi);
        if (THREE) tmem_st8(taddr + (uint32_t)BK_ + col, lo);
    }
}

// WIDE tiles: this thread's row of the raw A tile (128-byte swizzle), split
// as split_a_to_tmem does, but only hi goes to tensor memory (columns tslot +
// k); lo = round(x - hi) is stored in the A_lo tile at x's own swizzled
// position, the layout the shared-memory MMA reads.
template <int BK_>
__device__ __forceinline__ void split_a_hi_lo(uint32_t raw, uint32_t lo_tile, uint32_t taddr, int q,
                                              int half, int lane) {
    constexpr int KH = BK_ / 2;                       // k values per thread
    const int r = q * 32 + lane;
    const uint32_t sw = BK_ == 16 ? (uint32_t)((r >> 1) & 3) : (uint32_t)(r & 7);
    const uint32_t roff = (uint32_t)(r * BK_ * 4);
#pragma unroll
    for (int g = 0; g < KH / 8; ++g) {                // 8 k values per TMEM store
        float hi[8];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const uint32_t chunk = (uint32_t)(half * (KH / 4) + g * 2 + c);
            const uint32_t o = roff + ((chunk ^ sw) << 4);
            float4 v;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(raw + o));
            const float x[4] = {v.x, v.y, v.z, v.w};
            float lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                hi[4 * c + e] = tf32_round(x[e]);
                lo[e] = tf32_round(__fsub_rn(x[e], hi[4 * c + e]));
            }
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};"
                         :: "r"(lo_tile + o), "f"(lo[0]), "f"(lo[1]), "f"(lo[2]), "f"(lo[3]) : "memory");
        }
        tmem_st8(taddr + (uint32_t)(half * KH + g * 8), hi);
    }
}

// ---------------------------------------------------------------- kernel
__device__ __forceinline__ void raster(int t, int tiles_m, int tiles_n, int group_m, int &tm,
                                       int &tn) {
    const int per_group = group_m * tiles_n;
    const int g = t / per_group;
    const int first_m = g * group_m;
    const int gm = min(tiles_m - first_m, group_m);
    const int r = t - g * per_group;
    tm = first_m + r % gm;
    tn = r / gm;
}

// Decodes unit u: whole tiles first, then the last-wave tiles' column slices.
// TM rows per tile (128, or 256 for a CTA pair).
__device__ __forceinline__ void unit_of(const Params &p, int TM, int BN_, int u, int &m0, int &n0,
                                        int &bn, int &nsub) {
    int tile, sub = 0;
    nsub = 1;
    if (u < p.dp_tiles) {
        tile = u;
    } else {
        const int v = u - p.dp_tiles;
        nsub = p.tail_nsplit;
        tile = p.dp_tiles + v / nsub;
        sub = v % nsub;
    }
    int tm, tn;
    raster(tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
    bn = BN_ / nsub;
    m0 = tm * TM;
    n0 = tn * BN_ + sub * bn;
}

// One piece of a CTA's work: the k-blocks [kb0, kb1) of a tile (or of a
// column slice of one).  slot < 0: the piece is the whole tile and its
// epilogue writes C; else its partial sum goes to partial slot `slot`.
struct Piece {
    int m0, n0, bn, nsub, kb0, kb1, slot;
};

// Walks a CTA's pieces in order; every role of the CTA walks the same list.
struct Walk {
    long long i, i1;            // stream-K: iterations left
    int u;                      // otherwise: next unit
    int c;                      // the CTA (pair) index
    bool first;
};

__device__ __forceinline__ void walk_begin(const Params &p, int group, Walk &w) {
    w.u = group;
    w.c = group;
    w.first = true;
    w.i = w.i1 = 0;
    if (p.sk_ctas) {
        w.i = (long long)group * p.sk_iters / p.sk_ctas;
        w.i1 = (long long)(group + 1) * p.sk_iters / p.sk_ctas;
    }
}

__device__ __forceinline__ bool walk_next(const Params &p, int TM, int BN_, int groups, Walk &w,
                                          Piece &pc) {
    if (w.u < p.dp_units) {
        // whole units, one wave after another
        unit_of(p, TM, BN_, w.u, pc.m0, pc.n0, pc.bn, pc.nsub);
        pc.kb0 = 0;
        pc.kb1 = p.num_kb;
        pc.slot = -1;
        w.u += groups;
        return true;
    }
    if (!p.sk_ctas || w.i >= w.i1) return false;
    const int t = (int)(w.i / p.num_kb);
    pc.kb0 = (int)(w.i - (long long)t * p.num_kb);
    const long long left = w.i1 - w.i;
    pc.kb1 = left < (long long)(p.num_kb - pc.kb0) ? pc.kb0 + (int)left : p.num_kb;
    unit_of(p, TM, BN_, p.sk_tile0 + t, pc.m0, pc.n0, pc.bn, pc.nsub);   // whole tiles
    pc.slot = (pc.kb0 == 0 && pc.kb1 == p.num_kb) ? -1 : 2 * w.c + (w.first ? 0 : 1);
    w.i += pc.kb1 - pc.kb0;
    w.first = false;
    return true;
}

// Persistent over units: CTA (or CTA pair) c handles units c, c + count, ...
// The k-block stream of the TMA producer and of the MMA issuer runs on across
// units (stage and phase from a per-CTA k-block counter), and the two TMEM
// accumulators alternate between units, so the epilogue of one unit overlaps
// the main loop of the next.
//
// PAIR: a cluster of two CTAs computes 256-row tiles with cta_group::2 MMAs
// issued by the leader (rank 0).  Each CTA loads its 128 rows of A and half
// of the tile's B columns into its own shared memory and keeps its 128 rows
// of the accumulator in its own TMEM.  Both operands come pre-split (the
// host never pairs an operand split in shared memory): both CTAs' TMA loads
// count their bytes on the leader's full barrier, which the leader arms for
// both.  The leader's commits free the stage and announce the accumulator in
// both CTAs (multicast); every epilogue warp of both CTAs hands the
// accumulator back on the leader's acce barrier.  Halving B per SM cuts the
// shared-memory traffic per flop by a third.
template <int BN, bool THREE, bool PAIR, bool WIDE>
__global__ void __launch_bounds__(THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tm_ahi,
                   const __grid_constant__ CUtensorMap tm_alo,
                   const __grid_constant__ CUtensorMap tm_bhi,
                   const __grid_constant__ CUtensorMap tm_blo,
                   const __grid_constant__ CUtensorMap tm_bhi_tail,
                   const __grid_constant__ CUtensorMap tm_blo_tail, const Params p) {
    using K_ = Cfg<BN, THREE, PAIR, WIDE>;
    constexpr int BK = K_::BK;
    constexpr int NW = WORKERS / 32;                   // split / epilogue warps
    constexpr int TM = PAIR ? 2 * BM : BM;             // tile rows
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *epi = reinterpret_cast<float *>(smem + K_::STAGES * K_::STAGE_BYTES);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + K_::STAGES * K_::STAGE_BYTES +
                                                  K_::EPI_BYTES);
    // bars[0..S) full, [S..2S) empty, [2S..3S) split done, [3S, 3S+2)
    // accumulator full, [3S+2, 3S+4) accumulator empty
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * K_::STAGES + 4);
    const uint32_t smem0 = smem_u32(smem);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (K_::STAGES + s); };
    auto conv_bar = [&](int s) { return bar0 + 8u * (2 * K_::STAGES + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (3 * K_::STAGES + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (3 * K_::STAGES + 2 + b); };
    // a stage: A_hi | A_lo | B_hi | B_lo, B_lo right after the unit's B_hi
    // rows (so that [B_hi | B_lo] is one operand of twice the width)
    auto a_hi = [&](int s) { return smem0 + s * K_::STAGE_BYTES; };
    auto a_lo = [&](int s) { return a_hi(s) + K_::A_BYTES; };
    auto b_hi = [&](int s) { return a_hi(s) + K_::PARTS * K_::A_BYTES; };
    auto b_lo = [&](int s, int b_rows) { return b_hi(s) + (uint32_t)(b_rows * BK * 4); };
    const bool fused = p.fuse_a || p.fuse_b;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? cluster_rank() : 0u;
    const bool leader = rank == 0;
    const int group = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;   // CTA pair index
    const int groups = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < K_::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
            mbar_init(conv_bar(s), NW);                // one arrival per split warp
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);                 // tcgen05.commit
            mbar_init(acce_bar(b), PAIR ? 2 * NW : NW);   // every epilogue warp of the tile
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_map(&tm_ahi);
        prefetch_map(&tm_bhi);
        prefetch_map(&tm_bhi_tail);
        if (THREE) {
            prefetch_map(&tm_alo);
            prefetch_map(&tm_blo);
            prefetch_map(&tm_blo_tail);
        }
    }
    if (warp == 1) {
        if (PAIR) {
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                         :: "r"(smem_u32(tmem_slot)), "r"(K_::TMEM_COLS) : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                         :: "r"(smem_u32(tmem_slot)), "r"(K_::TMEM_COLS) : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    tc_fence_before();
    if (PAIR) cluster_sync_all();   // the peer's barriers exist before anything arrives on them
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Launched after the split pre-pass, the setup above ran while the
    // pre-pass finished; its outputs are read only after this wait.  The
    // stream-K fixup may start launching now (it waits for this grid).
    pdl_wait();
    pdl_trigger();

    const uint64_t lim = p.wait_ns;
    // A CTA that splits A into TMEM has one accumulator (the A slots take
    // the columns of the second), so its pieces take turns on it.
    const int nbuf = p.fuse_a ? 1 : 2;

    // Roles are dispatched per WARP: the epilogue's tcgen05.ld is warp-collective,
    // so no lane of the producer or MMA warp may fall into it.
    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int64_t g = 0;                             // k-blocks issued by this CTA
            bool ok = true;
            // a pair: the leader's full barrier counts both CTAs' bytes
            const uint32_t lead_full0 = PAIR ? leader_addr(full_bar(0)) : 0u;
            Walk w;
            walk_begin(p, group, w);
            Piece pc;
            while (ok && walk_next(p, TM, BN, groups, w, pc)) {
                const int m0 = pc.m0, n0 = pc.n0, bn = pc.bn, nsub = pc.nsub;
                const CUtensorMap *mb_hi = nsub == 1 ? &tm_bhi : &tm_bhi_tail;
                const CUtensorMap *mb_lo = nsub == 1 ? &tm_blo : &tm_blo_tail;
                const int b_rows = PAIR ? bn / 2 : bn;            // this CTA's B rows
                const int am = m0 + (int)rank * BM, bnn = n0 + (int)rank * b_rows;
                const uint32_t a_bytes = (uint32_t)K_::A_BYTES, b_bytes = (uint32_t)(b_rows * BK * 4);
                const uint32_t tx = (p.fuse_a ? a_bytes : K_::PARTS * a_bytes) +
                                    (p.fuse_b ? b_bytes : K_::PARTS * b_bytes);
                for (int kb = pc.kb0; kb < pc.kb1; ++kb, ++g) {
                    const int s = (int)(g % K_::STAGES);
                    const uint32_t ph = (uint32_t)(g / K_::STAGES) & 1u;
                    if (!mbar_wait(empty_bar(s), ph ^ 1u, lim)) { ok = false; break; }
                    const int kc = kb * BK;
                    if (PAIR && !leader) {
                        // the leader arms its barrier with these bytes too
                        const uint32_t fb = lead_full0 + 8u * s;
                        tma_load_2d_pair(a_hi(s), &tm_ahi, fb, kc, am);
                        tma_load_2d_pair(b_hi(s), mb_hi, fb, kc, bnn);
                        if (THREE) tma_load_2d_pair(a_lo(s), &tm_alo, fb, kc, am);
                        if (THREE) tma_load_2d_pair(b_lo(s, b_rows), mb_lo, fb, kc, bnn);
                        continue;
                    }
                    mbar_expect_tx(full_bar(s), PAIR ? 2u * tx : tx);
                    // a fused operand arrives raw in its hi tile and is split there
                    tma_load_2d(a_hi(s), &tm_ahi, full_bar(s), kc, am);
                    tma_load_2d(b_hi(s), mb_hi, full_bar(s), kc, bnn);
                    if (THREE && !p.fuse_a) tma_load_2d(a_lo(s), &tm_alo, full_bar(s), kc, am);
                    if (THREE && !p.fuse_b) tma_load_2d(b_lo(s, b_rows), mb_lo, full_bar(s), kc, bnn);
                }
            }
            // drain: the last arming of each stage must have landed before
            // exit (a pair's peer, whose loads count on the leader's barrier: consumed)
            for (int64_t q = (g > K_::STAGES ? g - K_::STAGES : 0); q < g; ++q) {
                const int s = (int)(q % K_::STAGES);
                const uint32_t ph = (uint32_t)(q / K_::STAGES) & 1u;
                if (PAIR && !leader) mbar_wait(empty_bar(s), ph, kDrainNs);
                else mbar_wait(full_bar(s), ph, kDrainNs);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ------------------------------------------ MMA issuer
            int64_t g = 0;
            int j = 0;                                 // pieces done by this CTA
            bool ok = true;
            Walk w;
            walk_begin(p, group, w);
            Piece pc;
            for (; ok && walk_next(p, TM, BN, groups, w, pc); ++j) {
                const int bn = pc.bn, kb0 = pc.kb0;
                const int b = j % nbuf;
                // the epilogue must have emptied this accumulator (piece j - nbuf)
                const uint32_t eph = ((uint32_t)(j / nbuf) & 1u) ^ 1u;
                if (!(PAIR ? mbar_wait_cluster(acce_bar(b), eph, lim) : mbar_wait(acce_bar(b), eph, lim)))
                    break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(b * K_::NACC * BN);
                constexpr int NA = K_::NACC;
                const uint32_t idesc = (1u << 4) | (2u << 7) | (2u << 10) |
                                       ((uint32_t)(bn >> 3) << 17) | ((uint32_t)(TM >> 4) << 24);
                for (int kb = kb0; kb < pc.kb1; ++kb, ++g) {
                    const int s = (int)(g % K_::STAGES);
                    const uint32_t ph = (uint32_t)(g / K_::STAGES) & 1u;
                    const uint32_t ready = fused ? conv_bar(s) : full_bar(s);
                    if (!(PAIR ? mbar_wait_cluster(ready, ph, lim) : mbar_wait(ready, ph, lim))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (!PAIR && p.fuse_a) {
                        // A split into this stage's TMEM slot by the split warps
                        const uint32_t at = tmem + (uint32_t)(K_::A_TMEM_COL + s * K_::A_SLOT_COLS);
#pragma unroll
                        for (int kk = 0; kk < BK / 8; ++kk) {
                            const uint32_t off = kk * 32;
                            const uint64_t bh = smem_desc<BK * 4>(b_hi(s) + off);
                            const uint32_t first = (kb == kb0 && kk == 0) ? 0u : 1u;
                            const uint32_t ah = at + (uint32_t)(kk * 8);
                            if (WIDE) {
                                // A_hi (TMEM) x [B_hi | B_lo] (N = 2 bn): hi*hi to BN..,
                                // hi*lo to BN + bn..; A_lo (shared memory) x B_hi: lo*hi to 0..
                                const uint32_t idesc2 = idesc + ((uint32_t)(bn >> 3) << 17);
                                const uint64_t al = smem_desc<BK * 4>(a_lo(s) + off);
                                umma_tf32_ta(d + (uint32_t)BN, ah, bh, idesc2, first);
                                umma_tf32(d, al, bh, idesc, first);
                            } else if (THREE) {
                                const uint64_t bl = smem_desc<BK * 4>(b_lo(s, bn) + off);
                                const uint32_t f2 = NA == 3 ? first : 1u;
                                umma_tf32_ta(d, ah + (uint32_t)BK, bh, idesc, first);
                                umma_tf32_ta(d + (NA == 3 ? (uint32_t)(BN + bn) : 0u), ah, bl, idesc, f2);
                                umma_tf32_ta(d + (NA == 3 ? BN : 0), ah, bh, idesc, f2);
                            } else {
                                const int ka = NA == 2 ? (kk & 1) : 0;
                                const uint32_t fa = (kb == kb0 && kk < NA) ? 0u : 1u;
                                umma_tf32_ta(d + (uint32_t)(ka * BN), ah, bh, idesc, fa);
                            }
                        }
                        umma_commit(empty_bar(s));
                        continue;
                    }
#pragma unroll
                    for (int kk = 0; kk < BK / 8; ++kk) {
                        const uint32_t off = kk * 32;            // 8 tf32 = 32 bytes
                        const uint64_t ah = smem_desc<BK * 4>(a_hi(s) + off);
                        const uint64_t bh = smem_desc<BK * 4>(b_hi(s) + off);
                        const uint32_t first = (kb == kb0 && kk == 0) ? 0u : 1u;
                        if (THREE) {
                            const uint64_t al = smem_desc<BK * 4>(a_lo(s) + off);
                            const uint64_t bl = smem_desc<BK * 4>(b_lo(s, PAIR ? bn / 2 : bn) + off);
                            if (PAIR) {
                                umma_tf32_pair(d, al, bh, idesc, first);
                                umma_tf32_pair(d, ah, bl, idesc, 1u);
                                umma_tf32_pair(d, ah, bh, idesc, 1u);
                            } else {
                                const uint32_t f2 = NA == 3 ? first : 1u;
                                umma_tf32(d, al, bh, idesc, first);
                                umma_tf32(d + (NA == 3 ? (uint32_t)(BN + bn) : 0u), ah, bl, idesc, f2);
                                umma_tf32(d + (NA == 3 ? BN : 0), ah, bh, idesc, f2);
                            }
                        } else {
                            if (PAIR) {
                                umma_tf32_pair(d, ah, bh, idesc, first);
                            } else {
                                const int ka = NA == 2 ? (kk & 1) : 0;
                                const uint32_t fa = (kb == kb0 && kk < NA) ? 0u : 1u;
                                umma_tf32(d + (uint32_t)(ka * BN), ah, bh, idesc, fa);
                            }
                        }
                    }
                    if (PAIR) umma_commit_pair(empty_bar(s));
                    else umma_commit(empty_bar(s));
                }
                // this unit's accumulator is ready
                if (PAIR) umma_commit_pair(accf_bar(b));
                else umma_commit(accf_bar(b));
            }
            // all MMAs of this CTA retired before TMEM can be freed
            if (j > 0) {
                const int b = (j - 1) % nbuf;
                mbar_wait(accf_bar(b), (uint32_t)((j - 1) / nbuf) & 1u, kDrainNs);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ split + epilogue (warps 2..9)
        // Warp w owns TMEM lanes (= rows of this CTA's part of the tile)
        // 32*(w%4) .. +31, and of them every other 32-column block (two warps
        // per lane quarter).  Each 32 x 32 block is read with tcgen05.ld
        // (lane = row), turned around through a padded shared tile, then
        // written row by row: every store instruction of the warp covers 32
        // consecutive columns of one row.
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        float *stg = epi + (warp - 2) * 32 * EPI_LD;
        const int ct = threadIdx.x - 64;
        int64_t g = 0;
        int j = 0;
        Walk w;
        walk_begin(p, group, w);
        Piece pc;
        for (; walk_next(p, TM, BN, groups, w, pc); ++j) {
            const int m0 = pc.m0, n0 = pc.n0, bn = pc.bn;
            const int b_rows = PAIR ? bn / 2 : bn;
            if (fused) {
                // during the main loop these warps split the raw operand tiles
                bool ok = true;
                for (int kb = pc.kb0; kb < pc.kb1; ++kb, ++g) {
                    const int s = (int)(g % K_::STAGES);
                    const uint32_t ph = (uint32_t)(g / K_::STAGES) & 1u;
                    if (!mbar_wait(full_bar(s), ph, lim)) { ok = false; break; }
                    if (p.fuse_a) {
                        // A's hi and lo go to tensor memory, where the MMA reads
                        // them: no shared-memory traffic for A in the MMAs
                        const uint32_t slot = tmem + ((uint32_t)(q * 32) << 16) +
                                              (uint32_t)(K_::A_TMEM_COL + s * K_::A_SLOT_COLS);
                        if (WIDE) split_a_hi_lo<BK>(a_hi(s), a_lo(s), slot, q, half, lane);
                        else split_a_to_tmem<THREE, BK>(a_hi(s), slot, q, half, lane);
                        tmem_st_wait();
                        tc_fence_before();
                    }
                    if (p.fuse_b) split_tile<THREE>(b_hi(s), b_lo(s, b_rows), b_rows * BK * 4 / 16, ct);
                    if (p.fuse_b || (WIDE && p.fuse_a)) {
                        // generic-proxy stores must be visible to the tensor core's reads
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(conv_bar(s));
                }
                if (!ok) break;
            }
            const int b = j % nbuf;
            const bool ready = mbar_wait(accf_bar(b), (uint32_t)(j / nbuf) & 1u, lim);
            tc_fence_after();
            if (!ready) break;
            const float alpha = p.alpha, beta = p.beta;
            const int row0 = m0 + (int)rank * BM + q * 32;
            const int rows_here = min(32, p.M - row0);
#pragma unroll 1
            for (int c = half; c < bn / 32; c += 2) {
                uint32_t r[32];
                const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) +
                                    (uint32_t)(b * K_::NACC * BN + c * 32);
                tmem_ld32(ta, r);
                float v[32];
                if (K_::NACC == 1) {
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) v[jj] = __uint_as_float(r[jj]);
                } else {
                    // 3xTF32 (lo*hi at 0, hi*hi at BN, hi*lo at 2 BN):
                    // hi*hi + (lo*hi + hi*lo); TF32: even + odd k-slices
                    float f[32];
                    uint32_t r2[32];
                    tmem_ld32(ta + (uint32_t)(K_::NACC == 3 ? BN + bn : BN), r2);
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj)
                        f[jj] = __fadd_rn(__uint_as_float(r[jj]), __uint_as_float(r2[jj]));
                    if (K_::NACC == 3) {
                        tmem_ld32(ta + (uint32_t)BN, r2);
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) f[jj] = __fadd_rn(__uint_as_float(r2[jj]), f[jj]);
                    }
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) v[jj] = f[jj];
                }
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) stg[lane * EPI_LD + jj] = v[jj];
                // a whole tile's NaN (or, in TF32, non-finite) sums are redone in
                // fp32 (shared tiles' in the fixup)
                const bool bad = pc.slot < 0 && __any_sync(0xffffffffu, any_nonfinite32(v));
                __syncwarp();
                if (bad) redo_block<THREE>(stg, EPI_LD, p.raw, p.M, p.N, row0, n0 + c * 32, lane);
                const int col = n0 + c * 32 + lane;
                if (pc.slot >= 0) {
                    // a share of a tile's k range: the raw sum, tile-local
                    // (a pair's CTAs each write their 128 rows)
                    float *__restrict__ dst = p.partial + (int64_t)pc.slot * (TM * BN) +
                                              ((int)rank * BM + q * 32) * BN + c * 32 + lane;
#pragma unroll 8
                    for (int rr = 0; rr < 32; ++rr) dst[rr * BN] = stg[rr * EPI_LD + lane];
                } else if (col < p.N && (p.row_scale || p.bias || p.act != SGEMM_ACT_NONE)) {
                    // fused epilogue: alpha * s_row, + bias_col, activation
                    float *__restrict__ dst = p.C + (int64_t)row0 * p.ldc + col;
#pragma unroll 4
                    for (int rr = 0; rr < rows_here; ++rr) {
                        const float a_r = epi_alpha(alpha, p.row_scale, row0 + rr);
                        const float v = stg[rr * EPI_LD + lane];
                        float t = beta == 0.0f
                                      ? __fmul_rn(a_r, v)
                                      : __fmaf_rn(a_r, v, __fmul_rn(beta, dst[(int64_t)rr * p.ldc]));
                        dst[(int64_t)rr * p.ldc] = epi_tail(t, p.bias, col, p.act);
                    }
                } else if (col < p.N) {
                    float *__restrict__ dst = p.C + (int64_t)row0 * p.ldc + col;
                    if (beta == 0.0f) {
#pragma unroll 8
                        for (int rr = 0; rr < rows_here; ++rr)
                            dst[(int64_t)rr * p.ldc] = __fmul_rn(alpha, stg[rr * EPI_LD + lane]);
                    } else {
                        // issue all 32 loads of C before the first store
                        float cin[32];
#pragma unroll
                        for (int rr = 0; rr < 32; ++rr)
                            cin[rr] = rr < rows_here ? dst[(int64_t)rr * p.ldc] : 0.0f;
#pragma unroll
                        for (int rr = 0; rr < 32; ++rr)
                            if (rr < rows_here)
                                dst[(int64_t)rr * p.ldc] =
                                    __fmaf_rn(alpha, stg[rr * EPI_LD + lane], __fmul_rn(beta, cin[rr]));
                    }
                }
                __syncwarp();
            }
            // this warp has read its part of accumulator b: hand it back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (PAIR) remote_arrive_cluster(leader_addr(acce_bar(b)));
                else mbar_arrive(acce_bar(b));
            }
        }
    }

    tc_fence_before();
    if (PAIR) cluster_sync_all();   // no CTA leaves while its peer may still signal it
    else __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        if (PAIR)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;"
                         :: "r"(tmem), "r"(K_::TMEM_COLS) : "memory");
        else
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                         :: "r"(tmem), "r"(K_::TMEM_COLS) : "memory");
    }
}

// ---------------------------------------------------------------- thin problems
// out(s, p) = sum_k Small(s, k) Big(p, k) for S <= 128 outputs per column of a
// large operand Big whose rows run along P in memory (Big(p, k) at
// big[k ld + p]: decode's weights stored [K][N], or a transposed matrix
// times a few vectors).  On the CUDA cores each element of Big feeds S FMAs,
// which from S = 12 up is the bound; here the tensor cores take them.  A CTA
// owns 128 columns p of Big and one K range (K split over CTAs, multiples of
// 32; the partial sums go to the thin path's sum kernel):
//   * raw Big tiles of 32 k x 128 p arrive by TMA in a ring of their own
//     (ThinCfg::RAW stages of 16 KB), freed as soon as the split warps have read
//     them, so that the HBM stream runs ahead of the split and the MMAs;
//   * 8 warps split each tile (hi = rna_tf32(x), lo = rna_tf32(x - hi)) and
//     turn it around into the K-major 128-byte-swizzled layout of an MMA
//     operand (128 rows p x 32 k), in a ring of ThinCfg::OPS operand stages;
//   * Small, split by the pre-pass into [S][Kp] hi and lo, comes by TMA as a
//     2 SMAX-row operand per stage (SMAX = 32, 64 or 128, the least >= S): rows
//     0..SMAX-1 Small_hi, SMAX.. Small_lo (rows past S read as zeros), so any
//     S up to SMAX costs the same MMAs;
//   * per 8 k the MMA thread issues Big_hi x that operand into D1 (columns
//     0..SMAX-1 hi*hi, SMAX.. hi*lo) and Big_lo x it into D2 (lo*hi, then
//     lo*lo, unused), M = 128, N = 2 SMAX, K = 8.  The k-slices of a block
//     take turns on NSETS accumulator sets (4 of D1 and D2 for SMAX = 32, 2
//     for 64, 1 for 128), which roughly halves the error against one set;
//   * the epilogue adds each product's 4 accumulators, then hi*hi + (lo*hi
//     + hi*lo) per output, and redoes NaN sums in fp32 over the CTA's K
//     range.
// The MMAs bound it: on GB300 an M = 128 kind::tf32 MMA costs ~120 cycles
// whatever its N up to 256 (here ~116 at N = 64, by clock64 on the MMA
// thread: ~930 of a block's ~1,090 cycles).  Swapping the operands (Small's
// hi and lo stacked as M = 128, Big's 256 columns as N) makes every MMA a
// full one but doubles the shared-memory traffic per byte of Big and leaves
// room for only two raw stages: measured slower (16 x 16384 x 8192 NN 154 ->
// 165 us).
constexpr int THIN_P = 128;            // columns p per CTA (the MMA's M)
constexpr int THIN_K = 32;             // k per block
constexpr int THIN_RAW_BYTES = THIN_K * THIN_P * 4;
constexpr int THIN_A_BYTES = THIN_P * THIN_K * 4;
// SMAX: rows of Small per part in the operand, S <= SMAX (32, 64 or 128).
// The MMA's N is 2 SMAX; each accumulator set holds D1 and D2 (2 x 2 SMAX
// columns), and 512 columns of TMEM hold NSETS of them, taken by the k-slices
// of a block in turn.  A larger Small operand per stage (16 KB at SMAX = 64,
// 32 KB at 128) leaves room for fewer stages.
template <int SMAX>
struct ThinCfg {
    static constexpr int RAW = SMAX == 32 ? 6 : 5;       // raw tile stages (16 KB)
    static constexpr int OPS = SMAX == 128 ? 2 : 3;       // operand stages (Big_hi, Big_lo, Small)
    static constexpr int B_BYTES = 2 * SMAX * THIN_K * 4;
    static constexpr int OP_BYTES = 2 * THIN_A_BYTES + B_BYTES;
    static constexpr int BARS = 2 * RAW + 3 * OPS + 1;
    static constexpr int SMEM = RAW * THIN_RAW_BYTES + OPS * OP_BYTES + 512 + 1024;
    static constexpr int SET_COLS = 4 * SMAX;
    static constexpr int NSETS = 512 / SET_COLS;
    static_assert(SMAX == 32 || SMAX == 64 || SMAX == 128, "operand height");
    static_assert(BARS * 8 + 8 <= 512, "thin barriers");
    static_assert(SMEM <= SMEM_LIMIT, "thin shared memory");
    static_assert(NSETS >= 1 && (THIN_K / 8) % NSETS == 0, "k-slices per accumulator set");
};

struct ThinParams {
    int S, P, K;
    int kchunk, ksplit;                // K range of CTA y: [y kchunk, min(K, +kchunk)), kchunk % 32 == 0
    const float *big;                  // Big(p, k) = big[k * big_ld + p]
    int64_t big_ld;
    const float *small;                // Small(s, k) = small[s * small_ss + k * small_sk]
    int64_t small_ss, small_sk;
    float *C;
    int64_t c_s, c_p;                  // C(s, p) = C[s * c_s + p * c_p]
    int rows_thin;                     // s is the row of C (M small), else its column
    float alpha, beta;
    const float *row_scale, *bias;
    int act;
    float *partial;                    // ksplit > 1: [ksplit][S][P]
    unsigned long long wait_ns;
};

// 32 lanes x 8 columns of 32-bit values from tensor memory.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// sum_{k0 <= k < k1} Small(s, k) Big(p, k) in fp32 by the whole warp (lanes
// take k = k0 + lane, + 32, ...; a butterfly adds them); every lane returns it.
__device__ __noinline__ float thin_dot_fp32_warp(const ThinParams p, int s, int pp, int k0, int k1,
                                                 int lane) {
    float acc = 0.0f;
    for (int k = k0 + lane; k < k1; k += 32)
        acc = __fmaf_rn(p.small[(int64_t)s * p.small_ss + (int64_t)k * p.small_sk],
                        p.big[(int64_t)k * p.big_ld + pp], acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
    return acc;
}

template <int SMAX>
__global__ void __launch_bounds__(THREADS, 1)
    tc_thin_kernel(const __grid_constant__ CUtensorMap tm_big,
                   const __grid_constant__ CUtensorMap tm_shi,
                   const __grid_constant__ CUtensorMap tm_slo, const ThinParams p) {
    using TC = ThinCfg<SMAX>;
    constexpr int R = TC::RAW, O = TC::OPS, NW = WORKERS / 32;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t smem0 = smem_u32(smem);
    auto raw_at = [&](int r) { return smem0 + (uint32_t)(r * THIN_RAW_BYTES); };
    auto hi_at = [&](int o) { return smem0 + (uint32_t)(R * THIN_RAW_BYTES + o * TC::OP_BYTES); };
    auto lo_at = [&](int o) { return hi_at(o) + (uint32_t)THIN_A_BYTES; };
    auto b_at = [&](int o) { return hi_at(o) + (uint32_t)(2 * THIN_A_BYTES); };
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + R * THIN_RAW_BYTES + O * TC::OP_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + TC::BARS);
    const uint32_t bar0 = smem_u32(bars);
    auto raw_full = [&](int r) { return bar0 + 8u * r; };
    auto raw_empty = [&](int r) { return bar0 + 8u * (R + r); };
    auto op_ready = [&](int o) { return bar0 + 8u * (2 * R + o); };      // split done
    auto op_bfull = [&](int o) { return bar0 + 8u * (2 * R + O + o); };  // Small landed
    auto op_empty = [&](int o) { return bar0 + 8u * (2 * R + 2 * O + o); };
    const uint32_t accf = bar0 + 8u * (2 * R + 3 * O);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int p0 = (int)blockIdx.x * THIN_P;
    const int k0 = (int)blockIdx.y * p.kchunk;
    const int k1 = min(p.K, k0 + p.kchunk);
    const int nblk = (k1 - k0 + THIN_K - 1) / THIN_K;
    const uint64_t lim = p.wait_ns;

    if (warp == 0 && lane == 0) {
        for (int r = 0; r < R; ++r) {
            mbar_init(raw_full(r), 1);
            mbar_init(raw_empty(r), NW);
        }
        for (int o = 0; o < O; ++o) {
            mbar_init(op_ready(o), NW);
            mbar_init(op_bfull(o), 1);
            mbar_init(op_empty(o), 1);
        }
        mbar_init(accf, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_map(&tm_big);
        prefetch_map(&tm_shi);
        prefetch_map(&tm_slo);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(tmem_slot)), "r"(512) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();      // the split of Small is complete
    pdl_trigger();

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both rings)
        if (lane == 0) {
            int ga = 0, gb = 0;
            uint64_t idle0 = 0;
            bool ok = true;
            while (ok && (ga < nblk || gb < nblk)) {
                bool moved = false;
                if (ga < nblk && mbar_test(raw_empty(ga % R), ((uint32_t)(ga / R) & 1u) ^ 1u)) {
                    const int r = ga % R;
                    mbar_expect_tx(raw_full(r), (uint32_t)THIN_RAW_BYTES);
                    tma_load_2d(raw_at(r), &tm_big, raw_full(r), p0, k0 + ga * THIN_K);
                    ++ga;
                    moved = true;
                }
                if (gb < nblk && mbar_test(op_empty(gb % O), ((uint32_t)(gb / O) & 1u) ^ 1u)) {
                    const int o = gb % O;
                    // both parts' boxes are SMAX rows; rows past S are zero-filled
                    mbar_expect_tx(op_bfull(o), (uint32_t)TC::B_BYTES);
                    tma_load_2d(b_at(o), &tm_shi, op_bfull(o), k0 + gb * THIN_K, 0);
                    tma_load_2d(b_at(o) + (uint32_t)(SMAX * THIN_K * 4), &tm_slo, op_bfull(o),
                                k0 + gb * THIN_K, 0);
                    ++gb;
                    moved = true;
                }
                if (moved) {
                    idle0 = 0;
                } else if (idle0 == 0) {
                    idle0 = global_timer_ns();
                } else if (global_timer_ns() - idle0 > lim) {
                    atomicExch(&g_error, (unsigned)SGEMM_ERR_TIMEOUT);
                    ok = false;
                }
            }
            // drain: the last filling of each slot of both rings has landed
            for (int q = (ga > R ? ga - R : 0); q < ga; ++q)
                mbar_wait(raw_full(q % R), (uint32_t)(q / R) & 1u, kDrainNs);
            for (int q = (gb > O ? gb - O : 0); q < gb; ++q)
                mbar_wait(op_bfull(q % O), (uint32_t)(q / O) & 1u, kDrainNs);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------ MMA issuer
            const uint32_t idesc = (1u << 4) | (2u << 7) | (2u << 10) |
                                   ((uint32_t)((2 * SMAX) >> 3) << 17) | ((uint32_t)(THIN_P >> 4) << 24);
            for (int g = 0; g < nblk; ++g) {
                const int o = g % O;
                const uint32_t ph = (uint32_t)(g / O) & 1u;
                if (!mbar_wait(op_ready(o), ph, lim) || !mbar_wait(op_bfull(o), ph, lim)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < THIN_K / 8; ++kk) {
                    const uint32_t off = (uint32_t)(kk * 32);
                    const uint64_t bd = smem_desc<THIN_K * 4>(b_at(o) + off);
                    // k-slice kk into set kk % NSETS: D1 at its column 0, D2 at 2 SMAX
                    const uint32_t acc = (g == 0 && kk < TC::NSETS) ? 0u : 1u;
                    const uint32_t d = tmem + (uint32_t)((kk % TC::NSETS) * TC::SET_COLS);
                    umma_tf32(d, smem_desc<THIN_K * 4>(hi_at(o) + off), bd, idesc, acc);
                    umma_tf32(d + (uint32_t)(2 * SMAX), smem_desc<THIN_K * 4>(lo_at(o) + off), bd, idesc,
                              acc);
                }
                umma_commit(op_empty(o));
            }
            umma_commit(accf);          // every MMA issued above has completed
            mbar_wait(accf, 0u, kDrainNs);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ split + epilogue (warps 2..9)
        const int t = threadIdx.x - 64;
        const int pl = t & (THIN_P - 1);             // this thread's column p of the tile
        const int kh = t >> 7;                       // its half of a block's 32 k
        const uint32_t swz = (uint32_t)(pl & 7);     // 128-byte swizzle of row pl
        bool ok = true;
        for (int g = 0; g < nblk; ++g) {
            const int r = g % R, o = g % O;
            if (!mbar_wait(raw_full(r), (uint32_t)(g / R) & 1u, lim)) { ok = false; break; }
            // raw tile: row k (128 floats of p); this thread's 16 k of column pl
            float hi[16], lo[16];
            const float *raw = reinterpret_cast<const float *>(smem + r * THIN_RAW_BYTES);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float x = raw[(kh * 16 + j) * THIN_P + pl];
                hi[j] = tf32_round(x);
                lo[j] = tf32_round(__fsub_rn(x, hi[j]));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(raw_empty(r));
            if (!mbar_wait(op_empty(o), ((uint32_t)(g / O) & 1u) ^ 1u, lim)) { ok = false; break; }
            const uint32_t row = (uint32_t)(pl * THIN_K * 4);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t pos = row + ((((uint32_t)(kh * 4 + c)) ^ swz) << 4);
                asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};"
                             :: "r"(hi_at(o) + pos), "f"(hi[4 * c]), "f"(hi[4 * c + 1]),
                                "f"(hi[4 * c + 2]), "f"(hi[4 * c + 3]) : "memory");
                asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};"
                             :: "r"(lo_at(o) + pos), "f"(lo[4 * c]), "f"(lo[4 * c + 1]),
                                "f"(lo[4 * c + 2]), "f"(lo[4 * c + 3]) : "memory");
            }
            // generic-proxy stores must be visible to the tensor core's reads
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(op_ready(o));
        }
        // ---- epilogue: warp w reads TMEM lanes 32 (w % 4).. (its 32 columns
        // p) and s = SMAX/2 half .. + SMAX/2 - 1, 8 at a time; out = hi*hi +
        // (lo*hi + hi*lo)
        const bool ready = ok && mbar_wait(accf, 0u, lim);
        tc_fence_after();
        if (ready) {
            const int q = warp & 3, half = (warp - 2) >> 2;
            const int pp = p0 + q * 32 + lane;
#pragma unroll 1
            for (int s0 = (SMAX / 2) * half; s0 < (SMAX / 2) * (half + 1) && s0 < p.S; s0 += 8) {
                // (warp-uniform bounds)
                const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)s0;
                // each product summed over the accumulator sets, in set order
                float hh[8], hl[8], lh[8];
#pragma unroll
                for (int j = 0; j < TC::NSETS; ++j) {
                    uint32_t a[8], b[8], c[8];
                    const uint32_t tk = ta + (uint32_t)(j * TC::SET_COLS);
                    tmem_ld8(tk, a);
                    tmem_ld8(tk + (uint32_t)SMAX, b);
                    tmem_ld8(tk + (uint32_t)(2 * SMAX), c);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        hh[e] = j == 0 ? __uint_as_float(a[e]) : __fadd_rn(hh[e], __uint_as_float(a[e]));
                        hl[e] = j == 0 ? __uint_as_float(b[e]) : __fadd_rn(hl[e], __uint_as_float(b[e]));
                        lh[e] = j == 0 ? __uint_as_float(c[e]) : __fadd_rn(lh[e], __uint_as_float(c[e]));
                    }
                }
                float v[8];
                bool nan = false;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    v[e] = __fadd_rn(hh[e], __fadd_rn(lh[e], hl[e]));
                    nan |= v[e] != v[e];
                }
                // NaN sums (a split of an infinity, or of a value that rounds to
                // one) are redone in fp32 by the warp, one output at a time
                uint32_t bad = 0;
                if (pp < p.P)
                    for (int e = 0; e < 8; ++e)
                        if (s0 + e < p.S && v[e] != v[e]) bad |= 1u << e;
                if (__any_sync(0xffffffffu, nan)) {
                    while (true) {
                        const uint32_t lanes = __ballot_sync(0xffffffffu, bad != 0);
                        if (lanes == 0) break;
                        const int src = __ffs(lanes) - 1;
                        const int e = __ffs(__shfl_sync(0xffffffffu, bad, src)) - 1;
                        const float d = thin_dot_fp32_warp(p, s0 + e, p0 + q * 32 + src, k0, k1, lane);
                        if (lane == src) {
                            v[e] = d;
                            bad &= ~(1u << e);
                        }
                    }
                }
                if (pp < p.P) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int sidx = s0 + e;
                        if (sidx >= p.S) break;
                        if (p.ksplit > 1) {
                            p.partial[((int64_t)blockIdx.y * p.S + sidx) * p.P + pp] = v[e];
                            continue;
                        }
                        float *dst = p.C + (int64_t)sidx * p.c_s + (int64_t)pp * p.c_p;
                        const int crow = p.rows_thin ? sidx : pp, ccol = p.rows_thin ? pp : sidx;
                        const float a = epi_alpha(p.alpha, p.row_scale, crow);
                        const float tt = p.beta == 0.0f ? __fmul_rn(a, v[e])
                                                        : __fmaf_rn(a, v[e], __fmul_rn(p.beta, *dst));
                        *dst = epi_tail(tt, p.bias, ccol, p.act);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     :: "r"(tmem), "r"(512) : "memory");
    }
}

// ---------------------------------------------------------------- stream-K fixup
// CTA (t, y) finishes tile t: when the tile's k-blocks were shared by
// several CTAs, it adds their partial sums in ascending k order (the CTAs'
// order) and applies the epilogue exactly as the main kernel does; a tile
// computed whole by one CTA was written by that CTA and is skipped.
// Iteration x belongs to CTA ((x + 1) * G - 1) / T, the last c with
// floor(c * T / G) <= x.
template <int BN, int TM>
__global__ void __launch_bounds__(256) sk_fixup_kernel(const Params p) {
    pdl_wait();   // the main kernel's partial sums are complete and visible
    const long long T = p.sk_iters, G = p.sk_ctas;
    const int t = p.sk_tile0 + (int)blockIdx.x;
    const long long first = (long long)blockIdx.x * p.num_kb, last = first + p.num_kb - 1;
    const int c_lo = (int)(((first + 1) * G - 1) / T);
    const int c_hi = (int)(((last + 1) * G - 1) / T);
    if (c_lo == c_hi) return;
    int m0, n0, bn, nsub;
    unit_of(p, TM, BN, t, m0, n0, bn, nsub);
    constexpr int ELEMS = TM * BN;
    // Only the first CTA can start before the tile (its piece is its range's
    // last, slot 2c + 1, unless its range starts exactly at the tile); every
    // later CTA's range starts inside the tile: slot 2c.
    const int lo_slot = 2 * c_lo + ((long long)c_lo * T / G >= first ? 0 : 1);
    const float4 *part = reinterpret_cast<const float4 *>(p.partial);
    const int lane = threadIdx.x & 31;
    // Every lane of a warp runs the same iterations (ELEMS / 4 and the stride
    // are multiples of 32), so the redo below can be warp-collective.
    for (int e4 = (int)(blockIdx.y * blockDim.x + threadIdx.x); e4 < ELEMS / 4;
         e4 += (int)(gridDim.y * blockDim.x)) {
        const int e = 4 * e4;
        const int r = e / BN, cc = e - r * BN;
        const int row = m0 + r, col = n0 + cc;
        const bool valid = row < p.M && col < p.N;
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (valid) {
            v = part[(int64_t)lo_slot * (ELEMS / 4) + e4];
            // the later partials four at a time: loads first, then the adds in order
            for (int c = c_lo + 1; c <= c_hi; c += 4) {
                float4 x[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (c + u <= c_hi) x[u] = part[(int64_t)(2 * (c + u)) * (ELEMS / 4) + e4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (c + u > c_hi) break;
                    v.x = __fadd_rn(v.x, x[u].x);
                    v.y = __fadd_rn(v.y, x[u].y);
                    v.z = __fadd_rn(v.z, x[u].z);
                    v.w = __fadd_rn(v.w, x[u].w);
                }
            }
        }
        // NaN (3xTF32) or non-finite (TF32) sums redone in fp32 by the warp
        const float2 z = __ffma2_rn(make_float2(v.x, v.y), make_float2(0.0f, 0.0f),
                                    __fmul2_rn(make_float2(v.z, v.w), make_float2(0.0f, 0.0f)));
        const float zs = __fadd_rn(z.x, z.y);
        if (__any_sync(0xffffffffu, zs != zs)) {
            uint32_t mask = 0;
            const float vq[4] = {v.x, v.y, v.z, v.w};
            if (valid)
                for (int q = 0; q < 4 && col + q < p.N; ++q)
                    if (p.three ? vq[q] != vq[q] : !(fabsf(vq[q]) < f32_inf())) mask |= 1u << q;
            while (true) {
                const uint32_t lanes = __ballot_sync(0xffffffffu, mask != 0);
                if (lanes == 0) break;
                const int src = __ffs(lanes) - 1;
                const int q = __ffs(__shfl_sync(0xffffffffu, mask, src)) - 1;
                const int srow = __shfl_sync(0xffffffffu, row, src);
                const int scol = __shfl_sync(0xffffffffu, col, src) + q;
                const float d = dot_fp32_warp(p.raw, srow, scol, lane);
                if (lane == src) {
                    if (q == 0) v.x = d;
                    else if (q == 1) v.y = d;
                    else if (q == 2) v.z = d;
                    else v.w = d;
                    mask &= ~(1u << q);
                }
            }
        }
        if (!valid) continue;
        const float vs[4] = {v.x, v.y, v.z, v.w};
        float *dst = p.C + (int64_t)row * p.ldc + col;
        const float a_r = epi_alpha(p.alpha, p.row_scale, row);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (col + q >= p.N) break;
            const float tt = p.beta == 0.0f ? __fmul_rn(a_r, vs[q])
                                            : __fmaf_rn(a_r, vs[q], __fmul_rn(p.beta, dst[q]));
            dst[q] = epi_tail(tt, p.bias, col + q, p.act);
        }
    }
}

// ---------------------------------------------------------------- split pre-pass
// One operand of the split pre-pass: out[r][k] (r < rows, k < Kp, row stride
// Kp) = op value at (r, k) for k < K, 0 for K <= k < Kp; hi = rna_tf32(x),
// lo = rna_tf32(x - hi).  trans: the source is stored k-major
// (src[k*ld + r]), else src[r*ld + k]; vec: the source rows are 16-byte
// aligned (base aligned, ld % 4 == 0).
struct SplitJob {
    const float *src;
    int64_t ld;
    int rows, K, Kp;
    float *hi, *lo;
    int trans, vec;
    int blocks;                 // CTAs of this job
};

__host__ __device__ inline int split_blocks(int rows, int Kp, bool trans) {
    // transposed: one 32 x 32 tile per CTA; direct: 1024 float4 per CTA
    return trans ? (Kp / 32) * ((rows + 31) / 32)
                 : (int)(((int64_t)rows * (Kp / 4) + 1023) / 1024);
}

template <bool THREE>
__device__ __forceinline__ void split_store4(const SplitJob &j, int64_t o, float4 x) {
    const float4 h = make_float4(tf32_round(x.x), tf32_round(x.y), tf32_round(x.z),
                                 tf32_round(x.w));
    *reinterpret_cast<float4 *>(j.hi + o) = h;
    if (THREE)
        *reinterpret_cast<float4 *>(j.lo + o) =
            make_float4(tf32_round(__fsub_rn(x.x, h.x)), tf32_round(__fsub_rn(x.y, h.y)),
                        tf32_round(__fsub_rn(x.z, h.z)), tf32_round(__fsub_rn(x.w, h.w)));
}

// Both operands in one launch: CTAs [0, j0.blocks) do j0, the rest j1.
// The direct case streams float4 groups (16-byte loads where the source
// allows, always 16-byte stores); the transposed case turns 32 x 32 tiles
// around through shared memory so that reads and writes are both coalesced.
template <bool THREE>
__global__ void __launch_bounds__(256) split_pair_kernel(const SplitJob j0, const SplitJob j1) {
    pdl_trigger();   // the main kernel may launch; it waits for this grid's writes
    __shared__ float tile[32][33];
    const bool second = (int)blockIdx.x >= j0.blocks;
    const SplitJob &j = second ? j1 : j0;
    const int b = second ? (int)blockIdx.x - j0.blocks : (int)blockIdx.x;
    if (j.trans) {
        const int tiles_k = j.Kp / 32;
        const int k0 = (b % tiles_k) * 32, r0 = (b / tiles_k) * 32;
        const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int k = k0 + ty + 8 * i, r = r0 + tx;
            tile[ty + 8 * i][tx] = (k < j.K && r < j.rows) ? j.src[(int64_t)k * j.ld + r] : 0.0f;
        }
        __syncthreads();
        // each thread then writes a float4 of one output row
        const int r = r0 + (threadIdx.x >> 3), kq = (threadIdx.x & 7) * 4;
        if (r < j.rows) {
            const float4 x = make_float4(tile[kq][r - r0], tile[kq + 1][r - r0],
                                         tile[kq + 2][r - r0], tile[kq + 3][r - r0]);
            split_store4<THREE>(j, (int64_t)r * j.Kp + k0 + kq, x);
        }
        return;
    }
    const int64_t per_row = j.Kp / 4;
    const int64_t total = (int64_t)j.rows * per_row;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t g = (int64_t)b * 1024 + i * 256 + threadIdx.x;
        if (g >= total) break;
        const int64_t r = g / per_row;
        const int k = (int)(g - r * per_row) * 4;
        const float *src = j.src + r * j.ld + k;
        float4 x;
        if (j.vec && k + 3 < j.K) {
            x = __ldg(reinterpret_cast<const float4 *>(src));
        } else {
            x.x = k < j.K ? __ldg(src) : 0.0f;
            x.y = k + 1 < j.K ? __ldg(src + 1) : 0.0f;
            x.z = k + 2 < j.K ? __ldg(src + 2) : 0.0f;
            x.w = k + 3 < j.K ? __ldg(src + 3) : 0.0f;
        }
        split_store4<THREE>(j, r * j.Kp + k, x);
    }
}

// ---------------------------------------------------------------- MMA rate probe
// The tensor pipe's kind::tf32 rate, measured: one CTA per SM (the dynamic
// shared memory admits one), one thread issues `reps` MMAs of 128 x 256 x 8
// back to back from zeroed shared-memory operands into one TMEM accumulator,
// commits them to a barrier and waits (bounded).  clock64 around the issue
// loop and the wait gives that SM's cycles for `reps` MMAs (0 on a timeout).
constexpr int PROBE_SMEM = 120 * 1024;
__device__ unsigned long long g_probe_cycles[1024];

__global__ void __launch_bounds__(128, 1) tf32_rate_probe_kernel(int reps, unsigned long long wait_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar;
    __shared__ uint32_t tslot;
    // A: 128 rows x 64 bytes, B: 256 rows x 64 bytes (K = 16 floats per row)
    for (int i = threadIdx.x; i < (128 + 256) * 64 / 16; i += blockDim.x)
        reinterpret_cast<float4 *>(base)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // the zero stores are read by the tensor core (async proxy)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (threadIdx.x < 32) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;"
                     :: "r"(smem_u32(&tslot)) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tslot;
    if (threadIdx.x == 0) {
        const uint32_t idesc = idesc_tf32(256);
        const uint64_t a = smem_desc<64>(smem_u32(base));
        const uint64_t b = smem_desc<64>(smem_u32(base + 128 * 64));
        const long long t0 = clock64();
        for (int i = 0; i < reps; ++i) umma_tf32(tmem, a, b, idesc, i > 0 ? 1u : 0u);
        umma_commit(smem_u32(&bar));
        const bool ok = mbar_wait(smem_u32(&bar), 0, wait_ns);
        const long long t1 = clock64();
        if (blockIdx.x < 1024) g_probe_cycles[blockIdx.x] = ok ? (unsigned long long)(t1 - t0) : 0ull;
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" :: "r"(tmem) : "memory");
    }
}

}  // namespace tc

// ---------------------------------------------------------------- host side
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 2-D map over a [rows][Kp] fp32 array: box bk (k) x box_rows, swizzled over
// the bk*4-byte row (64 or 128 bytes); rows past `rows` read as zeros.
static bool make_map(CUtensorMap *m, const float *base, int rows, int Kp, int box_rows, int bk) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)Kp, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)Kp * sizeof(float)};
    cuuint32_t box[2] = {(cuuint32_t)bk, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               bk == 16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static std::mutex g_tc_mu;
static uint64_t g_wait_ns = tc::kDefaultWaitNs;


void tc_set_wait_limit(uint64_t ns) {
    std::lock_guard<std::mutex> lk(g_tc_mu);
    g_wait_ns = ns ? ns : tc::kDefaultWaitNs;
}

int tc_take_device_error() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, tc::g_error, sizeof(v)) != cudaSuccess) return SGEMM_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(tc::g_error, &zero, sizeof(zero)) != cudaSuccess)
        return SGEMM_ERR_CUDA;
    return v == 0 ? SGEMM_OK : (int)v;
}

static int last_status() {
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) return SGEMM_OK;
    if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
        return SGEMM_ERR_UNSUPPORTED;
    return SGEMM_ERR_CUDA;
}

int tc_probe_tf32_rate(int reps, double *mac_per_clock) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SGEMM_ERR_CUDA;
    sms = std::min(sms, 1024);
    if (cudaFuncSetAttribute(tc::tf32_rate_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             tc::PROBE_SMEM) != cudaSuccess)
        return last_status();
    std::vector<unsigned long long> cyc((size_t)sms);
    for (int run = 0; run < 2; ++run) {            // the first run warms up
        count_launch();
        tc::tf32_rate_probe_kernel<<<sms, 128, tc::PROBE_SMEM>>>(reps, tc::kDefaultWaitNs);
        int st = last_status();
        if (st != SGEMM_OK) return st;
        if (cudaDeviceSynchronize() != cudaSuccess) return SGEMM_ERR_CUDA;
    }
    if (cudaMemcpyFromSymbol(cyc.data(), tc::g_probe_cycles, cyc.size() * sizeof(cyc[0])) !=
        cudaSuccess)
        return SGEMM_ERR_CUDA;
    for (unsigned long long c : cyc)
        if (c == 0) return SGEMM_ERR_TIMEOUT;
    std::sort(cyc.begin(), cyc.end());
    const double per_mma = (double)cyc[cyc.size() / 2] / reps;   // median SM
    *mac_per_clock = 128.0 * 256.0 * 8.0 / per_mma;
    return SGEMM_OK;
}

static tc::SplitJob split_job(const float *src, int64_t ld, bool trans, int rows, int K, int Kp,
                              float *hi, float *lo) {
    tc::SplitJob j{};
    j.src = src; j.ld = ld; j.rows = rows; j.K = K; j.Kp = Kp; j.hi = hi; j.lo = lo;
    j.trans = trans;
    j.vec = aligned16(src) && ld % 4 == 0;
    j.blocks = rows > 0 ? tc::split_blocks(rows, Kp, trans) : 0;
    return j;
}

// One launch for the operands that need the pre-pass (either may be absent).
static void launch_split_pair(bool three, const tc::SplitJob &a, const tc::SplitJob &b,
                              cudaStream_t s) {
    const int blocks = a.blocks + b.blocks;
    if (blocks == 0) return;
    count_launch();
    if (three) tc::split_pair_kernel<true><<<blocks, 256, 0, s>>>(a, b);
    else tc::split_pair_kernel<false><<<blocks, 256, 0, s>>>(a, b);
}

// dep: the split pre-pass was launched just before, so this launch is its
// programmatic dependent (the kernel's setup overlaps the pre-pass's tail).
template <int BN, bool THREE, bool PAIR, bool WIDE = false>
static int launch_main(const CUtensorMap *maps, const tc::Params &p, int grid, cudaStream_t s,
                       bool dep) {
    using K_ = tc::Cfg<BN, THREE, PAIR, WIDE>;
    auto kern = tc::tc_gemm_kernel<BN, THREE, PAIR, WIDE>;
    // the shared-memory opt-in is a per-device function attribute
    static uint64_t attr_done = 0;   // bit d: set on device d
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_CUDA;
    const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0;
    if (!bit || !(__atomic_load_n(&attr_done, __ATOMIC_ACQUIRE) & bit)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, K_::SMEM) !=
            cudaSuccess)
            return last_status();
        __atomic_fetch_or(&attr_done, bit, __ATOMIC_RELEASE);
    }
    timing_mark(s, true);
    if (PAIR) {
        // clusters of two CTAs (one per SM of a pair)
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(tc::THREADS);
        cfg.dynamicSmemBytes = K_::SMEM;
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = dep ? 2 : 1;
        count_launch();
        cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], p);
    } else if (dep) {
        launch_dependent(kern, dim3(grid), dim3(tc::THREADS), K_::SMEM, s, maps[0], maps[1],
                         maps[2], maps[3], maps[4], maps[5], p);
    } else {
        count_launch();
        kern<<<grid, tc::THREADS, K_::SMEM, s>>>(maps[0], maps[1], maps[2], maps[3], maps[4],
                                                   maps[5], p);
    }
    timing_mark(s, false);
    return last_status();
}

template <int BN, bool THREE>
static int launch_main_any(bool pair, const CUtensorMap *maps, const tc::Params &p, int grid,
                           cudaStream_t s, bool dep) {
    return pair ? launch_main<BN, THREE, true>(maps, p, grid, s, dep)
                : launch_main<BN, THREE, false>(maps, p, grid, s, dep);
}

// 2-D map over a caller's K-contiguous fp32 operand (`rows` rows of K values,
// row stride ld): box bk (k) x box_rows, swizzled like the split operands;
// k past K and rows past `rows` read as zeros.
static bool make_raw_map(CUtensorMap *m, const float *base, int rows, int K, int64_t ld,
                         int box_rows, int bk) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * sizeof(float)};
    cuuint32_t box[2] = {(cuuint32_t)bk, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               bk == 16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int run_tc_thin(const ThinCall &c, cudaStream_t s) {
    if (c.S < 1 || c.S > 128 || c.P < 1 || c.K < 1 || c.kchunk % tc::THIN_K != 0)
        return SGEMM_ERR_UNSUPPORTED;
    // Small(s, k) = small[s * ss + k * sk]: K-contiguous (sk == 1) or stored k-major (ss == 1)
    const bool s_direct = c.small_sk == 1, s_trans = !s_direct && c.small_ss == 1;
    if (!s_direct && !s_trans) return SGEMM_ERR_UNSUPPORTED;
    if (!aligned16(c.big) || c.big_ld % 4 != 0) return SGEMM_ERR_UNSUPPORTED;
    const int Kp = (int)((c.K + tc::KPAD - 1) / tc::KPAD) * tc::KPAD;
    auto up = [](size_t x) { return (x + 1023) & ~size_t(1023); };
    const size_t sm_elems = up((size_t)c.S * Kp * 4) / 4;
    void *ws = nullptr;
    int st = workspace(s, 2 * sm_elems * 4, &ws);
    if (st != SGEMM_OK) return st;
    float *s_hi = static_cast<float *>(ws), *s_lo = s_hi + sm_elems;
    // every check before the first launch: UNSUPPORTED means nothing ran
    EncodeTiledFn enc = encode_fn();
    if (!enc) return SGEMM_ERR_UNSUPPORTED;
    CUtensorMap maps[3];
    {
        cuuint64_t dims[2] = {(cuuint64_t)c.P, (cuuint64_t)c.K};
        cuuint64_t strides[1] = {(cuuint64_t)c.big_ld * sizeof(float)};
        cuuint32_t box[2] = {(cuuint32_t)tc::THIN_P, (cuuint32_t)tc::THIN_K};
        cuuint32_t es[2] = {1, 1};
        if (enc(&maps[0], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(c.big), dims, strides,
                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return SGEMM_ERR_UNSUPPORTED;
    }
    const int smax = c.S <= 32 ? 32 : c.S <= 64 ? 64 : 128;   // the operand's rows per part
    if (!make_map(&maps[1], s_hi, c.S, Kp, smax, tc::THIN_K) ||
        !make_map(&maps[2], s_lo, c.S, Kp, smax, tc::THIN_K))
        return SGEMM_ERR_UNSUPPORTED;
    auto kern = smax == 32 ? tc::tc_thin_kernel<32>
                : smax == 64 ? tc::tc_thin_kernel<64> : tc::tc_thin_kernel<128>;
    const int smem_bytes = smax == 32   ? tc::ThinCfg<32>::SMEM
                           : smax == 64 ? tc::ThinCfg<64>::SMEM : tc::ThinCfg<128>::SMEM;
    static uint64_t attr_done[3] = {0, 0, 0};   // bit d: the shared-memory opt-in is set on device d
    uint64_t &done = attr_done[smax == 32 ? 0 : smax == 64 ? 1 : 2];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_CUDA;
    const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0;
    if (!bit || !(__atomic_load_n(&done, __ATOMIC_ACQUIRE) & bit)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) !=
            cudaSuccess)
            return last_status();
        __atomic_fetch_or(&done, bit, __ATOMIC_RELEASE);
    }
    tc::SplitJob js = split_job(c.small, s_direct ? c.small_ss : c.small_sk, s_trans, c.S, c.K, Kp,
                                s_hi, s_lo);
    launch_split_pair(true, js, tc::SplitJob{}, s);
    st = last_status();
    if (st != SGEMM_OK) return st;
    tc::ThinParams p{};
    p.S = c.S; p.P = c.P; p.K = c.K;
    p.kchunk = c.kchunk; p.ksplit = c.ksplit;
    p.big = c.big; p.big_ld = c.big_ld;
    p.small = c.small; p.small_ss = c.small_ss; p.small_sk = c.small_sk;
    p.C = c.C; p.c_s = c.c_s; p.c_p = c.c_p;
    p.rows_thin = c.rows_thin;
    p.alpha = c.alpha; p.beta = c.beta;
    p.row_scale = c.row_scale; p.bias = c.bias; p.act = c.act;
    p.partial = c.partial;
    {
        std::lock_guard<std::mutex> lk(g_tc_mu);
        p.wait_ns = g_wait_ns;
    }
    const dim3 grid((unsigned)((c.P + tc::THIN_P - 1) / tc::THIN_P), (unsigned)c.ksplit);
    timing_mark(s, true);
    launch_dependent(kern, grid, dim3(tc::THREADS), smem_bytes, s, maps[0], maps[1], maps[2], p);
    timing_mark(s, false);
    return last_status();
}

int run_tc(const Plan &pl, char ta, char tb, int64_t M, int64_t N, int64_t K, float alpha,
           const float *A, int64_t lda, const float *B, int64_t ldb, float beta, float *C,
           int64_t ldc, cudaStream_t s, int sms, const Epilogue &epi) {
    const bool three = pl.path == SGEMM_PATH_3XTF32;
    const int BN = pl.tile_n;
    const int Kp = (int)((K + tc::KPAD - 1) / tc::KPAD) * tc::KPAD;
    // An operand whose rows already run along K in memory, 16-byte aligned
    // with a leading dimension that is a multiple of 4, is read raw by TMA and
    // split in shared memory; any other goes through the split pre-pass into
    // the canonical K-contiguous workspace layout.  (The plan decided this
    // from the same pointers; the checks here only guard the TMA rules.)
    const TcVariant v = tc_variant(pl);
    if ((v.fuse_a && !(is_notrans(ta) && aligned16(A) && lda % 4 == 0)) ||
        (v.fuse_b && !(!is_notrans(tb) && aligned16(B) && ldb % 4 == 0)))
        return SGEMM_ERR_UNSUPPORTED;
    const bool fuse_a = v.fuse_a, fuse_b = v.fuse_b;
    const bool sk = v.sk, pair = v.pair, sk_tail = v.sk_tail;
    const int TM = pair ? 2 * tc::BM : tc::BM;          // tile rows
    const int bdiv = pair ? 2 : 1;                      // B rows per CTA = tile columns / bdiv
    auto up = [](size_t x) { return (x + 1023) & ~size_t(1023); };
    const size_t a_elems = fuse_a ? 0 : up((size_t)M * Kp * 4) / 4;
    const size_t b_elems = fuse_b ? 0 : up((size_t)N * Kp * 4) / 4;
    const int parts = three ? 2 : 1;
    // stream-K: the iterations of the shared tiles (at full width) and their
    // sharing -- every tile, or those after the last full wave
    const int64_t tiles_all = ((M + TM - 1) / TM) * ((N + BN - 1) / BN);
    const int nkb_all = Kp / v.bk;
    const int slots = pair ? std::max(sms / 2, 1) : std::max(sms, 1);
    const int64_t sk_tile0 = sk_tail ? std::min<int64_t>(pl.dp_tiles, tiles_all) : 0;
    const int64_t sk_tiles = (sk || sk_tail) ? tiles_all - sk_tile0 : 0;
    const int64_t sk_iters = sk_tiles * nkb_all;
    const int sk_ctas = sk ? (int)std::min<int64_t>(pl.tc_sk, sk_iters)
                           : sk_tail ? (int)std::min<int64_t>(slots, sk_iters) : 0;
    const size_t part_elems = sk_ctas > 0 ? (size_t)2 * sk_ctas * TM * BN : 0;
    float *a_hi = nullptr, *b_hi = nullptr, *a_lo = nullptr, *b_lo = nullptr, *partial = nullptr;
    if (a_elems + b_elems + part_elems > 0) {
        void *ws = nullptr;
        int st = workspace(s, ((size_t)parts * (a_elems + b_elems) + part_elems) * 4, &ws);
        if (st != SGEMM_OK) return st;
        a_hi = static_cast<float *>(ws);
        b_hi = a_hi + a_elems;
        a_lo = three ? b_hi + b_elems : a_hi;
        b_lo = three ? a_lo + a_elems : b_hi;
        partial = a_hi + (size_t)parts * (a_elems + b_elems);
    }

    // canonical K-major operands: A as [M][Kp], B as [N][Kp]
    const bool a_trans = !is_notrans(ta);   // A stored K x M
    const bool b_trans = is_notrans(tb);    // B stored K x N
    tc::SplitJob ja{}, jb{};
    if (!fuse_a) ja = split_job(A, lda, a_trans, (int)M, (int)K, Kp, a_hi, three ? a_lo : nullptr);
    if (!fuse_b) jb = split_job(B, ldb, b_trans, (int)N, (int)K, Kp, b_hi, three ? b_lo : nullptr);
    launch_split_pair(three, ja, jb, s);
    const bool dep = ja.blocks + jb.blocks > 0;
    int st = last_status();
    if (st != SGEMM_OK) return st;

    const int nsplit = std::max(1, pl.tail_nsplit);
    // 64- and 128-wide 3xTF32 tiles that split A into TMEM stream raw A from
    // HBM: 32-wide k-blocks (128-byte rows) there (16384 x 64 x 8192: 2.3 ->
    // 4.5 TB/s of A in the TF32 mode, which always has them; 16384 x 128 x
    // 8192 3xTF32: 142 -> 170 TFLOP/s)
    const bool wide = v.wide;
    const int bk = v.bk;
    CUtensorMap maps[6];
    bool ok;
    if (fuse_a) {
        ok = make_raw_map(&maps[0], A, (int)M, (int)K, lda, tc::BM, bk);
        maps[1] = maps[0];
    } else {
        ok = make_map(&maps[0], a_hi, (int)M, Kp, tc::BM, bk) &&
             make_map(&maps[1], a_lo, (int)M, Kp, tc::BM, bk);
    }
    if (fuse_b) {
        ok = ok && make_raw_map(&maps[2], B, (int)N, (int)K, ldb, BN / bdiv, bk) &&
             make_raw_map(&maps[4], B, (int)N, (int)K, ldb, BN / nsplit / bdiv, bk);
        maps[3] = maps[2];
        maps[5] = maps[4];
    } else {
        ok = ok && make_map(&maps[2], b_hi, (int)N, Kp, BN / bdiv, bk) &&
             make_map(&maps[3], b_lo, (int)N, Kp, BN / bdiv, bk) &&
             make_map(&maps[4], b_hi, (int)N, Kp, BN / nsplit / bdiv, bk) &&
             make_map(&maps[5], b_lo, (int)N, Kp, BN / nsplit / bdiv, bk);
    }
    if (!ok) return SGEMM_ERR_UNSUPPORTED;

    tc::Params p{};
    p.C = C; p.ldc = ldc; p.M = (int)M; p.N = (int)N; p.K = (int)K;
    p.alpha = alpha; p.beta = beta;
    p.tiles_m = (int)((M + TM - 1) / TM);
    p.tiles_n = (int)((N + BN - 1) / BN);
    p.group_m = pair ? 8 : 16;
    p.dp_tiles = std::min(pl.dp_tiles, p.tiles_m * p.tiles_n);
    p.tail_nsplit = nsplit;
    p.num_kb = Kp / bk;
    p.fuse_a = fuse_a;
    p.fuse_b = fuse_b;
    p.row_scale = epi.row_scale;
    p.bias = epi.bias;
    p.act = epi.act;
    p.raw = tc::RawOps{A, B, lda, ldb, is_notrans(ta) ? 1 : 0, is_notrans(tb) ? 1 : 0, (int)K};
    p.three = three ? 1 : 0;
    p.units = p.dp_tiles + (p.tiles_m * p.tiles_n - p.dp_tiles) * nsplit;
    p.dp_units = p.units;
    if (sk_ctas > 0) {
        if (p.num_kb != nkb_all) return SGEMM_ERR_UNSUPPORTED;   // one k-block width
        // whole tiles up to sk_tile0 (none for stream-K over every tile),
        // then the shared ones; unit_of decodes every tile at full width
        p.dp_tiles = p.tiles_m * p.tiles_n;
        p.tail_nsplit = 1;
        p.units = p.dp_tiles;
        p.dp_units = (int)sk_tile0;
        p.sk_ctas = sk_ctas;
        p.sk_tile0 = (int)sk_tile0;
        p.sk_iters = sk_iters;
        p.partial = partial;
    }
    {
        std::lock_guard<std::mutex> lk(g_tc_mu);
        p.wait_ns = g_wait_ns;
    }
    // Persistent (one CTA per SM walking the units, epilogue of one unit
    // under the main loop of the next) unless an operand is split in the
    // kernel: the split warps are also the epilogue warps, so those CTAs take
    // one unit each.
    // Stream-K: one CTA (pair) per share of the iterations.
    const int groups = sk_ctas > 0 ? sk_ctas : (fuse_a || fuse_b) ? p.units : std::min(p.units, slots);
    const int grid = groups * (pair ? 2 : 1);
    int st2;
    if (BN == 256)
        st2 = three ? launch_main_any<256, true>(pair, maps, p, grid, s, dep)
                    : launch_main_any<256, false>(pair, maps, p, grid, s, dep);
    else if (BN == 128 && wide)
        st2 = launch_main<128, true, false, true>(maps, p, grid, s, dep);
    else if (BN == 128)
        st2 = three ? launch_main_any<128, true>(pair, maps, p, grid, s, dep)
                    : launch_main_any<128, false>(pair, maps, p, grid, s, dep);
    else if (wide)
        st2 = launch_main<64, true, false, true>(maps, p, grid, s, dep);
    else
        st2 = three ? launch_main_any<64, true>(pair, maps, p, grid, s, dep)
                    : launch_main_any<64, false>(pair, maps, p, grid, s, dep);
    if (st2 != SGEMM_OK || sk_ctas == 0) return st2;
    // the shared tiles' partial sums, added in k order, then the epilogue
    const dim3 fgrid((unsigned)sk_tiles, (unsigned)(TM * BN / 1024));   // one float4 per thread
    // a programmatic dependent of the main kernel: it launches while the
    // main kernel runs and waits for it in pdl_wait()
    auto fix = pair ? (BN == 256   ? tc::sk_fixup_kernel<256, 256>
                       : BN == 128 ? tc::sk_fixup_kernel<128, 256>
                                   : tc::sk_fixup_kernel<64, 256>)
                    : (BN == 256   ? tc::sk_fixup_kernel<256, 128>
                       : BN == 128 ? tc::sk_fixup_kernel<128, 128>
                                   : tc::sk_fixup_kernel<64, 128>);
    launch_dependent(fix, fgrid, dim3(256), 0, s, p);
    return last_status();
}

}  // namespace sgemm_gb300
