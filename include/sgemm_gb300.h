/*
 * sgemm_gb300.h - single-precision GEMM on one GB300 (sm_103a), C ABI.
 *
 *   C = alpha * op(A) * op(B) + beta * C
 *
 * The operation is the GEMM definition of "Optimising fp32 GEMM on A100",
 * section "What is GEMM?" (A is M x K, B is K x N, C is M x N, alpha and beta
 * scalars), with the alpha/beta epilogue of "CuTe-ly writing an SM86 SGEMM",
 * section "epilogue" (C_out = alpha*(AB) + beta*C_in).  The argument list
 * follows the BLAS xGEMM order; the host function of "CuTe-ly writing an SM86
 * SGEMM", section "host-side setup", takes the same sizes, scalars, pointers,
 * leading dimensions and stream.
 *
 * Storage: ROW-MAJOR.
 *   transA 'N': A is stored M x K, lda >= max(1, K), op(A)(i,k) = A[i*lda + k]
 *   transA 'T': A is stored K x M, lda >= max(1, M), op(A)(i,k) = A[k*lda + i]
 *   transB 'N': B is stored K x N, ldb >= max(1, N), op(B)(k,j) = B[k*ldb + j]
 *   transB 'T': B is stored N x K, ldb >= max(1, K), op(B)(k,j) = B[j*ldb + k]
 *   C is stored M x N, ldc >= max(1, N), C(i,j) = C[i*ldc + j]
 *   'n'/'t' are accepted; 'C'/'c' mean 'T' for real data.
 *   A column-major caller computes its C by swapping A<->B, M<->N and the two
 *   trans flags (C^T = op(B)^T op(A)^T).
 *
 * Pointers: A, B, C are DEVICE pointers owned by the caller; the library never
 * frees or retains them.  A and B are only read.  C is read only when
 * beta != 0 and written only inside its M x N window (the ld gap is never
 * touched).  A and B may be NULL when M, N, K or alpha make them unused.
 * C may not overlap A or B.
 *
 * Execution: every call is asynchronous on `stream` (a cudaStream_t; NULL is
 * the legacy default stream) and never synchronises.  Calls on different
 * streams may run concurrently.  The tensor-core paths use a library-owned
 * workspace (per device, grown on demand with cudaMallocAsync on the calling
 * stream, kept until sgemm_release_workspace()).
 *
 * Errors: arguments are checked before anything is launched.  A negative
 * return value -i names the i-th argument (1-based, BLAS style) as invalid:
 * -1 transA, -2 transB, -3 M, -4 N, -5 K, -7 A, -8 lda, -9 B, -10 ldb,
 * -12 C, -13 ldc.  Positive values are sgemm_status codes below.
 *
 * Quick returns (BLAS rules): M == 0 or N == 0 does nothing.  K == 0 or
 * alpha == 0 sets C = beta*C without reading A or B, and C = 0 when
 * beta == 0 (C is not read, so NaN in C does not propagate).
 *
 * Infinities and NaN in A or B give, on every path, the result of IEEE fp32
 * arithmetic: a sum that meets an infinity is that infinity (sign of the
 * product), or NaN where an infinity meets zero or one of the other sign; NaN
 * propagates.  The tensor-core paths split each value into two TF32 parts,
 * whose cross products turn a sum that meets an infinity, or a finite value
 * above (2 - 2^-11) * 2^127 (which rounds to an infinite TF32 part), into
 * NaN; so every output that comes out NaN (3xTF32) or not finite (TF32) is
 * recomputed in fp32 straight from A and B, by one warp with fused
 * multiply-adds.  A sum whose true value is infinite or NaN comes out of the
 * recomputation the same.  Calls without such values pay one check per
 * output; calls whose outputs are mostly non-finite run much slower.
 */
#ifndef SGEMM_GB300_H
#define SGEMM_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *sgemm_stream_t; /* same handle as cudaStream_t */

typedef enum {
    SGEMM_OK = 0,
    SGEMM_ERR_CUDA = 1,        /* a CUDA call or a kernel launch failed      */
    SGEMM_ERR_TIMEOUT = 2,     /* a bounded device-side wait ran out          */
    SGEMM_ERR_NOMEM = 3,       /* the workspace could not be allocated        */
    SGEMM_ERR_UNSUPPORTED = 4, /* the forced path cannot run this problem or
                                  this device (e.g. not compute capability 10.3) */
    SGEMM_ERR_ARG = 5,         /* an argument of an auxiliary entry point     */
    SGEMM_ERR_SCRATCH = 6      /* the problem needs more scratch than the
                                  fixed-size static array of
                                  sgemm_ffma_static_scratch holds            */
} sgemm_status;

/* Activation of the fused epilogue (sgemm_epilogue). */
typedef enum {
    SGEMM_ACT_NONE = 0,
    SGEMM_ACT_RELU = 1     /* max(x, 0); NaN passes through */
} sgemm_activation;

/* Arithmetic path.  AUTO lets the per-shape selector choose among the
   fp32-accurate paths: GEMV for min(M, N) <= 16, and up to 128 where its
   tensor-core form applies (see below for the details); else FFMA's small-problem kernel for small problems (2MNK <=
   1.2e8, K <= 512, at most 1024 tiles of 16 x 16); else 3xTF32 for K >= 32
   and FFMA for K < 32.  TF32 is never chosen by AUTO. */
typedef enum {
    SGEMM_PATH_AUTO = 0,
    SGEMM_PATH_FFMA = 1,   /* CUDA-core fp32 FMA, 128x128 block tiles, 8x16
                              register outer products ("Matmul II: register
                              blocking, warp tiling, tensor cores", sections
                              3-5); small problems (the rule above, with
                              split <= 1) run one launch of 16 x 16 tiles
                              instead.  Both sum each output in ascending k
                              with fused multiply-adds, so with split == 1
                              the result is bit-identical to the naive loop
                              ("How to get a matmul kernel into the top
                              percentile (worklog)", "Optimization 1").  On
                              a large grid a K-contiguous operand is first
                              copied transposed into the workspace by one
                              extra launch (sgemm_plan_info.pre_transpose);
                              the sums and their order do not change.     */
    SGEMM_PATH_3XTF32 = 2, /* tensor cores (tcgen05 kind::tf32, TMEM
                              accumulators, TMA operand loads) with each
                              operand split x = hi + lo into two TF32 parts
                              and the three products lo*hi + hi*lo + hi*hi
                              accumulated in fp32: fp32-level accuracy.      */
    SGEMM_PATH_TF32 = 3,   /* the same tensor-core kernel with only hi*hi:
                              single-pass TF32, LOWER accuracy than fp32
                              ("Optimising fp32 GEMM on A100", "Kernel 1").  */
    SGEMM_PATH_GEMV = 4    /* thin problems, min(M, N) <= 16 (128 on the
                              tensor cores): the large operand streamed once,
                              no tiles ("Matmul II", section 8: dedicated GEMV
                              kernels for decode's M = 1 to a few dozen).
                              CUDA-core fp32 FMAs, except with 12 <= min(M, N)
                              <= 128 and the large operand's rows along the
                              long dimension (16-byte aligned, leading
                              dimension a multiple of 4): those run 3xTF32 on
                              the tensor cores.  AUTO takes this path whenever
                              min(M, N) <= 16, except with K >= 32, min(M, N)
                              > 4 and the large operand's rows along K
                              (weights stored [N][K]): those go to the 3xTF32
                              tiles; and for 16 < min(M, N) <= 128 when the
                              tensor-core form applies, K >= 32 and max(M, N)
                              >= 8 min(M, N).  Forced on
                              any other problem it returns
                              SGEMM_ERR_UNSUPPORTED.                          */
} sgemm_path;

/*
 * sgemm - C = alpha*op(A)*op(B) + beta*C on `stream`, path chosen per shape.
 * Returns SGEMM_OK, a negative argument index, or an sgemm_status code.
 */
int sgemm(char transA, char transB, int64_t M, int64_t N, int64_t K,
          float alpha, const float *A, int64_t lda,
          const float *B, int64_t ldb,
          float beta, float *C, int64_t ldc, sgemm_stream_t stream);

/*
 * sgemm_ex - as sgemm, with the path forced (sgemm_path) and the split-K
 * factor forced (split >= 1, or 0 to let the selector decide).
 * FFMA path: split = 1 computes every output tile whole (bit-identical to
 * the naive ascending-k FMA loop); split > 1 sums K in `split` contiguous
 * slices per tile whose partial results are added in a fixed order; 0 lets
 * the selector share all tiles x k-tiles iterations equally among two CTAs
 * per SM ("stream-K": deterministic, not bit-identical to the naive loop
 * where a tile is shared).
 * Tensor-core paths: split = 1 computes every 128- or 256-row tile whole;
 * split > 1 shares all tiles x k-blocks iterations in equal contiguous
 * ranges among min(split x tiles, 8 x SMs, iterations) CTAs, one SM each
 * (stream-K; shared tiles' partial sums are added in k order by a second
 * kernel); 0 lets the selector choose stream-K when fewer 128-row tiles
 * than SMs would leave SMs idle.
 * Returns SGEMM_ERR_UNSUPPORTED when the forced path cannot run the problem.
 */
int sgemm_ex(char transA, char transB, int64_t M, int64_t N, int64_t K,
             float alpha, const float *A, int64_t lda,
             const float *B, int64_t ldb,
             float beta, float *C, int64_t ldc, sgemm_stream_t stream,
             int path, int split);

/*
 * sgemm_epilogue - the GEMM with a fused epilogue, on every path:
 *
 *   C(i,j) = act( alpha * s_i * (op(A) op(B))(i,j) + beta * C(i,j) + bias_j )
 *
 * "Optimising fp32 GEMM on A100", section "Performance comparison": GEMM
 * kernels are fused with the work before and after them as prologue and
 * epilogue; "CuTe-ly writing an SM86 SGEMM", section "epilogue": other
 * epilogues swap in for alpha/beta; "Matmul II", section 6: per-row scaling
 * as position-dependent work on the accumulator.
 *
 *   row_scale   device pointer to M fp32 values s_i, or NULL (all ones)
 *   bias        device pointer to N fp32 values bias_j, or NULL (zero)
 *   activation  sgemm_activation: SGEMM_ACT_NONE or SGEMM_ACT_RELU
 *   path, split as in sgemm_ex (0, 0: the selector)
 *
 * Evaluated once per output in fp32 in this order: a_i = alpha * s_i,
 * t = a_i * acc (beta == 0: C not read) or fma(a_i, acc, beta * C(i,j)),
 * t = t + bias_j, then the activation.  With row_scale = bias = NULL and
 * SGEMM_ACT_NONE it is sgemm_ex, bit for bit.  When K == 0 or alpha == 0
 * the product term is absent: C = act(beta * C + bias).  The vectors are
 * caller-owned device memory, read only, and must hold M and N values;
 * their sizes cannot be checked.  Other arguments and errors as sgemm_ex;
 * an unknown activation returns -16.
 */
int sgemm_epilogue(char transA, char transB, int64_t M, int64_t N, int64_t K,
                   float alpha, const float *A, int64_t lda,
                   const float *B, int64_t ldb,
                   float beta, float *C, int64_t ldc,
                   const float *row_scale, const float *bias, int activation,
                   sgemm_stream_t stream, int path, int split);

/*
 * sgemm_host - the same operation on HOST buffers (same arguments and
 * conventions as sgemm, but A, B and C point to host memory).  The library
 * cuts K into up to 4 chunks, uploads each chunk's slices of A and B (after
 * C when beta != 0) on an internal stream while the previous chunks'
 * GEMMs run, accumulates the chunks into C on the device (one extra fp32
 * rounding of C per chunk), runs the last chunk in row blocks and downloads
 * each block of C on a second internal stream as soon as it is final.  When
 * beta == 0 and M >= 4096 the rows of C are done in two halves: the top half's
 * copy home runs while A's bottom rows are still being uploaded.
 * Asynchronous on `stream`: C is complete once `stream` has synchronised.
 * For the copies to overlap and to run at full speed A, B and C must be
 * page-locked (cudaHostAlloc / cudaHostRegister); pageable buffers work but
 * their copies serialise.  Device staging buffers (4*(M*K + K*N + M*N)
 * bytes) are library-owned per (device, stream) like the workspace.
 * Returns as sgemm.
 */
int sgemm_host(char transA, char transB, int64_t M, int64_t N, int64_t K,
               float alpha, const float *A, int64_t lda,
               const float *B, int64_t ldb,
               float beta, float *C, int64_t ldc, sgemm_stream_t stream);

/*
 * sgemm_plan - the selector's decision for a problem, without launching
 * anything and without touching the GPU.  `path` and `split` as in
 * sgemm_ex (0 = let the selector decide); num_sms is the GPU's SM count.
 * a_aligned/b_aligned/c_aligned say whether the base pointer is 16-byte
 * aligned.  On success writes the chosen path (sgemm_path), the CTAs per
 * output tile rounded up (FFMA or tensor-core stream-K, or the column slices
 * of the tensor cores' last-wave tiles, or the thin path's CTAs along K on the
 * tensor cores; 1 = every tile whole), the tile rows and columns (the thin
 * path: min(M, N), and 0, or 128 columns of the large operand per CTA on the
 * tensor cores), whether the FFMA path uses 16-byte loads (1) or the 4-byte edge
 * path (0), and the number of CTAs of the main kernel.  Any output pointer
 * may be NULL.  Returns SGEMM_OK or a negative argument index as sgemm.
 */
int sgemm_plan(char transA, char transB, int64_t M, int64_t N, int64_t K,
               int64_t lda, int64_t ldb, int64_t ldc,
               int a_aligned, int b_aligned, int c_aligned,
               int path, int split, int num_sms,
               int *out_path, int *out_split, int *out_tile_m, int *out_tile_n,
               int *out_vector, int *out_ctas);

/*
 * The selector's whole decision for one problem, down to the kernel variant
 * (filled by sgemm_plan_detail).  Fields that do not apply to the chosen
 * path are 0.
 */
typedef struct {
    int path;          /* sgemm_path actually run                               */
    int tile_m;        /* tile rows: 128, or 256 on an SM pair; GEMV: min(M, N)  */
    int tile_n;        /* tile columns: 64, 128 or 256 (FFMA: 128, or 16 for the
                          small-problem kernel; GEMV: 0, or 128 columns of the
                          large operand per CTA on the tensor cores)          */
    int vector;        /* FFMA / GEMV: 16-byte operand loads (else 4-byte)      */
    int ctas;          /* CTAs of the main kernel, as sgemm_plan's out_ctas     */
    int split;         /* as sgemm_plan's out_split                             */
    int dp_tiles;      /* tiles computed whole before any shared or narrowed one */
    /* tensor cores only: */
    int pair;          /* 256-row tiles on a pair of SMs (tcgen05 cta_group::2) */
    int fuse_a;        /* A split inside the kernel, into tensor memory         */
    int fuse_b;        /* B split inside the kernel, in shared memory           */
    int wide;          /* 3xTF32 with 32-wide k-blocks: A_hi in tensor memory,
                          A_lo in shared memory, one MMA over [B_hi | B_lo]     */
    int accumulators;  /* independent accumulators per tile, summed by the
                          epilogue (1, 2 or 3; 8 in the thin path's
                          tensor-core form)                                   */
    int k_block;       /* k-block width of a pipeline stage, in floats          */
    int tail_nsplit;   /* column slices of each tile after the last full wave   */
    int sk_ctas;       /* stream-K over every tile: CTAs sharing the k-blocks   */
    int sk_tail;       /* 1: the tiles after the last full wave are shared in k
                          by all CTAs (pairs)                                   */
    /* FFMA tile path only: */
    int pre_transpose; /* K-contiguous operands copied transposed by a pre-pass
                          launch before the kernel: bit 0 op(A), bit 1 op(B)   */
} sgemm_plan_info;

/*
 * sgemm_plan_detail - sgemm_plan's decision with the kernel variant spelled
 * out (sgemm_plan_info), for tests and tools that must know which kernel a
 * shape reaches.  Same arguments and checks as sgemm_plan; `out` must not be
 * NULL (-15).  Touches no GPU.
 */
int sgemm_plan_detail(char transA, char transB, int64_t M, int64_t N, int64_t K,
                      int64_t lda, int64_t ldb, int64_t ldc,
                      int a_aligned, int b_aligned, int c_aligned,
                      int path, int split, int num_sms, sgemm_plan_info *out);

/* Static description of a status code (never NULL). */
const char *sgemm_status_string(int status);

/*
 * sgemm_device_error - synchronises `stream`, then returns and clears the
 * library's sticky device error words on the current device (one per path
 * with device-side waits; the tensor cores' is reported first): SGEMM_OK, or
 * SGEMM_ERR_TIMEOUT when a bounded device-side wait gave up (the kernel
 * then stopped early and its C is undefined).  SGEMM_ERR_CUDA if the
 * synchronisation itself failed.
 */
int sgemm_device_error(sgemm_stream_t stream);

/*
 * sgemm_set_wait_limit - spin limit for the device-side waits of the
 * tensor-core path and of the thin-problem kernel that stages its large
 * operand through shared memory, in nanoseconds of %globaltimer (0 restores
 * the default of 2 s).  A test hook: a tiny limit makes a wait run out on
 * purpose so that the timeout path can be checked without hanging anything.
 * In the staged thin-problem kernel a limit below 100 us bounds a single
 * mbarrier try_wait's suspension instead, so that a wait not complete within
 * it runs out whatever the timer's resolution.
 */
int sgemm_set_wait_limit(uint64_t nanoseconds);

/*
 * Measurement hook.  sgemm_timing_enable(n), n > 0, makes the library record
 * a CUDA event pair around the main GEMM kernel (the FFMA or tensor-core
 * kernel, not the split pre-pass or the split-K reduction) of each of its
 * next n launches on the current device, on the caller's stream; n = 0 turns
 * recording off.  sgemm_timing_read(ms, capacity) waits for the recorded
 * launches, writes their durations in milliseconds (oldest first, at most
 * capacity) and clears the record; it returns the count written or a
 * negative argument index / sgemm_status (as a negative number) on error.
 * Recording costs two event records per call; it is off by default.
 */
int sgemm_timing_enable(int n);
int sgemm_timing_read(float *ms, int capacity);

/*
 * sgemm_probe_tf32_rate - the tensor pipe's measured rate for the MMAs of the
 * tensor-core paths, the denominator of their roofline: one CTA per SM issues
 * `reps` (64 .. 2^20) tcgen05.mma kind::tf32 instructions of 128 x 256 x 8
 * back to back from zeroed shared-memory operands into tensor memory, timed
 * with the SM's cycle counter.  Writes the median over the SMs of the
 * multiply-adds per clock per SM to *mac_per_clock; the TF32 peak is then
 * SMs x *mac_per_clock x 2 flop x SM clock.  A measurement hook: launches
 * on the legacy default stream and synchronises the device.  Returns
 * SGEMM_OK, -1 / -2 for a bad argument, SGEMM_ERR_TIMEOUT when a probe's
 * bounded wait ran out, SGEMM_ERR_UNSUPPORTED off compute capability 10.3.
 */
int sgemm_probe_tf32_rate(int reps, double *mac_per_clock);

/*
 * sgemm_launch_count - the number of GPU kernels this library has launched in
 * this process, on every device and path: split pre-passes, main kernels,
 * stream-K and K-split reductions, and the C = beta*C quick return.  A
 * measurement hook: the difference of two readings counts the launches in
 * between.  Never fails.
 */
int64_t sgemm_launch_count(void);

/* Free the current device's workspace (synchronises the device). */
int sgemm_release_workspace(void);

/*
 * sgemm_ffma_static_scratch - the FFMA path (SGEMM_PATH_FFMA) for callers
 * that cannot allocate device memory.  The GEMM write-ups this library
 * follows have no counterpart: this entry point exists only for its users.
 *
 * Who needs it: code that runs where cudaMalloc/cudaMallocAsync must not be
 * called - a host framework that owns the whole device memory pool and
 * forbids allocations behind its back, or a latency-critical loop that may
 * not take the allocator's locks or risk an allocation failure mid-run.
 * sgemm and sgemm_ex may allocate their workspace on first use; this call
 * never does: it calls no cudaMalloc, cudaFree or allocating library routine.
 *
 * Same arguments and result as sgemm_ex(..., SGEMM_PATH_FFMA, split), with
 * `split` = 0 letting the selector choose.  The partial sums of tiles shared
 * by several CTAs go to a file-scope static __device__ array of 16 MiB (256
 * partial tiles of 128 x 128 floats, two per CTA) that every GPU which loads
 * the library holds until the process exits.  With split = 0, where the
 * selector would share k-tiles among more than 128 CTAs, the same k-tiles
 * are shared among 128 CTAs; a forced split that needs more returns
 * SGEMM_ERR_SCRATCH and launches nothing (split = 1 never needs scratch).
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  Every call on a device shares the one array:
 * calls whose kernels overlap on the GPU (different streams, or different
 * host threads without ordering) race on it and give undefined results.  The
 * array keeps the last call's contents; nothing in it needs to start at
 * zero, because every partial tile is written in full before it is read.
 */
int sgemm_ffma_static_scratch(char transA, char transB, int64_t M, int64_t N, int64_t K,
                              float alpha, const float *A, int64_t lda,
                              const float *B, int64_t ldb,
                              float beta, float *C, int64_t ldc, sgemm_stream_t stream,
                              int split);

/* Library version, 100*major + minor. */
int sgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SGEMM_GB300_H */
