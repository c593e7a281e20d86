// sgemm_host: the GEMM on HOST buffers, with the host<->device copies
// pipelined against the computation (declared in include/sgemm_gb300.h).
//
// K is cut into chunks: C = alpha*op(A)[:, K_0]*op(B)[K_0, :] + beta*C, then
// C += alpha*op(A)[:, K_c]*op(B)[K_c, :] for each later chunk.  An internal
// upload stream sends C (when beta != 0) and then each chunk's slices of
// op(A) and op(B); the caller's stream runs each chunk's GEMM (the selector's
// path on rows x N: every chunk keeps its tile parallelism and splits only
// its own slice of the operands) as soon as its slices have landed; the last
// chunk runs in row blocks, and an internal download stream sends each block
// of C home as soon as it is final.
// With beta == 0, at least two chunks and M >= 4096, the rows of C are done
// in two phases, top half then bottom half, because the link carries both
// directions at once (measured on GB300: ~320 GB/s together against ~205 and
// ~190 alone).  The first phase uploads op(B) and op(A)'s top rows chunk by
// chunk and computes the top rows whole.  Their copy home then runs while
// op(A)'s bottom rows come in, and the second phase computes those (op(B)
// resident) in kPhase2Chunks chunks, its last in row blocks sent home as
// above.  Each chunk after the first adds one fp32 rounding
// of C, well inside the 4*K*2^-24 bound.  The caller's stream finishes after
// the last download.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <map>
#include <mutex>

#include "../../include/sgemm_gb300.h"
#include "plan.h"
#include "tc_gemm.h"

namespace sgemm_gb300 {

constexpr int kMaxChunks = 4;
constexpr int kLastBlocks = 4;
constexpr int kMaxPhases = 2;
// The second phase sends only op(A)'s bottom rows (op(B) is resident), so its
// GEMMs, not its copies, are the tail: fewer, larger ones there.  Measured on
// GB300 against the one-phase pipeline (4096^3 NN 1.091 -> 1.025 ms, 6144 x
// 4096 x 4096 TN 1.458 -> 1.317, 8192 x 2048 x 4096 1.248 -> 1.147); with 4
// chunks and 4 row blocks there the gain was 0-8 %, with 1 chunk none.
constexpr int kPhase2Chunks = 2;    // K-chunks of the second phase
constexpr int kPhase2Blocks = 2;    // row blocks of its last chunk
static_assert(kPhase2Chunks >= 1 && kPhase2Chunks <= kMaxChunks, "second-phase chunks");
static_assert(kPhase2Blocks >= 1 && kPhase2Blocks <= kLastBlocks, "second-phase row blocks");

struct HostPipe {
    bool ready = false;
    cudaStream_t up = nullptr, down = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t uploaded[kMaxPhases * kMaxChunks] = {}, computed[kMaxPhases * kLastBlocks] = {};
};

static std::mutex g_host_mu;                 // one enqueue at a time per process
static std::map<int, HostPipe> g_pipes;

static int host_pipe(HostPipe **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_CUDA;
    HostPipe &h = g_pipes[dev];
    if (!h.ready) {
        bool ok = cudaStreamCreateWithFlags(&h.up, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&h.down, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&h.start, cudaEventDisableTiming) == cudaSuccess &&
                  cudaEventCreateWithFlags(&h.done, cudaEventDisableTiming) == cudaSuccess;
        for (int i = 0; ok && i < kMaxPhases * kMaxChunks; ++i)
            ok = cudaEventCreateWithFlags(&h.uploaded[i], cudaEventDisableTiming) == cudaSuccess;
        for (int i = 0; ok && i < kMaxPhases * kLastBlocks; ++i)
            ok = cudaEventCreateWithFlags(&h.computed[i], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) {
            cudaGetLastError();
            return SGEMM_ERR_CUDA;
        }
        h.ready = true;
    }
    *out = &h;
    return SGEMM_OK;
}

static int copy_status(cudaError_t e) {
    if (e == cudaSuccess) return SGEMM_OK;
    cudaGetLastError();
    return SGEMM_ERR_CUDA;
}

}  // namespace sgemm_gb300

using namespace sgemm_gb300;

extern "C" int sgemm_host(char transA, char transB, int64_t M, int64_t N, int64_t K, float alpha,
                          const float *A, int64_t lda, const float *B, int64_t ldb, float beta,
                          float *C, int64_t ldc, sgemm_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int st = check_args(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc);
    if (st != SGEMM_OK) return st;
    if (M == 0 || N == 0) return SGEMM_OK;
    const bool need_ab = K > 0 && alpha != 0.0f;
    const bool a_n = is_notrans(transA), b_n = is_notrans(transB);
    const int64_t Ke = need_ab ? K : 0;

    // chunks of K (multiples of 32, at least 512 deep), whole when K is short
    int nk = need_ab ? (int)std::min<int64_t>(kMaxChunks, Ke / 512) : 1;
    nk = std::max(nk, 1);

    // device staging: the chunks of A and of B packed one after another, C (ld = N)
    auto up = [](size_t e) { return (e * 4 + 255) & ~size_t(255); };
    const size_t a_elems = (size_t)M * Ke, b_elems = (size_t)Ke * N, c_elems = (size_t)M * N;
    void *ws = nullptr;
    st = workspace(s, up(a_elems) + up(b_elems) + up(c_elems), &ws, 1);
    if (st != SGEMM_OK) return st;
    float *dA = static_cast<float *>(ws);
    float *dB = reinterpret_cast<float *>(static_cast<char *>(ws) + up(a_elems));
    float *dC = reinterpret_cast<float *>(static_cast<char *>(ws) + up(a_elems) + up(b_elems));

    std::lock_guard<std::mutex> lk(g_host_mu);
    HostPipe *h = nullptr;
    st = host_pipe(&h);
    if (st != SGEMM_OK) return st;

    // nothing of this call may start before the work already on the caller's stream
    if ((st = copy_status(cudaEventRecord(h->start, s))) != SGEMM_OK) return st;
    if ((st = copy_status(cudaStreamWaitEvent(h->up, h->start, 0))) != SGEMM_OK) return st;
    if ((st = copy_status(cudaStreamWaitEvent(h->down, h->start, 0))) != SGEMM_OK) return st;

    // phases: row ranges of C done one after the other.  Two only when C is
    // not read (beta == 0): with beta != 0 the call's uploads grow by C and
    // bound it, and a download beside them slows them (4096^3 NT, beta 0.5:
    // 1.42 ms in one phase, 1.46-1.50 in two); and only from 4096 rows (at
    // 2048 the halves' GEMMs are too small to gain).
    const int nph = (need_ab && beta == 0.0f && nk >= 2 && M >= 4096) ? 2 : 1;
    int64_t prow[kMaxPhases + 1] = {0, M, M};
    if (nph == 2) prow[1] = (M / 2 + 127) / 128 * 128;
    // op(B) staged in its stored shape (K x N for 'N', N x K for 'T'), so that
    // any K range of it is one strided operand
    const int64_t ldb_d = b_n ? N : std::max<int64_t>(1, Ke);
    auto b_at = [&](int64_t k0) { return b_n ? dB + k0 * N : dB + k0; };
    size_t a_off = 0;
    for (int ph = 0; ph < nph; ++ph) {
        const int64_t r0 = prow[ph], rows = prow[ph + 1] - prow[ph];
        // the second phase's operands are short to send (op(B) is resident):
        // fewer, larger GEMMs there
        const int nkp = ph == 0 ? nk : std::max(1, std::min(nk, kPhase2Chunks));
        const int64_t kcp = ((Ke + nkp - 1) / nkp + 31) / 32 * 32;
        if (beta != 0.0f) {
            st = copy_status(cudaMemcpy2DAsync(dC + r0 * N, N * 4, C + r0 * ldc, ldc * 4, N * 4, rows,
                                               cudaMemcpyHostToDevice, h->up));
            if (st != SGEMM_OK) return st;
        }
        for (int c = 0; c < nkp; ++c) {
            const int64_t k0 = (int64_t)c * kcp;
            const int64_t kc = need_ab ? std::max<int64_t>(0, std::min<int64_t>(kcp, Ke - k0)) : 0;
            // the chunk's slices: op(A)[r0:r0+rows, k0:k0+kc] packed, and
            // (first phase) op(B)[k0:k0+kc, :] into its place
            float *a_c = dA + a_off;
            const int64_t lda_c = a_n ? std::max<int64_t>(1, kc) : rows;
            if (kc > 0) {
                if (a_n)   // rows r0.. of A, columns k0..
                    st = copy_status(cudaMemcpy2DAsync(a_c, kc * 4, A + r0 * lda + k0, lda * 4, kc * 4,
                                                       rows, cudaMemcpyHostToDevice, h->up));
                else       // rows k0 .. k0+kc of the stored K x M array, columns r0..
                    st = copy_status(cudaMemcpy2DAsync(a_c, rows * 4, A + k0 * lda + r0, lda * 4,
                                                       rows * 4, kc, cudaMemcpyHostToDevice, h->up));
                if (st != SGEMM_OK) return st;
                a_off += (size_t)rows * kc;
                if (ph == 0) {
                    if (b_n)   // rows k0 .. k0+kc of the stored K x N array
                        st = copy_status(cudaMemcpy2DAsync(b_at(k0), N * 4, B + k0 * ldb, ldb * 4,
                                                           N * 4, kc, cudaMemcpyHostToDevice, h->up));
                    else       // N rows, columns k0.. of each
                        st = copy_status(cudaMemcpy2DAsync(b_at(k0), ldb_d * 4, B + k0, ldb * 4, kc * 4,
                                                           N, cudaMemcpyHostToDevice, h->up));
                    if (st != SGEMM_OK) return st;
                }
            }
            cudaEvent_t up_ev = h->uploaded[ph * kMaxChunks + c];
            if ((st = copy_status(cudaEventRecord(up_ev, h->up))) != SGEMM_OK) return st;
            if ((st = copy_status(cudaStreamWaitEvent(s, up_ev, 0))) != SGEMM_OK) return st;
            const float beta_c = c == 0 ? beta : 1.0f;
            const float *a_arg = kc > 0 ? a_c : nullptr, *b_arg = kc > 0 ? b_at(k0) : nullptr;
            float *c_ph = dC + r0 * N;
            if (c + 1 < nkp) {
                st = gemm_impl(transA, transB, rows, N, kc, alpha, a_arg, lda_c, b_arg, ldb_d, beta_c,
                               c_ph, N, s, SGEMM_PATH_AUTO, 0);
                if (st != SGEMM_OK) return st;
                continue;
            }
            // last chunk: the first phase whole (its copy home runs under the
            // next phase's uploads), the last phase in row blocks, each sent
            // home as soon as it is final
            const int nbmax = nph == 1 ? kLastBlocks : kPhase2Blocks;
            const int nb = ph + 1 < nph ? 1
                                        : (int)std::max<int64_t>(1, std::min<int64_t>(nbmax, rows / 512));
            const int64_t per = ((rows + nb - 1) / nb + 127) / 128 * 128;
            for (int b = 0; b < nb; ++b) {
                const int64_t q0 = (int64_t)b * per;
                if (q0 >= rows) break;
                const int64_t qn = std::min<int64_t>(per, rows - q0);
                const float *a_blk = a_arg ? (a_n ? a_arg + q0 * lda_c : a_arg + q0) : nullptr;
                st = gemm_impl(transA, transB, qn, N, kc, alpha, a_blk, lda_c, b_arg, ldb_d, beta_c,
                               c_ph + q0 * N, N, s, SGEMM_PATH_AUTO, 0);
                if (st != SGEMM_OK) return st;
                cudaEvent_t done_ev = h->computed[ph * kLastBlocks + b];
                if ((st = copy_status(cudaEventRecord(done_ev, s))) != SGEMM_OK) return st;
                if ((st = copy_status(cudaStreamWaitEvent(h->down, done_ev, 0))) != SGEMM_OK) return st;
                st = copy_status(cudaMemcpy2DAsync(C + (r0 + q0) * ldc, ldc * 4, c_ph + q0 * N, N * 4,
                                                   N * 4, qn, cudaMemcpyDeviceToHost, h->down));
                if (st != SGEMM_OK) return st;
            }
        }
    }
    if ((st = copy_status(cudaEventRecord(h->done, h->down))) != SGEMM_OK) return st;
    return copy_status(cudaStreamWaitEvent(s, h->done, 0));
}
