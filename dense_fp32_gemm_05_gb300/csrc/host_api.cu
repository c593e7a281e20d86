// sgemm_host: the GEMM on HOST buffers, with the host<->device copies
// pipelined against the computation (declared in include/sgemm_gb300.h).
//
// K is cut into chunks: C = alpha*op(A)[:, K_0]*op(B)[K_0, :] + beta*C, then
// C += alpha*op(A)[:, K_c]*op(B)[K_c, :] for each later chunk.  An internal
// upload stream sends C (when beta != 0) and then each chunk's slices of A
// and B; the caller's stream runs each chunk's GEMM (the selector's path, on
// the whole M x N, so every chunk keeps full tile parallelism and splits only
// its own slice of the operands) as soon as its slices have landed; the last
// chunk runs in row blocks and an internal download stream sends each block
// of C back as soon as it is final.  So the uploads overlap the computation
// of earlier chunks and the download overlaps the last chunk.  Each chunk
// after the first adds one fp32 rounding of C, well inside the 4*K*2^-24
// bound.  The caller's stream finishes after the last download.
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

struct HostPipe {
    bool ready = false;
    cudaStream_t up = nullptr, down = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t uploaded[kMaxChunks] = {}, computed[kLastBlocks] = {};
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
        for (int i = 0; ok && i < kMaxChunks; ++i)
            ok = cudaEventCreateWithFlags(&h.uploaded[i], cudaEventDisableTiming) == cudaSuccess;
        for (int i = 0; ok && i < kLastBlocks; ++i)
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
    const int64_t kc_full = ((Ke + nk - 1) / nk + 31) / 32 * 32;

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

    if (beta != 0.0f) {
        st = copy_status(cudaMemcpy2DAsync(dC, N * 4, C, ldc * 4, N * 4, M,
                                           cudaMemcpyHostToDevice, h->up));
        if (st != SGEMM_OK) return st;
    }

    size_t a_off = 0, b_off = 0;
    for (int c = 0; c < nk; ++c) {
        const int64_t k0 = (int64_t)c * kc_full;
        const int64_t kc = need_ab ? std::max<int64_t>(0, std::min<int64_t>(kc_full, Ke - k0)) : 0;
        // the chunk's slices, packed: op(A)[:, k0:k0+kc] and op(B)[k0:k0+kc, :]
        float *a_c = dA + a_off, *b_c = dB + b_off;
        int64_t lda_c = a_n ? std::max<int64_t>(1, kc) : M;
        int64_t ldb_c = b_n ? N : std::max<int64_t>(1, kc);
        if (kc > 0) {
            if (a_n)   // M rows, columns k0.. of each
                st = copy_status(cudaMemcpy2DAsync(a_c, kc * 4, A + k0, lda * 4, kc * 4, M,
                                                   cudaMemcpyHostToDevice, h->up));
            else       // rows k0 .. k0+kc of the stored K x M array
                st = copy_status(cudaMemcpy2DAsync(a_c, M * 4, A + k0 * lda, lda * 4, M * 4, kc,
                                                   cudaMemcpyHostToDevice, h->up));
            if (st != SGEMM_OK) return st;
            if (b_n)   // rows k0 .. k0+kc of the stored K x N array
                st = copy_status(cudaMemcpy2DAsync(b_c, N * 4, B + k0 * ldb, ldb * 4, N * 4, kc,
                                                   cudaMemcpyHostToDevice, h->up));
            else       // N rows, columns k0.. of each
                st = copy_status(cudaMemcpy2DAsync(b_c, kc * 4, B + k0, ldb * 4, kc * 4, N,
                                                   cudaMemcpyHostToDevice, h->up));
            if (st != SGEMM_OK) return st;
            a_off += (size_t)M * kc;
            b_off += (size_t)kc * N;
        }
        if ((st = copy_status(cudaEventRecord(h->uploaded[c], h->up))) != SGEMM_OK) return st;
        if ((st = copy_status(cudaStreamWaitEvent(s, h->uploaded[c], 0))) != SGEMM_OK) return st;
        const float beta_c = c == 0 ? beta : 1.0f;
        const float *a_arg = kc > 0 ? a_c : nullptr, *b_arg = kc > 0 ? b_c : nullptr;
        if (c + 1 < nk) {
            st = gemm_impl(transA, transB, M, N, kc, alpha, a_arg, lda_c, b_arg, ldb_c, beta_c,
                           dC, N, s, SGEMM_PATH_AUTO, 0);
            if (st != SGEMM_OK) return st;
            continue;
        }
        // last chunk: row blocks, each sent home as soon as it is final
        const int nb = (int)std::max<int64_t>(1, std::min<int64_t>(kLastBlocks, M / 512));
        const int64_t per = ((M + nb - 1) / nb + 127) / 128 * 128;
        for (int b = 0; b < nb; ++b) {
            const int64_t r0 = (int64_t)b * per;
            if (r0 >= M) break;
            const int64_t rows = std::min<int64_t>(per, M - r0);
            const float *a_blk = a_arg ? (a_n ? a_arg + r0 * lda_c : a_arg + r0) : nullptr;
            st = gemm_impl(transA, transB, rows, N, kc, alpha, a_blk, a_n ? lda_c : M, b_arg,
                           ldb_c, beta_c, dC + r0 * N, N, s, SGEMM_PATH_AUTO, 0);
            if (st != SGEMM_OK) return st;
            if ((st = copy_status(cudaEventRecord(h->computed[b], s))) != SGEMM_OK) return st;
            if ((st = copy_status(cudaStreamWaitEvent(h->down, h->computed[b], 0))) != SGEMM_OK)
                return st;
            st = copy_status(cudaMemcpy2DAsync(C + r0 * ldc, ldc * 4, dC + r0 * N, N * 4, N * 4,
                                               rows, cudaMemcpyDeviceToHost, h->down));
            if (st != SGEMM_OK) return st;
        }
    }
    if ((st = copy_status(cudaEventRecord(h->done, h->down))) != SGEMM_OK) return st;
    return copy_status(cudaStreamWaitEvent(s, h->done, 0));
}
