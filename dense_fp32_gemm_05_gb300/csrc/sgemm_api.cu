// C-ABI entry points of the single-precision GEMM library: argument checks,
// the per-shape selector, workspace handling and kernel launches.
// The interface is declared and documented in include/sgemm_gb300.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/sgemm_gb300.h"
#include "ffma_kernel.cuh"
#include "ffma_small.cuh"
#include "plan.h"
#include "gemv.h"
#include "tc_gemm.h"

namespace sgemm_gb300 {

// ------------------------------------------------------------ device state
struct DeviceState {
    bool ready = false;
    int sms = 0;
    int cc_major = 0, cc_minor = 0;
};

static std::mutex g_mu;
static std::map<int, DeviceState> g_dev;
// per (device, stream, slot) workspace so that concurrent streams never share
// one; slot 0 is the kernels' scratch, slot 1 the staging buffers of sgemm_host
struct WsKey {
    int dev;
    cudaStream_t stream;
    int slot;
    bool operator<(const WsKey &o) const {
        if (dev != o.dev) return dev < o.dev;
        if (stream != o.stream) return stream < o.stream;
        return slot < o.slot;
    }
};
static std::map<WsKey, std::pair<void *, size_t>> g_ws;

static int device_state(DeviceState **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return SGEMM_ERR_CUDA;
        d.ready = true;
    }
    *out = &d;
    return SGEMM_OK;
}

// Returns a workspace of at least `bytes` private to (device, stream, slot).
// It is allocated and, when it must grow, freed in stream order on `stream`.
int workspace(cudaStream_t stream, size_t bytes, void **out, int which) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    auto &slot = g_ws[WsKey{dev, stream, which}];
    if (slot.second < bytes) {
        if (slot.first) cudaFreeAsync(slot.first, stream);
        slot = {nullptr, 0};
        size_t want = std::max<size_t>(bytes, size_t(1) << 20);
        void *p = nullptr;
        if (cudaMallocAsync(&p, want, stream) != cudaSuccess) {
            cudaGetLastError();
            return SGEMM_ERR_NOMEM;
        }
        slot = {p, want};
    }
    *out = slot.first;
    return SGEMM_OK;
}

// ------------------------------------------------------------ timing hook
// A ring of event pairs recorded around main-kernel launches (see
// sgemm_timing_enable in the header).  Guarded by g_mu.
struct TimingRing {
    int dev = -1;
    std::vector<cudaEvent_t> ev;   // 2 per slot
    int slots = 0, next = 0, count = 0;
    bool open = false;             // a begin without its end yet
};
static TimingRing g_timing;

// Kernel launches made by the library in this process (every path).
static std::atomic<long long> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

void timing_mark(cudaStream_t s, bool begin) {
    std::lock_guard<std::mutex> lk(g_mu);
    TimingRing &t = g_timing;
    if (t.slots == 0) return;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != t.dev) return;
    if (begin) {
        cudaEventRecord(t.ev[2 * t.next], s);
        t.open = true;
    } else if (t.open) {
        cudaEventRecord(t.ev[2 * t.next + 1], s);
        t.open = false;
        t.next = (t.next + 1) % t.slots;
        t.count = std::min(t.count + 1, t.slots);
    }
}

static int launch_status() {
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) return SGEMM_OK;
    if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
        return SGEMM_ERR_UNSUPPORTED;
    return SGEMM_ERR_CUDA;
}

static int grid_for(int64_t total, int sms) {
    int64_t blocks = (total + 255) / 256;
    return (int)std::max<int64_t>(1, std::min<int64_t>(blocks, (int64_t)sms * 8));
}

// ------------------------------------------------------------ FFMA launch
// dep: launched as the programmatic dependent of the transpose pre-pass
template <bool AK, bool BK_, bool V>
static void launch_ffma_t(const ffma::Params &p, int grid, cudaStream_t s, bool dep) {
    auto kern = ffma::ffma_gemm_kernel<AK, BK_, V>;
    if (dep) {
        launch_dependent(kern, dim3(grid), dim3(ffma::THREADS), 0, s, p);
        return;
    }
    count_launch();
    kern<<<grid, ffma::THREADS, 0, s>>>(p);
}

// Fills the FFMA kernel parameters of a plan (shared by sgemm_ex and the
// static-scratch entry point).
static ffma::Params ffma_params(const Plan &pl, int64_t M, int64_t N, int64_t K, float alpha,
                                const float *A, int64_t lda, const float *B, int64_t ldb,
                                float beta, float *C, int64_t ldc,
                                const Epilogue &epi = Epilogue{}) {
    ffma::Params p{};
    p.A = A; p.B = B; p.C = C; p.partial = nullptr;
    p.lda = lda; p.ldb = ldb; p.ldc = ldc;
    p.M = (int)M; p.N = (int)N; p.K = (int)K;
    p.alpha = alpha; p.beta = beta;
    p.tiles_m = (int)((M + ffma::BM - 1) / ffma::BM);
    p.tiles_n = (int)((N + ffma::BN - 1) / ffma::BN);
    p.group_m = pl.group_m;
    p.kt = (int)((K + ffma::BK - 1) / ffma::BK);
    const int64_t tiles = (int64_t)p.tiles_m * p.tiles_n;
    p.dp_tiles = (int)std::min<int64_t>(pl.dp_tiles, tiles);
    p.sk_iters = (tiles - p.dp_tiles) * p.kt;
    p.sk_ctas = p.sk_iters == 0 ? 0 : (int)std::max<int64_t>(1, std::min<int64_t>(pl.ctas, p.sk_iters));
    p.c_vec = pl.c_vector;
    p.row_scale = epi.row_scale;
    p.bias = epi.bias;
    p.act = epi.act;
    return p;
}

// True when some share starts or ends inside a tile (partials + fixup needed).
static bool ffma_has_partials(const ffma::Params &p) {
    if (p.sk_ctas == 0) return false;
    return !(p.sk_iters % p.sk_ctas == 0 && (p.sk_iters / p.sk_ctas) % p.kt == 0);
}

static int ffma_grid(const ffma::Params &p) { return p.dp_tiles + p.sk_ctas; }
static int ffma_fix_tiles(const ffma::Params &p) {
    return p.tiles_m * p.tiles_n - p.dp_tiles;
}

static int launch_ffma(const ffma::Params &p, char ta, char tb, bool vec, cudaStream_t s,
                       bool dep = false) {
    const bool ak = is_notrans(ta), bk = !is_notrans(tb);
    const int grid = ffma_grid(p);
    if (ak && !bk && vec) launch_ffma_t<true, false, true>(p, grid, s, dep);
    else if (ak && !bk && !vec) launch_ffma_t<true, false, false>(p, grid, s, dep);
    else if (ak && bk && vec) launch_ffma_t<true, true, true>(p, grid, s, dep);
    else if (ak && bk && !vec) launch_ffma_t<true, true, false>(p, grid, s, dep);
    else if (!ak && !bk && vec) launch_ffma_t<false, false, true>(p, grid, s, dep);
    else if (!ak && !bk && !vec) launch_ffma_t<false, false, false>(p, grid, s, dep);
    else if (!ak && bk && vec) launch_ffma_t<false, true, true>(p, grid, s, dep);
    else launch_ffma_t<false, true, false>(p, grid, s, dep);
    return launch_status();
}

template <bool AK, bool BK_>
static void launch_ffma_small_t(const ffma_small::Params &p, unsigned tiles, cudaStream_t s) {
    count_launch();
    ffma_small::ffma_small_kernel<AK, BK_><<<tiles, ffma_small::THREADS, 0, s>>>(p);
}

// The small-problem kernel: one launch, one CTA per 16 x 16 tile.
static int run_ffma_small(char ta, char tb, int64_t M, int64_t N, int64_t K, float alpha,
                          const float *A, int64_t lda, const float *B, int64_t ldb, float beta,
                          float *C, int64_t ldc, cudaStream_t s, const Epilogue &epi) {
    ffma_small::Params p{};
    p.A = A; p.B = B; p.C = C;
    p.lda = lda; p.ldb = ldb; p.ldc = ldc;
    p.M = (int)M; p.N = (int)N; p.K = (int)K;
    p.alpha = alpha; p.beta = beta;
    p.tiles_n = (int)((N + ffma_small::TN - 1) / ffma_small::TN);
    p.row_scale = epi.row_scale;
    p.bias = epi.bias;
    p.act = epi.act;
    const int64_t tiles = ((M + ffma_small::TM - 1) / ffma_small::TM) * p.tiles_n;
    if (tiles > INT32_MAX) return SGEMM_ERR_UNSUPPORTED;
    const bool ak = is_notrans(ta), bk = !is_notrans(tb);
    timing_mark(s, true);
    if (ak && bk) launch_ffma_small_t<true, true>(p, (unsigned)tiles, s);
    else if (ak) launch_ffma_small_t<true, false>(p, (unsigned)tiles, s);
    else if (bk) launch_ffma_small_t<false, true>(p, (unsigned)tiles, s);
    else launch_ffma_small_t<false, false>(p, (unsigned)tiles, s);
    timing_mark(s, false);
    return launch_status();
}

static int run_ffma(const Plan &pl, char ta, char tb, int64_t M, int64_t N, int64_t K,
                    float alpha, const float *A, int64_t lda, const float *B, int64_t ldb,
                    float beta, float *C, int64_t ldc, cudaStream_t s, const Epilogue &epi) {
    if (pl.small)
        return run_ffma_small(ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, s, epi);
    // a K-contiguous operand copied transposed first (pl.t_a, pl.t_b): the
    // kernel then reads it as op(A) 'T' ([K][Mp]) or op(B) 'N' ([K][Np]),
    // rows padded to 16 bytes
    auto up = [](size_t bytes) { return (bytes + 255) & ~size_t(255); };
    const int64_t mp = (M + 3) / 4 * 4, np = (N + 3) / 4 * 4;
    const size_t a_t = pl.t_a ? up((size_t)K * mp * 4) : 0, b_t = pl.t_b ? up((size_t)K * np * 4) : 0;
    const char ta_k = pl.t_a ? 'T' : ta, tb_k = pl.t_b ? 'N' : tb;
    const float *a_k = A, *b_k = B;
    int64_t lda_k = lda, ldb_k = ldb;
    ffma::Params p = ffma_params(pl, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, epi);
    const bool partials = ffma_has_partials(p);
    const size_t part_bytes = partials ? (size_t)2 * p.sk_ctas * ffma::BM * ffma::BN * sizeof(float) : 0;
    if (a_t + b_t + part_bytes > 0) {
        void *ws = nullptr;
        int st = workspace(s, a_t + b_t + part_bytes, &ws);
        if (st != SGEMM_OK) return st;
        char *w = static_cast<char *>(ws);
        if (pl.t_a) { a_k = reinterpret_cast<float *>(w); lda_k = mp; }
        if (pl.t_b) { b_k = reinterpret_cast<float *>(w + a_t); ldb_k = np; }
        if (partials) p.partial = reinterpret_cast<float *>(w + a_t + b_t);
    }
    const bool pre = pl.t_a || pl.t_b;
    if (pre) {
        ffma::TransposeJob ja{}, jb{};
        if (pl.t_a) {   // A stored M x K -> [K][mp]
            ja = ffma::TransposeJob{A, lda, const_cast<float *>(a_k), mp, (int)M, (int)K,
                                    (int)((K + 31) / 32), 0};
            ja.tiles = (int)(((M + 31) / 32) * ja.tiles_c);
        }
        if (pl.t_b) {   // B stored N x K -> [K][np]
            jb = ffma::TransposeJob{B, ldb, const_cast<float *>(b_k), np, (int)N, (int)K,
                                    (int)((K + 31) / 32), 0};
            jb.tiles = (int)(((N + 31) / 32) * jb.tiles_c);
        }
        count_launch();
        ffma::transpose_pair_kernel<<<ja.tiles + jb.tiles, 256, 0, s>>>(ja, jb);
        int st = launch_status();
        if (st != SGEMM_OK) return st;
        p.A = a_k;
        p.B = b_k;
        p.lda = lda_k;
        p.ldb = ldb_k;
    }
    const bool vec = (pl.t_a || (aligned16(A) && lda % 4 == 0)) && (pl.t_b || (aligned16(B) && ldb % 4 == 0));
    timing_mark(s, true);
    int st = pre ? launch_ffma(p, ta_k, tb_k, vec, s, true) : launch_ffma(p, ta, tb, pl.vector != 0, s);
    timing_mark(s, false);
    if (st != SGEMM_OK) return st;
    if (partials) {
        launch_dependent(ffma::sk_fixup_kernel, dim3(ffma_fix_tiles(p), ffma::FIX_PARTS), dim3(256), 0,
                         s, p);
        st = launch_status();
    }
    return st;
}

int gemm_impl(char ta, char tb, int64_t M, int64_t N, int64_t K, float alpha,
                     const float *A, int64_t lda, const float *B, int64_t ldb, float beta,
                     float *C, int64_t ldc, cudaStream_t s, int path, int split,
                     const Epilogue &epi) {
    int st = check_args(ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc);
    if (st != SGEMM_OK) return st;
    if (path < SGEMM_PATH_AUTO || path > SGEMM_PATH_GEMV) return SGEMM_ERR_ARG;
    if (split < 0) return SGEMM_ERR_ARG;
    if (M == 0 || N == 0) return SGEMM_OK;

    DeviceState *d = nullptr;
    st = device_state(&d);
    if (st != SGEMM_OK) return st;
    if (!(d->cc_major == 10 && d->cc_minor == 3)) return SGEMM_ERR_UNSUPPORTED;

    if (K == 0 || alpha == 0.0f) {
        if (beta == 1.0f && !epi.bias && epi.act == SGEMM_ACT_NONE) return SGEMM_OK;
        count_launch();
        ffma::scale_c_kernel<<<grid_for(M * N, d->sms), 256, 0, s>>>((int)M, (int)N, beta, C, ldc,
                                                                     epi.bias, epi.act);
        return launch_status();
    }
    Plan pl;
    st = make_plan(ta, tb, M, N, K, lda, ldb, ldc, aligned16(A), aligned16(B), aligned16(C),
                   path, split, d->sms, &pl);
    if (st != SGEMM_OK) return st;
    if (pl.path == SGEMM_PATH_GEMV)
        return run_gemv(ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, s, d->sms, epi);
    if (pl.path == SGEMM_PATH_FFMA)
        return run_ffma(pl, ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, s, epi);
    return run_tc(pl, ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, s, d->sms, epi);
}

}  // namespace sgemm_gb300

using namespace sgemm_gb300;

extern "C" int sgemm(char transA, char transB, int64_t M, int64_t N, int64_t K, float alpha,
                     const float *A, int64_t lda, const float *B, int64_t ldb, float beta,
                     float *C, int64_t ldc, sgemm_stream_t stream) {
    return gemm_impl(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                     reinterpret_cast<cudaStream_t>(stream), SGEMM_PATH_AUTO, 0);
}

extern "C" int sgemm_ex(char transA, char transB, int64_t M, int64_t N, int64_t K, float alpha,
                        const float *A, int64_t lda, const float *B, int64_t ldb, float beta,
                        float *C, int64_t ldc, sgemm_stream_t stream, int path, int split) {
    return gemm_impl(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                     reinterpret_cast<cudaStream_t>(stream), path, split);
}

extern "C" int sgemm_epilogue(char transA, char transB, int64_t M, int64_t N, int64_t K,
                              float alpha, const float *A, int64_t lda, const float *B,
                              int64_t ldb, float beta, float *C, int64_t ldc,
                              const float *row_scale, const float *bias, int activation,
                              sgemm_stream_t stream, int path, int split) {
    if (activation != SGEMM_ACT_NONE && activation != SGEMM_ACT_RELU) return -16;
    Epilogue epi;
    epi.row_scale = row_scale;
    epi.bias = bias;
    epi.act = activation;
    return gemm_impl(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                     reinterpret_cast<cudaStream_t>(stream), path, split, epi);
}

extern "C" int sgemm_plan(char transA, char transB, int64_t M, int64_t N, int64_t K,
                          int64_t lda, int64_t ldb, int64_t ldc, int a_aligned, int b_aligned,
                          int c_aligned, int path, int split, int num_sms, int *out_path,
                          int *out_split, int *out_tile_m, int *out_tile_n, int *out_vector,
                          int *out_ctas) {
    int st = check_args(transA, transB, M, N, K, 1.0f, nullptr, lda, nullptr, ldb, 0.0f,
                        nullptr, ldc, /*pointers_checked=*/false);
    if (st != SGEMM_OK) return st;
    if (path < SGEMM_PATH_AUTO || path > SGEMM_PATH_GEMV || split < 0 || num_sms <= 0)
        return SGEMM_ERR_ARG;
    Plan pl;
    st = make_plan(transA, transB, M, N, K, lda, ldb, ldc, a_aligned != 0, b_aligned != 0,
                   c_aligned != 0, path, split, num_sms, &pl);
    if (st != SGEMM_OK) return st;
    if (out_path) *out_path = pl.path;
    // tensor cores: the CTAs (pairs) sharing one tile -- stream-K's split, or
    // the column slices of the last-wave tiles
    if (out_split) *out_split = (pl.path == SGEMM_PATH_3XTF32 || pl.path == SGEMM_PATH_TF32) &&
                                        pl.tc_sk == 0 && pl.tc_sk_tail == 0
                                    ? pl.tail_nsplit : pl.split;
    if (out_tile_m) *out_tile_m = pl.tile_m;
    if (out_tile_n) *out_tile_n = pl.tile_n;
    if (out_vector) *out_vector = pl.vector;
    if (pl.path == SGEMM_PATH_GEMV &&
        thin_on_tensor_cores(transA, transB, M, N, lda, ldb, a_aligned != 0, b_aligned != 0)) {
        // the thin path's tensor-core form: 128 columns of the large operand
        // per CTA, and split = the CTAs along K
        if (out_tile_n) *out_tile_n = 128;
        if (out_split)
            *out_split = thin_tc_geometry(std::max(M, N), std::max<int64_t>(K, 1), num_sms).ksplit;
    }
    if (out_ctas) {
        if (pl.path == SGEMM_PATH_FFMA) {
            *out_ctas = pl.dp_tiles + pl.ctas;
        } else if (pl.path == SGEMM_PATH_GEMV) {
            *out_ctas = gemv_ctas(transA, transB, M, N, K, lda, ldb, a_aligned != 0,
                                  b_aligned != 0, num_sms);
        } else if (pl.tc_sk > 0) {
            *out_ctas = pl.tc_sk;   // stream-K: one CTA per share of the iterations
        } else {
            // units of work; one CTA each (two for SM pairs), or one CTA (pair)
            // per SM (pair) walking them when no operand is split in the kernel
            const int64_t tiles = ((M + pl.tile_m - 1) / pl.tile_m) * ((N + pl.tile_n - 1) / pl.tile_n);
            const int64_t units = pl.dp_tiles + (tiles - pl.dp_tiles) * pl.tail_nsplit;
            const bool fa = pl.fuse_a && is_notrans(transA) && a_aligned && lda % 4 == 0;
            const bool fb = pl.fuse_b && !is_notrans(transB) && b_aligned && ldb % 4 == 0;
            const int64_t slots = pl.pair ? std::max(num_sms / 2, 1) : num_sms;
            const int64_t groups = pl.tc_sk_tail ? slots : (fa || fb) ? units : std::min<int64_t>(units, slots);
            *out_ctas = (int)(groups * (pl.pair ? 2 : 1));
        }
    }
    return SGEMM_OK;
}

extern "C" int sgemm_plan_detail(char transA, char transB, int64_t M, int64_t N, int64_t K,
                                 int64_t lda, int64_t ldb, int64_t ldc, int a_aligned,
                                 int b_aligned, int c_aligned, int path, int split, int num_sms,
                                 sgemm_plan_info *out) {
    if (out == nullptr) return -15;
    sgemm_plan_info info{};
    int st = sgemm_plan(transA, transB, M, N, K, lda, ldb, ldc, a_aligned, b_aligned, c_aligned,
                        path, split, num_sms, &info.path, &info.split, &info.tile_m,
                        &info.tile_n, &info.vector, &info.ctas);
    if (st != SGEMM_OK) return st;
    Plan pl;
    make_plan(transA, transB, M, N, K, lda, ldb, ldc, a_aligned != 0, b_aligned != 0,
              c_aligned != 0, path, split, num_sms, &pl);
    info.dp_tiles = pl.path == SGEMM_PATH_GEMV ? 0 : pl.dp_tiles;
    if (pl.path == SGEMM_PATH_GEMV &&
        thin_on_tensor_cores(transA, transB, M, N, lda, ldb, a_aligned != 0, b_aligned != 0)) {
        // the tensor-core form (tile_n and split from sgemm_plan above):
        // 32-wide k-blocks, 8 accumulators
        info.k_block = 32;
        info.accumulators = 8;
    }
    if (pl.path == SGEMM_PATH_3XTF32 || pl.path == SGEMM_PATH_TF32) {
        const TcVariant v = tc_variant(pl);
        info.pair = v.pair;
        info.fuse_a = v.fuse_a;
        info.fuse_b = v.fuse_b;
        info.wide = v.wide;
        info.accumulators = v.nacc;
        info.k_block = v.bk;
        info.tail_nsplit = (v.sk || v.sk_tail) ? 1 : pl.tail_nsplit;
        info.sk_ctas = v.sk ? pl.tc_sk : 0;
        info.sk_tail = v.sk_tail;
    } else if (pl.path == SGEMM_PATH_FFMA) {
        info.k_block = pl.small ? ffma_small::KC : ffma::BK;
        info.pre_transpose = pl.t_a | (pl.t_b << 1);
    }
    *out = info;
    return SGEMM_OK;
}

extern "C" const char *sgemm_status_string(int status) {
    if (status < 0) return "invalid argument (the negated value is its 1-based position)";
    switch (status) {
    case SGEMM_OK: return "success";
    case SGEMM_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case SGEMM_ERR_TIMEOUT: return "a bounded device-side wait timed out";
    case SGEMM_ERR_NOMEM: return "workspace allocation failed";
    case SGEMM_ERR_UNSUPPORTED: return "path or device not supported for this problem";
    case SGEMM_ERR_ARG: return "invalid argument to an auxiliary entry point";
    case SGEMM_ERR_SCRATCH: return "problem needs more than the static scratch array holds";
    default: return "unknown status";
    }
}

extern "C" int sgemm_device_error(sgemm_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SGEMM_ERR_CUDA;
    // both words are read (and cleared); the tensor cores' is reported first
    const int t = tc_take_device_error();
    const int g = gemv_take_device_error();
    return t != SGEMM_OK ? t : g;
}

extern "C" int sgemm_set_wait_limit(uint64_t nanoseconds) {
    tc_set_wait_limit(nanoseconds);
    gemv_set_wait_limit(nanoseconds);
    return SGEMM_OK;
}

extern "C" int64_t sgemm_launch_count(void) {
    return g_launches.load(std::memory_order_relaxed);
}

extern "C" int sgemm_probe_tf32_rate(int reps, double *mac_per_clock) {
    if (reps < 64 || reps > (1 << 20)) return -1;
    if (mac_per_clock == nullptr) return -2;
    DeviceState *d = nullptr;
    int st = device_state(&d);
    if (st != SGEMM_OK) return st;
    if (!(d->cc_major == 10 && d->cc_minor == 3)) return SGEMM_ERR_UNSUPPORTED;
    return tc_probe_tf32_rate(reps, mac_per_clock);
}

extern "C" int sgemm_timing_enable(int n) {
    if (n < 0 || n > 100000) return -1;
    int dev = 0;
    if (n > 0 && cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    TimingRing &t = g_timing;
    for (cudaEvent_t e : t.ev) cudaEventDestroy(e);
    t = TimingRing{};
    if (n == 0) return SGEMM_OK;
    t.ev.resize(2 * (size_t)n, nullptr);
    for (auto &e : t.ev) {
        if (cudaEventCreate(&e) != cudaSuccess) {
            for (cudaEvent_t x : t.ev) if (x) cudaEventDestroy(x);
            t = TimingRing{};
            return SGEMM_ERR_CUDA;
        }
    }
    t.dev = dev;
    t.slots = n;
    return SGEMM_OK;
}

extern "C" int sgemm_timing_read(float *ms, int capacity) {
    if (ms == nullptr && capacity > 0) return -1;
    if (capacity < 0) return -2;
    std::lock_guard<std::mutex> lk(g_mu);
    TimingRing &t = g_timing;
    const int n = std::min(t.count, capacity);
    const int first = (t.next - t.count + t.slots) % std::max(t.slots, 1);
    for (int i = 0; i < n; ++i) {
        const int slot = (first + i) % t.slots;
        if (cudaEventSynchronize(t.ev[2 * slot + 1]) != cudaSuccess ||
            cudaEventElapsedTime(&ms[i], t.ev[2 * slot], t.ev[2 * slot + 1]) != cudaSuccess)
            return -SGEMM_ERR_CUDA;
    }
    t.count = 0;
    return n;
}

extern "C" int sgemm_release_workspace(void) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return SGEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto it = g_ws.begin(); it != g_ws.end();) {
        if (it->first.dev == dev) {
            if (it->second.first) cudaFree(it->second.first);
            it = g_ws.erase(it);
        } else {
            ++it;
        }
    }
    return SGEMM_OK;
}

extern "C" int sgemm_version(void) { return 100; }

// ------------------------------------------------------------------------
// sgemm_ffma_static_scratch: the FFMA split-K launch with its partial sums in
// a fixed-size static device array instead of the allocated workspace, for
// callers that cannot allocate device memory (see include/sgemm_gb300.h).
namespace sgemm_gb300 {

constexpr int kStaticPartialTiles = 256;                       // 16 MiB
constexpr size_t kStaticPartialFloats =
    (size_t)kStaticPartialTiles * ffma::BM * ffma::BN;

// Every GPU that loads the library holds this array until the process exits.
// It holds 2 slots per CTA of the stream-K decomposition (a CTA's first and
// last partial tile), so plans with up to 128 sharing CTAs fit.
static __device__ __align__(256) float g_static_partials[kStaticPartialFloats];

// Device address of g_static_partials per device, looked up once with that
// device current.  (In host code the symbol's name is only a host-side
// stand-in; passing it to a kernel would be wrong.)
static std::mutex g_static_mu;
static std::map<int, float *> g_static_addr;

static int static_partials(float **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_static_mu);
    auto it = g_static_addr.find(dev);
    if (it == g_static_addr.end()) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_partials) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return SGEMM_ERR_CUDA;
        }
        it = g_static_addr.emplace(dev, static_cast<float *>(p)).first;
    }
    *out = it->second;
    return SGEMM_OK;
}

}  // namespace sgemm_gb300

extern "C" int sgemm_ffma_static_scratch(char transA, char transB, int64_t M, int64_t N,
                                         int64_t K, float alpha, const float *A, int64_t lda,
                                         const float *B, int64_t ldb, float beta, float *C,
                                         int64_t ldc, sgemm_stream_t stream, int split) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int st = check_args(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc);
    if (st != SGEMM_OK) return st;
    if (split < 0) return SGEMM_ERR_ARG;
    if (M == 0 || N == 0) return SGEMM_OK;
    DeviceState *d = nullptr;
    st = device_state(&d);
    if (st != SGEMM_OK) return st;
    if (!(d->cc_major == 10 && d->cc_minor == 3)) return SGEMM_ERR_UNSUPPORTED;
    if (K == 0 || alpha == 0.0f) {
        if (beta == 1.0f) return SGEMM_OK;
        count_launch();
        ffma::scale_c_kernel<<<grid_for(M * N, d->sms), 256, 0, s>>>((int)M, (int)N, beta, C, ldc,
                                                                     nullptr, SGEMM_ACT_NONE);
        return launch_status();
    }
    Plan pl;
    st = make_plan(transA, transB, M, N, K, lda, ldb, ldc, aligned16(A), aligned16(B),
                   aligned16(C), SGEMM_PATH_FFMA, split, d->sms, &pl);
    if (st != SGEMM_OK) return st;
    if (pl.small)   // one launch, no partial sums
        return run_ffma_small(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, s,
                              Epilogue{});
    ffma::Params p = ffma_params(pl, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc);
    bool partials = ffma_has_partials(p);
    if (partials && 2LL * p.sk_ctas > kStaticPartialTiles) {
        if (split != 0) return SGEMM_ERR_SCRATCH;    // the caller's split does not fit
        // the selector's stream-K share does not fit: the same iterations
        // shared by as many CTAs as the array holds slots for
        p.sk_ctas = kStaticPartialTiles / 2;
        partials = ffma_has_partials(p);
    }
    if (partials) {
        st = static_partials(&p.partial);
        if (st != SGEMM_OK) return st;
    }
    st = launch_ffma(p, transA, transB, pl.vector != 0, s);
    if (st != SGEMM_OK) return st;
    if (partials) {
        launch_dependent(ffma::sk_fixup_kernel, dim3(ffma_fix_tiles(p), ffma::FIX_PARTS), dim3(256), 0,
                         s, p);
        st = launch_status();
    }
    return st;
}
