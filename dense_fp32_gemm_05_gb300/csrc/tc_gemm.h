// Tensor-core (tcgen05 kind::tf32) path: 3xTF32 and single-pass TF32.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "epilogue.cuh"
#include "plan.h"

namespace sgemm_gb300 {

// Runs the tensor-core path chosen in `pl` (SGEMM_PATH_3XTF32 or _TF32).
int run_tc(const Plan &pl, char ta, char tb, int64_t M, int64_t N, int64_t K, float alpha,
           const float *A, int64_t lda, const float *B, int64_t ldb, float beta, float *C,
           int64_t ldc, cudaStream_t s, int sms, const Epilogue &epi = Epilogue{});

// A thin problem on the tensor cores (3xTF32): out(s, p) = sum_k Small(s, k)
// Big(p, k) for S <= 128, Big stored with its rows along P (Big(p, k) =
// big[k * big_ld + p], 16-byte aligned, big_ld % 4 == 0), Small(s, k) =
// small[s * small_ss + k * small_sk] with small_sk == 1 or small_ss == 1.
// K is cut into ksplit ranges of kchunk (a multiple of 32); with ksplit > 1
// the raw sums go to partial[y][s][p] for the thin path's sum kernel,
// otherwise C(s, p) = C[s * c_s + p * c_p] gets the epilogue (rows_thin: s
// is C's row).  Launches the split of Small and the kernel (a programmatic
// dependent); returns SGEMM_ERR_UNSUPPORTED, launching nothing, when the
// operands do not qualify.
struct ThinCall {
    int S, P, K;
    int kchunk, ksplit;
    const float *big;
    int64_t big_ld;
    const float *small;
    int64_t small_ss, small_sk;
    float *C;
    int64_t c_s, c_p;
    int rows_thin;
    float alpha, beta;
    const float *row_scale, *bias;
    int act;
    float *partial;
};
int run_tc_thin(const ThinCall &c, cudaStream_t s);

// Measures the tensor pipe's kind::tf32 MMA rate on the current device
// (MAC per clock per SM, median over the SMs); synchronises the device.
int tc_probe_tf32_rate(int reps, double *mac_per_clock);

// Reads and clears the current device's sticky device error word.
int tc_take_device_error();

// Sets the bounded-wait limit (ns; 0 = default).
void tc_set_wait_limit(uint64_t ns);

// Measurement hook: records an event before (begin = true) or after the main
// kernel launch on `s` when timing is enabled (no-op otherwise).
void timing_mark(cudaStream_t s, bool begin);

// Library-owned per-(device, stream, slot) workspace, grown on demand.
int workspace(cudaStream_t stream, size_t bytes, void **out, int which = 0);

// The whole device-pointer GEMM call (checks, quick returns, selector, launch).
int gemm_impl(char ta, char tb, int64_t M, int64_t N, int64_t K, float alpha, const float *A,
              int64_t lda, const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
              cudaStream_t s, int path, int split, const Epilogue &epi = Epilogue{});

}  // namespace sgemm_gb300
