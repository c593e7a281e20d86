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
