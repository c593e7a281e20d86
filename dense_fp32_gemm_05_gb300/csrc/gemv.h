// Thin GEMMs (min(M, N) <= kGemvMaxSmall) on the CUDA cores: the large
// operand is streamed once.  Defined in gemv.cu.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

#include "epilogue.cuh"

namespace sgemm_gb300 {

constexpr int64_t kGemvMaxSmall = 16;
// ... and up to kThinTcMaxS on the tensor cores (tc_thin_kernel)
constexpr int64_t kThinTcMaxS = 128;

// CTAs of the main GEMV launch for this problem (what run_gemv launches).
int gemv_ctas(char ta, char tb, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
              bool a_al, bool b_al, int sms);

// Whether the thin problem runs on the tensor cores (tc_thin_kernel): S =
// min(M, N) >= 12 and the large operand's rows along the long dimension,
// 16-byte aligned with a leading dimension that is a multiple of 4.
bool thin_on_tensor_cores(char ta, char tb, int64_t M, int64_t N, int64_t lda, int64_t ldb,
                          bool a_al, bool b_al);

// The tensor-core form's K split and grid for P columns of the large operand.
struct ThinTc {
    int kchunk, ksplit, ctas;
};
ThinTc thin_tc_geometry(int64_t P, int64_t K, int sms);

// Bounded-wait limit of the staged kernel (ns; 0 = the default 2 s).
void gemv_set_wait_limit(uint64_t ns);

// Reads and clears the current device's sticky error word of this path.
int gemv_take_device_error();

// Arguments already validated (check_args), M, N, K > 0, alpha != 0.
int run_gemv(char ta, char tb, int64_t M, int64_t N, int64_t K, float alpha, const float *A,
             int64_t lda, const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
             cudaStream_t s, int sms, const Epilogue &epi = Epilogue{});

}  // namespace sgemm_gb300
