// The fused epilogue shared by every path:
//   D(i,j) = act(alpha * s_i * acc + beta * C(i,j) + bias_j)
// evaluated in fp32 in one fixed order: a_i = alpha * s_i (alpha when there
// is no row scale), t = a_i * acc (beta == 0) or fma(a_i, acc, beta * c),
// then t + bias_j, then the activation.  With no row scale, bias or
// activation the result is bit for bit the plain alpha/beta epilogue
// ("CuTe-ly writing an SM86 SGEMM", section "epilogue").
#pragma once
#include <cuda_runtime.h>

#include "../../include/sgemm_gb300.h"

namespace sgemm_gb300 {

struct Epilogue {
    const float *row_scale = nullptr;   // M values or null (all ones)
    const float *bias = nullptr;        // N values or null (zero)
    int act = SGEMM_ACT_NONE;
    bool plain() const { return !row_scale && !bias && act == SGEMM_ACT_NONE; }
};

__device__ __forceinline__ float epi_alpha(float alpha, const float *row_scale, int row) {
    return row_scale ? __fmul_rn(alpha, __ldg(row_scale + row)) : alpha;
}

// t + bias_col, then the activation (ReLU: x < 0 -> 0, NaN passes through)
__device__ __forceinline__ float epi_tail(float t, const float *bias, int col, int act) {
    if (bias) t = __fadd_rn(t, __ldg(bias + col));
    if (act == SGEMM_ACT_RELU && t < 0.0f) t = 0.0f;
    return t;
}

}  // namespace sgemm_gb300
