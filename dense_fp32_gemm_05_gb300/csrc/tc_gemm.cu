// Tensor-core path (placeholder until the tcgen05 kernel lands).
#include "tc_gemm.h"

namespace sgemm_gb300 {

int run_tc(const Plan &, char, char, int64_t, int64_t, int64_t, float, const float *, int64_t,
           const float *, int64_t, float, float *, int64_t, cudaStream_t, int) {
    return SGEMM_ERR_UNSUPPORTED;
}

int tc_take_device_error() { return SGEMM_OK; }

void tc_set_wait_limit(uint64_t) {}

}  // namespace sgemm_gb300
