// kq_tc.cu -- tensor-core prefill GEMM (not yet enabled: every shape takes the exact MMQ kernel).
#include "kq_tc.cuh"

namespace kq {

bool tc_eligible(kq_dtype, int64_t, int64_t, int64_t) { return false; }
size_t tc_workspace_bytes(kq_dtype, int64_t, int64_t, int64_t) { return 0; }
kq_status tc_gemm(kq_dtype wt, const uint8_t *, const uint8_t *, int64_t, int64_t, int64_t, float *, int64_t, uint8_t *,
                  cudaStream_t) {
    return fail(KQ_ERR_UNSUPPORTED_DTYPE, "tc_gemm: dtype %s has no tensor-core path", dtype_name(wt));
}

}  // namespace kq
