// kq_tc.cuh -- tensor-core (tcgen05) prefill GEMM interface (internal).
#pragma once
#include "kq_internal.cuh"

namespace kq {

// True when the tensor-core kernel handles this shape (large-M prefill of a supported dtype).
bool tc_eligible(kq_dtype wt, int64_t M, int64_t N, int64_t K);
// Workspace bytes the tensor-core path needs for this shape (0 when it is not eligible).
size_t tc_workspace_bytes(kq_dtype wt, int64_t M, int64_t N, int64_t K);
kq_status tc_gemm(kq_dtype wt, const uint8_t *w, const uint8_t *xq, int64_t M, int64_t N, int64_t K, float *y,
                  int64_t ldy, uint8_t *workspace, cudaStream_t st);

}  // namespace kq
