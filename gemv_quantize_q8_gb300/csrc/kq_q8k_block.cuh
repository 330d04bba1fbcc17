// kq_q8k_block.cuh -- the Q8_K block arithmetic shared by every kernel that writes Q8_K rows.
//
// silu_mul is the SwiGLU element h = silu(g)*u; q8k_block_codes quantizes one 256-element block
// held by a warp and q8k_block_store writes it as Q8_K bytes.  The standalone and SwiGLU quantizers,
// the RMSNorm producer, the routed gate/up GEMM's fused SwiGLU epilogue and the fp32-input GEMM's
// prologue (codes straight into the tensor-core panel) all call these, so their blocks are identical
// by construction.
#pragma once
#include "kq_internal.cuh"

namespace kq {

__device__ __forceinline__ float silu_mul(float g, float u) {
    float e = expf(-g);
    float den = __fadd_rn(1.0f, e);
    float s = __fdiv_rn(g, den);
    return __fmul_rn(s, u);
}

__device__ __forceinline__ int q8k_code(float p) {
    if (isnan(p)) return 0;
    if (p >= 127.0f) return 127;
    if (p <= -127.0f) return -127;
    return __float2int_rn(p);
}

// The Q8_K block arithmetic.  One warp, lane l holding elements 8l..8l+7 of the block: q receives
// lane l's eight codes, pair the sum of the codes of lanes l and l^1 (bsum l/2 of the block, valid
// on even lanes) and d the block scale.  An all-zero (or all-NaN) block gives q = 0, pair = 0, d = 0.
__device__ __forceinline__ void q8k_block_codes(const float (&v)[8], int (&q)[8], int &pair, float &d) {
    // lane-local ascending scan, first occurrence wins (strict >)
    float amax = 0.0f, mx = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float ax = fabsf(v[i]);
        if (ax > amax) { amax = ax; mx = v[i]; }
    }
    // block amax and its first occurrence: amax is never negative or NaN, so its bits order like its
    // value, and the lowest lane holding the maximum holds the first occurrence
    const uint32_t key = __float_as_uint(amax);
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
    const int src = __ffs(__ballot_sync(0xffffffffu, key == kmax)) - 1;
    mx = __shfl_sync(0xffffffffu, mx, src);
    if (kmax == 0u) {  // zero block
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = 0;
        pair = 0;
        d = 0.0f;
        return;
    }
    const float iscale = __fdiv_rn(-127.0f, mx);
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        q[i] = q8k_code(__fmul_rn(iscale, v[i]));
        sum += q[i];
    }
    pair = sum + __shfl_xor_sync(0xffffffffu, sum, 1);
    d = __fdiv_rn(1.0f, iscale);
}

// The 292-byte Q8_K block (f32 d, int8 q[256], int16 bsums[16]) of the warp's 256 values at o.
__device__ __forceinline__ void q8k_block_store(const float (&v)[8], uint8_t *__restrict__ o) {
    const int lane = threadIdx.x & 31;
    int q[8], pair;
    float d;
    q8k_block_codes(v, q, pair, d);
    uint32_t w0 = (q[0] & 0xff) | ((q[1] & 0xff) << 8) | ((q[2] & 0xff) << 16) | ((uint32_t)(q[3] & 0xff) << 24);
    uint32_t w1 = (q[4] & 0xff) | ((q[5] & 0xff) << 8) | ((q[6] & 0xff) << 16) | ((uint32_t)(q[7] & 0xff) << 24);
    uint32_t *qs = reinterpret_cast<uint32_t *>(o + 4 + lane * 8);
    qs[0] = w0;
    qs[1] = w1;
    if ((lane & 1) == 0) reinterpret_cast<int16_t *>(o + 260)[lane >> 1] = (int16_t)pair;
    if (lane == 0) *reinterpret_cast<float *>(o) = d;
}

}  // namespace kq
