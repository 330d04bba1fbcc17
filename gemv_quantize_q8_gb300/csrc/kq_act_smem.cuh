// kq_act_smem.cuh -- warp-level activation quantizers that write into shared memory.
//
// Same arithmetic as the standalone quantizers in kq_quant.cu, but the block lands in a
// shared-memory layout the matmul kernels read directly: q int8 [256 per block] (16-byte
// aligned), d f32, bsums int16 [16].  Used by the decode GEMV's fused-quant prologue, which
// quantizes the activation once per thread block instead of launching a separate kernel
// (strix-llama.cpp PR #18 "Optimize ROCM Prefill and Decode", fused-quant MMVQ commit).
#pragma once
#include "kq_q8k_block.cuh"

namespace kq {

// One warp quantizes 256 fp32 values at x (any 4-byte alignment) into Q8_K fields.
__device__ __forceinline__ void warp_quantize_q8k_smem(const float *__restrict__ x, int8_t *q, float *d,
                                                       int16_t *bs) {
    const int lane = threadIdx.x & 31;
    float v[8];
    if ((reinterpret_cast<uintptr_t>(x) & 15) == 0) {
        const float4 a = reinterpret_cast<const float4 *>(x)[2 * lane];
        const float4 b = reinterpret_cast<const float4 *>(x)[2 * lane + 1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = x[lane * 8 + i];
    }
    float amax = 0.0f, mx = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float ax = fabsf(v[i]);
        if (ax > amax) { amax = ax; mx = v[i]; }
    }
    // Block amax and the signed value of its first occurrence: amax is never negative or NaN, so its
    // bit pattern orders like its value; the lowest lane holding the maximum holds the first
    // occurrence (within a lane the strict > above keeps the first).  One max-reduction, one ballot
    // and one shuffle -- a short dependency chain on the decode call's critical path.
    const uint32_t key = __float_as_uint(amax);
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
    const int src = __ffs(__ballot_sync(0xffffffffu, key == kmax)) - 1;
    mx = __shfl_sync(0xffffffffu, mx, src);
    amax = __uint_as_float(kmax);
    int qv[8], sum = 0;
    float iscale = 0.0f;
    if (amax != 0.0f) iscale = __fdiv_rn(-127.0f, mx);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        qv[i] = amax == 0.0f ? 0 : q8k_code(__fmul_rn(iscale, v[i]));
        sum += qv[i];
    }
    uint32_t w0 = (qv[0] & 0xff) | ((qv[1] & 0xff) << 8) | ((qv[2] & 0xff) << 16) | ((uint32_t)(qv[3] & 0xff) << 24);
    uint32_t w1 = (qv[4] & 0xff) | ((qv[5] & 0xff) << 8) | ((qv[6] & 0xff) << 16) | ((uint32_t)(qv[7] & 0xff) << 24);
    *reinterpret_cast<uint2 *>(q + lane * 8) = make_uint2(w0, w1);
    int pair = sum + __shfl_xor_sync(0xffffffffu, sum, 1);
    if ((lane & 1) == 0) bs[lane >> 1] = (int16_t)pair;
    if (lane == 0) *d = amax == 0.0f ? 0.0f : __fdiv_rn(1.0f, iscale);
}

// One warp quantizes 128 fp32 values (four Q8_1 blocks) at x into q int8 [128] and d f32 [4]
// (d rounded through f16, which is what a stored Q8_1 block carries into the dot product).
__device__ __forceinline__ void warp_quantize_q8_1x4_smem(const float *__restrict__ x, int8_t *q, float *d) {
    const int lane = threadIdx.x & 31;
    const int t = lane & 7;
    float v[4];
    if ((reinterpret_cast<uintptr_t>(x) & 15) == 0) {
        const float4 a = reinterpret_cast<const float4 *>(x)[lane];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = x[lane * 4 + i];
    }
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int s = 4; s >= 1; s >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, s));
    const float dd = __fdiv_rn(amax, 127.0f);
    int qv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float r = amax == 0.0f ? 0.0f : roundf(__fdiv_rn(v[i], dd));
        if (!isfinite(r)) r = 0.0f;
        r = fminf(fmaxf(r, -127.0f), 127.0f);
        qv[i] = (int)r;
    }
    *reinterpret_cast<uint32_t *>(q + lane * 4) =
        (qv[0] & 0xff) | ((qv[1] & 0xff) << 8) | ((qv[2] & 0xff) << 16) | ((uint32_t)(qv[3] & 0xff) << 24);
    if (t == 0) d[lane >> 3] = __half2float(__float2half_rn(dd));
}

}  // namespace kq
