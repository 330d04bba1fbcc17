// kq_quant.cu -- activation quantizers: Q8_K, Q8_1 and their fused SwiGLU variants.
//
// Q8_K follows the warp-cooperative quantizer of vllm.cpp PR #2890 ("fuse silu-mul with Q8_K quant
// epilogue"): each lane owns a contiguous chunk of the 256-element block, scans it in ascending
// order keeping the first maximum, and the lanes combine with an xor butterfly that prefers the
// lower chunk index on ties -- the same element a sequential scan would pick.  Here one 32-lane
// warp owns one block (8 elements per lane).  amax is seeded at 0 (the page's NaN fix), so NaN
// never wins and an all-zero block is the zero block.
//
// Q8_1 follows strix-llama.cpp PR #18 ("Optimize ROCM Prefill and Decode", fused-quant MMVQ
// commit): d = amax/127 with IEEE division, q = roundf(x/d), and the block sum taken in xor-butterfly
// order.  Eight lanes own one 32-element block (4 elements each); the butterfly strides 16, 8, 4
// cross lanes and strides 2, 1 stay inside a lane, which reproduces the 32-lane order exactly.
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

template <bool VEC>
__device__ __forceinline__ void load8(const float *p, float v[8]) {
    if (VEC) {
        float4 a = *reinterpret_cast<const float4 *>(p);
        float4 b = *reinterpret_cast<const float4 *>(p + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = p[i];
    }
}

// One warp quantizes one 256-element block; lane l holds elements 8l..8l+7.
// SWIGLU: the block's inputs are h = silu(g)*u computed here (optionally stored to h_out).
template <bool VEC, bool SWIGLU>
__global__ void quantize_q8k_kernel(const float *__restrict__ x, const float *__restrict__ u, int64_t M,
                                    int64_t nb, int64_t ld, uint8_t *__restrict__ out, float *__restrict__ h_out) {
    const int lane = threadIdx.x & 31;
    const int64_t blk = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (blk >= M * nb) return;
    const int64_t m = blk / nb, b = blk % nb;
    const int64_t off = m * ld + b * 256 + lane * 8;
    float v[8];
    load8<VEC>(x + off, v);
    if (SWIGLU) {
        float uv[8];
        load8<VEC>(u + off, uv);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = silu_mul(v[i], uv[i]);
        if (h_out) {
            float *hp = h_out + m * (nb * 256) + b * 256 + lane * 8;
#pragma unroll
            for (int i = 0; i < 8; ++i) hp[i] = v[i];
        }
    }
    // lane-local ascending scan, first occurrence wins (strict >)
    float amax = 0.0f, mx = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float ax = fabsf(v[i]);
        if (ax > amax) { amax = ax; mx = v[i]; }
    }
    int src = lane;  // chunk index holding the current maximum
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        float oa = __shfl_xor_sync(0xffffffffu, amax, s);
        float om = __shfl_xor_sync(0xffffffffu, mx, s);
        int os = __shfl_xor_sync(0xffffffffu, src, s);
        if (oa > amax || (oa == amax && os < src)) { amax = oa; mx = om; src = os; }
    }
    uint8_t *o = out + blk * kQ8KBytes;
    if (amax == 0.0f) {  // zero block
        uint32_t *o32 = reinterpret_cast<uint32_t *>(o);
        for (int i = lane; i < kQ8KBytes / 4; i += 32) o32[i] = 0u;
        return;
    }
    const float iscale = __fdiv_rn(-127.0f, mx);
    int q[8];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        q[i] = q8k_code(__fmul_rn(iscale, v[i]));
        sum += q[i];
    }
    uint32_t w0 = (q[0] & 0xff) | ((q[1] & 0xff) << 8) | ((q[2] & 0xff) << 16) | ((uint32_t)(q[3] & 0xff) << 24);
    uint32_t w1 = (q[4] & 0xff) | ((q[5] & 0xff) << 8) | ((q[6] & 0xff) << 16) | ((uint32_t)(q[7] & 0xff) << 24);
    uint32_t *qs = reinterpret_cast<uint32_t *>(o + 4 + lane * 8);
    qs[0] = w0;
    qs[1] = w1;
    int pair = sum + __shfl_xor_sync(0xffffffffu, sum, 1);
    if ((lane & 1) == 0) reinterpret_cast<int16_t *>(o + 260)[lane >> 1] = (int16_t)pair;
    if (lane == 0) *reinterpret_cast<float *>(o) = __fdiv_rn(1.0f, iscale);
}

__device__ __forceinline__ uint16_t f16_bits(float f) {
    if (isnan(f)) return 0x7e00u;  // one canonical NaN
    return __half_as_ushort(__float2half_rn(f));
}

// Eight lanes quantize one 32-element block; lane t (0..7 within its group) holds elements 4t..4t+3.
template <bool VEC, bool SWIGLU>
__global__ void quantize_q8_1_kernel(const float *__restrict__ x, const float *__restrict__ u, int64_t M,
                                     int64_t nb, int64_t ld, uint8_t *__restrict__ out, float *__restrict__ h_out) {
    const int lane = threadIdx.x & 31;
    const int t = lane & 7;
    const int64_t blk = ((int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32) * 4 + (lane >> 3);
    const bool active = blk < M * nb;
    const int64_t bb = active ? blk : 0;
    const int64_t m = bb / nb, b = bb % nb;
    const int64_t off = m * ld + b * 32 + t * 4;
    float v[4];
    if (active) {
        if (VEC) {
            float4 a = *reinterpret_cast<const float4 *>(x + off);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = x[off + i];
        }
        if (SWIGLU) {
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = silu_mul(v[i], u[off + i]);
            if (h_out) {
#pragma unroll
                for (int i = 0; i < 4; ++i) h_out[m * (nb * 32) + b * 32 + t * 4 + i] = v[i];
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = 0.0f;
    }
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int s = 4; s >= 1; s >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, s));
    const float d = __fdiv_rn(amax, 127.0f);
    int q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float r = amax == 0.0f ? 0.0f : roundf(__fdiv_rn(v[i], d));
        if (!isfinite(r)) r = 0.0f;
        r = fminf(fmaxf(r, -127.0f), 127.0f);
        q[i] = (int)r;
    }
    // xor butterfly over element index i = 4t + e: strides 16, 8, 4 pair lanes t^4, t^2, t^1;
    // strides 2, 1 pair e^2, e^1 inside the lane.
    float p[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
    for (int s = 4; s >= 1; s >>= 1) {
#pragma unroll
        for (int e = 0; e < 4; ++e) p[e] = __fadd_rn(p[e], __shfl_xor_sync(0xffffffffu, p[e], s));
    }
    float p2[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) p2[e] = __fadd_rn(p[e], p[e ^ 2]);
    const float sum = __fadd_rn(p2[0], p2[1]);
    if (!active) return;
    uint8_t *o = out + blk * kQ81Bytes;
    *reinterpret_cast<uint32_t *>(o + 4 + t * 4) =
        (q[0] & 0xff) | ((q[1] & 0xff) << 8) | ((q[2] & 0xff) << 16) | ((uint32_t)(q[3] & 0xff) << 24);
    if (t == 0) {
        *reinterpret_cast<uint32_t *>(o) = (uint32_t)f16_bits(d) | ((uint32_t)f16_bits(sum) << 16);
    }
}

static kq_status quant_common(const char *name, const float *x, const float *u, int64_t M, int64_t K, int64_t ld,
                              void *xq, float *h_out, int block, bool swiglu, cudaStream_t st) {
    if (!x || !xq || (swiglu && !u)) return fail(KQ_ERR_INVALID_ARG, "%s: null pointer", name);
    if (M <= 0 || K <= 0 || K % block)
        return fail(KQ_ERR_INVALID_ARG, "%s: need M > 0 and K a positive multiple of %d (M=%lld K=%lld)", name, block,
                    (long long)M, (long long)K);
    if (ld < K) return fail(KQ_ERR_INVALID_ARG, "%s: leading dimension %lld < K %lld", name, (long long)ld, (long long)K);
    if (!aligned(x, 4) || !aligned(xq, 4) || (u && !aligned(u, 4)) || (h_out && !aligned(h_out, 4)))
        return fail(KQ_ERR_ALIGNMENT, "%s: pointers must be 4-byte aligned", name);
    const bool vec = aligned(x, 16) && (!u || aligned(u, 16)) && ld % 4 == 0;
    const int64_t nb = K / block;
    const int threads = 256;
    uint8_t *o = static_cast<uint8_t *>(xq);
    if (block == 256) {
        int64_t warps = M * nb;
        int64_t grid = (warps + 7) / 8;
        if (swiglu) {
            if (vec) quantize_q8k_kernel<true, true><<<grid, threads, 0, st>>>(x, u, M, nb, ld, o, h_out);
            else quantize_q8k_kernel<false, true><<<grid, threads, 0, st>>>(x, u, M, nb, ld, o, h_out);
        } else {
            if (vec) quantize_q8k_kernel<true, false><<<grid, threads, 0, st>>>(x, nullptr, M, nb, ld, o, nullptr);
            else quantize_q8k_kernel<false, false><<<grid, threads, 0, st>>>(x, nullptr, M, nb, ld, o, nullptr);
        }
    } else {
        int64_t warps = (M * nb + 3) / 4;
        int64_t grid = (warps + 7) / 8;
        if (swiglu) {
            if (vec) quantize_q8_1_kernel<true, true><<<grid, threads, 0, st>>>(x, u, M, nb, ld, o, h_out);
            else quantize_q8_1_kernel<false, true><<<grid, threads, 0, st>>>(x, u, M, nb, ld, o, h_out);
        } else {
            if (vec) quantize_q8_1_kernel<true, false><<<grid, threads, 0, st>>>(x, nullptr, M, nb, ld, o, nullptr);
            else quantize_q8_1_kernel<false, false><<<grid, threads, 0, st>>>(x, nullptr, M, nb, ld, o, nullptr);
        }
    }
    kq_status s = check_launch(name);
    if (s == KQ_OK) count_launch(R_QUANT);
    return s;
}

}  // namespace kq

using namespace kq;

extern "C" {

kq_status kq_quantize_q8k(const float *x, int64_t M, int64_t K, int64_t ldx, void *xq, kq_stream_t stream) {
    return quant_common("kq_quantize_q8k", x, nullptr, M, K, ldx, xq, nullptr, 256, false, (cudaStream_t)stream);
}

kq_status kq_quantize_q8_1(const float *x, int64_t M, int64_t K, int64_t ldx, void *xq, kq_stream_t stream) {
    return quant_common("kq_quantize_q8_1", x, nullptr, M, K, ldx, xq, nullptr, 32, false, (cudaStream_t)stream);
}

kq_status kq_swiglu_quantize_q8_1(const float *g, const float *u, int64_t M, int64_t K, int64_t ld, void *xq,
                                  float *h_out, kq_stream_t stream) {
    return quant_common("kq_swiglu_quantize_q8_1", g, u, M, K, ld, xq, h_out, 32, true, (cudaStream_t)stream);
}

kq_status kq_swiglu_quantize_q8k(const float *g, const float *u, int64_t M, int64_t K, int64_t ld, void *xq,
                                 float *h_out, kq_stream_t stream) {
    return quant_common("kq_swiglu_quantize_q8k", g, u, M, K, ld, xq, h_out, 256, true, (cudaStream_t)stream);
}

}  // extern "C"
