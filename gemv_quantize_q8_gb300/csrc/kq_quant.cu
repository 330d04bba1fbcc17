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
#include "kq_q8k_block.cuh"
#include "kq_sm100.cuh"

namespace kq {

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
    q8k_block_store(v, out + blk * kQ8KBytes);
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

// Fused RMSNorm + Q8_K producer (vllm.cpp PR #2890, fused norm-quant epilogue: the norm row kernel
// emits the row's Q8_K blocks beside its normalized output).  One block per row:
//   ss = sum_i x_i^2 -- thread t < 256 adds x[t]^2, x[t+256]^2, ... in order, each of the first 8
//        warps combines its 32 sums in xor-butterfly order (strides 16 .. 1), thread 0 adds the 8
//        warp sums in order;
//   r  = 1 / sqrt(ss / K + eps) (IEEE division and square root);  y_i = (x_i * r) * gamma_i;
// then warp w quantises blocks w, w+NW, ... of y with the standalone Q8_K body (and stores y when
// y_out != NULL).  Every operation is rounded on its own, so codes and y match the CPU oracle's.
// With few rows (THREADS = 1024) the x and gamma values of each warp's first two blocks, which do not
// depend on r, are loaded before the reduction, so a decode row pays one memory round trip for them;
// with many rows (THREADS = 256) the rows in flight hide the latency and registers stay free.
// The few-row launch allows programmatic dependent launch, as the decode GEMV does: gamma (a weight,
// never written by the kernel before this one) is read before the dependency wait, x after it.
template <bool VEC, int THREADS>
__global__ void __launch_bounds__(THREADS) rmsnorm_q8k_kernel(const float *__restrict__ x, const float *__restrict__ gamma,
                                                              float eps, int64_t K, int64_t ldx, uint8_t *__restrict__ out,
                                                              float *__restrict__ y_out) {
    constexpr int NW = THREADS / 32;
    constexpr int PF = THREADS >= 1024 ? 2 : 0;  // blocks per warp loaded before the reduction
    __shared__ float wsum[8];
    __shared__ float rs;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t row = blockIdx.x;
    const float *xr = x + row * ldx;
    const int64_t nb = K / 256;
    float pv[PF > 0 ? PF : 1][8], pg[PF > 0 ? PF : 1][8];
    if (PF > 0) sm100::grid_launch_dependents();
#pragma unroll
    for (int j = 0; j < PF; ++j)
        if (warp + j * NW < nb) load8<VEC>(gamma + (warp + j * NW) * 256 + lane * 8, pg[j]);
    if (PF > 0) sm100::grid_dependency_wait();
#pragma unroll
    for (int j = 0; j < PF; ++j)
        if (warp + j * NW < nb) load8<VEC>(xr + (warp + j * NW) * 256 + lane * 8, pv[j]);
    if (tid < 256) {
        float s = 0.0f;
        for (int64_t i = tid; i < K; i += 256) {
            const float v = xr[i];
            s = __fadd_rn(s, __fmul_rn(v, v));
        }
#pragma unroll
        for (int st = 16; st >= 1; st >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, st));
        if (lane == 0) wsum[warp] = s;
    }
    __syncthreads();
    if (tid == 0) {
        float total = 0.0f;
        for (int w = 0; w < 8; ++w) total = __fadd_rn(total, wsum[w]);
        const float mean = __fdiv_rn(total, (float)K);
        rs = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
    }
    __syncthreads();
    const float r = rs;
    auto emit = [&](int64_t b, float (&v)[8], const float (&gv)[8]) {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(__fmul_rn(v[i], r), gv[i]);
        if (y_out) {
            float *yp = y_out + row * K + b * 256 + lane * 8;
#pragma unroll
            for (int i = 0; i < 8; ++i) yp[i] = v[i];
        }
        q8k_block_store(v, out + (row * nb + b) * kQ8KBytes);
    };
#pragma unroll
    for (int j = 0; j < PF; ++j)
        if (warp + j * NW < nb) emit(warp + j * NW, pv[j], pg[j]);
    for (int64_t b = warp + PF * NW; b < nb; b += NW) {
        float v[8], gv[8];
        load8<VEC>(xr + b * 256 + lane * 8, v);
        load8<VEC>(gamma + b * 256 + lane * 8, gv);
        emit(b, v, gv);
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

kq_status kq_rmsnorm_quantize_q8k(const float *x, const float *gamma, float eps, int64_t M, int64_t K, int64_t ldx,
                                  void *xq, float *y_out, kq_stream_t stream) {
    const char *name = "kq_rmsnorm_quantize_q8k";
    if (!x || !gamma || !xq) return fail(KQ_ERR_INVALID_ARG, "%s: null pointer", name);
    if (M <= 0 || K <= 0 || K % 256 || M > 0x7fffffff)
        return fail(KQ_ERR_INVALID_ARG, "%s: need M > 0 and K a positive multiple of 256 (M=%lld K=%lld)", name,
                    (long long)M, (long long)K);
    if (ldx < K) return fail(KQ_ERR_INVALID_ARG, "%s: leading dimension %lld < K %lld", name, (long long)ldx, (long long)K);
    if (!(eps >= 0.0f) || !isfinite(eps)) return fail(KQ_ERR_INVALID_ARG, "%s: eps must be finite and >= 0", name);
    if (!aligned(x, 4) || !aligned(gamma, 4) || !aligned(xq, 4) || (y_out && !aligned(y_out, 4)))
        return fail(KQ_ERR_ALIGNMENT, "%s: pointers must be 4-byte aligned", name);
    const bool vec = aligned(x, 16) && aligned(gamma, 16) && ldx % 4 == 0 && (!y_out || aligned(y_out, 16));
    cudaStream_t st = (cudaStream_t)stream;
    uint8_t *o = static_cast<uint8_t *>(xq);
    // a few rows (decode): 32 warps per row so the Q8_K blocks are quantised in one round; many rows:
    // 8 warps per row, several rows per SM
    if (M <= 64) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)M, 1, 1);
        cfg.blockDim = dim3(1024, 1, 1);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = vec ? cudaLaunchKernelEx(&cfg, rmsnorm_q8k_kernel<true, 1024>, x, gamma, eps, K, ldx, o, y_out)
                            : cudaLaunchKernelEx(&cfg, rmsnorm_q8k_kernel<false, 1024>, x, gamma, eps, K, ldx, o, y_out);
        if (e != cudaSuccess) return fail(KQ_ERR_CUDA, "%s: launch failed: %s", name, cudaGetErrorString(e));
    } else {
        if (vec) rmsnorm_q8k_kernel<true, 256><<<(unsigned)M, 256, 0, st>>>(x, gamma, eps, K, ldx, o, y_out);
        else rmsnorm_q8k_kernel<false, 256><<<(unsigned)M, 256, 0, st>>>(x, gamma, eps, K, ldx, o, y_out);
    }
    kq_status s = check_launch(name);
    if (s == KQ_OK) count_launch(R_QUANT);
    return s;
}

}  // extern "C"
