// kq_gemv.cu -- decode GEMV (one activation column) over native block-quantised weights.
//
// Design (GB300): the weight stream is the whole cost, so every byte is read once with 16-byte
// (or 8-byte) coalesced loads, and the next chunk's loads are issued before the current chunk is
// consumed.  A thread block owns one 16-row group and a contiguous range of 256-element chunks;
// rows with long K are split across the CTAs of a thread-block cluster, whose partial results are
// combined through distributed shared memory (no workspace, no atomics).
//
// Each (row, chunk) term is formed exactly as the prefill GEMM forms it -- integer sub-block dots
// (dp4a), integer scale/min sums reduced across the 8 lanes of a row with shuffles, then one fp32
// expression per super-block -- and the terms of a row are added in ascending K order by a single
// thread.  The result is therefore bit-identical to the sequential CPU accumulation order, the
// property the keep-quant provider of vllm.cpp PR #2890 gates on, and it does not depend on the
// launch shape (strix-llama.cpp PR #18 keeps batch-one MMVQ on a fixed reduction order for the
// same reason).
//
// With x != NULL the activation is quantised inside the kernel (fused-quant MMVQ of
// strix-llama.cpp PR #18): each CTA quantises the part of x its K range needs into shared memory,
// after its first weight loads are already in flight.
#include <cooperative_groups.h>

#include "kq_act_smem.cuh"
#include "kq_internal.cuh"

namespace cg = cooperative_groups;

namespace kq {

constexpr int kGemvThreads = 256;  // 2 chunk slots x 16 rows x 8 lanes

template <int DT>
struct GemvTraits;
template <>
struct GemvTraits<KQ_Q4_K> { static constexpr int terms = 1; static constexpr bool q81 = false; };
template <>
struct GemvTraits<KQ_Q6_K> { static constexpr int terms = 1; static constexpr bool q81 = false; };
template <>
struct GemvTraits<KQ_Q8_0> { static constexpr int terms = 8; static constexpr bool q81 = true; };

// Registers holding one lane's slice of one chunk.  Lane t of a row owns kblock c = t/2 and the
// 16-byte half seg = t%2 of that kblock's codes: elements 64c+16seg+i (low nibbles) and
// 64c+32+16seg+i (high nibbles), i < 16.  (Q8_0: lane t owns 32-element block t.)
struct LaneRegs {
    uint4 a;     // Q4_K/Q6_K: 16 code bytes (low 4 bits); Q8_0: codes 0..15
    uint4 b;     // Q4_K: header (d, dmin, scales); Q6_K: 16 high-bit bytes; Q8_0: codes 16..31
    uint32_t c;  // Q6_K: scale bytes of sub-blocks 4c..4c+3; Q8_0: f16 d
    uint32_t d;  // Q6_K: f16 d
};

template <int DT>
__device__ __forceinline__ void gemv_load(const uint8_t *__restrict__ chunk, int r, int t, LaneRegs &R) {
    const int c = t >> 1, seg = t & 1;
    if (DT == KQ_Q4_K) {
        R.a = __ldg(reinterpret_cast<const uint4 *>(chunk + c * 512 + r * 32 + seg * 16));
        R.b = __ldg(reinterpret_cast<const uint4 *>(chunk + 2048 + r * 16));
    } else if (DT == KQ_Q6_K) {
        R.a = __ldg(reinterpret_cast<const uint4 *>(chunk + c * 512 + r * 32 + seg * 16));
        R.b = __ldg(reinterpret_cast<const uint4 *>(chunk + 2048 + c * 256 + r * 16));
        R.c = __ldg(reinterpret_cast<const uint32_t *>(chunk + 3072 + r * 16 + 4 * c));
        R.d = __ldg(reinterpret_cast<const uint16_t *>(chunk + 3328 + r * 2));
    } else {
        const uint8_t *codes = chunk + c * 1024 + r * 64 + 32 * seg;
        R.a = __ldg(reinterpret_cast<const uint4 *>(codes));
        R.b = __ldg(reinterpret_cast<const uint4 *>(codes + 16));
        R.c = __ldg(reinterpret_cast<const uint16_t *>(chunk + 4096 + r * 16 + 2 * t));
    }
}

__device__ __forceinline__ int sext8(uint32_t w, int i) { return (int)(int8_t)((w >> (8 * i)) & 0xff); }

// Computes this lane's integer contributions for one chunk and, on lane 0 of the row, the exact
// fp32 term(s) of the super-block.  q/da/bs point at the chunk's activation in shared memory.
template <int DT>
__device__ __forceinline__ void gemv_compute(const LaneRegs &R, int t, const int8_t *__restrict__ q,
                                             const float *__restrict__ da, const int16_t *__restrict__ bs,
                                             float *term_out) {
    const int c = t >> 1, seg = t & 1;
    if (DT == KQ_Q4_K || DT == KQ_Q6_K) {
        const int4 qlo = *reinterpret_cast<const int4 *>(q + 64 * c + 16 * seg);
        const int4 qhi = *reinterpret_cast<const int4 *>(q + 64 * c + 32 + 16 * seg);
        const uint32_t w[4] = {R.a.x, R.a.y, R.a.z, R.a.w};
        const uint32_t hb[4] = {R.b.x, R.b.y, R.b.z, R.b.w};
        const int ql[4] = {qlo.x, qlo.y, qlo.z, qlo.w}, qh[4] = {qhi.x, qhi.y, qhi.z, qhi.w};
        int plo = 0, phi = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t lo = w[i] & 0x0f0f0f0fu, hi = (w[i] >> 4) & 0x0f0f0f0fu;
            if (DT == KQ_Q6_K) {
                lo = __vsub4(lo | (((hb[i] >> (2 * seg)) & 0x03030303u) << 4), 0x20202020u);
                hi = __vsub4(hi | (((hb[i] >> (4 + 2 * seg)) & 0x03030303u) << 4), 0x20202020u);
            }
            plo = dp4a((int)lo, ql[i], plo);
            phi = dp4a((int)hi, qh[i], phi);
        }
        if (DT == KQ_Q4_K) {
            uint8_t s12[12];
            const uint32_t hw[3] = {R.b.y, R.b.z, R.b.w};
#pragma unroll
            for (int i = 0; i < 12; ++i) s12[i] = (hw[i / 4] >> (8 * (i % 4))) & 0xff;
            int sc0, m0, sc1, m1;
            q4k_scale_min(s12, 2 * c, sc0, m0);
            q4k_scale_min(s12, 2 * c + 1, sc1, m1);
            int sumi = sc0 * plo + sc1 * phi;
            // bsums of the lane's two 16-element groups; the partner lane (t ^ 1) adds the other
            // half of each sub-block, so the row-wide integer sum over lanes is exact.
            int summ = m0 * bs[4 * c + seg] + m1 * bs[4 * c + 2 + seg];
#pragma unroll
            for (int s = 4; s >= 1; s >>= 1) {
                sumi += __shfl_xor_sync(0xffffffffu, sumi, s);
                summ += __shfl_xor_sync(0xffffffffu, summ, s);
            }
            if (t == 0) {
                const float dw = half_bits_to_float((uint16_t)(R.b.x & 0xffff));
                const float dmin = half_bits_to_float((uint16_t)(R.b.x >> 16));
                const float a = da[0];
                float t1 = __fmul_rn(a, dw);
                float t2 = __fmul_rn(t1, (float)sumi);
                float t3 = __fmul_rn(a, dmin);
                float t4 = __fmul_rn(t3, (float)summ);
                term_out[0] = __fsub_rn(t2, t4);
            }
        } else {
            // sub-blocks of 16: low run = 4c+seg, high run = 4c+2+seg (scale bytes seg and 2+seg of R.c)
            int sumi = sext8(R.c, seg) * plo + sext8(R.c, 2 + seg) * phi;
#pragma unroll
            for (int s = 4; s >= 1; s >>= 1) sumi += __shfl_xor_sync(0xffffffffu, sumi, s);
            if (t == 0) {
                const float dw = half_bits_to_float((uint16_t)R.d);
                const float t1 = __fmul_rn(da[0], dw);
                term_out[0] = __fmul_rn(t1, (float)sumi);
            }
        }
    } else {
        const int4 q0 = *reinterpret_cast<const int4 *>(q + 32 * t);
        const int4 q1 = *reinterpret_cast<const int4 *>(q + 32 * t + 16);
        int p = 0;
        p = dp4a((int)R.a.x, q0.x, p); p = dp4a((int)R.a.y, q0.y, p);
        p = dp4a((int)R.a.z, q0.z, p); p = dp4a((int)R.a.w, q0.w, p);
        p = dp4a((int)R.b.x, q1.x, p); p = dp4a((int)R.b.y, q1.y, p);
        p = dp4a((int)R.b.z, q1.z, p); p = dp4a((int)R.b.w, q1.w, p);
        const float dw = half_bits_to_float((uint16_t)R.c);
        const float t1 = __fmul_rn(dw, da[t]);
        term_out[t] = __fmul_rn(t1, (float)p);
    }
}

// grid: (S, groups); cluster (S, 1, 1).  CTA rank k of a cluster covers chunks [k*cpr, ...).
template <int DT, bool FUSED>
__global__ void __launch_bounds__(kGemvThreads) gemv_kernel(const uint8_t *__restrict__ w,
                                                            const float *__restrict__ x,
                                                            const uint8_t *__restrict__ xq, int64_t N,
                                                            int nchunk, int cpr, float *__restrict__ y) {
    using Tr = GemvTraits<DT>;
    extern __shared__ __align__(16) uint8_t smem[];
    const int S = gridDim.x;
    const int rank = blockIdx.x;
    const int64_t g = blockIdx.y;
    const int c_begin = rank * cpr;
    const int c_end = min(nchunk, c_begin + cpr);
    const int nloc = max(0, c_end - c_begin);

    // shared layout: q [cpr*256] | da [cpr*terms_per_chunk_d] | bs [cpr*16] | terms [16][cpr*terms]
    constexpr int kDaPerChunk = Tr::q81 ? 8 : 1;
    int8_t *q_s = reinterpret_cast<int8_t *>(smem);
    float *da_s = reinterpret_cast<float *>(smem + cpr * 256);
    int16_t *bs_s = reinterpret_cast<int16_t *>(smem + cpr * 256 + cpr * kDaPerChunk * 4);
    float *terms = reinterpret_cast<float *>(smem + cpr * 256 + cpr * kDaPerChunk * 4 + cpr * 32);

    const int tid = threadIdx.x;
    const int slot = tid >> 7, r = (tid >> 3) & 15, t = tid & 7;
    const int cb = chunk_bytes(DT);
    const uint8_t *wg = w + (g * nchunk) * (int64_t)cb;

    // issue the first chunk's weight loads before touching the activation
    LaneRegs cur;
    int c = c_begin + slot;
    if (c < c_end) gemv_load<DT>(wg + (int64_t)c * cb, r, t, cur);

    // ---- activation prologue: quantise (FUSED) or copy the K range into shared memory
    const int warp = tid >> 5, lane = tid & 31;
    if (FUSED) {
        if (!Tr::q81) {
            for (int cc = warp; cc < nloc; cc += kGemvThreads / 32)
                warp_quantize_q8k_smem(x + (int64_t)(c_begin + cc) * 256, q_s + cc * 256, da_s + cc, bs_s + cc * 16);
        } else {
            for (int part = warp; part < nloc * 2; part += kGemvThreads / 32)
                warp_quantize_q8_1x4_smem(x + (int64_t)c_begin * 256 + part * 128, q_s + part * 128, da_s + part * 4);
        }
    } else {
        if (!Tr::q81) {
            for (int cc = warp; cc < nloc; cc += kGemvThreads / 32) {
                const uint8_t *blk = xq + (int64_t)(c_begin + cc) * kQ8KBytes;
                const uint32_t *src = reinterpret_cast<const uint32_t *>(blk + 4);
                reinterpret_cast<uint2 *>(q_s + cc * 256)[lane] = make_uint2(src[2 * lane], src[2 * lane + 1]);
                if (lane < 16) bs_s[cc * 16 + lane] = reinterpret_cast<const int16_t *>(blk + 260)[lane];
                if (lane == 0) da_s[cc] = *reinterpret_cast<const float *>(blk);
            }
        } else {
            for (int b = tid; b < nloc * 8; b += kGemvThreads) {
                const uint8_t *blk = xq + ((int64_t)c_begin * 8 + b) * kQ81Bytes;
                const uint32_t *src = reinterpret_cast<const uint32_t *>(blk + 4);
                uint32_t *dst = reinterpret_cast<uint32_t *>(q_s + b * 32);
#pragma unroll
                for (int i = 0; i < 8; ++i) dst[i] = src[i];
                da_s[b] = half_bits_to_float(*reinterpret_cast<const uint16_t *>(blk));
            }
        }
    }
    __syncthreads();

    // ---- main loop: two chunk slots in flight per row, next chunk prefetched into registers
    const int tstride = cpr * Tr::terms;
    for (; c < c_end; c += 2) {
        LaneRegs nxt;
        const int cn = c + 2;
        if (cn < c_end) gemv_load<DT>(wg + (int64_t)cn * cb, r, t, nxt);
        const int cl = c - c_begin;
        gemv_compute<DT>(cur, t, q_s + cl * 256, da_s + cl * kDaPerChunk, bs_s + cl * 16,
                         terms + r * tstride + cl * Tr::terms);
        cur = nxt;
    }

    // ---- ordered reduction: one thread per row adds the row's terms in ascending K order
    if (S == 1) {
        __syncthreads();
        if (tid < 16) {
            const int64_t n = g * 16 + tid;
            float acc = 0.0f;
            for (int i = 0; i < nloc * Tr::terms; ++i) acc = __fadd_rn(acc, terms[tid * tstride + i]);
            if (n < N) y[n] = acc;
        }
    } else {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        if (rank == 0 && tid < 16) {
            const int64_t n = g * 16 + tid;
            float acc = 0.0f;
            for (int k = 0; k < S; ++k) {
                const float *rt = cluster.map_shared_rank(terms, k);
                const int kb = k * cpr, ke = min(nchunk, kb + cpr);
                const int cnt = max(0, ke - kb) * Tr::terms;
                for (int i = 0; i < cnt; ++i) acc = __fadd_rn(acc, rt[tid * tstride + i]);
            }
            if (n < N) y[n] = acc;
        }
        cluster.sync();
    }
}

template <int DT, bool FUSED>
static kq_status launch_gemv(const uint8_t *w, const float *x, const uint8_t *xq, int64_t N, int64_t K, float *y,
                             cudaStream_t st) {
    using Tr = GemvTraits<DT>;
    const int nchunk = (int)(K / 256);
    const int64_t groups = (N + 15) / 16;
    // split K across a cluster when there are too few row groups to fill the GPU
    int S = 1;
    while (S < 8 && groups * S < 4 * 152 && nchunk >= 4 * S * 2) S *= 2;
    const int cpr = (nchunk + S - 1) / S;
    constexpr int kDaPerChunk = Tr::q81 ? 8 : 1;
    const size_t smem = (size_t)cpr * 256 + (size_t)cpr * kDaPerChunk * 4 + (size_t)cpr * 32 +
                        (size_t)16 * cpr * Tr::terms * 4;
    if (smem > 200 * 1024) return fail(KQ_ERR_INVALID_ARG, "kq_gemv: K=%lld too large", (long long)K);
    if (groups > 65535) return fail(KQ_ERR_INVALID_ARG, "kq_gemv: N=%lld too large", (long long)N);
    auto kern = gemv_kernel<DT, FUSED>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return fail(KQ_ERR_CUDA, "kq_gemv: %s", cudaGetErrorString(e));
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S, (unsigned)groups, 1);
    cfg.blockDim = dim3(kGemvThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, w, x, xq, N, nchunk, cpr, y);
    if (e != cudaSuccess) return fail(KQ_ERR_CUDA, "kq_gemv: launch failed: %s", cudaGetErrorString(e));
    count_launch(R_GEMV);
    return KQ_OK;
}

}  // namespace kq

using namespace kq;

extern "C" kq_status kq_gemv(kq_dtype wt, const void *w, const float *x, const void *xq, int64_t N, int64_t K,
                             float *y, kq_stream_t stream) {
    if (wt != KQ_Q4_K && wt != KQ_Q6_K && wt != KQ_Q8_0)
        return fail(KQ_ERR_UNSUPPORTED_DTYPE, "kq_gemv: weight dtype %s is not Q4_K, Q6_K or Q8_0", dtype_name(wt));
    if (!w || !y || (!x && !xq) || (x && xq))
        return fail(KQ_ERR_INVALID_ARG, "kq_gemv: need w, y and exactly one of x / xq");
    if (N <= 0 || K <= 0 || K % 256)
        return fail(KQ_ERR_INVALID_ARG, "kq_gemv: need N > 0 and K a positive multiple of 256 (N=%lld K=%lld)",
                    (long long)N, (long long)K);
    if (!aligned(w, 16) || !aligned(y, 4) || (x && !aligned(x, 4)) || (xq && !aligned(xq, 4)))
        return fail(KQ_ERR_ALIGNMENT, "kq_gemv: w must be 16-byte aligned, x/xq/y 4-byte aligned");
    cudaStream_t st = (cudaStream_t)stream;
    const uint8_t *wb = static_cast<const uint8_t *>(w);
    const uint8_t *xb = static_cast<const uint8_t *>(xq);
    switch (wt) {
    case KQ_Q4_K: return x ? launch_gemv<KQ_Q4_K, true>(wb, x, xb, N, K, y, st) : launch_gemv<KQ_Q4_K, false>(wb, x, xb, N, K, y, st);
    case KQ_Q6_K: return x ? launch_gemv<KQ_Q6_K, true>(wb, x, xb, N, K, y, st) : launch_gemv<KQ_Q6_K, false>(wb, x, xb, N, K, y, st);
    default: return x ? launch_gemv<KQ_Q8_0, true>(wb, x, xb, N, K, y, st) : launch_gemv<KQ_Q8_0, false>(wb, x, xb, N, K, y, st);
    }
}
