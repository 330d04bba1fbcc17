// kq_gemv.cu -- decode GEMV (one activation column) over native block-quantised weights.
//
// Design (GB300): the weight stream is the whole cost.  A thread block owns 32 rows (two native row
// groups) and a range of 256-element chunks; each warp owns one chunk and streams its codes into
// shared memory with bulk copies (cp.async.bulk + mbarrier), so all of the block's bytes are in
// flight at once, and waits for them asleep rather than spinning.  A lane owns one row of that
// chunk (128-256 code bytes), which keeps the instruction count per weight byte low; 32 rows per
// block also halve the activation work each block repeats.
// Rows with long K are split across the CTAs of a thread-block cluster, whose partial results are
// combined through distributed shared memory (no workspace, no atomics).  Launches allow
// programmatic dependent launch: the next kernel in the stream is scheduled early and waits on the
// hardware dependency before touching memory, which hides the launch gap between decode kernels.
//
// Each (row, chunk) term is formed exactly as the CPU oracle forms it -- integer sub-block dots
// (dp4a), integer scale/min sums, then one fp32 expression per super-block -- and the terms of a
// row are added in ascending K order by a single thread.  The result is therefore bit-identical to the sequential CPU accumulation order, the
// property the keep-quant provider of vllm.cpp PR #2890 gates on, and it does not depend on the
// launch shape (strix-llama.cpp PR #18 keeps batch-one MMVQ on a fixed reduction order for the
// same reason).
//
// With x != NULL the activation is quantised inside the kernel (fused-quant MMVQ of
// strix-llama.cpp PR #18): each warp quantises the 256 activation values of its own chunk into
// shared memory while its weight copies are in flight.
//
// Long K without a cluster: gemv16_kernel (one column) and gemv16_mc_kernel (up to 8 pre-quantised
// columns) give each 16-row group one block over the whole K, so successive calls are not clustered
// launches; several columns stage their activation blocks with every load issued before the first
// store.
#include <cooperative_groups.h>

#include "kq_act_smem.cuh"
#include "kq_internal.cuh"
#include "kq_sm100.cuh"

namespace cg = cooperative_groups;

namespace kq {

using namespace sm100;

#ifndef GEMV16_OK
#define GEMV16_OK 1
#endif

constexpr int kGemvRows = 32;
// gemv16_kernel: at most 20 warps (40 chunks, K <= 10240), registers for two blocks per SM -- this
// call's and the next one's
constexpr int kGemv16MaxWarps = 20;      // rows per thread block (two native row groups), one per lane
constexpr int kGemvMaxWarps = 32;

template <int DT>
struct GemvTraits;
template <>
struct GemvTraits<KQ_Q4_K> { static constexpr int terms = 1; static constexpr bool q81 = false; };
template <>
struct GemvTraits<KQ_Q5_K> { static constexpr int terms = 1; static constexpr bool q81 = false; };
template <>
struct GemvTraits<KQ_Q6_K> { static constexpr int terms = 1; static constexpr bool q81 = false; };
template <>
struct GemvTraits<KQ_Q8_0> { static constexpr int terms = 8; static constexpr bool q81 = true; };

__device__ __forceinline__ int sext8(uint32_t w, int i) { return (int)(int8_t)((w >> (8 * i)) & 0xff); }

// Two-way dot products of the two signed 16-bit halves of a with two bytes of b (bytes 0-1: lo, 2-3: hi;
// signed or unsigned bytes), plus c.
__device__ __forceinline__ int dp2a_lo_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp2a_lo_ss(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.lo.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp2a_hi_ss(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.hi.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Dot product of four unsigned bytes of a with four signed bytes of b, plus c.
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Per-warp shared region: the chunk's codes for the block's two row groups, then the chunk's
// activation for each of the MC activation columns (320 bytes each: q[256], d, bsums).
template <int DT, int MC>
struct GemvWarpSmem {
    static constexpr int CB = chunk_bytes(DT);
    static constexpr int Q_OFF = 2 * CB;          // column m at Q_OFF + m*XB: int8 q[256]
    static constexpr int D_OFF = Q_OFF + 256;     // f32 d: 1 (Q8_K) or 8 (Q8_1)
    static constexpr int B_OFF = D_OFF + 32;      // int16 bsums[16]
    static constexpr int XB = 320;                // one column's activation (multiple of 16)
    static constexpr int BYTES = Q_OFF + MC * XB;
};

// One lane = one row: the exact fp32 term(s) of (row, chunk) from the integer sub-block dots.
// Q4_K, Q5_K: term = (d_a*d_w)*sumi - (d_a*dmin)*summ; Q6_K: term = (d_a*d_w)*sumi;
// Q8_0: 8 terms (d_w*d_a)*P_b, one per 32-element block.
template <int DT>
__device__ __forceinline__ void gemv_row_chunk(const uint8_t *__restrict__ chunk, int r,
                                               const int8_t *__restrict__ q, const float *__restrict__ da,
                                               const int16_t *__restrict__ bs, float *__restrict__ term) {
    if (DT == KQ_Q4_K || DT == KQ_Q5_K || DT == KQ_Q6_K) {
        constexpr bool K4 = DT == KQ_Q4_K || DT == KQ_Q5_K;  // 8 sub-blocks of 32 with (d, dmin, scales, mins)
        int P[16];  // Q4_K/Q5_K: 8 sub-blocks of 32; Q6_K: 16 sub-blocks of 16
        uint32_t q5h[8];  // Q5_K: the row's 32 high-bit bytes (byte l pairs with code byte l of every kblock)
        if (DT == KQ_Q5_K) {
            const uint4 a = *reinterpret_cast<const uint4 *>(chunk + 2304 + r * 32);
            const uint4 b = *reinterpret_cast<const uint4 *>(chunk + 2304 + r * 32 + 16);
            q5h[0] = a.x; q5h[1] = a.y; q5h[2] = a.z; q5h[3] = a.w; q5h[4] = b.x; q5h[5] = b.y; q5h[6] = b.z; q5h[7] = b.w;
        }
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
            const uint4 v0 = *reinterpret_cast<const uint4 *>(chunk + kb * 512 + r * 32);
            const uint4 v1 = *reinterpret_cast<const uint4 *>(chunk + kb * 512 + r * 32 + 16);
            const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            uint32_t hb[4] = {0u, 0u, 0u, 0u};
            if (DT == KQ_Q6_K) {
                const uint4 h = *reinterpret_cast<const uint4 *>(chunk + 2048 + kb * 256 + r * 16);
                hb[0] = h.x; hb[1] = h.y; hb[2] = h.z; hb[3] = h.w;
            }
            const int4 qa0 = *reinterpret_cast<const int4 *>(q + 64 * kb);
            const int4 qa1 = *reinterpret_cast<const int4 *>(q + 64 * kb + 16);
            const int4 qb0 = *reinterpret_cast<const int4 *>(q + 64 * kb + 32);
            const int4 qb1 = *reinterpret_cast<const int4 *>(q + 64 * kb + 48);
            const int ql[8] = {qa0.x, qa0.y, qa0.z, qa0.w, qa1.x, qa1.y, qa1.z, qa1.w};
            const int qh[8] = {qb0.x, qb0.y, qb0.z, qb0.w, qb1.x, qb1.y, qb1.z, qb1.w};
            int plo[2] = {0, 0}, phi[2] = {0, 0};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int seg = i >> 2;  // elements 64kb+16seg+.. (low nibbles) / 64kb+32+16seg+.. (high)
                const uint32_t lo4 = w[i] & 0x0f0f0f0fu;
                if (DT == KQ_Q4_K) {
                    // high nibbles left in place: the bytes are 16*c, so the dot is 16 times the
                    // sub-block's (divided out, exactly, below) and no shift is needed per word
                    plo[seg] = dp4a((int)lo4, ql[i], plo[seg]);
                    phi[seg] = dp4a_us(w[i] & 0xf0f0f0f0u, qh[i], phi[seg]);
                } else if (DT == KQ_Q5_K) {  // fifth bit: bit 2kb of byte l (low nibbles), bit 2kb+1 (high)
                    const uint32_t lo = lo4 | (((q5h[i] >> (2 * kb)) & 0x01010101u) << 4);
                    const uint32_t hi = ((w[i] >> 4) & 0x0f0f0f0fu) | (((q5h[i] >> (2 * kb + 1)) & 0x01010101u) << 4);
                    plo[seg] = dp4a((int)lo, ql[i], plo[seg]);
                    phi[seg] = dp4a((int)hi, qh[i], phi[seg]);
                } else {
                    // Q6_K: the unsigned 6-bit codes c; the -32 offset comes off once per sub-block
                    // below (sum (c-32)*q = sum c*q - 32*bsum, the activation's bsum of those 16)
                    const uint32_t lo = lo4 | (((hb[i & 3] >> (2 * seg)) & 0x03030303u) << 4);
                    const uint32_t hi = ((w[i] >> 4) & 0x0f0f0f0fu) | (((hb[i & 3] >> (4 + 2 * seg)) & 0x03030303u) << 4);
                    plo[seg] = dp4a((int)lo, ql[i], plo[seg]);
                    phi[seg] = dp4a((int)hi, qh[i], phi[seg]);
                }
            }
            if (K4) {
                P[2 * kb] = plo[0] + plo[1];  // sub-block 2kb   (elements 64kb .. 64kb+31)
                // sub-block 2kb+1 (elements 64kb+32 .. 64kb+63); Q4_K's sums are of 16*c, a multiple of 16
                P[2 * kb + 1] = DT == KQ_Q4_K ? (phi[0] + phi[1]) >> 4 : phi[0] + phi[1];
            } else {
                P[4 * kb] = plo[0];      // sub-block 4kb   (elements 64kb .. +15), sum c*q
                P[4 * kb + 1] = plo[1];  // sub-block 4kb+1 (64kb+16 .. +31)
                P[4 * kb + 2] = phi[0];  // sub-block 4kb+2 (64kb+32 .. +47)
                P[4 * kb + 3] = phi[1];  // sub-block 4kb+3 (64kb+48 .. +63)
            }
        }
        if (K4) {
            const uint4 hv = *reinterpret_cast<const uint4 *>(chunk + 2048 + r * 16);
            // the eight 6-bit scales and mins, four per word, from the 12 packed bytes (GGUF's packing:
            // sub-blocks 0-3 in the low 6 bits of bytes 0-3 / 4-7; 4-7 from the nibbles of bytes 8-11
            // and the top two bits of bytes 0-3 / 4-7)
            const uint32_t scw[2] = {hv.y & 0x3f3f3f3fu, (hv.w & 0x0f0f0f0fu) | ((hv.y >> 2) & 0x30303030u)};
            const uint32_t mw[2] = {hv.z & 0x3f3f3f3fu, ((hv.w >> 4) & 0x0f0f0f0fu) | ((hv.z >> 2) & 0x30303030u)};
            const uint4 b0 = *reinterpret_cast<const uint4 *>(bs);
            const uint4 b1 = *reinterpret_cast<const uint4 *>(bs + 8);
            const uint32_t bw[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
            int sumi = 0, summ = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                sumi += (int)((scw[j >> 2] >> (8 * (j & 3))) & 0xff) * P[j];
                // m_j*(bs_2j + bs_2j+1): the two int16 halves of bsum word j against m_j in both bytes
                summ = dp2a_lo_su(bw[j], __byte_perm(mw[j >> 2], 0u, 0x4400u | ((j & 3) * 0x11u)), summ);
            }
            const float dw = half_bits_to_float((uint16_t)(hv.x & 0xffff));
            const float dmin = half_bits_to_float((uint16_t)(hv.x >> 16));
            const float a = da[0];
            const float t1 = __fmul_rn(a, dw);
            const float t2 = __fmul_rn(t1, (float)sumi);
            const float t3 = __fmul_rn(a, dmin);
            const float t4 = __fmul_rn(t3, (float)summ);
            term[0] = __fsub_rn(t2, t4);
        } else {
            const uint4 sv = *reinterpret_cast<const uint4 *>(chunk + 3072 + r * 16);
            const uint32_t sw4[4] = {sv.x, sv.y, sv.z, sv.w};
            const uint4 b0 = *reinterpret_cast<const uint4 *>(bs);
            const uint4 b1 = *reinterpret_cast<const uint4 *>(bs + 8);
            const uint32_t bw[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
            // sum_j sc_j*(P_j - 32*bs_j): the codes' dots, then the offset through the bsums (sc_j with
            // bsum j: two per word of each, two-way dot products)
            int sumi = 0, sumb = 0;
#pragma unroll
            for (int j = 0; j < 16; ++j) sumi += sext8(sw4[j / 4], j % 4) * P[j];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                sumb = dp2a_lo_ss(bw[2 * k], sw4[k], sumb);
                sumb = dp2a_hi_ss(bw[2 * k + 1], sw4[k], sumb);
            }
            sumi -= 32 * sumb;
            const float dw = half_bits_to_float(*reinterpret_cast<const uint16_t *>(chunk + 3328 + r * 2));
            const float t1 = __fmul_rn(da[0], dw);
            term[0] = __fmul_rn(t1, (float)sumi);
        }
    } else {
        const uint4 dv = *reinterpret_cast<const uint4 *>(chunk + 4096 + r * 16);
        const uint32_t dw4[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const uint8_t *codes = chunk + (b >> 1) * 1024 + r * 64 + 32 * (b & 1);
            const uint4 a0 = *reinterpret_cast<const uint4 *>(codes);
            const uint4 a1 = *reinterpret_cast<const uint4 *>(codes + 16);
            const int4 q0 = *reinterpret_cast<const int4 *>(q + 32 * b);
            const int4 q1 = *reinterpret_cast<const int4 *>(q + 32 * b + 16);
            int p = 0;
            p = dp4a((int)a0.x, q0.x, p); p = dp4a((int)a0.y, q0.y, p);
            p = dp4a((int)a0.z, q0.z, p); p = dp4a((int)a0.w, q0.w, p);
            p = dp4a((int)a1.x, q1.x, p); p = dp4a((int)a1.y, q1.y, p);
            p = dp4a((int)a1.z, q1.z, p); p = dp4a((int)a1.w, q1.w, p);
            const float dw = half_bits_to_float((uint16_t)((dw4[b >> 1] >> (16 * (b & 1))) & 0xffff));
            const float t1 = __fmul_rn(dw, da[b]);
            term[b] = __fmul_rn(t1, (float)p);
        }
    }
}

// One lane = one row, M <= MC activation columns (Q4_K, Q5_K, Q6_K): the terms of gemv_row_chunk for
// every column, each weight word unpacked once and dotted against all columns.  A column's integer sum
// sum_j sc_j*P_j is gathered sub-block by sub-block (exact integers in any order), so every term is
// formed exactly as gemv_row_chunk forms it.  Column m's activation block sits at q + m*xb (int8
// q[256], then f32 d at +256, int16 bsums at +288); term m goes to term[m * tstep].
template <int DT, int MC>
__device__ __forceinline__ void gemv_row_chunk_mc(const uint8_t *__restrict__ chunk, int r, const uint8_t *__restrict__ q,
                                                  int xb, int M, float *__restrict__ term, int tstep) {
    constexpr bool K4 = DT == KQ_Q4_K || DT == KQ_Q5_K;
    const uint4 hv = *reinterpret_cast<const uint4 *>(chunk + (K4 ? 2048 : 3072) + r * 16);
    // per-sub-block scales: Q4_K/Q5_K four 6-bit scales per word, Q6_K four int8 scales per word
    uint32_t scw[4], mw[2];
    if (K4) {
        scw[0] = hv.y & 0x3f3f3f3fu;
        scw[1] = (hv.w & 0x0f0f0f0fu) | ((hv.y >> 2) & 0x30303030u);
        mw[0] = hv.z & 0x3f3f3f3fu;
        mw[1] = ((hv.w >> 4) & 0x0f0f0f0fu) | ((hv.z >> 2) & 0x30303030u);
        scw[2] = scw[3] = 0u;
    } else {
        scw[0] = hv.x; scw[1] = hv.y; scw[2] = hv.z; scw[3] = hv.w;
        mw[0] = mw[1] = 0u;
    }
    uint32_t q5h[8];
    if (DT == KQ_Q5_K) {
        const uint4 a = *reinterpret_cast<const uint4 *>(chunk + 2304 + r * 32);
        const uint4 b = *reinterpret_cast<const uint4 *>(chunk + 2304 + r * 32 + 16);
        q5h[0] = a.x; q5h[1] = a.y; q5h[2] = a.z; q5h[3] = a.w; q5h[4] = b.x; q5h[5] = b.y; q5h[6] = b.z; q5h[7] = b.w;
    }
    int sumi[MC];
#pragma unroll
    for (int m = 0; m < MC; ++m) sumi[m] = 0;
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
        const uint4 v0 = *reinterpret_cast<const uint4 *>(chunk + kb * 512 + r * 32);
        const uint4 v1 = *reinterpret_cast<const uint4 *>(chunk + kb * 512 + r * 32 + 16);
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint32_t hb[4] = {0u, 0u, 0u, 0u};
        if (DT == KQ_Q6_K) {
            const uint4 h = *reinterpret_cast<const uint4 *>(chunk + 2048 + kb * 256 + r * 16);
            hb[0] = h.x; hb[1] = h.y; hb[2] = h.z; hb[3] = h.w;
        }
        // the kblock's words unpacked once: lo = codes of the first 32 elements, hi = of the last 32
        // (Q4_K: 16*c left in place)
        uint32_t lo[8], hi[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int seg = i >> 2;
            lo[i] = w[i] & 0x0f0f0f0fu;
            if (DT == KQ_Q4_K) {
                hi[i] = w[i] & 0xf0f0f0f0u;
            } else if (DT == KQ_Q5_K) {
                lo[i] |= ((q5h[i] >> (2 * kb)) & 0x01010101u) << 4;
                hi[i] = ((w[i] >> 4) & 0x0f0f0f0fu) | (((q5h[i] >> (2 * kb + 1)) & 0x01010101u) << 4);
            } else {
                lo[i] |= ((hb[i & 3] >> (2 * seg)) & 0x03030303u) << 4;
                hi[i] = ((w[i] >> 4) & 0x0f0f0f0fu) | (((hb[i & 3] >> (4 + 2 * seg)) & 0x03030303u) << 4);
            }
        }
#pragma unroll
        for (int m = 0; m < MC; ++m) {
            if (m >= M) break;
            const int8_t *qm = reinterpret_cast<const int8_t *>(q + m * xb) + 64 * kb;
            const int4 qa0 = *reinterpret_cast<const int4 *>(qm);
            const int4 qa1 = *reinterpret_cast<const int4 *>(qm + 16);
            const int4 qb0 = *reinterpret_cast<const int4 *>(qm + 32);
            const int4 qb1 = *reinterpret_cast<const int4 *>(qm + 48);
            const int ql[8] = {qa0.x, qa0.y, qa0.z, qa0.w, qa1.x, qa1.y, qa1.z, qa1.w};
            const int qh[8] = {qb0.x, qb0.y, qb0.z, qb0.w, qb1.x, qb1.y, qb1.z, qb1.w};
            int plo[2] = {0, 0}, phi[2] = {0, 0};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                plo[i >> 2] = dp4a((int)lo[i], ql[i], plo[i >> 2]);
                phi[i >> 2] = DT == KQ_Q4_K ? dp4a_us(hi[i], qh[i], phi[i >> 2]) : dp4a((int)hi[i], qh[i], phi[i >> 2]);
            }
            if (K4) {  // sub-blocks 2kb (lo) and 2kb+1 (hi)
                const int s_lo = (int)((scw[kb >> 1] >> (16 * (kb & 1))) & 0xff);
                const int s_hi = (int)((scw[kb >> 1] >> (16 * (kb & 1) + 8)) & 0xff);
                const int ph = DT == KQ_Q4_K ? (phi[0] + phi[1]) >> 4 : phi[0] + phi[1];
                sumi[m] += s_lo * (plo[0] + plo[1]) + s_hi * ph;
            } else {  // sub-blocks 4kb .. 4kb+3, sum c*q (the -32 offset below)
                sumi[m] += sext8(scw[kb], 0) * plo[0] + sext8(scw[kb], 1) * plo[1] + sext8(scw[kb], 2) * phi[0] +
                           sext8(scw[kb], 3) * phi[1];
            }
        }
    }
    const float dw = K4 ? half_bits_to_float((uint16_t)(hv.x & 0xffff))
                        : half_bits_to_float(*reinterpret_cast<const uint16_t *>(chunk + 3328 + r * 2));
    const float dmin = K4 ? half_bits_to_float((uint16_t)(hv.x >> 16)) : 0.0f;
#pragma unroll
    for (int m = 0; m < MC; ++m) {
        if (m >= M) break;
        const uint8_t *xm = q + m * xb;
        const uint4 b0 = *reinterpret_cast<const uint4 *>(xm + 288);
        const uint4 b1 = *reinterpret_cast<const uint4 *>(xm + 304);
        const uint32_t bw[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        const float a = *reinterpret_cast<const float *>(xm + 256);
        if (K4) {
            int summ = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                summ = dp2a_lo_su(bw[j], __byte_perm(mw[j >> 2], 0u, 0x4400u | ((j & 3) * 0x11u)), summ);
            const float t1 = __fmul_rn(a, dw);
            const float t2 = __fmul_rn(t1, (float)sumi[m]);
            const float t3 = __fmul_rn(a, dmin);
            const float t4 = __fmul_rn(t3, (float)summ);
            term[m * tstep] = __fsub_rn(t2, t4);
        } else {
            int sumb = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                sumb = dp2a_lo_ss(bw[2 * k], scw[k], sumb);
                sumb = dp2a_hi_ss(bw[2 * k + 1], scw[k], sumb);
            }
            const float t1 = __fmul_rn(a, dw);
            term[m * tstep] = __fmul_rn(t1, (float)(sumi[m] - 32 * sumb));
        }
    }
}

// Stage the Q8_K blocks of M <= MC activation columns (column m's block at src + m*src_stride) into
// shared memory at dst + m*xb in the layout the dot reads (int8 q[256], f32 d at +256, int16 bsums at
// +288).  Every column's loads are issued before the first store, so the warp waits for one memory
// round trip instead of one per column.
template <int MC>
__device__ __forceinline__ void stage_q8k_cols(const uint8_t *__restrict__ src, int64_t src_stride, int M,
                                               uint8_t *__restrict__ dst, int xb) {
    const int lane = threadIdx.x & 31;
    uint32_t a[MC], b[MC];
    int16_t bsv[MC];
    float dv[MC];
#pragma unroll
    for (int m = 0; m < MC; ++m) {
        if (m < M) {
            const uint8_t *blk = src + m * src_stride;
            const uint32_t *q32 = reinterpret_cast<const uint32_t *>(blk + 4);
            a[m] = q32[2 * lane];
            b[m] = q32[2 * lane + 1];
            bsv[m] = reinterpret_cast<const int16_t *>(blk + 260)[lane & 15];
            dv[m] = *reinterpret_cast<const float *>(blk);
        }
    }
#pragma unroll
    for (int m = 0; m < MC; ++m) {
        if (m < M) {
            uint8_t *d = dst + m * xb;
            reinterpret_cast<uint2 *>(d)[lane] = make_uint2(a[m], b[m]);
            if (lane < 16) reinterpret_cast<int16_t *>(d + 288)[lane] = bsv[m];
            if (lane == 0) *reinterpret_cast<float *>(d + 256) = dv[m];
        }
    }
}

// grid: (S, ceil(N/32)); cluster (S, 1, 1) when S > 1; block: 32 * cpr threads.  Warp w of cluster
// rank k owns chunk k*cpr + w for all 32 rows of the block (lane = row): it bulk-copies that chunk's
// codes for the block's two row groups into its own shared region, quantises (or copies) the
// chunk's activation there, and forms the 32 rows' terms.  No warp waits for another until the
// final ordered reduction.  MC > 1 (batched decode, M <= MC activation rows given quantised): the
// staged weight chunk serves every activation column; each (row, column) output is formed exactly as
// for one column.  y[m*ldy + n].
template <int DT, bool FUSED, int MC>
__global__ void __launch_bounds__(kGemvRows * kGemvMaxWarps) gemv_kernel(const uint8_t *__restrict__ w,
                                                                         const float *__restrict__ x,
                                                                         const uint8_t *__restrict__ xq,
                                                                         int64_t N, int nchunk, int cpr,
                                                                         float *__restrict__ y, int M,
                                                                         int64_t ldy) {
    static_assert(!FUSED || MC == 1, "the fused quantise prologue takes one activation column");
    using Tr = GemvTraits<DT>;
    using WS = GemvWarpSmem<DT, MC>;
    constexpr int CB = chunk_bytes(DT);
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t bars[kGemvMaxWarps];
    __shared__ uint64_t gather_bar;  // cluster rank 0: one arrival per other rank once its terms landed
    __shared__ int abort_flag;
    const int S = gridDim.x;
    const int rank = blockIdx.x;
    const int64_t rb = blockIdx.y;                   // 32-row block = row groups 2rb, 2rb+1
    const int64_t groups_total = (N + 15) / 16;
    const int64_t g0 = rb * 2;
    const int ngroups = (int)min((int64_t)2, groups_total - g0);
    const int c_begin = rank * cpr;
    const int nloc = max(0, min(nchunk, c_begin + cpr) - c_begin);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tstride = MC * cpr * Tr::terms;  // a row's terms: [column][local chunk][term]
    // Eight K-quant columns and no cluster: a lane's terms go into the 32 bytes of its row's first-
    // kblock codes (read by that lane alone, and read by then) instead of the terms buffer, which
    // lets a third block share the SM
    const bool inplace = MC == 8 && !Tr::q81 && S == 1;
    // shared layout: per-warp buffers [cpr][WS] | terms [32][tstride] | (S > 1) gather [S-1][32][tstride]
    float *terms = reinterpret_cast<float *>(smem + (size_t)cpr * WS::BYTES);
    float *gather = terms + kGemvRows * tstride;

    // Let the next kernel in the stream get scheduled; it waits on this grid before touching memory.
    // Fed a quantised row, the trigger goes first (measured: the pre-quantised Q4_K [9728 x 2560] call
    // 10% faster); with the fused quantizer it goes after the set-up (there, first was 2% slower).
    if (!FUSED) grid_launch_dependents();
    if (threadIdx.x == 0) {
        for (int i = 0; i < cpr; ++i) mbar_init(&bars[i], 1);
        if (S > 1) mbar_init(&gather_bar, S - 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (S > 1) cluster_arrive_relaxed();  // "my barriers are initialised"; waited for before any remote access
    if (FUSED) grid_launch_dependents();

    const bool active = warp < nloc;
    const int c = c_begin + warp;
    uint8_t *ws = smem + (size_t)warp * WS::BYTES;
    // The weight is staged once and never written by the kernel that runs just before this one in
    // the stream, so its copy starts before the dependency wait and overlaps that kernel's tail.
    if (active && lane == 0) {
        mbar_arrive_expect_tx(&bars[warp], ngroups * CB);
        for (int gi = 0; gi < ngroups; ++gi)
            bulk_load(ws + gi * CB, w + ((g0 + gi) * nchunk + c) * (int64_t)CB, CB, &bars[warp]);
    }
    // Everything below reads memory (the activation) that an earlier kernel may have written.
    grid_dependency_wait();
    if (active) {
        int8_t *q_s = reinterpret_cast<int8_t *>(ws + WS::Q_OFF);
        float *da_s = reinterpret_cast<float *>(ws + WS::D_OFF);
        int16_t *bs_s = reinterpret_cast<int16_t *>(ws + WS::B_OFF);
        if (MC > 1) {
            // batched decode: column m's chunk c is block (m, c) of the quantised activation rows
            if (!Tr::q81) {
                stage_q8k_cols<MC>(xq + (int64_t)c * kQ8KBytes, (int64_t)nchunk * kQ8KBytes, M,
                                   reinterpret_cast<uint8_t *>(q_s), WS::XB);
            } else {
                for (int m = 0; m < M; ++m) {
                    int8_t *qm = q_s + m * WS::XB;
                    float *dm = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(da_s) + m * WS::XB);
                    const int b = lane >> 2, part = lane & 3;  // 8 blocks x 4 lanes
                    const uint8_t *blk = xq + (((int64_t)m * nchunk + c) * 8 + b) * kQ81Bytes;
                    const uint32_t *src = reinterpret_cast<const uint32_t *>(blk + 4 + 8 * part);
                    reinterpret_cast<uint2 *>(qm + 32 * b)[part] = make_uint2(src[0], src[1]);
                    if (part == 0) dm[b] = half_bits_to_float(*reinterpret_cast<const uint16_t *>(blk));
                }
            }
        } else if (FUSED) {
            if (!Tr::q81) {
                warp_quantize_q8k_smem(x + (int64_t)c * 256, q_s, da_s, bs_s);
            } else {
                warp_quantize_q8_1x4_smem(x + (int64_t)c * 256, q_s, da_s);
                warp_quantize_q8_1x4_smem(x + (int64_t)c * 256 + 128, q_s + 128, da_s + 4);
            }
        } else if (!Tr::q81) {
            const uint8_t *blk = xq + (int64_t)c * kQ8KBytes;
            const uint32_t *src = reinterpret_cast<const uint32_t *>(blk + 4);
            reinterpret_cast<uint2 *>(q_s)[lane] = make_uint2(src[2 * lane], src[2 * lane + 1]);
            if (lane < 16) bs_s[lane] = reinterpret_cast<const int16_t *>(blk + 260)[lane];
            if (lane == 0) da_s[0] = *reinterpret_cast<const float *>(blk);
        } else {
            const int b = lane >> 2, part = lane & 3;  // 8 blocks x 4 lanes
            const uint8_t *blk = xq + ((int64_t)c * 8 + b) * kQ81Bytes;
            const uint32_t *src = reinterpret_cast<const uint32_t *>(blk + 4 + 8 * part);  // 4-byte aligned
            reinterpret_cast<uint2 *>(q_s + 32 * b)[part] = make_uint2(src[0], src[1]);
            if (part == 0) da_s[b] = half_bits_to_float(*reinterpret_cast<const uint16_t *>(blk));
        }
        __syncwarp();
        if (mbar_wait_sleep(&bars[warp], 0, &abort_flag)) {
            const int gi = lane >> 4;
            if (gi < ngroups) {
                if (MC > 1 && DT != KQ_Q8_0)  // several columns: each weight word unpacked once for all
                    gemv_row_chunk_mc<DT, MC>(ws + gi * CB, lane & 15, reinterpret_cast<const uint8_t *>(q_s), WS::XB, M,
                                              inplace ? reinterpret_cast<float *>(ws + gi * CB + (lane & 15) * 32)
                                                      : terms + lane * tstride + warp * Tr::terms,
                                              inplace ? 1 : cpr * Tr::terms);
                else
                    for (int m = 0; m < (MC > 1 ? M : 1); ++m)
                        gemv_row_chunk<DT>(ws + gi * CB, lane & 15, q_s + m * WS::XB,
                                           reinterpret_cast<const float *>(reinterpret_cast<const uint8_t *>(da_s) + m * WS::XB),
                                           reinterpret_cast<const int16_t *>(reinterpret_cast<const uint8_t *>(bs_s) + m * WS::XB),
                                           terms + lane * tstride + (m * cpr + warp) * Tr::terms);
            }
        } else if (lane == 0) {
            int no_abort = 0;  // drain this warp's copies (bounded) before the block may exit
            mbar_wait(&bars[warp], 0, &no_abort, 100000000ull);
        }
    }

    // ---- ordered reduction: one thread per row adds the row's terms in ascending K order
    const int ncol = MC > 1 ? M : 1;
    if (S == 1) {
        __syncthreads();
        for (int t = threadIdx.x; t < kGemvRows * ncol; t += blockDim.x) {
            // in place, column fastest: a warp's reads of one chunk then cover whole 32-byte rows
            const int r = inplace ? t / ncol : t & (kGemvRows - 1), m = inplace ? t % ncol : t / kGemvRows;
            const int64_t n = rb * kGemvRows + r;
            float acc = 0.0f;
            if (inplace) {
                // chunk i's terms for row r: warp i's buffer, row group r/16, row r%16's first code bytes
                for (int i = 0; i < nloc; ++i)
                    acc = __fadd_rn(acc, reinterpret_cast<const float *>(smem + (size_t)i * WS::BYTES + (r >> 4) * CB +
                                                                       (r & 15) * 32)[m]);
            } else {
                const float *tr = terms + r * tstride + m * cpr * Tr::terms;
                for (int i = 0; i < nloc * Tr::terms; ++i) acc = __fadd_rn(acc, tr[i]);
            }
            if (n < N) y[m * ldy + n] = abort_flag ? __int_as_float(0x7fc00000) : acc;
        }
    } else {
        // Every rank pushes its terms into rank 0's gather buffer and signals rank 0's barrier; only
        // rank 0 waits, then adds each row's terms in ascending K order.
        cg::cluster_group cluster = cg::this_cluster();
        cluster_wait();  // every CTA of the cluster has initialised its barriers
        __syncthreads();
        const int per = kGemvRows * tstride;
        if (rank != 0) {
            float *dst = cluster.map_shared_rank(gather, 0) + (size_t)(rank - 1) * per;
            for (int i = threadIdx.x; i < per; i += blockDim.x) dst[i] = terms[i];
            fence_acq_rel_cluster();
            __syncthreads();
            if (threadIdx.x == 0) {
                if (abort_flag) *cluster.map_shared_rank(&abort_flag, 0) = 1;
                fence_acq_rel_cluster();
                mbar_arrive_remote(&gather_bar, 0);
            }
        } else {
            const bool got = mbar_wait_sleep(&gather_bar, 0, &abort_flag);
            for (int t = threadIdx.x; t < kGemvRows * ncol; t += blockDim.x) {
                const int r = t & (kGemvRows - 1), m = t / kGemvRows;
                const int64_t n = rb * kGemvRows + r;
                float acc = 0.0f;
                for (int k = 0; k < S; ++k) {
                    const int kb = k * cpr, ke = min(nchunk, kb + cpr);
                    const int cnt = max(0, ke - kb) * Tr::terms;
                    const float *src = (k == 0 ? terms : gather + (size_t)(k - 1) * per) + r * tstride + m * cpr * Tr::terms;
                    for (int i = 0; i < cnt; ++i) acc = __fadd_rn(acc, src[i]);
                }
                if (n < N) y[m * ldy + n] = (!got || abort_flag) ? __int_as_float(0x7fc00000) : acc;
            }
        }
    }
}

// Long-K GEMV without a cluster: one block per 16-row group over the whole of K.  grid: ceil(N/16);
// block: 32 * ceil(nchunk/2) threads (at most kGemv16MaxWarps warps).  Warp w stages chunks 2w and 2w+1 of the group (one bulk copy
// each) and their activation blocks; half-warp h (lane >> 4) then forms the terms of chunk 2w+h, a
// lane per row (lane & 15), exactly as gemv_kernel does, and one thread per row adds the row's terms
// in ascending K order.  Every block covers its rows over the whole K, so no partial sums cross
// blocks and the launch needs no cluster: the next call's blocks start beside it under programmatic
// dependent launch, and with 16 rows per block the blocks of a 2560-row GEMV cover every SM.
template <int DT, bool FUSED>
__global__ void __launch_bounds__(32 * kGemv16MaxWarps, 2) gemv16_kernel(const uint8_t *__restrict__ w,
                                                                           const float *__restrict__ x,
                                                                           const uint8_t *__restrict__ xq,
                                                                           int64_t N, int nchunk,
                                                                           float *__restrict__ y) {
    using Tr = GemvTraits<DT>;
    using WS = GemvWarpSmem<DT, 2>;  // two chunks' codes (one row group each) and two activation blocks
    constexpr int CB = chunk_bytes(DT);
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t bars[kGemvMaxWarps];
    __shared__ int abort_flag;
    const int64_t g = blockIdx.x;  // row group: rows 16g .. 16g+15
    const int nw = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tstride = nchunk * Tr::terms;
    float *terms = reinterpret_cast<float *>(smem + (size_t)nw * WS::BYTES);  // [16][nchunk][terms]

    if (threadIdx.x == 0) {
        for (int i = 0; i < nw; ++i) mbar_init(&bars[i], 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    grid_launch_dependents();

    const int c0 = 2 * warp, nc = min(2, nchunk - c0);
    uint8_t *ws = smem + (size_t)warp * WS::BYTES;
    // the weights are never written by the kernel before this one: their copies start before the wait
    if (lane == 0) {
        mbar_arrive_expect_tx(&bars[warp], nc * CB);
        for (int h = 0; h < nc; ++h) bulk_load(ws + h * CB, w + (g * nchunk + c0 + h) * (int64_t)CB, CB, &bars[warp]);
    }
    grid_dependency_wait();
    // a pre-quantised row: both chunks' Q8_K blocks staged with every load issued before the first store
    if (!FUSED && !Tr::q81)
        stage_q8k_cols<2>(xq + (int64_t)c0 * kQ8KBytes, kQ8KBytes, nc, ws + WS::Q_OFF, WS::XB);
    for (int h = 0; h < nc && (FUSED || Tr::q81); ++h) {
        int8_t *q_s = reinterpret_cast<int8_t *>(ws + WS::Q_OFF + h * WS::XB);
        float *da_s = reinterpret_cast<float *>(ws + WS::D_OFF + h * WS::XB);
        int16_t *bs_s = reinterpret_cast<int16_t *>(ws + WS::B_OFF + h * WS::XB);
        const int c = c0 + h;
        if (FUSED) {
            if (!Tr::q81) {
                warp_quantize_q8k_smem(x + (int64_t)c * 256, q_s, da_s, bs_s);
            } else {
                warp_quantize_q8_1x4_smem(x + (int64_t)c * 256, q_s, da_s);
                warp_quantize_q8_1x4_smem(x + (int64_t)c * 256 + 128, q_s + 128, da_s + 4);
            }
        } else {
            const int b = lane >> 2, part = lane & 3;  // 8 blocks x 4 lanes
            const uint8_t *blk = xq + ((int64_t)c * 8 + b) * kQ81Bytes;
            const uint32_t *src = reinterpret_cast<const uint32_t *>(blk + 4 + 8 * part);
            reinterpret_cast<uint2 *>(q_s + 32 * b)[part] = make_uint2(src[0], src[1]);
            if (part == 0) da_s[b] = half_bits_to_float(*reinterpret_cast<const uint16_t *>(blk));
        }
    }
    __syncwarp();
    if (mbar_wait_sleep(&bars[warp], 0, &abort_flag)) {
        const int h = lane >> 4;
        if (h < nc)
            gemv_row_chunk<DT>(ws + h * CB, lane & 15, reinterpret_cast<const int8_t *>(ws + WS::Q_OFF + h * WS::XB),
                               reinterpret_cast<const float *>(ws + WS::D_OFF + h * WS::XB),
                               reinterpret_cast<const int16_t *>(ws + WS::B_OFF + h * WS::XB),
                               terms + (lane & 15) * tstride + (c0 + h) * Tr::terms);
    } else if (lane == 0) {
        int no_abort = 0;  // drain this warp's copies (bounded) before the block may exit
        mbar_wait(&bars[warp], 0, &no_abort, 100000000ull);
    }
    __syncthreads();
    if (threadIdx.x < 16) {  // ordered reduction: one thread per row, ascending K
        const int64_t n = g * 16 + threadIdx.x;
        const float *tr = terms + threadIdx.x * tstride;
        float acc = 0.0f;
        for (int i = 0; i < tstride; ++i) acc = __fadd_rn(acc, tr[i]);
        if (n < N) y[n] = abort_flag ? __int_as_float(0x7fc00000) : acc;
    }
}

// Batched long-K decode (M <= MC pre-quantised activation rows, K-quant weights) without a cluster:
// one block per 16-row group over the whole K, as gemv16_kernel, with every staged weight chunk dotted
// against all M columns (gemv_row_chunk_mc: each weight word unpacked once).  Warp w stages chunks 2w
// and 2w+1 of the group (one bulk copy each) and their M activation blocks; half-warp h forms the
// terms of chunk 2w+h for its 16 rows, and one thread per (row, column) adds that column's terms in
// ascending K order -- every output formed exactly as for one column.  A lane's M terms for its chunk
// go into the 32 bytes of that row's first kblock codes, which only that lane reads and has read by
// then, so the terms need no shared memory of their own; y[m*ldy + n].  Q4_K with two columns keeps
// to two blocks per SM (registers and shared memory), so the next call's blocks can start beside it.
template <int DT, int MC>
__global__ void __launch_bounds__(32 * kGemv16MaxWarps, (MC == 2 && DT == KQ_Q4_K) ? 2 : 1) gemv16_mc_kernel(const uint8_t *__restrict__ w,
                                                                              const uint8_t *__restrict__ xq,
                                                                              int64_t N, int nchunk,
                                                                              float *__restrict__ y, int M,
                                                                              int64_t ldy) {
    constexpr int CB = chunk_bytes(DT);
    constexpr int XB = GemvWarpSmem<DT, 1>::XB;    // one column's activation block: q[256], d, bsums
    constexpr int WB = 2 * CB + 2 * MC * XB;       // per warp: two chunks' codes, then their activations
    static_assert(MC * 4 <= 32, "a row's terms fit its first kblock's 32 code bytes");
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t bars[kGemvMaxWarps];
    __shared__ int abort_flag;
    const int64_t g = blockIdx.x;  // row group: rows 16g .. 16g+15
    const int nw = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < nw; ++i) mbar_init(&bars[i], 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    grid_launch_dependents();

    const int c0 = 2 * warp, nc = min(2, nchunk - c0);
    uint8_t *ws = smem + (size_t)warp * WB;
    // the weights are never written by the kernel before this one: their copies start before the wait
    if (lane == 0) {
        mbar_arrive_expect_tx(&bars[warp], nc * CB);
        for (int h = 0; h < nc; ++h) bulk_load(ws + h * CB, w + (g * nchunk + c0 + h) * (int64_t)CB, CB, &bars[warp]);
    }
    grid_dependency_wait();
    // column m's chunk c is Q8_K block (m, c) of the activation rows
    for (int h = 0; h < nc; ++h)
        stage_q8k_cols<MC>(xq + (int64_t)(c0 + h) * kQ8KBytes, (int64_t)nchunk * kQ8KBytes, M, ws + 2 * CB + h * MC * XB,
                           XB);
    __syncwarp();
    if (mbar_wait_sleep(&bars[warp], 0, &abort_flag)) {
        const int h = lane >> 4;
        if (h < nc)
            gemv_row_chunk_mc<DT, MC>(ws + h * CB, lane & 15, ws + 2 * CB + h * MC * XB, XB, M,
                                      reinterpret_cast<float *>(ws + h * CB + (lane & 15) * 32), 1);
    } else if (lane == 0) {
        int no_abort = 0;  // drain this warp's copies (bounded) before the block may exit
        mbar_wait(&bars[warp], 0, &no_abort, 100000000ull);
    }
    __syncthreads();
    for (int t = threadIdx.x; t < 16 * M; t += blockDim.x) {  // ordered reduction: one thread per (row, column)
        const int r = t & 15, m = t >> 4;
        const int64_t n = g * 16 + r;
        float acc = 0.0f;
        for (int i = 0; i < nchunk; ++i)  // chunk i's terms: warp i/2's buffer, chunk slot i%2, row r
            acc = __fadd_rn(acc, reinterpret_cast<const float *>(smem + (size_t)(i >> 1) * WB + (i & 1) * CB + r * 32)[m]);
        if (n < N) y[m * ldy + n] = abort_flag ? __int_as_float(0x7fc00000) : acc;
    }
}

// Number of SMs of the current device (looked up once per device).
static int gemv_sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
        cache[dev] = n;
    }
    return cache[dev];
}

template <int DT, bool FUSED, int MC>
static kq_status launch_gemv(const uint8_t *w, const float *x, const uint8_t *xq, int64_t N, int64_t K, float *y,
                             cudaStream_t st, int M = 1, int64_t ldy = 0) {
    using Tr = GemvTraits<DT>;
    using WS = GemvWarpSmem<DT, MC>;
    const int nchunk = (int)(K / 256);
    const int64_t rblocks = (N + kGemvRows - 1) / kGemvRows;
    // Smallest power-of-two cluster split (at most 8) with at most 32 chunks per block.
    int S = 1;
    while (S < 8 && (nchunk + S - 1) / S > kGemvMaxWarps) S *= 2;
    if ((nchunk + S - 1) / S > kGemvMaxWarps)
        return fail(KQ_ERR_INVALID_ARG, "kq_gemv: K=%lld too large (at most %d)", (long long)K,
                    8 * kGemvMaxWarps * 256);
    // Then split further only while the blocks do not cover the SMs once, or a block needs more shared
    // memory than lets two of them share an SM (measured on the decode shapes: fewer, larger blocks
    // shorten each call's dependent chain, as long as the next call's blocks can still start beside
    // them), keeping >= 5 chunks per block.
    auto smem_for = [&](int s) {
        const int c = (nchunk + s - 1) / s;
        // no terms buffer where the kernel keeps eight K-quant columns' terms in place (no cluster)
        const bool inplace = MC == 8 && !Tr::q81 && s == 1;
        return (size_t)c * WS::BYTES + (inplace ? 0 : (size_t)s * kGemvRows * c * Tr::terms * MC * 4);
    };
    while (S < 8 && (rblocks * S < gemv_sm_count() || smem_for(S) > 112 * 1024) && (nchunk + 2 * S - 1) / (2 * S) >= 5)
        S *= 2;
    while (S < 8 && smem_for(S) > 220 * 1024) S *= 2;  // several activation columns need more room
    const int cpr = (nchunk + S - 1) / S;
    const size_t smem = smem_for(S);
    if (smem > 220 * 1024) return fail(KQ_ERR_INVALID_ARG, "kq_gemv: K=%lld too large", (long long)K);
    if (ldy == 0) ldy = N;
    if (rblocks > 65535) return fail(KQ_ERR_INVALID_ARG, "kq_gemv: N=%lld too large", (long long)N);
    if (MC == 1 && S > 1 && GEMV16_OK) {
        // one column whose K the cluster split would share out: 16-row blocks over the whole K
        // instead, when they fit (at most 40 chunks, the row group's whole K in shared memory)
        using WS2 = GemvWarpSmem<DT, 2>;
        const int nw = (nchunk + 1) / 2;
        const size_t smem16 = (size_t)nw * WS2::BYTES + (size_t)16 * nchunk * Tr::terms * 4;
        const int64_t groups = (N + 15) / 16;
        // only where two calls' blocks fit on an SM together: otherwise the next call cannot start
        // beside this one and the cluster split, with less post-wait work per warp, is as fast
        if (nw <= kGemv16MaxWarps && 2 * smem16 <= 220 * 1024 && groups <= 0x7fffffff) {
            auto k16 = gemv16_kernel<DT, FUSED>;
            cudaError_t e = cudaFuncSetAttribute(k16, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem16);
            if (e != cudaSuccess) return fail(KQ_ERR_CUDA, "kq_gemv: %s", cudaGetErrorString(e));
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)groups, 1, 1);
            cfg.blockDim = dim3(32 * nw, 1, 1);
            cfg.dynamicSmemBytes = smem16;
            cfg.stream = st;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            e = cudaLaunchKernelEx(&cfg, k16, w, x, xq, N, nchunk, y);
            if (e != cudaSuccess) return fail(KQ_ERR_CUDA, "kq_gemv: launch failed: %s", cudaGetErrorString(e));
            count_launch(R_GEMV);
            return KQ_OK;
        }
    }
    if constexpr (MC > 1 && DT != KQ_Q8_0) if (S > 1 && GEMV16_OK) {
        // several columns whose K the cluster split would share out: 16-row blocks over the whole K
        // instead (no cluster), one per SM, where the group's whole K and its activations fit
        constexpr int WB = 2 * chunk_bytes(DT) + 2 * MC * GemvWarpSmem<DT, 1>::XB;
        const int nw = (nchunk + 1) / 2;
        const size_t smem16 = (size_t)nw * WB;
        const int64_t groups = (N + 15) / 16;
        if (nw <= kGemv16MaxWarps && smem16 <= 226 * 1024 && groups <= 0x7fffffff) {
            auto k16 = gemv16_mc_kernel<DT, MC>;
            cudaError_t e = cudaFuncSetAttribute(k16, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem16);
            if (e != cudaSuccess) return fail(KQ_ERR_CUDA, "kq_gemv: %s", cudaGetErrorString(e));
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)groups, 1, 1);
            cfg.blockDim = dim3(32 * nw, 1, 1);
            cfg.dynamicSmemBytes = smem16;
            cfg.stream = st;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            e = cudaLaunchKernelEx(&cfg, k16, w, xq, N, nchunk, y, M, ldy);
            if (e != cudaSuccess) return fail(KQ_ERR_CUDA, "kq_gemv: launch failed: %s", cudaGetErrorString(e));
            count_launch(R_GEMV);
            return KQ_OK;
        }
    }
    auto kern = gemv_kernel<DT, FUSED, MC>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(KQ_ERR_CUDA, "kq_gemv: %s", cudaGetErrorString(e));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S, (unsigned)rblocks, 1);
    cfg.blockDim = dim3(32 * cpr, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (S > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = S;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    e = cudaLaunchKernelEx(&cfg, kern, w, x, xq, N, nchunk, cpr, y, M, ldy);
    if (e != cudaSuccess) return fail(KQ_ERR_CUDA, "kq_gemv: launch failed: %s", cudaGetErrorString(e));
    count_launch(R_GEMV);
    return KQ_OK;
}

template <int DT>
static kq_status gemv_batched_dt(const uint8_t *w, const uint8_t *xq, int64_t M, int64_t N, int64_t K, float *y,
                                 int64_t ldy, cudaStream_t st) {
    if (M == 1) return launch_gemv<DT, false, 1>(w, nullptr, xq, N, K, y, st, 1, ldy);
    if (M == 2) return launch_gemv<DT, false, 2>(w, nullptr, xq, N, K, y, st, (int)M, ldy);
    if (M <= 4) return launch_gemv<DT, false, 4>(w, nullptr, xq, N, K, y, st, (int)M, ldy);
    return launch_gemv<DT, false, 8>(w, nullptr, xq, N, K, y, st, (int)M, ldy);
}

// Batched decode (1 <= M <= kGemvMaxBatch quantised activation rows): the GEMV with every staged
// weight chunk serving all M columns.  Returns KQ_ERR_INVALID_ARG when the shape does not fit the
// kernel's shared memory (the caller then takes the general path).
kq_status gemv_batched(kq_dtype wt, const uint8_t *w, const uint8_t *xq, int64_t M, int64_t N, int64_t K, float *y,
                       int64_t ldy, cudaStream_t st) {
    if (M < 1 || M > kGemvMaxBatch) return fail(KQ_ERR_INVALID_ARG, "gemv_batched: M=%lld", (long long)M);
    switch (wt) {
    case KQ_Q4_K: return gemv_batched_dt<KQ_Q4_K>(w, xq, M, N, K, y, ldy, st);
    case KQ_Q5_K: return gemv_batched_dt<KQ_Q5_K>(w, xq, M, N, K, y, ldy, st);
    case KQ_Q6_K: return gemv_batched_dt<KQ_Q6_K>(w, xq, M, N, K, y, ldy, st);
    default: return gemv_batched_dt<KQ_Q8_0>(w, xq, M, N, K, y, ldy, st);
    }
}

}  // namespace kq

using namespace kq;

extern "C" kq_status kq_gemv(kq_dtype wt, const void *w, const float *x, const void *xq, int64_t N, int64_t K,
                             float *y, kq_stream_t stream) {
    if (wt != KQ_Q4_K && wt != KQ_Q5_K && wt != KQ_Q6_K && wt != KQ_Q8_0)
        return fail(KQ_ERR_UNSUPPORTED_DTYPE, "kq_gemv: weight dtype %s is not Q4_K, Q5_K, Q6_K or Q8_0",
                    dtype_name(wt));
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
    case KQ_Q4_K: return x ? launch_gemv<KQ_Q4_K, true, 1>(wb, x, xb, N, K, y, st) : launch_gemv<KQ_Q4_K, false, 1>(wb, x, xb, N, K, y, st);
    case KQ_Q5_K: return x ? launch_gemv<KQ_Q5_K, true, 1>(wb, x, xb, N, K, y, st) : launch_gemv<KQ_Q5_K, false, 1>(wb, x, xb, N, K, y, st);
    case KQ_Q6_K: return x ? launch_gemv<KQ_Q6_K, true, 1>(wb, x, xb, N, K, y, st) : launch_gemv<KQ_Q6_K, false, 1>(wb, x, xb, N, K, y, st);
    default: return x ? launch_gemv<KQ_Q8_0, true, 1>(wb, x, xb, N, K, y, st) : launch_gemv<KQ_Q8_0, false, 1>(wb, x, xb, N, K, y, st);
    }
}
