// kq_tc.cu -- tensor-core prefill GEMM for Q4_K / Q6_K weights x Q8_K activations on sm_103a.
//
// sm_103a has no integer tcgen05 MMA, so the integer block dots are carried EXACTLY on the f16
// tensor pipe (tcgen05.mma kind::f16, fp32 accumulation in TMEM):
//   * activation codes q (|q| <= 127) are exact in f16; a prologue writes them as an f16 panel that
//     TMA loads with 128-byte swizzle.  One activation tile is staged per CTA and shared by every
//     MMA of the CTA (the cooperative activation share of vllm.cpp PR #3035).
//   * weights stay packed in HBM; converter warps unpack one 64-element kblock at a time in shared
//     memory into the integer products sc_j*c (Q4_K, <= 945) or, for Q6_K, into two tiles
//     lo = (sc & 15)*(c-32) and hi = (sc >> 4)*(c-32) (|.| <= 480), all exact in f16.
//   * each super-block (256 elements) accumulates into its own TMEM tile: the sums are integers
//     below 2^24 for any realistic input, so the fp32 accumulator holds them exactly.  Q4_K's min
//     term sum_j m_j*bsum is a 16-wide extension MMA (bsums and mins are exact in f16) into a second
//     tile; Q6_K's second tile holds the hi half, recombined exactly as lo + 16*hi.
//   * epilogue warps promote each super-block to fp32 while the MMA warp fills the other TMEM
//     buffer: acc += d_a*(d_w*S1 - dmin*S2) (Q4_K) or acc += d_a*d_w*(S_lo + 16*S_hi) (Q6_K).
// The integer parts are therefore the oracle's integers; only the fp32 scaling uses fused
// multiply-adds, which keeps the result within a few ulps of the sequential CPU order.
//
// Roles (448 threads): warps 0-7 epilogue (TMEM lane quarter = warp % 4, column half = warp / 4),
// warps 8-11 weight converters, warp 12 TMA producer, warp 13 MMA issuer and TMEM owner.
// Waiting warps sleep on their mbarrier (try_wait with a suspend hint) instead of spinning, so
// they do not steal issue slots or shared-memory bandwidth from the converter and epilogue warps.
// Every mbarrier wait is bounded (2 s): on expiry the CTA records an error in the workspace's
// device flag and leaves after draining its own copies and MMAs; it never spins forever.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kq_sm100.cuh"
#include "kq_tc.cuh"

namespace kq {

using namespace sm100;

constexpr int TC_M = 128, TC_N = 128, TC_KB = 64;
constexpr int TC_THREADS = 448;
constexpr int TILE_BYTES = TC_M * TC_KB * 2;  // 16 KB: 128 rows x 64 f16

template <int DT>
struct TcCfg;
template <>
struct TcCfg<KQ_Q4_K> {
    static constexpr int NSA = 4, NSB = 4;
    static constexpr int B_STAGE = TILE_BYTES;   // one tile
    static constexpr int CB = kQ4KChunk;        // packed chunk bytes per row group
    static constexpr int HSLOT = 128 * 8;        // per-row (d, -dmin) float pairs of one super-block
    static constexpr bool EXT = true;
};
template <>
struct TcCfg<KQ_Q6_K> {
    static constexpr int NSA = 4, NSB = 3;
    static constexpr int B_STAGE = 2 * TILE_BYTES;  // lo and hi tiles
    static constexpr int CB = kQ6KChunk;
    static constexpr int HSLOT = 128 * 8;          // per-row (d, 0) float pairs of one super-block
    static constexpr bool EXT = false;
};

template <int DT>
struct TcLayout {
    using C = TcCfg<DT>;
    static constexpr int A_OFF = 0;
    static constexpr int B_OFF = A_OFF + C::NSA * TILE_BYTES;
    static constexpr int EA_OFF = B_OFF + C::NSB * C::B_STAGE;
    static constexpr int EB_OFF = EA_OFF + (C::EXT ? 2 * 4096 : 0);
    static constexpr int P_OFF = EB_OFF + (C::EXT ? 2 * 4096 : 0);
    static constexpr int H_OFF = P_OFF + 2 * 8 * C::CB;
    static constexpr int BAR_OFF = (H_OFF + 4 * C::HSLOT + 7) & ~7;
    static constexpr int NBAR = 2 * C::NSA + 2 * C::NSB + 2 * 2 + 3 * 2 + 2 * 4 + 2 * 2 + 1;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr int TOTAL = MISC_OFF + 16;
    static constexpr int ALLOC = TOTAL + 1024;  // slack for 1024-byte alignment of the base
};
static_assert(TcLayout<KQ_Q4_K>::ALLOC <= 227 * 1024, "Q4_K tensor-core smem budget");
static_assert(TcLayout<KQ_Q6_K>::ALLOC <= 227 * 1024, "Q6_K tensor-core smem budget");

struct TcParams {
    const uint8_t *w;      // native weights
    const float *da;       // [nsb][M_pad] activation scales
    float *y;
    int64_t ldy;
    int M, N, K, M_pad;
    int nsplit, sb_per_split;  // split-K: cluster rank z covers super-blocks [z*sb_per_split, ...)
    unsigned long long *err;   // device flag (workspace header)
};

// Packed fp32 pair arithmetic (one instruction for two lanes of work).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(d)
        : "l"(*reinterpret_cast<uint64_t *>(&a)), "l"(*reinterpret_cast<uint64_t *>(&b)),
          "l"(*reinterpret_cast<uint64_t *>(&c)));
    return *reinterpret_cast<float2 *>(&d);
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;"
        : "=l"(d)
        : "l"(*reinterpret_cast<uint64_t *>(&a)), "l"(*reinterpret_cast<uint64_t *>(&b)));
    return *reinterpret_cast<float2 *>(&d);
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// Q4_K: 16 code bytes (low nibble -> first 16 elements, high nibble -> the 16 elements 32 later)
// into f16 products sc*c written as 4 swizzled 16-byte chunks of the B tile row.  The magic
// exponents make (0x6400 | n) = 1024 + n and (0x5400 | 16n) = 64 + n, so one fused multiply-add
// per pair gives sc*n exactly.
__device__ __forceinline__ void convert_q4k_unit(uint4 v, int sc_lo, int sc_hi, uint8_t *brow, int row, int seg) {
    const __half2 slo = __float2half2_rn((float)sc_lo), shi = __float2half2_rn((float)sc_hi);
    const __half2 nlo = __float2half2_rn(-1024.0f * sc_lo), nhi = __float2half2_rn(-64.0f * sc_hi);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t lo[8], hi[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t d01 = __byte_perm(w[i], 0u, 0x4140), d23 = __byte_perm(w[i], 0u, 0x4342);
        lo[2 * i] = h2u(__hfma2(u2h((d01 & 0x000F000Fu) | 0x64006400u), slo, nlo));
        lo[2 * i + 1] = h2u(__hfma2(u2h((d23 & 0x000F000Fu) | 0x64006400u), slo, nlo));
        hi[2 * i] = h2u(__hfma2(u2h((d01 & 0x00F000F0u) | 0x54005400u), shi, nhi));
        hi[2 * i + 1] = h2u(__hfma2(u2h((d23 & 0x00F000F0u) | 0x54005400u), shi, nhi));
    }
    const int sw = row & 7;
    *reinterpret_cast<uint4 *>(brow + (((2 * seg) ^ sw) << 4)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    *reinterpret_cast<uint4 *>(brow + (((2 * seg + 1) ^ sw) << 4)) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
    *reinterpret_cast<uint4 *>(brow + (((4 + 2 * seg) ^ sw) << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4 *>(brow + (((5 + 2 * seg) ^ sw) << 4)) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
}

// Q6_K: 16 low-nibble bytes + 16 high-bit bytes -> 6-bit codes c; writes (sc&15)*(c-32) into the lo
// tile row and (sc>>4)*(c-32) into the hi tile row (sub-block scales of the low and high runs).
__device__ __forceinline__ void convert_q6k_unit(uint4 v, uint4 h, int sc_a, int sc_b, uint8_t *brow_lo,
                                                 uint8_t *brow_hi, int row, int seg) {
    const int la = sc_a & 15, ha = sc_a >> 4, lb = sc_b & 15, hb = sc_b >> 4;
    const __half2 mla = __float2half2_rn((float)la), nla = __float2half2_rn(-1056.0f * la);
    const __half2 mha = __float2half2_rn((float)ha), nha = __float2half2_rn(-1056.0f * ha);
    const __half2 mlb = __float2half2_rn((float)lb), nlb = __float2half2_rn(-1056.0f * lb);
    const __half2 mhb = __float2half2_rn((float)hb), nhb = __float2half2_rn(-1056.0f * hb);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w}, q[4] = {h.x, h.y, h.z, h.w};
    uint32_t alo[8], ahi[8], blo[8], bhi[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t ca = (w[i] & 0x0f0f0f0fu) | (((q[i] >> (2 * seg)) & 0x03030303u) << 4);
        const uint32_t cb = ((w[i] >> 4) & 0x0f0f0f0fu) | (((q[i] >> (4 + 2 * seg)) & 0x03030303u) << 4);
        const __half2 a01 = u2h(__byte_perm(ca, 0u, 0x4140) | 0x64006400u);
        const __half2 a23 = u2h(__byte_perm(ca, 0u, 0x4342) | 0x64006400u);
        const __half2 b01 = u2h(__byte_perm(cb, 0u, 0x4140) | 0x64006400u);
        const __half2 b23 = u2h(__byte_perm(cb, 0u, 0x4342) | 0x64006400u);
        alo[2 * i] = h2u(__hfma2(a01, mla, nla)); alo[2 * i + 1] = h2u(__hfma2(a23, mla, nla));
        ahi[2 * i] = h2u(__hfma2(a01, mha, nha)); ahi[2 * i + 1] = h2u(__hfma2(a23, mha, nha));
        blo[2 * i] = h2u(__hfma2(b01, mlb, nlb)); blo[2 * i + 1] = h2u(__hfma2(b23, mlb, nlb));
        bhi[2 * i] = h2u(__hfma2(b01, mhb, nhb)); bhi[2 * i + 1] = h2u(__hfma2(b23, mhb, nhb));
    }
    const int sw = row & 7;
    const int c0 = ((2 * seg) ^ sw) << 4, c1 = ((2 * seg + 1) ^ sw) << 4;
    const int c2 = ((4 + 2 * seg) ^ sw) << 4, c3 = ((5 + 2 * seg) ^ sw) << 4;
    *reinterpret_cast<uint4 *>(brow_lo + c0) = make_uint4(alo[0], alo[1], alo[2], alo[3]);
    *reinterpret_cast<uint4 *>(brow_lo + c1) = make_uint4(alo[4], alo[5], alo[6], alo[7]);
    *reinterpret_cast<uint4 *>(brow_lo + c2) = make_uint4(blo[0], blo[1], blo[2], blo[3]);
    *reinterpret_cast<uint4 *>(brow_lo + c3) = make_uint4(blo[4], blo[5], blo[6], blo[7]);
    *reinterpret_cast<uint4 *>(brow_hi + c0) = make_uint4(ahi[0], ahi[1], ahi[2], ahi[3]);
    *reinterpret_cast<uint4 *>(brow_hi + c1) = make_uint4(ahi[4], ahi[5], ahi[6], ahi[7]);
    *reinterpret_cast<uint4 *>(brow_hi + c2) = make_uint4(bhi[0], bhi[1], bhi[2], bhi[3]);
    *reinterpret_cast<uint4 *>(brow_hi + c3) = make_uint4(bhi[4], bhi[5], bhi[6], bhi[7]);
}

template <int DT>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmE, TcParams P) {
    using C = TcCfg<DT>;
    using L = TcLayout<DT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = sm + L::A_OFF;
    uint8_t *sB = sm + L::B_OFF;
    uint8_t *sEA = sm + L::EA_OFF;
    uint8_t *sEB = sm + L::EB_OFF;
    uint8_t *sP = sm + L::P_OFF;
    uint8_t *sH = sm + L::H_OFF;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::BAR_OFF);
    uint64_t *a_full = bars, *a_empty = a_full + C::NSA;
    uint64_t *b_full = a_empty + C::NSA, *b_empty = b_full + C::NSB;
    uint64_t *p_full = b_empty + C::NSB, *p_empty = p_full + 2;
    uint64_t *e_full = p_empty + 2, *be_full = e_full + 2, *e_empty = be_full + 2;
    uint64_t *h_full = e_empty + 2, *h_empty = h_full + 4;  // per-super-block row-scale ring (4 slots)
    uint64_t *acc_full = h_empty + 4, *acc_empty = acc_full + 2;
    uint64_t *mma_done = acc_empty + 2;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(sm + L::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::MISC_OFF + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * TC_N, m0 = blockIdx.y * TC_M;
    const int nchunk = P.K / 256;
    const int sb0 = blockIdx.z * P.sb_per_split;
    const int nsb = min(nchunk, sb0 + P.sb_per_split) - sb0;  // super-blocks of this CTA (t = sb - sb0)
    const int groups_total = (P.N + 15) / 16;
    const int g0 = n0 / 16;
    const int valid_groups = min(8, groups_total - g0);
    const int rows_valid = valid_groups * 16;

    if (tid == 0) {
        for (int i = 0; i < C::NSA; ++i) { mbar_init(&a_full[i], 1); mbar_init(&a_empty[i], 1); }
        for (int i = 0; i < C::NSB; ++i) { mbar_init(&b_full[i], 128); mbar_init(&b_empty[i], 1); }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&p_full[i], 1); mbar_init(&p_empty[i], 128);
            mbar_init(&e_full[i], 1); mbar_init(&be_full[i], 128); mbar_init(&e_empty[i], 1);
            mbar_init(&acc_full[i], 1); mbar_init(&acc_empty[i], 8);
        }
        for (int i = 0; i < 4; ++i) { mbar_init(&h_full[i], 128); mbar_init(&h_empty[i], 8); }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 13) tmem_alloc(tmem_holder, 512);
    if (warp == 12 && lane == 0) {
        prefetch_tmap(&tmA);
        if (C::EXT) prefetch_tmap(&tmE);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_holder;
    float acc[64];       // epilogue: this thread's 64 outputs (token row, column half)
    bool epi_ok = false;

    if (warp == 12) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int last_a[C::NSA], last_p[2], last_e[2];
            for (int i = 0; i < C::NSA; ++i) last_a[i] = -1;
            for (int i = 0; i < 2; ++i) { last_p[i] = -1; last_e[i] = -1; }
            bool ok = true;
            for (int sb = 0; sb < nsb && ok; ++sb) {
                const int gsb = sb0 + sb;
                const int p = sb & 1, pph = (sb >> 1) & 1;
                if (!(ok = mbar_wait_sleep(&p_empty[p], pph ^ 1, abort_flag))) break;
                mbar_arrive_expect_tx(&p_full[p], valid_groups * C::CB);
                for (int gi = 0; gi < valid_groups; ++gi)
                    bulk_load(sP + (p * 8 + gi) * C::CB, P.w + ((int64_t)(g0 + gi) * nchunk + gsb) * C::CB, C::CB,
                              &p_full[p]);
                last_p[p] = pph;
                if (C::EXT) {
                    const int e = sb & 1, eph = (sb >> 1) & 1;
                    if (!(ok = mbar_wait_sleep(&e_empty[e], eph ^ 1, abort_flag))) break;
                    mbar_arrive_expect_tx(&e_full[e], 4096);
                    tma_load_2d(sEA + e * 4096, &tmE, &e_full[e], gsb * 16, m0);
                    last_e[e] = eph;
                }
                for (int kb = 0; kb < 4; ++kb) {
                    const int kk = sb * 4 + kb, s = kk % C::NSA, ph = (kk / C::NSA) & 1;
                    if (!(ok = mbar_wait_sleep(&a_empty[s], ph ^ 1, abort_flag))) break;
                    mbar_arrive_expect_tx(&a_full[s], TILE_BYTES);
                    tma_load_2d(sA + s * TILE_BYTES, &tmA, &a_full[s], gsb * 256 + kb * TC_KB, m0);
                    last_a[s] = ph;
                }
            }
            if (!ok) {
                // drain: wait (bounded) for every copy this thread issued to land before leaving
                volatile int no_abort = 0;
                for (int i = 0; i < C::NSA; ++i)
                    if (last_a[i] >= 0) { no_abort = 0; mbar_wait(&a_full[i], last_a[i], &no_abort, 100000000ull); }
                for (int i = 0; i < 2; ++i) {
                    if (last_p[i] >= 0) { no_abort = 0; mbar_wait(&p_full[i], last_p[i], &no_abort, 100000000ull); }
                    if (last_e[i] >= 0) { no_abort = 0; mbar_wait(&e_full[i], last_e[i], &no_abort, 100000000ull); }
                }
            }
        }
    } else if (warp == 13) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(TC_M, TC_N);
            const uint32_t sA_u = smem_u32(sA), sB_u = smem_u32(sB), sEA_u = smem_u32(sEA), sEB_u = smem_u32(sEB);
            bool ok = true;
            for (int sb = 0; sb < nsb && ok; ++sb) {
                const int buf = sb & 1;
                if (!(ok = mbar_wait_sleep(&acc_empty[buf], ((sb >> 1) & 1) ^ 1, abort_flag))) break;
                tc_fence_after();
                const uint32_t d1 = tbase + buf * TC_N, d2 = tbase + 256 + buf * TC_N;
                for (int kb = 0; kb < 4 && ok; ++kb) {
                    const int kk = sb * 4 + kb;
                    const int sa = kk % C::NSA, sbb = kk % C::NSB;
                    if (!(ok = mbar_wait_sleep(&a_full[sa], (kk / C::NSA) & 1, abort_flag))) break;
                    if (!(ok = mbar_wait_sleep(&b_full[sbb], (kk / C::NSB) & 1, abort_flag))) break;
                    tc_fence_after();
#pragma unroll
                    for (int k16 = 0; k16 < 4; ++k16) {
                        const uint64_t ad = smem_desc(sA_u + sa * TILE_BYTES + k16 * 32, 1024, 2);
                        const uint64_t bd = smem_desc(sB_u + sbb * C::B_STAGE + k16 * 32, 1024, 2);
                        const uint32_t accum = (kb | k16) != 0;
                        mma_f16(d1, ad, bd, idesc, accum);
                        if (!C::EXT) {
                            const uint64_t bd2 = smem_desc(sB_u + sbb * C::B_STAGE + TILE_BYTES + k16 * 32, 1024, 2);
                            mma_f16(d2, ad, bd2, idesc, accum);
                        }
                    }
                    mma_commit(&a_empty[sa]);
                    mma_commit(&b_empty[sbb]);
                }
                if (!ok) break;
                if (C::EXT) {
                    const int e = sb & 1, eph = (sb >> 1) & 1;
                    if (!(ok = mbar_wait_sleep(&e_full[e], eph, abort_flag))) break;
                    if (!(ok = mbar_wait_sleep(&be_full[e], eph, abort_flag))) break;
                    tc_fence_after();
                    mma_f16(d2, smem_desc(sEA_u + e * 4096, 256, 6), smem_desc(sEB_u + e * 4096, 256, 6), idesc, 0);
                    mma_commit(&e_empty[e]);
                }
                mma_commit(&acc_full[buf]);
            }
            // every MMA this thread issued has finished before TMEM is released
            mma_commit(mma_done);
            volatile int no_abort = 0;
            mbar_wait(mma_done, 0, &no_abort, 100000000ull);
        }
    } else if (warp >= 8) {
        // ------------------------------------------------------------ weight converters
        // Thread ct owns B-tile row ct for the whole super-block: its scales are decoded once, and
        // eight consecutive threads write eight different rows, whose swizzled 16-byte chunks fall
        // in eight different bank groups.
        const int row = tid - 256;
        const bool rvalid = row < rows_valid;
        bool ok = true;
        for (int sb = 0; sb < nsb && ok; ++sb) {
            const int p = sb & 1;
            if (!(ok = mbar_wait_sleep(&p_full[p], (sb >> 1) & 1, abort_flag))) break;
            const uint8_t *chunk = sP + p * 8 * C::CB + (row >> 4) * C::CB;
            int sc[16], mn[8];
#pragma unroll
            for (int j = 0; j < 16; ++j) sc[j] = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) mn[j] = 0;
            float2 dpair = make_float2(0.0f, 0.0f);  // (d, -dmin) of this row for the epilogue
            if (rvalid) {
                if (C::EXT) {
                    const uint4 hv = *reinterpret_cast<const uint4 *>(chunk + 2048 + (row & 15) * 16);
                    dpair = make_float2(half_bits_to_float((uint16_t)(hv.x & 0xffff)),
                                        -half_bits_to_float((uint16_t)(hv.x >> 16)));
                    uint8_t s12[12];
                    const uint32_t hw[3] = {hv.y, hv.z, hv.w};
#pragma unroll
                    for (int i = 0; i < 12; ++i) s12[i] = (hw[i / 4] >> (8 * (i % 4))) & 0xff;
#pragma unroll
                    for (int j = 0; j < 8; ++j) q4k_scale_min(s12, j, sc[j], mn[j]);
                } else {
                    const uint4 sv = *reinterpret_cast<const uint4 *>(chunk + 3072 + (row & 15) * 16);
                    const uint32_t sw4[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
                    for (int j = 0; j < 16; ++j) sc[j] = (int)(int8_t)((sw4[j / 4] >> (8 * (j % 4))) & 0xff);
                    dpair = make_float2(half_bits_to_float(*reinterpret_cast<const uint16_t *>(chunk + 3328 + (row & 15) * 2)),
                                        0.0f);
                }
            }
            {
                const int h = sb & 3;
                if (!(ok = mbar_wait_sleep(&h_empty[h], ((sb >> 2) & 1) ^ 1, abort_flag))) break;
                reinterpret_cast<float2 *>(sH + h * C::HSLOT)[row] = dpair;
                mbar_arrive(&h_full[h]);
            }
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
                const int kk = sb * 4 + kb, s = kk % C::NSB;
                if (!(ok = mbar_wait_sleep(&b_empty[s], ((kk / C::NSB) & 1) ^ 1, abort_flag))) break;
                uint8_t *brow = sB + s * C::B_STAGE + row * 128;
                if (!rvalid) {
                    const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        *reinterpret_cast<uint4 *>(brow + j * 16) = z;
                        if (!C::EXT) *reinterpret_cast<uint4 *>(brow + TILE_BYTES + j * 16) = z;
                    }
                } else {
                    const uint8_t *codes = chunk + kb * 512 + (row & 15) * 32;
                    const uint4 v0 = *reinterpret_cast<const uint4 *>(codes);
                    const uint4 v1 = *reinterpret_cast<const uint4 *>(codes + 16);
                    if (C::EXT) {
                        convert_q4k_unit(v0, sc[2 * kb], sc[2 * kb + 1], brow, row, 0);
                        convert_q4k_unit(v1, sc[2 * kb], sc[2 * kb + 1], brow, row, 1);
                    } else {
                        const uint4 h = *reinterpret_cast<const uint4 *>(chunk + 2048 + kb * 256 + (row & 15) * 16);
                        convert_q6k_unit(v0, h, sc[4 * kb], sc[4 * kb + 2], brow, brow + TILE_BYTES, row, 0);
                        convert_q6k_unit(v1, h, sc[4 * kb + 1], sc[4 * kb + 3], brow, brow + TILE_BYTES, row, 1);
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(&b_full[s]);
            }
            if (!ok) break;
            if (C::EXT) {
                // extension B row: the 8 sub-block mins, each repeated for its two bsum groups
                const int e = sb & 1;
                if (!(ok = mbar_wait_sleep(&e_empty[e], ((sb >> 1) & 1) ^ 1, abort_flag))) break;
                uint32_t mm[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) mm[j] = h2u(__float2half2_rn((float)mn[j]));
                uint8_t *erow = sEB + e * 4096 + row * 32;
                const int sw = (row >> 2) & 1;  // 32-byte swizzle: 16-byte chunk index ^= address bit 7
                *reinterpret_cast<uint4 *>(erow + ((0 ^ sw) << 4)) = make_uint4(mm[0], mm[1], mm[2], mm[3]);
                *reinterpret_cast<uint4 *>(erow + ((1 ^ sw) << 4)) = make_uint4(mm[4], mm[5], mm[6], mm[7]);
                fence_proxy_async_smem();
                mbar_arrive(&be_full[e]);
            }
            mbar_arrive(&p_empty[p]);
        }
    } else {
        // ------------------------------------------------------------ epilogue: per-super-block promotion
        const int wq = warp & 3, half = warp >> 2;
        const int m = m0 + 32 * wq + lane;
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[i] = 0.0f;
        const uint32_t lane_base = tbase + ((uint32_t)(32 * wq) << 16);
        float da_next = P.da[(int64_t)sb0 * P.M_pad + m];
        bool ok = true;
        for (int sb = 0; sb < nsb && ok; ++sb) {
            const int buf = sb & 1, h = sb & 3;
            const float da = da_next;
            if (sb + 1 < nsb) da_next = P.da[(int64_t)(sb0 + sb + 1) * P.M_pad + m];
            if (!(ok = mbar_wait_sleep(&acc_full[buf], (sb >> 1) & 1, abort_flag))) break;
            if (!(ok = mbar_wait_sleep(&h_full[h], (sb >> 2) & 1, abort_flag))) break;
            tc_fence_after();
            const float4 *dsc = reinterpret_cast<const float4 *>(sH + h * C::HSLOT) + half * 32;
            const float2 da2 = make_float2(da, da);
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                const int col = half * 64 + ch * 16;
                float s1[16], s2[16];
                tmem_ld16(lane_base + buf * TC_N + col, s1);
                tmem_ld16(lane_base + 256 + buf * TC_N + col, s2);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    const float4 sc2 = dsc[ch * 8 + i / 2];  // (d, -dmin) of columns col+i, col+i+1
                    float2 &a = *reinterpret_cast<float2 *>(&acc[ch * 16 + i]);
                    if (C::EXT) {
                        // acc += da * (d*S1 - dmin*S2)
                        const float2 u = fmul2(make_float2(s2[i], s2[i + 1]), make_float2(sc2.y, sc2.w));
                        const float2 v = ffma2(make_float2(s1[i], s1[i + 1]), make_float2(sc2.x, sc2.z), u);
                        a = ffma2(v, da2, a);
                    } else {
                        // acc += (da*d) * (S_lo + 16*S_hi)
                        const float2 v = ffma2(make_float2(16.0f, 16.0f), make_float2(s2[i], s2[i + 1]),
                                               make_float2(s1[i], s1[i + 1]));
                        const float2 t = fmul2(da2, make_float2(sc2.x, sc2.z));
                        a = ffma2(t, v, a);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&acc_empty[buf]);
                mbar_arrive(&h_empty[h]);
            }
        }
        epi_ok = ok;
        if (ok && P.nsplit == 1 && m < P.M) {
            float *yr = P.y + (int64_t)m * P.ldy + n0 + half * 64;
            const int nrem = P.N - (n0 + half * 64);
            if (nrem >= 64 && (reinterpret_cast<uintptr_t>(yr) & 15) == 0) {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    reinterpret_cast<float4 *>(yr)[i] =
                        make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
            } else {
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    if (i < nrem) yr[i] = acc[i];
            }
        }
    }

    __syncthreads();
    if (P.nsplit > 1) {
        // Split-K across the CTAs of a cluster: every CTA parks its fp32 tile in its own (now idle)
        // pipeline buffers, then each CTA sums a slice of rows over all CTAs of the cluster in rank
        // order through distributed shared memory and writes it -- deterministic, no workspace.
        constexpr int RS = TC_N + 4;  // padded row stride (floats): conflict-free row-per-lane writes
        float *red = reinterpret_cast<float *>(sA);
        if (warp < 8) {
            const int ml = 32 * (warp & 3) + lane;
            float *rr = red + ml * RS + (warp >> 2) * 64;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                reinterpret_cast<float4 *>(rr)[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
        }
        cooperative_groups::cluster_group cluster = cooperative_groups::this_cluster();
        cluster.sync();
        const int S = P.nsplit, rank = blockIdx.z;
        const int rows_per = (TC_M + S - 1) / S;
        const int r0 = rank * rows_per, r1 = min(TC_M, r0 + rows_per);
        for (int idx = tid; idx < (r1 - r0) * TC_N; idx += TC_THREADS) {
            const int ml = r0 + idx / TC_N, nl = idx % TC_N;
            float v = 0.0f;
            for (int k = 0; k < S; ++k) v += cluster.map_shared_rank(red, k)[ml * RS + nl];
            const int mm = m0 + ml, nn = n0 + nl;
            if (mm < P.M && nn < P.N) P.y[(int64_t)mm * P.ldy + nn] = v;
        }
        cluster.sync();
    }
    (void)epi_ok;
    if (tid == 0 && *abort_flag) atomicAdd(P.err, 1ull);
    if (warp == 13) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// Activation prologue: Q8_K rows -> f16 code panel [M_pad][K], f16 bsum panel [M_pad][nsb*16],
// f32 scale panel [nsb][M_pad]; rows past M are zero.  One warp per (row, super-block).
// Also clears the workspace's device flag.
__global__ void act_panel_kernel(const uint8_t *__restrict__ xq, int M, int M_pad, int nsb, __half *__restrict__ A,
                                 __half *__restrict__ E, float *__restrict__ D, unsigned long long *__restrict__ err) {
    if (blockIdx.x == 0 && threadIdx.x == 0) *err = 0ull;  // the GEMM that follows counts timeouts here
    const int64_t wid = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (wid >= (int64_t)M_pad * nsb) return;
    const int m = (int)(wid / nsb), sb = (int)(wid % nsb);
    const int64_t K = (int64_t)nsb * 256;
    uint4 out = make_uint4(0, 0, 0, 0);
    __half bsv = __float2half(0.0f);
    float d = 0.0f;
    if (m < M) {
        const uint8_t *blk = xq + ((int64_t)m * nsb + sb) * kQ8KBytes;
        const uint32_t w0 = *reinterpret_cast<const uint32_t *>(blk + 4 + lane * 8);
        const uint32_t w1 = *reinterpret_cast<const uint32_t *>(blk + 8 + lane * 8);
        __half hv[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            hv[i] = __int2half_rn((int)(int8_t)((w0 >> (8 * i)) & 0xff));
            hv[4 + i] = __int2half_rn((int)(int8_t)((w1 >> (8 * i)) & 0xff));
        }
        out = *reinterpret_cast<uint4 *>(hv);
        if (lane < 16) bsv = __int2half_rn((int)reinterpret_cast<const int16_t *>(blk + 260)[lane]);
        d = *reinterpret_cast<const float *>(blk);
    }
    *reinterpret_cast<uint4 *>(A + (int64_t)m * K + sb * 256 + lane * 8) = out;
    if (lane < 16) E[(int64_t)m * nsb * 16 + sb * 16 + lane] = bsv;
    if (lane == 0) D[(int64_t)sb * M_pad + m] = d;
}

// ------------------------------------------------------------------ host side
struct TcWs {
    size_t off_flag, off_a, off_e, off_d, total;
    int M_pad;
};

static size_t al256(size_t v) { return (v + 255) & ~(size_t)255; }

static TcWs tc_ws(int64_t M, int64_t K) {
    TcWs w{};
    w.M_pad = (int)((M + TC_M - 1) / TC_M * TC_M);
    const int64_t nsb = K / 256;
    size_t o = 0;
    w.off_flag = o; o += 256;
    w.off_a = o; o += al256((size_t)w.M_pad * K * 2);
    w.off_e = o; o += al256((size_t)w.M_pad * nsb * 16 * 2);
    w.off_d = o; o += al256((size_t)w.M_pad * nsb * 4);
    w.total = o;
    return w;
}

bool tc_eligible(kq_dtype wt, int64_t M, int64_t N, int64_t K) {
    if (wt != KQ_Q4_K && wt != KQ_Q6_K) return false;
    if (M < 128 || N < 128) return false;
    if (K % 256 || K > (1 << 20) || M > (1 << 22) || N > (1 << 22)) return false;
    return true;
}

// Split-K factor: the number of CTAs per output tile (a cluster along z) that best fills whole
// waves of the 152 SMs, with at least 4 super-blocks per CTA; 1 when the tiles alone fill the GPU.
static int tc_splits(int64_t M, int64_t N, int64_t K) {
    const int64_t tiles = ((M + TC_M - 1) / TC_M) * ((N + TC_N - 1) / TC_N);
    const int nsb = (int)(K / 256);
    const int num_sms = 152;
    if (tiles >= 2 * num_sms) return 1;
    int best = 1;
    double best_eff = 0.0;
    for (int S = 1; S <= 8; ++S) {
        const int per = (nsb + S - 1) / S;
        if (S > 1 && per < 4) break;
        if ((nsb + per - 1) / per != S) continue;  // S must be exactly realisable
        const int64_t ctas = tiles * S;
        const double eff = (double)ctas / (double)(((ctas + num_sms - 1) / num_sms) * num_sms);
        if (eff > best_eff + 1e-9) { best_eff = eff; best = S; }
    }
    return best;
}

size_t tc_workspace_bytes(kq_dtype wt, int64_t M, int64_t N, int64_t K) {
    if (!tc_eligible(wt, M, N, K)) return 0;
    return tc_ws(M, K).total;
}

static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

template <int DT>
static kq_status launch_tc(const uint8_t *w, int64_t M, int64_t N, int64_t K, float *y, int64_t ldy, uint8_t *ws,
                           const TcWs &L, cudaStream_t st) {
    using Lay = TcLayout<DT>;
    auto encode = get_encode();
    if (!encode) return fail(KQ_ERR_CUDA, "kq_gemm: cuTensorMapEncodeTiled unavailable");
    const int64_t nsb = K / 256;
    CUtensorMap tmA, tmE;
    {
        cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)L.M_pad};
        cuuint64_t strides[1] = {(cuuint64_t)K * 2};
        cuuint32_t box[2] = {TC_KB, TC_M};
        cuuint32_t es[2] = {1, 1};
        CUresult r = encode(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, ws + L.off_a, dims, strides, box, es,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(KQ_ERR_CUDA, "kq_gemm: tensor map A encode failed (%d)", (int)r);
    }
    {
        cuuint64_t dims[2] = {(cuuint64_t)nsb * 16, (cuuint64_t)L.M_pad};
        cuuint64_t strides[1] = {(cuuint64_t)nsb * 32};
        cuuint32_t box[2] = {16, TC_M};
        cuuint32_t es[2] = {1, 1};
        CUresult r = encode(&tmE, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, ws + L.off_e, dims, strides, box, es,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(KQ_ERR_CUDA, "kq_gemm: tensor map E encode failed (%d)", (int)r);
    }
    TcParams p{};
    p.w = w;
    p.da = reinterpret_cast<const float *>(ws + L.off_d);
    p.y = y;
    p.ldy = ldy;
    p.M = (int)M; p.N = (int)N; p.K = (int)K; p.M_pad = L.M_pad;
    const int S = tc_splits(M, N, K);
    p.nsplit = S;
    p.sb_per_split = (int)((nsb + S - 1) / S);
    p.err = reinterpret_cast<unsigned long long *>(ws + L.off_flag);
    auto kern = tc_gemm_kernel<DT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::ALLOC);
    if (e != cudaSuccess) return fail(KQ_ERR_CUDA, "kq_gemm: %s", cudaGetErrorString(e));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((N + TC_N - 1) / TC_N), (unsigned)(L.M_pad / TC_M), (unsigned)S);
    cfg.blockDim = dim3(TC_THREADS, 1, 1);
    cfg.dynamicSmemBytes = Lay::ALLOC;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = (unsigned)S;
    cfg.attrs = attr;
    cfg.numAttrs = S > 1 ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kern, tmA, tmE, p);
    if (e != cudaSuccess) return fail(KQ_ERR_CUDA, "kq_gemm (tensor core): launch failed: %s", cudaGetErrorString(e));
    return KQ_OK;
}

kq_status tc_gemm(kq_dtype wt, const uint8_t *w, const uint8_t *xq, int64_t M, int64_t N, int64_t K, float *y,
                  int64_t ldy, uint8_t *workspace, cudaStream_t st) {
    const TcWs L = tc_ws(M, K);
    if ((N + TC_N - 1) / TC_N > 65535 || L.M_pad / TC_M > 65535)
        return fail(KQ_ERR_INVALID_ARG, "kq_gemm: shape too large for the tensor-core grid");
    const int64_t nsb = K / 256;
    const int64_t warps = (int64_t)L.M_pad * nsb;
    act_panel_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(
        xq, (int)M, L.M_pad, (int)nsb, reinterpret_cast<__half *>(workspace + L.off_a),
        reinterpret_cast<__half *>(workspace + L.off_e), reinterpret_cast<float *>(workspace + L.off_d),
        reinterpret_cast<unsigned long long *>(workspace + L.off_flag));
    kq_status s = check_launch("kq_gemm (activation panel)");
    if (s != KQ_OK) return s;
    s = wt == KQ_Q4_K ? launch_tc<KQ_Q4_K>(w, M, N, K, y, ldy, workspace, L, st)
                      : launch_tc<KQ_Q6_K>(w, M, N, K, y, ldy, workspace, L, st);
    if (s == KQ_OK) count_launch(R_MMQ_TC, 2);
    return s;
}

}  // namespace kq
