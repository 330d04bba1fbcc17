// kq_tc.cu -- tensor-core prefill GEMM for Q4_K / Q6_K weights x Q8_K activations on sm_103a.
//
// sm_103a has no integer tcgen05 MMA, so the integer block dots are carried EXACTLY on the f16
// tensor pipe (tcgen05.mma kind::f16, fp32 accumulation in TMEM):
//   * activation codes q (|q| <= 127) are exact in f16; a prologue writes them as an f16 panel that
//     TMA loads with 128-byte swizzle into a shared-memory ring.  One activation tile serves every
//     weight row of the CTA (the cooperative activation share of vllm.cpp PR #3035).
//   * weights stay packed in HBM; converter warps unpack each 64-element kblock of their row into
//     the integer products sc_j*c (Q4_K, <= 945) or, for Q6_K, into ((sc & 15)/16)*(c-32) and
//     (sc >> 4)*(c-32) (at most 9 significant bits), all exact in f16, and store them straight into
//     TENSOR MEMORY, where the MMA reads them as its A operand.  Converted
//     weights never touch shared memory, so shared-memory bandwidth goes to the activation tiles.
//   * each super-block (256 elements) accumulates into its own TMEM tile (weight rows = lanes,
//     tokens = columns): the sums are integers below 2^24 for any realistic input, so the fp32
//     accumulator holds them exactly.  Q4_K's min term sum_j m_j*bsum_j is a 16-wide extension MMA
//     (mins and bsums are exact in f16) into a second tile; Q6_K's two halves share one tile, which
//     holds the super-block's integer sum over 16.
//   * epilogue warps promote each super-block to fp32 while the MMA fills the other TMEM buffer:
//     acc += d_a*(d_w*S1 - dmin*S2) (Q4_K) or acc += (d_a*16*d_w)*S (Q6_K).
// Q5_K follows Q4_K (a fifth code bit), Q8_0 x Q8_1 reads every 32-block's dot out of its own
// accumulator; an opt-in folded-scale mode instead dequantises to f16 in the converters and
// accumulates a whole tile in one accumulator (not bit-exact).  Schedule: persistent CTAs over whole
// tiles, split-K clusters for few tiles, or both (a split tail) when the last wave would be short; a
// dense GEMM starts under programmatic dependent launch beside the end of its activation prologue.
// The integer parts are therefore the oracle's integers; only the fp32 scaling uses fused
// multiply-adds, which keeps the result within a few ulps of the sequential CPU order.
//
// Roles (896 threads, 28 warps): warps 0-15 epilogue (TMEM lane quarter = warp % 4, token quarter =
// warp / 4), warps 16-23 weight converters (lane quarter = warp % 4; warps 16-19 convert kblocks 0
// and 2 of every super-block, warps 20-23 kblocks 1 and 3), warp 24 producer of the packed weights,
// bsums and activation scales, warp 26 producer of the activation tiles (a stream of its own, so it
// runs ahead without waiting on the other rings), warps 25 and 27 MMA issuers for the even and odd
// super-blocks (warp 25 also owns the TMEM allocation).
// Waiting warps sleep on their mbarrier (try_wait with a suspend hint) instead of spinning, so
// they do not steal issue slots or shared-memory bandwidth from the converter and epilogue warps.
// Every mbarrier wait is bounded (2 s): on expiry the CTA records an error in the workspace's
// device flag and leaves after draining its own copies and MMAs; it never spins forever.
#include <algorithm>
#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kq_q8k_block.cuh"
#include "kq_sm100.cuh"
#include "kq_tc.cuh"

namespace kq {

using namespace sm100;

constexpr int TC_ROWS = 128;  // weight rows per CTA: MMA M, TMEM lanes
constexpr int TC_TOK = 128;   // tokens per CTA: MMA N, TMEM columns of one accumulator
constexpr int TC_KB = 64;     // K elements per kblock (one activation tile, one TMEM A stage)
constexpr int TC_EPI_WARPS = 16, TC_CONV_WARPS = 8;
constexpr int TC_WARP_PROD = TC_EPI_WARPS + TC_CONV_WARPS, TC_WARP_MMA = TC_WARP_PROD + 1;
constexpr int TC_WARP_ACT = TC_WARP_MMA + 1, TC_WARP_MMA2 = TC_WARP_ACT + 1;
constexpr int TC_THREADS = (TC_WARP_MMA2 + 1) * 32;
constexpr int ACT_TILE = TC_TOK * TC_KB * 2;  // 16 KB: 128 tokens x 64 f16
constexpr int NACT = 8;                       // activation ring: two super-blocks ahead
constexpr int NPAIR = NACT / 2;               // the ring is handed over in pairs of kblocks
constexpr int TMEM_COLS = 512;

template <int DT>
struct TcCfg;
template <>
struct TcCfg<KQ_Q4_K> {
    static constexpr int CB = kQ4KChunk;  // packed chunk bytes per 16-row group
    static constexpr bool EXT = true;     // min term through the extension MMA
    static constexpr bool Q8 = false;     // per-32-block scales (Q8_0 x Q8_1)
    static constexpr bool Q5 = false;     // fifth code bit from the row's high-bit bytes (Q5_K)
    static constexpr bool FOLD = false;   // scales folded into the f16 operands (one accumulator per tile)
    static constexpr int TOK = TC_TOK;    // tokens per tile (MMA N)
    static constexpr int BASE = KQ_Q4_K;  // the weight format
    static constexpr int NACT = 8;        // activation-ring tiles (64 K each)
    static constexpr int A_COLS = 32;     // TMEM columns of one converted kblock (64 f16)
    static constexpr int NACC = 2;        // accumulator buffers
    static constexpr int BPS = 1;         // accumulator read-outs per step (scale blocks per 256 K)
    static constexpr int H_ROW = 8;       // bytes of row scales per step: f32 (d, -dmin)
    static constexpr int NP = 2;          // packed-weight ring slots (super-blocks in flight)
    static constexpr int NE = 2;          // extension-operand ring slots (mins, bsums)
    static constexpr uint32_t TM_S2 = 256, TM_A = 384;
};
template <>
struct TcCfg<KQ_Q5_K> {  // Q4_K's header and min term; 5-bit codes, sc*c <= 63*31 exact in f16
    static constexpr int CB = kQ5KChunk;
    static constexpr bool EXT = true, Q8 = false, Q5 = true, FOLD = false;
    static constexpr int TOK = TC_TOK, NACT = 8, BASE = KQ_Q5_K;
    static constexpr int A_COLS = 32, NACC = 2, BPS = 1, H_ROW = 8, NP = 2, NE = 2;
    static constexpr uint32_t TM_S2 = 256, TM_A = 384;
};
template <>
struct TcCfg<KQ_Q6_K> {
    static constexpr int CB = kQ6KChunk;
    static constexpr bool EXT = false, Q8 = false, Q5 = false, FOLD = false;
    static constexpr int TOK = TC_TOK, NACT = 8, BASE = KQ_Q6_K;
    static constexpr int A_COLS = 64;     // lo tile (32 columns) then 16*hi tile (32 columns)
    static constexpr int NACC = 2, BPS = 1, H_ROW = 8;  // f32 (d, 0)
    static constexpr int NP = 2, NE = 2;
    static constexpr uint32_t TM_S2 = 0, TM_A = 256;
};
template <>
struct TcCfg<KQ_Q8_0> {
    static constexpr int CB = kQ80Chunk;
    static constexpr bool EXT = false, Q8 = true, Q5 = false, FOLD = false;
    static constexpr int TOK = TC_TOK, NACT = 8, BASE = KQ_Q8_0;
    static constexpr int A_COLS = 32;
    // every 32-element block has its own weight and activation scale, so every block's integer
    // dot P_b is read out of its own accumulator: three buffers rotate along the blocks
    static constexpr int NACC = 3, BPS = 8, H_ROW = 16;  // the row's 8 f16 block scales
    static constexpr int NP = 2, NE = 2;
    static constexpr uint32_t TM_S2 = 0, TM_A = 384;
};
// Folded scales (an opt-in throughput mode): the block scales are multiplied into the f16 operands --
// the converters write the dequantised weight f16(d*sc*c - dmin*m) (Q4_K, Q5_K), f16(d*sc*(c-32))
// (Q6_K) or f16(d_w*w) (Q8_0), the activation panel holds f16(d_a*q) -- so every product is the
// scaled one and a tile accumulates over the whole of K in one fp32 TMEM buffer, read out once per
// tile.  Without a per-step read-out the accumulator need not be double-buffered, which leaves room
// for 256-token tiles (one 128 x 256 accumulator + four kblock stages): every converted weight then
// serves twice the tokens.  Not bit-exact: each operand is rounded to f16.
// Few output tiles (small M) take 128-token tiles instead, two accumulators alternating per tile, and
// split K across a cluster as the exact kernels do.
constexpr int KQ_Q4_KF = 101, KQ_Q6_KF = 102, KQ_Q8_0F = 103, KQ_Q5_KF = 106;  // internal, not kq_dtype values
constexpr int KQ_FOLD128 = 100;  // added to a folded code: the 128-token form
template <int BASEDT, int CHUNK, int T>
struct TcFoldCfg {
    static constexpr int CB = CHUNK;
    static constexpr int BASE = BASEDT;  // the weight format
    static constexpr bool EXT = false, Q8 = false, Q5 = BASEDT == KQ_Q5_K, FOLD = true;
    static constexpr int TOK = T;                 // 256: two pairs of 32 KB activation tiles; 128: four of 16 KB
    static constexpr int NACT = T == 256 ? 4 : 8;
    static constexpr int A_COLS = 32;
    static constexpr int NACC = T == 256 ? 1 : 2, BPS = 1, H_ROW = 16;  // accumulators (of TOK columns)
    static constexpr int NP = 2, NE = 2;
    static constexpr uint32_t TM_S2 = 0, TM_A = 256;
};
template <> struct TcCfg<KQ_Q4_KF> : TcFoldCfg<KQ_Q4_K, kQ4KChunk, 256> {};
template <> struct TcCfg<KQ_Q5_KF> : TcFoldCfg<KQ_Q5_K, kQ5KChunk, 256> {};
template <> struct TcCfg<KQ_Q6_KF> : TcFoldCfg<KQ_Q6_K, kQ6KChunk, 256> {};
template <> struct TcCfg<KQ_Q8_0F> : TcFoldCfg<KQ_Q8_0, kQ80Chunk, 256> {};
template <> struct TcCfg<KQ_Q4_KF + KQ_FOLD128> : TcFoldCfg<KQ_Q4_K, kQ4KChunk, 128> {};
template <> struct TcCfg<KQ_Q5_KF + KQ_FOLD128> : TcFoldCfg<KQ_Q5_K, kQ5KChunk, 128> {};
template <> struct TcCfg<KQ_Q6_KF + KQ_FOLD128> : TcFoldCfg<KQ_Q6_K, kQ6KChunk, 128> {};
template <> struct TcCfg<KQ_Q8_0F + KQ_FOLD128> : TcFoldCfg<KQ_Q8_0, kQ80Chunk, 128> {};
// TMEM map: accumulator buffers at columns 0, 128 (and 256 for Q8_0); Q4_K min-term tile at 256;
// converted kblock stages from TM_A on (4 stages = one super-block).
static_assert(TcCfg<KQ_Q4_K>::TM_A + 4 * TcCfg<KQ_Q4_K>::A_COLS <= TMEM_COLS, "Q4_K TMEM map");
static_assert(TcCfg<KQ_Q6_K>::TM_A + 4 * TcCfg<KQ_Q6_K>::A_COLS <= TMEM_COLS, "Q6_K TMEM map");
static_assert(TcCfg<KQ_Q8_0>::NACC * 128 <= (int)TcCfg<KQ_Q8_0>::TM_A &&
                  TcCfg<KQ_Q8_0>::TM_A + 4 * TcCfg<KQ_Q8_0>::A_COLS <= TMEM_COLS, "Q8_0 TMEM map");

template <int DT>
struct TcLayout {
    using C = TcCfg<DT>;
    static constexpr int ACTT = C::TOK * TC_KB * 2;  // one activation tile: TOK tokens x 64 f16
    static constexpr int NPAIR = C::NACT / 2;        // the ring is handed over in pairs of kblocks
    static constexpr int ACT_OFF = 0;
    static constexpr int P_OFF = ACT_OFF + C::NACT * ACTT;
    static constexpr int EA_OFF = (P_OFF + C::NP * 8 * C::CB + 1023) & ~1023;
    static constexpr int EB_OFF = EA_OFF + (C::EXT ? C::NE * 4096 : 0);
    static constexpr int H_OFF = EB_OFF + (C::EXT ? C::NE * 4096 : 0);
    static constexpr int DA_OFF = H_OFF + 4 * TC_ROWS * C::H_ROW;
    static constexpr int BAR_OFF = DA_OFF + 4 * C::TOK * 4 * C::BPS;
    static constexpr int NBAR = 2 * NPAIR + 2 * 3 + 2 * 3 + 3 * 4 + 2 * 3 + 2 + 4 + 1;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr int TOTAL = MISC_OFF + 16;
    static constexpr int ALLOC = TOTAL + 1024;  // slack for 1024-byte alignment of the base
};
static_assert(TcLayout<KQ_Q4_K>::ALLOC <= 227 * 1024, "Q4_K tensor-core smem budget");
static_assert(TcLayout<KQ_Q6_K>::ALLOC <= 227 * 1024, "Q6_K tensor-core smem budget");
static_assert(TcLayout<KQ_Q5_K>::ALLOC <= 227 * 1024, "Q5_K tensor-core smem budget");
static_assert(TcLayout<KQ_Q8_0>::ALLOC <= 227 * 1024, "Q8_0 tensor-core smem budget");
static_assert(TcLayout<KQ_Q8_0F>::ALLOC <= 227 * 1024, "folded Q8_0 tensor-core smem budget");
static_assert(TcLayout<KQ_Q6_KF>::ALLOC <= 227 * 1024, "folded Q6_K tensor-core smem budget");
static_assert(TcLayout<KQ_Q5_KF>::ALLOC <= 227 * 1024, "folded Q5_K tensor-core smem budget");
static_assert(TcCfg<KQ_Q8_0F>::TOK <= (int)TcCfg<KQ_Q8_0F>::TM_A &&
                  TcCfg<KQ_Q8_0F>::TM_A + 4 * TcCfg<KQ_Q8_0F>::A_COLS <= TMEM_COLS, "folded TMEM map");
// the split-K reduction parks a 128 x (128 + 4) fp32 tile in the activation ring
static_assert(TC_TOK * (TC_ROWS + 4) * 4 <= NACT * ACT_TILE, "split-K staging fits the activation ring");

struct TcParams {
    const uint8_t *w;      // native weights
    const float *da;       // [nsb][M_pad] activation scales
    float *y;
    int64_t ldy;
    int M, N, K, M_pad;
    int nsplit, sb_per_split;  // split-K: cluster rank z covers super-blocks [z*sb_per_split, ...)
    unsigned long long *err;   // device flag (workspace header)
    // Routed experts (grouped != 0): blockIdx.y indexes a table of (expert e, 128-row tile j); the
    // rows of expert e sit at panel rows poff[e] .. (padded to 4), its (token, slot) pair ids are
    // lists[offset[e] .. offset[e] + count[e]), and its weights start at row group e * N/16.
    int grouped;
    const int *tiles, *tile_count, *count, *offset, *poff, *lists;
    // Tile schedule: tiles are numbered token-tile-major (weight-row tile fastest): m_tiles x n_tiles
    // (dense) or *tile_count x n_tiles (grouped), so CTAs running at the same time share activation
    // tiles.  persistent: CTA b runs tiles b, b + gridDim.x, ...; otherwise CTA (x, y) runs tile
    // y*n_tiles + x alone (the split-K launch).
    int persistent, n_tiles, m_tiles;
    // Tile range of this launch (plain tiles): units [unit_base, unit_limit).  A dense GEMM whose last
    // wave would leave most SMs idle runs its whole waves in a persistent launch and the leftover tiles
    // in a second, split-K launch.
    int unit_base, unit_limit;
    // Fused SwiGLU -> Q8_K (swq != 0; routed gate/up weights: N = 2F rows per expert, gate rows [0, F),
    // up rows [F, 2F)).  The scheduled unit is four tiles of one token tile: gate rows 256b..256b+255
    // as two 128-row tiles, then the up rows of the same columns.  The epilogue parks the gate tiles
    // in this CTA's slice of scr, replaces them by h = silu(gate)*up when the up tiles arrive (each
    // thread meets its own gate values again), and after the fourth tile quantizes every token's 256
    // h values into Q8_K block b of its pair's row of hq.  scr is rewritten by every unit, so it
    // stays in L2; the fp32 gate/up rows never reach HBM.
    int swq;
    float *scr;    // [gridDim.x][2][TC_TOK][256] fp32 (units alternate halves)
    uint8_t *hq;   // [pairs][F/256] Q8_K blocks
    // Debug instantiation only (DBG): the integer sums every super-block (Q8_0: every 32-block)
    // accumulates in TMEM, read out before the fp32 promotion: dbg[out row][n][block][2] int32 =
    // (sum_j sc_j*P_j, Q4_K/Q5_K min term sum_j m_j*(bs_2j + bs_2j+1) or 0), out row = token row
    // (dense) or (token, slot) pair (routed).
    int *dbg;
    int dbg_nblk;
    // Wall-time limit of every pipeline wait (ns), and a test hook: withhold != 0 keeps the activation
    // producer idle, so the first wait for an activation tile cannot complete and runs into the limit.
    unsigned long long wait_ns;
    int withhold;
};

struct TcTile {
    int n0, m0, tok_valid, g0, valid_groups, list_base;
};

// Geometry of tile `tile`: weight rows n0.., first panel row m0, stored token rows, first weight row
// group, row groups present, and (grouped) the first pair-list entry.
template <bool SWQ, int TOK>
__device__ __forceinline__ TcTile tc_tile(const TcParams &P, int tile, int m_tiles) {
    TcTile T;
    const int nt = tile % P.n_tiles, mt = tile / P.n_tiles;
    (void)m_tiles;
    // fused SwiGLU units: weight-row tile nt = 4b + s is gate (s < 2) or up (s >= 2) half s & 1 of block b
    T.n0 = SWQ ? ((nt & 2) ? P.N / 2 : 0) + 256 * (nt >> 2) + TC_ROWS * (nt & 1) : nt * TC_ROWS;
    T.valid_groups = min(8, (P.N + 15) / 16 - T.n0 / 16);
    if (P.grouped) {
        const int e = P.tiles[2 * mt], j = P.tiles[2 * mt + 1];
        T.m0 = P.poff[e] + j * TOK;
        T.tok_valid = min(TOK, P.count[e] - j * TOK);
        T.g0 = e * (P.N / 16) + T.n0 / 16;
        T.list_base = P.offset[e] + j * TOK;
    } else {
        T.m0 = mt * TOK;
        T.tok_valid = P.M - T.m0;
        T.g0 = T.n0 / 16;
        T.list_base = 0;
    }
    return T;
}

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

// Q4_K kblock of one row (32 code bytes: low nibbles = sub-block 2kb, high nibbles = sub-block
// 2kb+1) -> 32 TMEM columns of f16 pairs sc*c.  The magic exponents make (0x6400 | n) = 1024 + n and
// (0x5400 | 16n) = 64 + n, so one fused multiply-add per pair gives sc*n exactly.
__device__ __forceinline__ void convert_q4k_kblock(uint4 v0, uint4 v1, int sc_lo, int sc_hi, uint32_t (&r)[32]) {
    const __half2 slo = __float2half2_rn((float)sc_lo), shi = __float2half2_rn((float)sc_hi);
    const __half2 nlo = __float2half2_rn(-1024.0f * sc_lo), nhi = __float2half2_rn(-64.0f * sc_hi);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t d01 = __byte_perm(w[i], 0u, 0x4140), d23 = __byte_perm(w[i], 0u, 0x4342);
        r[2 * i] = h2u(__hfma2(u2h((d01 & 0x000F000Fu) | 0x64006400u), slo, nlo));
        r[2 * i + 1] = h2u(__hfma2(u2h((d23 & 0x000F000Fu) | 0x64006400u), slo, nlo));
        r[16 + 2 * i] = h2u(__hfma2(u2h((d01 & 0x00F000F0u) | 0x54005400u), shi, nhi));
        r[16 + 2 * i + 1] = h2u(__hfma2(u2h((d23 & 0x00F000F0u) | 0x54005400u), shi, nhi));
    }
}

// Q5_K kblock kb of one row: the Q4_K conversion with each code's fifth bit taken from the row's
// high-bit words hq (byte l pairs with code byte l: bit 2kb for the low nibble, bit 2kb+1 for the high
// one) and placed above the nibble: (0x6400 | (n + 16h)) = 1024 + c and (0x5400 | 16(n + 16h)) = 64 + c.
__device__ __forceinline__ void convert_q5k_kblock(uint4 v0, uint4 v1, const uint32_t (&hq)[8], int kb, int sc_lo,
                                                   int sc_hi, uint32_t (&r)[32]) {
    const __half2 slo = __float2half2_rn((float)sc_lo), shi = __float2half2_rn((float)sc_hi);
    const __half2 nlo = __float2half2_rn(-1024.0f * sc_lo), nhi = __float2half2_rn(-64.0f * sc_hi);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t d01 = __byte_perm(w[i], 0u, 0x4140), d23 = __byte_perm(w[i], 0u, 0x4342);
        const uint32_t h01 = __byte_perm(hq[i], 0u, 0x4140), h23 = __byte_perm(hq[i], 0u, 0x4342);
        const uint32_t l01 = ((h01 >> (2 * kb)) & 0x00010001u) << 4, l23 = ((h23 >> (2 * kb)) & 0x00010001u) << 4;
        const uint32_t u01 = ((h01 >> (2 * kb + 1)) & 0x00010001u) << 8, u23 = ((h23 >> (2 * kb + 1)) & 0x00010001u) << 8;
        r[2 * i] = h2u(__hfma2(u2h((d01 & 0x000F000Fu) | l01 | 0x64006400u), slo, nlo));
        r[2 * i + 1] = h2u(__hfma2(u2h((d23 & 0x000F000Fu) | l23 | 0x64006400u), slo, nlo));
        r[16 + 2 * i] = h2u(__hfma2(u2h((d01 & 0x00F000F0u) | u01 | 0x54005400u), shi, nhi));
        r[16 + 2 * i + 1] = h2u(__hfma2(u2h((d23 & 0x00F000F0u) | u23 | 0x54005400u), shi, nhi));
    }
}

// Q6_K sub-block of one row (16 elements: 4 nibble words whose codes sit in the low nibbles (HI =
// false) or the high nibbles (HI = true) of each byte, 4 high-bit words whose 2-bit fields for this
// sub-block sit at bit HS) -> 8 lo columns ((sc & 15)/16)*(c-32) and 8 hi columns (sc >> 4)*(c-32), so
// the two MMAs of a 16-K slice accumulate (sc/16)*sum((c-32)*q): the super-block's integer sum over 16,
// which the epilogue scales back with 16*d (exact: a power of two).  The byte permute with 0x64 bytes
// builds (0x6400 | c) = 1024 + c directly and one fused multiply-add per pair gives each product
// exactly (at most 9 significant bits, the lo ones with 4 fractional bits).
template <bool HI, int HS>
__device__ __forceinline__ void convert_q6k_sub(const uint32_t (&nib)[4], const uint32_t (&hb)[4], int sc,
                                                uint32_t (&lo)[8], uint32_t (&hi)[8]) {
    const int l = sc & 15, hs = sc >> 4;
    const __half2 ml = __float2half2_rn(0.0625f * l), nl = __float2half2_rn(-66.0f * l);
    const __half2 mh = __float2half2_rn((float)hs), nh = __float2half2_rn(-1056.0f * hs);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // high bits of the sub-block to bits 4-5 of every byte, the code's low 4 bits to bits 0-3
        const uint32_t h = (HS <= 4 ? (hb[i] << (4 - HS)) : (hb[i] >> (HS - 4))) & 0x30303030u;
        const uint32_t c = (HI ? ((nib[i] >> 4) & 0x0f0f0f0fu) : (nib[i] & 0x0f0f0f0fu)) | h;
        const __half2 x01 = u2h(__byte_perm(c, 0x64646464u, 0x4140));
        const __half2 x23 = u2h(__byte_perm(c, 0x64646464u, 0x4342));
        lo[2 * i] = h2u(__hfma2(x01, ml, nl));
        lo[2 * i + 1] = h2u(__hfma2(x23, ml, nl));
        hi[2 * i] = h2u(__hfma2(x01, mh, nh));
        hi[2 * i + 1] = h2u(__hfma2(x23, mh, nh));
    }
}

// Folded-scale conversions (opt-in mode): each code becomes its dequantised f16 weight.
// Q4_K/Q5_K kblock: x = c*S + M with S = f16(d*sc), M = f16(-dmin*m) of the element's sub-block (low
// nibbles: sub-block 2kb, high nibbles: 2kb+1), the code recovered exactly from the magic-biased f16
// first (1024 + c - 1024, 64 + c - 64), then one fused multiply-add (one rounding).  With Q5 the fifth
// code bit comes from the row's high-bit words as in convert_q5k_kblock.
template <bool Q5>
__device__ __forceinline__ void convert_q4k_kblock_fold(uint4 v0, uint4 v1, const uint32_t (&hq)[8], int kb,
                                                        __half2 s_lo, __half2 m_lo, __half2 s_hi, __half2 m_hi,
                                                        uint32_t (&r)[32]) {
    const __half2 c1024 = __float2half2_rn(1024.0f), c64 = __float2half2_rn(64.0f);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t d01 = __byte_perm(w[i], 0u, 0x4140), d23 = __byte_perm(w[i], 0u, 0x4342);
        uint32_t l01 = 0, l23 = 0, u01 = 0, u23 = 0;
        if (Q5) {
            const uint32_t h01 = __byte_perm(hq[i], 0u, 0x4140), h23 = __byte_perm(hq[i], 0u, 0x4342);
            l01 = ((h01 >> (2 * kb)) & 0x00010001u) << 4;
            l23 = ((h23 >> (2 * kb)) & 0x00010001u) << 4;
            u01 = ((h01 >> (2 * kb + 1)) & 0x00010001u) << 8;
            u23 = ((h23 >> (2 * kb + 1)) & 0x00010001u) << 8;
        }
        r[2 * i] = h2u(__hfma2(__hsub2(u2h((d01 & 0x000F000Fu) | l01 | 0x64006400u), c1024), s_lo, m_lo));
        r[2 * i + 1] = h2u(__hfma2(__hsub2(u2h((d23 & 0x000F000Fu) | l23 | 0x64006400u), c1024), s_lo, m_lo));
        r[16 + 2 * i] = h2u(__hfma2(__hsub2(u2h((d01 & 0x00F000F0u) | u01 | 0x54005400u), c64), s_hi, m_hi));
        r[16 + 2 * i + 1] = h2u(__hfma2(__hsub2(u2h((d23 & 0x00F000F0u) | u23 | 0x54005400u), c64), s_hi, m_hi));
    }
}

// Q6_K sub-block (as convert_q6k_sub): x = (c - 32)*S with S = f16(d*sc): one exact subtraction, one
// rounding multiply.
template <bool HI, int HS>
__device__ __forceinline__ void convert_q6k_sub_fold(const uint32_t (&nib)[4], const uint32_t (&hb)[4], __half2 sd,
                                                     uint32_t (&o)[8]) {
    const __half2 c1056 = __float2half2_rn(1056.0f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t h = (HS <= 4 ? (hb[i] << (4 - HS)) : (hb[i] >> (HS - 4))) & 0x30303030u;
        const uint32_t c = (HI ? ((nib[i] >> 4) & 0x0f0f0f0fu) : (nib[i] & 0x0f0f0f0fu)) | h;
        o[2 * i] = h2u(__hmul2(__hsub2(u2h(__byte_perm(c, 0x64646464u, 0x4140)), c1056), sd));
        o[2 * i + 1] = h2u(__hmul2(__hsub2(u2h(__byte_perm(c, 0x64646464u, 0x4342)), c1056), sd));
    }
}

__device__ __forceinline__ __half2 h2dup(float v) { return __float2half2_rn(v); }

// SWQ: fused SwiGLU -> Q8_K epilogue (routed gate/up); DBG: the debug read-out of the integer sums
// (P.dbg).  Each is a separate instantiation, so the plain GEMM's register allocation is untouched.
template <int DT, bool SWQ, bool DBG>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmE, TcParams P) {
    using C = TcCfg<DT>;
    using L = TcLayout<DT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *sAct = sm + L::ACT_OFF;
    uint8_t *sP = sm + L::P_OFF;
    uint8_t *sEA = sm + L::EA_OFF;  // Q4_K: per-row mins (extension A operand), written by converters
    uint8_t *sEB = sm + L::EB_OFF;  // Q4_K: per-token bsums (extension B operand), loaded by TMA
    uint8_t *sH = sm + L::H_OFF;    // per-row (d, -dmin) of a super-block, 4-slot ring
    uint8_t *sDA = sm + L::DA_OFF;  // per-token activation scales of a super-block, same ring
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::BAR_OFF);
    // k_full/k_empty: one slot per pair of kblocks -- its two activation tiles (TMA) and its two
    // converted kblocks (TMEM, from both converter groups) complete the same phase, and a single MMA
    // commit frees both, so the MMA thread waits once per 128 K-elements.
    uint64_t *k_full = bars, *k_empty = k_full + L::NPAIR;
    uint64_t *p_full = k_empty + L::NPAIR, *p_empty = p_full + 3;   // up to 3 packed-weight slots
    uint64_t *e_full = p_empty + 3, *e_empty = e_full + 3;       // Q4_K: bsums (TMA) + mins (converters)
    uint64_t *h_full = e_empty + 3, *da_full = h_full + 4, *h_empty = da_full + 4;
    uint64_t *acc_full = h_empty + 4, *acc_empty = acc_full + 3;
    uint64_t *mma_done = acc_empty + 3;  // one per MMA issuer
    uint64_t *sw_bar = mma_done + 2;     // fused SwiGLU: the four epilogue warps of each token quarter
    uint64_t *s2_empty = sw_bar + 4;     // Q5_K: phase t completes once super-block t's min term is read
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(sm + L::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::MISC_OFF + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nchunk = P.K / 256;
    const int sb0 = blockIdx.z * P.sb_per_split;
    const int nsb = min(nchunk, sb0 + P.sb_per_split) - sb0;  // super-blocks per tile
    const int m_tiles = P.grouped ? *P.tile_count : P.m_tiles;
    const int ntiles = P.n_tiles * m_tiles;
    // scheduled units: single tiles, or (fused SwiGLU) runs of four consecutive tiles
    const int nunits = min(SWQ ? ntiles >> 2 : ntiles, P.unit_limit);
    const int unit0 = P.unit_base + (P.persistent ? (int)blockIdx.x : (int)(blockIdx.y * P.n_tiles + blockIdx.x));
    const int ustride = P.persistent ? (int)gridDim.x : nunits - P.unit_base;
    if (unit0 >= nunits) return;  // no tile for this CTA: it leaves before any setup
    // One step = one (tile, super-block); every role walks steps 0 .. nsteps-1 in the same order, so
    // the rings and accumulators run on across tile boundaries without draining.
    const int nsteps = (nunits - unit0 + ustride - 1) / ustride * (SWQ ? 4 : 1) * nsb;
    // roles keep (tile i, super-block t) counters along the steps instead of dividing by nsb
    auto tile_of = [&](int i) {
        return tc_tile<SWQ, C::TOK>(P, SWQ ? (unit0 + (i >> 2) * ustride) * 4 + (i & 3) : unit0 + i * ustride, m_tiles);
    };

    if (tid == 0) {
        for (int i = 0; i < L::NPAIR; ++i) { mbar_init(&k_full[i], 32 * TC_CONV_WARPS + 1); mbar_init(&k_empty[i], 1); }
        for (int i = 0; i < C::NP; ++i) { mbar_init(&p_full[i], 1); mbar_init(&p_empty[i], 32 * TC_CONV_WARPS); }
        for (int i = 0; i < C::NE; ++i) { mbar_init(&e_full[i], 32 * TC_CONV_WARPS / 2 + 1); mbar_init(&e_empty[i], 1); }
        for (int i = 0; i < C::NACC; ++i) { mbar_init(&acc_full[i], 1); mbar_init(&acc_empty[i], TC_EPI_WARPS); }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&h_full[i], 32 * TC_CONV_WARPS / 2); mbar_init(&da_full[i], 1);
            mbar_init(&h_empty[i], TC_EPI_WARPS);
        }
        mbar_init(&mma_done[0], 1);
        mbar_init(&mma_done[1], 1);
        for (int i = 0; i < 4; ++i) mbar_init(&sw_bar[i], 4);
        mbar_init(s2_empty, TC_EPI_WARPS);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == TC_WARP_MMA) tmem_alloc(tmem_holder, TMEM_COLS);
    if (warp == TC_WARP_ACT && lane == 0) prefetch_tmap(&tmA);
    if (C::EXT && warp == TC_WARP_PROD && lane == 0) prefetch_tmap(&tmE);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_holder;
    float acc[32];  // epilogue: this thread's 32 outputs (one weight row, a quarter of the tokens)

    if (warp == TC_WARP_PROD) {
        // ------------------------------------------------------------ weight-side producer
        if (lane == 0) {
            int last_p[3], last_e[3], last_d[4];
            for (int i = 0; i < 3; ++i) { last_p[i] = -1; last_e[i] = -1; }
            for (int i = 0; i < 4; ++i) last_d[i] = -1;
            bool ok = true;
            TcTile T{};
            for (int st = 0, ti = 0, tt = 0; st < nsteps && ok; ++st) {
                if (tt == 0) T = tile_of(ti);
                const int gsb = sb0 + tt;
                if (++tt == nsb) { tt = 0; ++ti; }
                const int p = st % C::NP, pph = (st / C::NP) & 1;
                if (!(ok = mbar_wait_sleep(&p_empty[p], pph ^ 1, abort_flag, P.wait_ns))) break;
                mbar_arrive_expect_tx(&p_full[p], T.valid_groups * C::CB);
                for (int gi = 0; gi < T.valid_groups; ++gi)
                    bulk_load(sP + (p * 8 + gi) * C::CB, P.w + ((int64_t)(T.g0 + gi) * nchunk + gsb) * C::CB, C::CB,
                              &p_full[p]);
                last_p[p] = pph;
                // The packed weights are never written by the prologue kernel just before this one; the
                // bsum and scale panels are: under programmatic dependent launch, wait for it here, after
                // the first weight copy is on its way (a no-op in a launch without the attribute).
                if (st == 0) grid_dependency_wait();
                if (C::EXT) {
                    const int e = st % C::NE, eph = (st / C::NE) & 1;
                    if (!(ok = mbar_wait_sleep(&e_empty[e], eph ^ 1, abort_flag, P.wait_ns))) break;
                    mbar_arrive_expect_tx(&e_full[e], 4096);
                    tma_load_2d(sEB + e * 4096, &tmE, &e_full[e], gsb * 16, T.m0);
                    last_e[e] = eph;
                }
                if (!C::FOLD) {  // the folded path has no per-step scales
                    const int h = st & 3, hph = (st >> 2) & 1;
                    if (!(ok = mbar_wait_sleep(&h_empty[h], hph ^ 1, abort_flag, P.wait_ns))) break;
                    // the scale panel has one row of M_pad floats per scale block (256 or 32 K)
                    mbar_arrive_expect_tx(&da_full[h], C::BPS * C::TOK * 4);
                    for (int b = 0; b < C::BPS; ++b)
                        bulk_load(sDA + (h * C::BPS + b) * C::TOK * 4,
                                  P.da + (int64_t)(gsb * C::BPS + b) * P.M_pad + T.m0, C::TOK * 4, &da_full[h]);
                    last_d[h] = hph;
                }
            }
            if (!ok) {
                // drain: wait (bounded) for every copy this thread issued to land before leaving.  A phase
                // that also counts converter arrivals may never complete after an abort; the 100 ms bound
                // still leaves the copy far more time than it needs to land.
                volatile int no_abort = 0;
                for (int i = 0; i < 3; ++i) {
                    if (last_p[i] >= 0) { no_abort = 0; mbar_wait(&p_full[i], last_p[i], &no_abort, 100000000ull); }
                    if (last_e[i] >= 0) { no_abort = 0; mbar_wait(&e_full[i], last_e[i], &no_abort, 100000000ull); }
                }
                for (int i = 0; i < 4; ++i)
                    if (last_d[i] >= 0) { no_abort = 0; mbar_wait(&da_full[i], last_d[i], &no_abort, 100000000ull); }
            }
        }
    } else if (warp == TC_WARP_ACT) {
        // ------------------------------------------------------------ activation-tile producer
        if (lane == 0) {
            int last_k[L::NPAIR];
            for (int i = 0; i < L::NPAIR; ++i) last_k[i] = -1;
            bool ok = true;
            int m0 = 0, ti = 0, tt = 0;
            grid_dependency_wait();  // the activation panel is the prologue kernel's output
            for (int pp = 0; pp < nsteps * 2 && ok && !P.withhold; ++pp) {
                if ((pp & 1) == 0 && tt == 0) m0 = tile_of(ti).m0;
                const int s = pp % L::NPAIR, ph = (pp / L::NPAIR) & 1;
                if (!(ok = mbar_wait_sleep(&k_empty[s], ph ^ 1, abort_flag, P.wait_ns))) break;
                mbar_arrive_expect_tx(&k_full[s], 2 * L::ACTT);
                const int x = (sb0 + tt) * 256 + (pp & 1) * 2 * TC_KB;
                if ((pp & 1) && ++tt == nsb) { tt = 0; ++ti; }
                tma_load_2d(sAct + (2 * s) * L::ACTT, &tmA, &k_full[s], x, m0);
                tma_load_2d(sAct + (2 * s + 1) * L::ACTT, &tmA, &k_full[s], x + TC_KB, m0);
                last_k[s] = ph;
            }
            if (!ok) {
                // bounded drain (see the weight-side producer)
                volatile int no_abort = 0;
                for (int i = 0; i < L::NPAIR; ++i)
                    if (last_k[i] >= 0) { no_abort = 0; mbar_wait(&k_full[i], last_k[i], &no_abort, 100000000ull); }
            }
        }
    } else if (warp == TC_WARP_MMA || warp == TC_WARP_MMA2) {
        // ------------------------------------------------------------ MMA issuers
        // Two issuers on different SM sub-partitions: TC_WARP_MMA takes the even super-blocks
        // (accumulator buffer 0), TC_WARP_MMA2 the odd ones (buffer 1).  One thread sharing its
        // sub-partition with busy warps cannot issue MMAs as fast as the tensor pipe retires them;
        // two interleaved streams can.  Their MMAs touch disjoint pair slots, TMEM stages and
        // accumulators, so no ordering between the issuers is needed beyond the barriers.
        // Lean issue loop: descriptors are built once and stepped by adding to their address field,
        // one wait and one commit cover a pair of kblocks.  Q4_K's min-term tile is single: the
        // extension MMA of super-block t waits until the epilogue is done with t-1 (Q5_K: until it has
        // read t-1's min term).
        if (lane == 0) {
            const int w = warp == TC_WARP_MMA ? 0 : 1;
            constexpr uint32_t idesc = idesc_f16_f32(TC_ROWS, C::TOK);
            const uint64_t dAct = smem_desc(smem_u32(sAct), 1024, 2);
            const uint64_t dEA = smem_desc(smem_u32(sEA), 256, 6), dEB = smem_desc(smem_u32(sEB), 256, 6);
            const uint32_t d1 = tbase + w * C::TOK;
            bool ok = true;
            if (C::Q8) {
                // Q8_0: each 32-element block (two K16 MMAs) fills its own accumulator buffer, the
                // buffers rotating along the global block index g = 8*step + block.  One issuer takes
                // every step: a parity wait only tells apart consecutive phases, so a buffer's user
                // must never run more than one use ahead of its releases, which a single in-order
                // issuer guarantees (a second issuer could reach use u while use u-2 is still held).
                for (int t = 0; t < nsteps && ok && w == 0; ++t) {
                    int g = 8 * t, buf = g % C::NACC, use = g / C::NACC;
                    for (int pr = 0; pr < 2 && ok; ++pr) {
                        const int pp = 2 * t + pr, s = pp % L::NPAIR;
                        if (!(ok = mbar_wait_sleep(&k_full[s], (pp / L::NPAIR) & 1, abort_flag, P.wait_ns))) break;
                        for (int h = 0; h < 2 && ok; ++h) {
                            const uint64_t bd = dAct + (uint64_t)((2 * s + h) * (L::ACTT >> 4));
                            const uint32_t a0 = tbase + C::TM_A + (2 * pr + h) * C::A_COLS;
                            for (int blk = 0; blk < 2; ++blk) {
                                if (!(ok = mbar_wait_sleep(&acc_empty[buf], (use & 1) ^ 1, abort_flag, P.wait_ns))) break;
                                tc_fence_after();
                                const uint32_t dq = tbase + buf * C::TOK;
                                mma_f16_ts(dq, a0 + blk * 16, bd + (uint64_t)(blk * 4), idesc, 0);
                                mma_f16_ts(dq, a0 + blk * 16 + 8, bd + (uint64_t)(blk * 4 + 2), idesc, 1);
                                mma_commit(&acc_full[buf]);
                                if (++buf == C::NACC) { buf = 0; ++use; }
                            }
                        }
                        if (!ok) break;
                        mma_commit(&k_empty[s]);
                    }
                }
            }
            if (C::FOLD) {
                // folded scales: one issuer (the MMAs into a tile's accumulator then go in one fixed
                // order, so the result is deterministic); a tile's steps all accumulate into the one
                // 128 x TOK accumulator, committed once at the tile's last step
                for (int t = 0, ti = 0, tt = 0; t < nsteps && ok && w == 0; ++t) {
                    const bool first = tt == 0, last = tt == nsb - 1;
                    // tile ti's accumulator: buffer ti % NACC, its use count ti / NACC
                    const int ab = C::NACC == 1 ? 0 : (ti & 1), use = C::NACC == 1 ? ti : (ti >> 1);
                    if (first) {  // the epilogue has read this buffer's previous tile out
                        if (!(ok = mbar_wait_sleep(&acc_empty[ab], (use & 1) ^ 1, abort_flag, P.wait_ns))) break;
                        tc_fence_after();
                    }
                    for (int pr = 0; pr < 2 && ok; ++pr) {
                        const int pp = 2 * t + pr, s = pp % L::NPAIR;
                        uint32_t aa[8];
                        uint64_t bb[8];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint64_t bd = dAct + (uint64_t)((2 * s + h) * (L::ACTT >> 4));
                            const uint32_t a0 = tbase + C::TM_A + (2 * pr + h) * C::A_COLS;
#pragma unroll
                            for (int k16 = 0; k16 < 4; ++k16) {
                                aa[h * 4 + k16] = a0 + k16 * 8;
                                bb[h * 4 + k16] = bd + (uint64_t)(k16 * 2);
                            }
                        }
                        if (!(ok = mbar_wait_sleep(&k_full[s], (pp / L::NPAIR) & 1, abort_flag, P.wait_ns))) break;
                        tc_fence_after();
                        mma8_f16_ts(tbase + ab * C::TOK, aa, bb, idesc, (first && pr == 0) ? 0u : 1u);
                        mma_commit(&k_empty[s]);
                    }
                    if (!ok) break;
                    if (last) mma_commit(&acc_full[ab]);
                    if (++tt == nsb) { tt = 0; ++ti; }
                }
            }
            for (int t = w; t < nsteps && ok && !C::Q8 && !C::FOLD; t += 2) {  // t: step
                if (!(ok = mbar_wait_sleep(&acc_empty[w], ((t >> 1) & 1) ^ 1, abort_flag, P.wait_ns))) break;
                tc_fence_after();
                for (int pr = 0; pr < 2 && ok; ++pr) {
                    const int pp = 2 * t + pr, s = pp % L::NPAIR;
                    // operands of the pair's MMAs, computed while the pair is still being filled, so the MMAs
                    // go out back to back with no integer work between them
                    uint32_t aa[2][8];
                    uint64_t bb[2][8];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint64_t bd = dAct + (uint64_t)((2 * s + h) * (L::ACTT >> 4));
                        const uint32_t a0 = tbase + C::TM_A + (2 * pr + h) * C::A_COLS;
#pragma unroll
                        for (int k16 = 0; k16 < 4; ++k16) {
                            if (C::EXT) {  // one MMA per 16 K: A column k16*8 of kblock h
                                aa[0][h * 4 + k16] = a0 + k16 * 8;
                                bb[0][h * 4 + k16] = bd + (uint64_t)(k16 * 2);
                            } else {       // Q6_K: the lo and the 16*hi product of the same 16 K
                                aa[h][2 * k16] = a0 + k16 * 8;
                                aa[h][2 * k16 + 1] = a0 + 32 + k16 * 8;
                                bb[h][2 * k16] = bb[h][2 * k16 + 1] = bd + (uint64_t)(k16 * 2);
                            }
                        }
                    }
                    if (!(ok = mbar_wait_sleep(&k_full[s], (pp / L::NPAIR) & 1, abort_flag, P.wait_ns))) break;
                    tc_fence_after();
                    mma8_f16_ts(d1, aa[0], bb[0], idesc, pr);
                    if (!C::EXT) mma8_f16_ts(d1, aa[1], bb[1], idesc, 1);
                    mma_commit(&k_empty[s]);
                }
                if (!ok) break;
                if (C::EXT) {
                    const int e = t % C::NE;
                    if (!(ok = mbar_wait_sleep(&e_full[e], (t / C::NE) & 1, abort_flag, P.wait_ns))) break;
                    if (t > 0 && !(ok = C::Q5 ? mbar_wait_sleep(s2_empty, (t - 1) & 1, abort_flag, P.wait_ns)
                                              : mbar_wait_sleep(&acc_empty[(t - 1) & 1], ((t - 1) >> 1) & 1, abort_flag,
                                                                P.wait_ns)))
                        break;
                    tc_fence_after();
                    mma_f16(tbase + C::TM_S2, dEA + (uint64_t)(e * (4096 >> 4)), dEB + (uint64_t)(e * (4096 >> 4)),
                            idesc, 0);
                    mma_commit(&e_empty[e]);
                }
                mma_commit(&acc_full[w]);
            }
            // every MMA this thread issued has finished before TMEM is released
            mma_commit(&mma_done[w]);
            volatile int no_abort = 0;
            mbar_wait(&mma_done[w], 0, &no_abort, 100000000ull);
        }
    } else if (warp >= TC_EPI_WARPS) {
        // ------------------------------------------------------------ weight converters
        // Thread (group, row) converts kblocks {group, group+2} of its weight row into its TMEM lane.
        // The kblocks go first, since the MMA waits on them; afterwards group 0 publishes the row's
        // super-block scales for the epilogue and, for Q4_K, group 1 publishes the mins operand of the
        // extension MMA -- both are needed only once the super-block's main MMAs are done.
        const int cw = warp - TC_EPI_WARPS, grp = cw >> 2, q = cw & 3;
        const int row = 32 * q + lane;
        const uint32_t lane_base = tbase + ((uint32_t)(32 * q) << 16);
        bool ok = true, rvalid = false;
        // folded scales, K-quant weights: step t's kblocks {grp, grp+2} of this row as dequantised f16
        auto fold_convert_kquant = [&](int t, int grp, int row, bool rvalid, const uint8_t *chunk, int r16,
                                       uint32_t lane_base) -> bool {
            constexpr bool K4 = C::BASE == KQ_Q4_K || C::BASE == KQ_Q5_K;
            uint4 cv[2][2], qh[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint8_t *codes = chunk + (grp + 2 * j) * 512 + r16 * 32;
                cv[j][0] = *reinterpret_cast<const uint4 *>(codes);
                cv[j][1] = *reinterpret_cast<const uint4 *>(codes + 16);
                qh[j] = K4 ? make_uint4(0, 0, 0, 0)
                           : *reinterpret_cast<const uint4 *>(chunk + 2048 + (grp + 2 * j) * 256 + r16 * 16);
            }
            const uint4 hv = *reinterpret_cast<const uint4 *>(chunk + (K4 ? 2048 : 3072) + r16 * 16);
            float d = K4 ? half_bits_to_float((uint16_t)(hv.x & 0xffff))
                         : half_bits_to_float(*reinterpret_cast<const uint16_t *>(chunk + 3328 + r16 * 2));
            float dmin = K4 ? half_bits_to_float((uint16_t)(hv.x >> 16)) : 0.0f;
            if (!rvalid) d = dmin = 0.0f;  // rows past N were not loaded
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int kb = grp + 2 * j;
                if (t > 0) {
                    const int pq = 2 * (t - 1) + j;
                    if (!mbar_wait_sleep(&k_empty[pq % L::NPAIR], (pq / L::NPAIR) & 1, abort_flag, P.wait_ns))
                        return false;
                }
                tc_fence_after();
                const uint32_t ta = lane_base + C::TM_A + kb * C::A_COLS;
                if (K4) {
                    // the scales and mins of sub-blocks 2kb and 2kb+1 from the 12 packed bytes
                    const uint32_t lo = grp ? (hv.y >> 16) : hv.y;   // scale bytes 2g, 2g+1
                    const uint32_t mz = grp ? (hv.z >> 16) : hv.z;   // min bytes 2g, 2g+1 (bytes 4+2g, 5+2g)
                    const uint32_t hi8 = grp ? (hv.w >> 16) : hv.w;  // bytes 8+2g, 9+2g
                    int sc0, sc1, m0, m1;
                    if (j == 0) {
                        sc0 = lo & 63; sc1 = (lo >> 8) & 63;
                        m0 = mz & 63; m1 = (mz >> 8) & 63;
                    } else {
                        sc0 = (hi8 & 0x0f) | (((lo >> 6) & 3) << 4);
                        sc1 = ((hi8 >> 8) & 0x0f) | (((lo >> 14) & 3) << 4);
                        m0 = ((hi8 >> 4) & 0x0f) | (((mz >> 6) & 3) << 4);
                        m1 = ((hi8 >> 12) & 0x0f) | (((mz >> 14) & 3) << 4);
                    }
                    uint32_t q5w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                    if (C::Q5) {
                        const uint4 a = *reinterpret_cast<const uint4 *>(chunk + 2304 + r16 * 32);
                        const uint4 b = *reinterpret_cast<const uint4 *>(chunk + 2304 + r16 * 32 + 16);
                        q5w[0] = a.x; q5w[1] = a.y; q5w[2] = a.z; q5w[3] = a.w;
                        q5w[4] = b.x; q5w[5] = b.y; q5w[6] = b.z; q5w[7] = b.w;
                    }
                    uint32_t r[32];
                    convert_q4k_kblock_fold<C::Q5>(cv[j][0], cv[j][1], q5w, kb, h2dup(d * (float)sc0),
                                                   h2dup(-dmin * (float)m0), h2dup(d * (float)sc1),
                                                   h2dup(-dmin * (float)m1), r);
                    tmem_st32(ta, r);
                } else {
                    const uint32_t ws = j ? (grp ? hv.w : hv.z) : (grp ? hv.y : hv.x);  // scales 4kb..4kb+3
                    const uint32_t hb[4] = {qh[j].x, qh[j].y, qh[j].z, qh[j].w};
                    const uint32_t n0[4] = {cv[j][0].x, cv[j][0].y, cv[j][0].z, cv[j][0].w};
                    const uint32_t n1[4] = {cv[j][1].x, cv[j][1].y, cv[j][1].z, cv[j][1].w};
                    uint32_t o[8];
                    convert_q6k_sub_fold<false, 0>(n0, hb, h2dup(d * (float)(int8_t)(ws & 0xff)), o);
                    tmem_st8(ta, o);
                    convert_q6k_sub_fold<false, 2>(n1, hb, h2dup(d * (float)(int8_t)((ws >> 8) & 0xff)), o);
                    tmem_st8(ta + 8, o);
                    convert_q6k_sub_fold<true, 4>(n0, hb, h2dup(d * (float)(int8_t)((ws >> 16) & 0xff)), o);
                    tmem_st8(ta + 16, o);
                    convert_q6k_sub_fold<true, 6>(n1, hb, h2dup(d * (float)(int8_t)(ws >> 24)), o);
                    tmem_st8(ta + 24, o);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&k_full[(2 * t + j) % L::NPAIR]);
            }
            return true;
        };
        for (int t = 0, ti = 0, tt = 0; t < nsteps && ok; ++t) {  // t: step
            if (tt == 0) rvalid = row < tile_of(ti).valid_groups * 16;
            if (++tt == nsb) { tt = 0; ++ti; }
            const int p = t % C::NP;
            if (!(ok = mbar_wait_sleep(&p_full[p], (t / C::NP) & 1, abort_flag, P.wait_ns))) break;
            // rows past N were not loaded: their scales are forced to 0, so they convert to zeros
            const uint8_t *chunk = sP + p * 8 * C::CB + (row >> 4) * C::CB;
            const int r16 = row & 15;
            if (C::FOLD && C::BASE != KQ_Q8_0) {
                if (!(ok = fold_convert_kquant(t, grp, row, rvalid, chunk, r16, lane_base))) break;
                mbar_arrive(&p_empty[p]);
                continue;
            }
            if (C::Q8 || C::FOLD) {
                // Q8_0: the row's 64 codes of kblock kb sit at kb*1024 + r16*64; its 8 f16 block
                // scales at 4096 + r16*16.  Codes go to f16 exactly: (0x6400 | (c ^ 0x80)) = 1152 + c;
                // the folded path then multiplies each code by its block's f16 scale (one rounding).
                uint4 cv[2][4];
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        cv[j][i] = reinterpret_cast<const uint4 *>(chunk + (grp + 2 * j) * 1024 + r16 * 64)[i];
                uint4 dv = *reinterpret_cast<const uint4 *>(chunk + 4096 + r16 * 16);
                if (!rvalid) dv = make_uint4(0, 0, 0, 0);
                const __half2 c1152 = __float2half2_rn(1152.0f);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    if (t > 0) {
                        const int pq = 2 * (t - 1) + j;
                        if (!(ok = mbar_wait_sleep(&k_empty[pq % L::NPAIR], (pq / L::NPAIR) & 1, abort_flag, P.wait_ns))) break;
                    }
                    tc_fence_after();
                    uint32_t r[32];
                    // folded: kblock kb = grp + 2j holds blocks 2kb (codes 0-31) and 2kb+1 (32-63), whose
                    // scales are the two halves of word kb of the row's scale vector
                    const uint32_t dword = (grp + 2 * j == 0) ? dv.x : (grp + 2 * j == 1) ? dv.y
                                         : (grp + 2 * j == 2) ? dv.z : dv.w;
                    const __half2 dlo = u2h((dword & 0xffffu) * 0x10001u), dhi = u2h((dword >> 16) * 0x10001u);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t wv[4] = {cv[j][i].x ^ 0x80808080u, cv[j][i].y ^ 0x80808080u,
                                                cv[j][i].z ^ 0x80808080u, cv[j][i].w ^ 0x80808080u};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            __half2 a = __hsub2(u2h(__byte_perm(wv[k], 0x64646464u, 0x4140)), c1152);
                            __half2 b = __hsub2(u2h(__byte_perm(wv[k], 0x64646464u, 0x4342)), c1152);
                            if (C::FOLD) {
                                a = __hmul2(a, i < 2 ? dlo : dhi);
                                b = __hmul2(b, i < 2 ? dlo : dhi);
                            }
                            r[8 * i + 2 * k] = h2u(a);
                            r[8 * i + 2 * k + 1] = h2u(b);
                        }
                    }
                    tmem_st32(lane_base + C::TM_A + (grp + 2 * j) * C::A_COLS, r);
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(&k_full[(2 * t + j) % L::NPAIR]);
                }
                if (!ok) break;
                if (grp == 0 && !C::FOLD) {
                    const int h = t & 3;
                    if (!(ok = mbar_wait_sleep(&h_empty[h], ((t >> 2) & 1) ^ 1, abort_flag, P.wait_ns))) break;
                    reinterpret_cast<uint4 *>(sH + h * TC_ROWS * C::H_ROW)[row] = dv;
                    mbar_arrive(&h_full[h]);
                }
                mbar_arrive(&p_empty[p]);
                continue;
            }
            // every shared-memory read of the super-block is issued up front
            uint4 cv[2][2], qh[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint8_t *codes = chunk + (grp + 2 * j) * 512 + r16 * 32;
                cv[j][0] = *reinterpret_cast<const uint4 *>(codes);
                cv[j][1] = *reinterpret_cast<const uint4 *>(codes + 16);
                if (!C::EXT) qh[j] = *reinterpret_cast<const uint4 *>(chunk + 2048 + (grp + 2 * j) * 256 + r16 * 16);
            }
            // Q4_K/Q5_K: d, dmin and the 12 packed scale bytes; Q6_K: the 16 int8 sub-block scales
            uint4 hv = *reinterpret_cast<const uint4 *>(chunk + (C::EXT ? 2048 : 3072) + r16 * 16);

            if (!rvalid) hv = make_uint4(0, 0, 0, 0);
            int ksc[2][4];  // sub-block scales of kblocks grp and grp+2
            if (C::EXT) {
                // 6-bit scales: sub-block j < 4 in byte j; j >= 4 from the low nibble of byte j+4 and
                // the top two bits of byte j-4.  Group g needs sub-blocks 2g, 2g+1, 2g+4, 2g+5.
                const uint32_t lo = grp ? (hv.y >> 16) : hv.y;   // bytes 2g, 2g+1
                const uint32_t hi8 = grp ? (hv.w >> 16) : hv.w;  // bytes 8+2g, 9+2g
                ksc[0][0] = lo & 63;
                ksc[0][1] = (lo >> 8) & 63;
                ksc[1][0] = (hi8 & 0x0f) | (((lo >> 6) & 3) << 4);
                ksc[1][1] = ((hi8 >> 8) & 0x0f) | (((lo >> 14) & 3) << 4);
                ksc[0][2] = ksc[0][3] = ksc[1][2] = ksc[1][3] = 0;
            } else {
                const uint32_t wa = grp ? hv.y : hv.x, wb = grp ? hv.w : hv.z;  // sub-blocks 4kb..4kb+3
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    ksc[0][k] = (int)(int8_t)((wa >> (8 * k)) & 0xff);
                    ksc[1][k] = (int)(int8_t)((wb >> (8 * k)) & 0xff);
                }
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                // kblock grp+2j belongs to pair j of the super-block; its TMEM stage is free once the
                // MMA of the same pair one super-block earlier has completed
                const int kb = grp + 2 * j;
                if (t > 0) {
                    const int pq = 2 * (t - 1) + j;
                    if (!(ok = mbar_wait_sleep(&k_empty[pq % L::NPAIR], (pq / L::NPAIR) & 1, abort_flag, P.wait_ns))) break;
                }
                tc_fence_after();
                const uint32_t ta = lane_base + C::TM_A + kb * C::A_COLS;
                if (C::EXT) {
                    uint32_t r[32];
                    if (C::Q5) {
                        // the row's 32 high-bit bytes, loaded per kblock to keep them out of the wait
                        const uint4 a = *reinterpret_cast<const uint4 *>(chunk + 2304 + r16 * 32);
                        const uint4 b = *reinterpret_cast<const uint4 *>(chunk + 2304 + r16 * 32 + 16);
                        const uint32_t q5w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                        convert_q5k_kblock(cv[j][0], cv[j][1], q5w, kb, ksc[j][0], ksc[j][1], r);
                    } else {
                        convert_q4k_kblock(cv[j][0], cv[j][1], ksc[j][0], ksc[j][1], r);
                    }
                    tmem_st32(ta, r);
                } else {
                    const uint32_t hb[4] = {qh[j].x, qh[j].y, qh[j].z, qh[j].w};
                    // sub-block 4kb+k: low nibbles of bytes 0-15 / 16-31, then high nibbles
                    const uint32_t n0[4] = {cv[j][0].x, cv[j][0].y, cv[j][0].z, cv[j][0].w};
                    const uint32_t n1[4] = {cv[j][1].x, cv[j][1].y, cv[j][1].z, cv[j][1].w};
                    uint32_t lo[8], hi[8];
                    convert_q6k_sub<false, 0>(n0, hb, ksc[j][0], lo, hi);
                    tmem_st8(ta, lo);
                    tmem_st8(ta + 32, hi);
                    convert_q6k_sub<false, 2>(n1, hb, ksc[j][1], lo, hi);
                    tmem_st8(ta + 8, lo);
                    tmem_st8(ta + 40, hi);
                    convert_q6k_sub<true, 4>(n0, hb, ksc[j][2], lo, hi);
                    tmem_st8(ta + 16, lo);
                    tmem_st8(ta + 48, hi);
                    convert_q6k_sub<true, 6>(n1, hb, ksc[j][3], lo, hi);
                    tmem_st8(ta + 24, lo);
                    tmem_st8(ta + 56, hi);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&k_full[(2 * t + j) % L::NPAIR]);
            }
            if (!ok) break;
            if (grp == 0) {
                // the row's (d, -dmin) for the epilogue
                const int h = t & 3;
                if (!(ok = mbar_wait_sleep(&h_empty[h], ((t >> 2) & 1) ^ 1, abort_flag, P.wait_ns))) break;
                float2 dpair = make_float2(0.0f, 0.0f);
                if (C::EXT)
                    dpair = make_float2(half_bits_to_float((uint16_t)(hv.x & 0xffff)),
                                        -half_bits_to_float((uint16_t)(hv.x >> 16)));
                else if (rvalid)  // Q6_K: 16*d, as the accumulator holds the integer sum over 16
                    dpair = make_float2(
                        16.0f * half_bits_to_float(*reinterpret_cast<const uint16_t *>(chunk + 3328 + r16 * 2)), 0.0f);
                reinterpret_cast<float2 *>(sH + h * TC_ROWS * 8)[row] = dpair;
                mbar_arrive(&h_full[h]);
            } else if (C::EXT) {
                // extension A row: the 8 sub-block mins, each repeated for its two bsum groups
                const int e = t % C::NE;
                if (!(ok = mbar_wait_sleep(&e_empty[e], ((t / C::NE) & 1) ^ 1, abort_flag, P.wait_ns))) break;
                uint8_t s12[12];
                const uint32_t hw[3] = {hv.y, hv.z, hv.w};
#pragma unroll
                for (int i = 0; i < 12; ++i) s12[i] = (hw[i / 4] >> (8 * (i % 4))) & 0xff;
                uint32_t mm[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    int s, m;
                    q4k_scale_min(s12, j, s, m);
                    mm[j] = h2u(__float2half2_rn((float)m));
                }
                uint8_t *erow = sEA + e * 4096 + row * 32;
                const int sw = (row >> 2) & 1;  // 32-byte swizzle: 16-byte chunk index ^= address bit 7
                *reinterpret_cast<uint4 *>(erow + ((0 ^ sw) << 4)) = make_uint4(mm[0], mm[1], mm[2], mm[3]);
                *reinterpret_cast<uint4 *>(erow + ((1 ^ sw) << 4)) = make_uint4(mm[4], mm[5], mm[6], mm[7]);
                fence_proxy_async_smem();
                mbar_arrive(&e_full[e]);
            }
            mbar_arrive(&p_empty[p]);
        }
    } else {
        // ------------------------------------------------------------ epilogue: per-super-block promotion
        const int q = warp & 3, tq = warp >> 2;  // TMEM lane quarter (weight rows), token quarter
        const int row = 32 * q + lane;
        const uint32_t lane_base = tbase + ((uint32_t)(32 * q) << 16);
        bool ok = true;
        // fused SwiGLU: the previous unit's h rows are quantized while the next unit runs, one token per
        // warp per step, from the other half of this CTA's double-buffered scratch
        int sw_u = 0;                 // units this warp has finished: the pending one is sw_u - 1
        int pj = 0, pend = -1;        // pending unit: next token of this quarter, end (-1: none)
        int plist = 0, pb = 0;        // its pair-list offset (token quarter included), its column block
        bool pwait = true;            // its barrier phase has been waited for
        auto swq_token = [&](int j) {  // quantize token j of the pending unit into its hq block
            const float *hs = P.scr + ((int64_t)blockIdx.x * 2 + ((sw_u - 1) & 1)) * (C::TOK * 256) + (tq * 32 + j) * 256;
            const float4 *hv = reinterpret_cast<const float4 *>(hs) + 2 * lane;
            const float4 h0 = hv[0], h1 = hv[1];
            const float v[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
            q8k_block_store(v, P.hq + ((int64_t)P.lists[plist + j] * (P.N / 512) + pb) * kQ8KBytes);
        };
        // DBG: component `comp` of block `blk` for this thread's row and the 8 tokens j0 .. j0+7 of the
        // tile, converted from the fp32 accumulator (an exact integer) to int32
        auto dbg_put = [&](const TcTile &T, int j0, int blk, int comp, const float (&v)[8]) {
            const int n = T.n0 + row;
            if (n >= P.N) return;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int j = j0 + i;
                if (j >= T.tok_valid) break;
                const int64_t mrow = P.grouped ? (int64_t)P.lists[T.list_base + j] : (int64_t)(T.m0 + j);
                P.dbg[((mrow * P.N + n) * P.dbg_nblk + blk) * 2 + comp] = __float2int_rn(v[i]);
            }
        };
        for (int t = 0, ti = 0, tt = 0; t < nsteps && ok; ++t) {  // t: step
            const int buf = t & 1, h = t & 3;
            const int tile_i = ti;
            const int gsb = sb0 + tt;  // this step's super-block along K
            const bool first = tt == 0, last = tt == nsb - 1;
            if (++tt == nsb) { tt = 0; ++ti; }
            if (first) {
#pragma unroll
                for (int i = 0; i < 32; ++i) acc[i] = 0.0f;
            }
            if (C::FOLD) {
                // folded scales: the tile's accumulator holds the finished sums; read once, at the tile's
                // last step: warp (lane quarter q, token quarter tq) takes rows 32q.. and tokens 64tq..,
                // in two halves of 32 tokens, then releases the accumulator for the next tile
                if (!last) continue;
                constexpr int TPW = C::TOK / 4;  // tokens of one warp's token quarter
                const int ab = C::NACC == 1 ? 0 : (tile_i & 1), use = C::NACC == 1 ? tile_i : (tile_i >> 1);
                if (!(ok = mbar_wait_sleep(&acc_full[ab], use & 1, abort_flag, P.wait_ns))) break;
                tc_fence_after();
                const TcTile T = tile_of(tile_i);
                for (int hh = 0; hh < TPW / 32; ++hh) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float v[8];
                        tmem_ld8(lane_base + ab * C::TOK + tq * TPW + hh * 32 + c * 8, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[c * 8 + i] = v[i];
                    }
                    // a split-K tile keeps its sums in acc for the cluster reduction after the loop
                    if (P.nsplit == 1 && T.n0 + row < P.N) {
                        const int mrem = T.tok_valid - tq * TPW - hh * 32;
                        float *yc = P.y + (int64_t)(T.m0 + tq * TPW + hh * 32) * P.ldy + T.n0 + row;
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (i < mrem) yc[(int64_t)i * P.ldy] = acc[i];
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[ab]);
                continue;
            } else if (C::Q8) {
                // Q8_0: per 32-element block b, acc += (d_w*d_a)*P_b with each product rounded on its
                // own and the blocks added in ascending K order -- the CPU oracle's arithmetic, so the
                // result is bit-identical to it
                if (!(ok = mbar_wait_sleep(&h_full[h], (t >> 2) & 1, abort_flag, P.wait_ns))) break;
                if (!(ok = mbar_wait_sleep(&da_full[h], (t >> 2) & 1, abort_flag, P.wait_ns))) break;
                const uint4 dwv = reinterpret_cast<const uint4 *>(sH + h * TC_ROWS * C::H_ROW)[row];
                int g = 8 * t, qb = g % C::NACC, use = g / C::NACC;
                for (int b = 0; b < 8 && ok; ++b) {
                    if (!(ok = mbar_wait_sleep(&acc_full[qb], use & 1, abort_flag, P.wait_ns))) break;
                    tc_fence_after();
                    // block b's f16 scale, picked from the four words with selects (no local array)
                    const uint32_t dword = (b & 4) ? ((b & 2) ? dwv.w : dwv.z) : ((b & 2) ? dwv.y : dwv.x);
                    const float dw = half_bits_to_float((uint16_t)((b & 1) ? (dword >> 16) : (dword & 0xffff)));
                    const float2 dw2 = make_float2(dw, dw);
                    const float4 *dap = reinterpret_cast<const float4 *>(sDA + (h * 8 + b) * C::TOK * 4) + tq * 8;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float pv[8];
                        tmem_ld8(lane_base + qb * C::TOK + tq * 32 + c * 8, pv);
                        tmem_wait_ld();
                        if (DBG) {
                            const TcTile T = tile_of(tile_i);
                            const float zero[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                            dbg_put(T, tq * 32 + c * 8, gsb * 8 + b, 0, pv);
                            dbg_put(T, tq * 32 + c * 8, gsb * 8 + b, 1, zero);
                        }
                        const float4 da0 = dap[2 * c], da1 = dap[2 * c + 1];
                        const float da[8] = {da0.x, da0.y, da0.z, da0.w, da1.x, da1.y, da1.z, da1.w};
#pragma unroll
                        for (int i = 0; i < 8; i += 2) {
                            const float2 sc = fmul2(dw2, make_float2(da[i], da[i + 1]));
                            const float2 tv = fmul2(sc, make_float2(pv[i], pv[i + 1]));
                            // the sums are scalar adds with explicit rounding: the compiler fuses packed
                            // f32x2 multiplies and adds into fused multiply-adds, which would round once
                            // instead of twice and leave the CPU order
                            acc[c * 8 + i] = __fadd_rn(acc[c * 8 + i], tv.x);
                            acc[c * 8 + i + 1] = __fadd_rn(acc[c * 8 + i + 1], tv.y);
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&acc_empty[qb]);
                    if (++qb == C::NACC) { qb = 0; ++use; }
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(&h_empty[h]);
            } else {
            // the step's scales are published long before its sums are complete: their barriers are
            // passed first, so nothing but the accumulator's own wait sits between the MMA and the reads
            if (!(ok = mbar_wait_sleep(&h_full[h], (t >> 2) & 1, abort_flag, P.wait_ns))) break;
            if (!(ok = mbar_wait_sleep(&da_full[h], (t >> 2) & 1, abort_flag, P.wait_ns))) break;
            if (!(ok = mbar_wait_sleep(&acc_full[buf], (t >> 1) & 1, abort_flag, P.wait_ns))) break;
            tc_fence_after();
            const float2 rs = reinterpret_cast<const float2 *>(sH + h * TC_ROWS * 8)[row];  // (d, -dmin)
            const float4 *dap = reinterpret_cast<const float4 *>(sDA + h * C::TOK * 4) + tq * 8;
            const float2 dw2 = make_float2(rs.x, rs.x), nm2 = make_float2(rs.y, rs.y);
            if (C::Q5) {
                // Q5_K: the min-term tile is single and the next super-block's extension MMA waits for
                // it, so it is read first, folded in as acc += da*(-dmin*S2) and released on its own
                // barrier before the main accumulator (acc += da*(d*S1)).  With Q5_K's heavier
                // conversion this takes the epilogue's second half off the chain that paces the steps
                // (measured faster for Q5_K only; Q4_K reads both tiles together below: with Q4_K the
                // early release, also with the next step's main MMAs held behind this extension MMA,
                // measured 1-9% slower).
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float s2[8];
                    tmem_ld8(lane_base + C::TM_S2 + tq * 32 + c * 8, s2);
                    tmem_wait_ld();
                    if (DBG) dbg_put(tile_of(tile_i), tq * 32 + c * 8, gsb, 1, s2);
                    const float4 da0 = dap[2 * c], da1 = dap[2 * c + 1];
                    const float da[8] = {da0.x, da0.y, da0.z, da0.w, da1.x, da1.y, da1.z, da1.w};
#pragma unroll
                    for (int i = 0; i < 8; i += 2) {
                        float2 &a = *reinterpret_cast<float2 *>(&acc[c * 8 + i]);
                        a = ffma2(fmul2(make_float2(s2[i], s2[i + 1]), nm2), make_float2(da[i], da[i + 1]), a);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(s2_empty);
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t col = tq * 32 + c * 8;
                float s1[8], s2[8];
                constexpr bool S2LATE = C::EXT && !C::Q5;
                tmem_ld8(lane_base + buf * C::TOK + col, s1);
                if (S2LATE) tmem_ld8(lane_base + C::TM_S2 + col, s2);
                tmem_wait_ld();
                if (DBG) {
                    const TcTile T = tile_of(tile_i);
                    if (!C::EXT) {  // Q6_K: the accumulator holds the integer sum over 16 (exact)
                        float s16[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) s16[i] = 16.0f * s1[i];
                        dbg_put(T, (int)col, gsb, 0, s16);
                    } else {
                        dbg_put(T, (int)col, gsb, 0, s1);
                    }
                    if (!C::EXT) {
                        const float zero[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                        dbg_put(T, (int)col, gsb, 1, zero);
                    } else if (S2LATE) {
                        dbg_put(T, (int)col, gsb, 1, s2);
                    }
                }
                const float4 da0 = dap[2 * c], da1 = dap[2 * c + 1];
                const float da[8] = {da0.x, da0.y, da0.z, da0.w, da1.x, da1.y, da1.z, da1.w};
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    float2 &a = *reinterpret_cast<float2 *>(&acc[c * 8 + i]);
                    const float2 dap2 = make_float2(da[i], da[i + 1]);
                    if (S2LATE) {
                        // acc += da * (d*S1 - dmin*S2)
                        const float2 u = fmul2(make_float2(s2[i], s2[i + 1]), nm2);
                        const float2 v = ffma2(make_float2(s1[i], s1[i + 1]), dw2, u);
                        a = ffma2(v, dap2, a);
                    } else if (C::EXT) {
                        a = ffma2(fmul2(make_float2(s1[i], s1[i + 1]), dw2), dap2, a);  // acc += da*(d*S1)
                    } else {
                        // acc += (da*d) * S
                        a = ffma2(fmul2(dap2, dw2), make_float2(s1[i], s1[i + 1]), a);
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
            if (SWQ && pend >= 0) {
                // the accumulator is released; one token of the pending unit (after its four warps met)
                if (!pwait) {
                    if (!(ok = mbar_wait_sleep(&sw_bar[tq], (sw_u - 1) & 1, abort_flag, P.wait_ns))) break;
                    pwait = true;
                }
                if (pj < pend) { swq_token(pj); pj += 4; }
            }
            if (!last || P.nsplit != 1) continue;
            const TcTile T = tile_of(tile_i);
            if (SWQ) {
                // fused SwiGLU -> Q8_K.  Tile s of the unit holds column 128*(s & 1) + row of the block
                // for this thread's 32 tokens: gate (s < 2) is parked, up (s >= 2) turns it into h.
                const int s = tile_i & 3;
                const int mrem = T.tok_valid - tq * 32;
                float *sc = P.scr + ((int64_t)blockIdx.x * 2 + (sw_u & 1)) * (C::TOK * 256) + tq * 32 * 256 +
                            TC_ROWS * (s & 1) + row;
                if (s < 2) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (i < mrem) sc[i * 256] = acc[i];
                } else {
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {  // eight gate loads in flight, then their h
                        float gv[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) gv[i] = c + i < mrem ? sc[(c + i) * 256] : 0.0f;
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            if (c + i < mrem) sc[(c + i) * 256] = silu_mul(gv[i], acc[c + i]);
                    }
                }
                if (s != 3) continue;
                // finish the pending unit, then publish this one: its four warps' h columns complete
                // every token's block once all four have arrived
                if (pend >= 0) {
                    if (!pwait && !(ok = mbar_wait_sleep(&sw_bar[tq], (sw_u - 1) & 1, abort_flag, P.wait_ns))) break;
                    for (; pj < pend; pj += 4) swq_token(pj);
                }
                __threadfence_block();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sw_bar[tq]);
                pj = q;
                pend = max(0, min(32, mrem));
                plist = T.list_base + tq * 32;
                pb = (T.n0 - P.N / 2) >> 8;
                pwait = false;
                ++sw_u;
                continue;
            }
            if (T.n0 + row < P.N) {
                // the tile's last super-block: store (a split-K tile is reduced across the cluster below)
                const int mrem = T.tok_valid - tq * 32;
                if (P.grouped) {
                    // token row -> its (token, slot) output row
                    const int *lp = P.lists + T.list_base + tq * 32;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (i < mrem) P.y[(int64_t)lp[i] * P.ldy + T.n0 + row] = acc[i];
                } else {
                    float *yc = P.y + (int64_t)(T.m0 + tq * 32) * P.ldy + T.n0 + row;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (i < mrem) yc[(int64_t)i * P.ldy] = acc[i];
                }
            }
        }
        if (SWQ && ok && pend >= 0) {  // the last unit's tokens
            if (pwait || mbar_wait_sleep(&sw_bar[tq], (sw_u - 1) & 1, abort_flag, P.wait_ns))
                for (; pj < pend; pj += 4) swq_token(pj);
        }
    }

    __syncthreads();
    if (P.nsplit > 1) {
        // Split-K across the CTAs of a cluster: every CTA parks its fp32 tile in its own (now idle)
        // activation ring, then each CTA sums a slice of token rows over all CTAs of the cluster in
        // rank order through distributed shared memory and writes it -- deterministic, no workspace.
        constexpr int RS = TC_ROWS + 4;  // padded token-row stride (floats)
        float *red = reinterpret_cast<float *>(sAct);
        if (warp < TC_EPI_WARPS) {
            const int row = 32 * (warp & 3) + lane, tq = warp >> 2;
#pragma unroll
            for (int i = 0; i < 32; ++i) red[(tq * 32 + i) * RS + row] = acc[i];
        }
        cooperative_groups::cluster_group cluster = cooperative_groups::this_cluster();
        cluster.sync();
        const int S = P.nsplit, rank = blockIdx.z;
        const int rows_per = (C::TOK + S - 1) / S;
        const int r0 = rank * rows_per, r1 = min(C::TOK, r0 + rows_per);
        for (int idx = tid; idx < (r1 - r0) * TC_ROWS; idx += TC_THREADS) {
            const int ml = r0 + idx / TC_ROWS, nl = idx % TC_ROWS;
            float v = 0.0f;
            for (int k = 0; k < S; ++k) v += cluster.map_shared_rank(red, k)[ml * RS + nl];
            const TcTile T = tile_of(0);
            const int mm = T.m0 + ml, nn = T.n0 + nl;
            if (mm < P.M && nn < P.N) P.y[(int64_t)mm * P.ldy + nn] = v;
        }
        cluster.sync();
    }
    if (tid == 0 && *abort_flag) {
        grid_dependency_wait();  // the prologue clears the flag: count only after it has finished
        atomicAdd(P.err, 1ull);
    }
    if (warp == TC_WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tbase, TMEM_COLS);
    }
}

// Activation prologue: Q8_K rows -> f16 code panel [M_pad][K], f16 bsum panel [M_pad][nsb*16],
// f32 scale panel [nsb][M_pad]; rows past M are zero.  One warp per (row, super-block).
// Also clears the workspace's device flag.
__global__ void act_panel_kernel(const uint8_t *__restrict__ xq, int M, int M_pad, int nsb, __half *__restrict__ A,
                                 __half *__restrict__ E, float *__restrict__ D, unsigned long long *__restrict__ err) {
    if (blockIdx.x == 0 && threadIdx.x == 0) *err = 0ull;  // the GEMM that follows counts timeouts here
    grid_launch_dependents();  // the GEMM may start its setup and weight loads beside this grid
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

// Activation prologue straight from fp32 rows (kq_gemm_f32): each warp quantises one 256-element
// block of row m with the Q8_K block arithmetic (q8k_block_codes, the standalone quantizer's) and
// writes the codes, the 16 bsums and d into the panels as act_panel_kernel would from the Q8_K block
// -- the same panels, without the Q8_K round trip through memory.  One warp per (row, super-block);
// rows past M are zero.  Also clears the workspace's device flag.
template <bool VEC>
__global__ void act_panel_f32_kernel(const float *__restrict__ x, int64_t ldx, int M, int M_pad, int nsb,
                                     __half *__restrict__ A, __half *__restrict__ E, float *__restrict__ D,
                                     unsigned long long *__restrict__ err) {
    if (blockIdx.x == 0 && threadIdx.x == 0) *err = 0ull;
    grid_launch_dependents();  // the GEMM may start its setup and weight loads beside this grid
    const int64_t wid = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (wid >= (int64_t)M_pad * nsb) return;
    const int m = (int)(wid / nsb), sb = (int)(wid % nsb);
    const int64_t K = (int64_t)nsb * 256;
    int q[8] = {0, 0, 0, 0, 0, 0, 0, 0}, pair = 0;
    float d = 0.0f;
    if (m < M) {
        const float *p = x + (int64_t)m * ldx + sb * 256 + lane * 8;
        float v[8];
        if (VEC) {
            const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = p[i];
        }
        q8k_block_codes(v, q, pair, d);
    }
    __half hv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) hv[i] = __int2half_rn(q[i]);
    *reinterpret_cast<uint4 *>(A + (int64_t)m * K + sb * 256 + lane * 8) = *reinterpret_cast<uint4 *>(hv);
    if ((lane & 1) == 0) E[(int64_t)m * nsb * 16 + sb * 16 + (lane >> 1)] = __int2half_rn(pair);
    if (lane == 0) D[(int64_t)sb * M_pad + m] = d;
}

// Activation prologue of the folded K-quant path from fp32 rows: each warp quantises one 256-element
// block of row m with the Q8_K block arithmetic (q8k_block_codes, the standalone quantizer's) and writes
// f16(d*q) for its 8 elements -- the panel act_panel_fold_kernel builds from the Q8_K block, without the
// Q8_K round trip through memory.  One warp per (row, super-block); rows past M are zero.  Also clears
// the workspace's device flag.
template <bool VEC>
__global__ void act_panel_f32_fold_kernel(const float *__restrict__ x, int64_t ldx, int M, int M_pad, int nsb,
                                          __half *__restrict__ A, unsigned long long *__restrict__ err) {
    if (blockIdx.x == 0 && threadIdx.x == 0) *err = 0ull;
    grid_launch_dependents();  // the GEMM may start its setup and weight loads beside this grid
    const int64_t wid = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (wid >= (int64_t)M_pad * nsb) return;
    const int m = (int)(wid / nsb), sb = (int)(wid % nsb);
    const int64_t K = (int64_t)nsb * 256;
    int q[8] = {0, 0, 0, 0, 0, 0, 0, 0}, pair = 0;
    float d = 0.0f;
    if (m < M) {
        const float *p = x + (int64_t)m * ldx + sb * 256 + lane * 8;
        float v[8];
        if (VEC) {
            const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = p[i];
        }
        q8k_block_codes(v, q, pair, d);
    }
    __half hv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) hv[i] = __float2half_rn(d * (float)q[i]);
    *reinterpret_cast<uint4 *>(A + (int64_t)m * K + sb * 256 + lane * 8) = *reinterpret_cast<uint4 *>(hv);
}

// Activation prologue for Q8_0 weights: Q8_1 rows -> f16 code panel [M_pad][K] and f32 scale panel
// [K/32][M_pad] (the f16 block scale widened); rows past M are zero.  One warp per (row, 256
// elements): lane l takes elements 8l .. 8l+7 of block l/4.  Also clears the workspace's device flag.
__global__ void act_panel_q81_kernel(const uint8_t *__restrict__ xq, int M, int M_pad, int nsb, __half *__restrict__ A,
                                     float *__restrict__ D, unsigned long long *__restrict__ err) {
    if (blockIdx.x == 0 && threadIdx.x == 0) *err = 0ull;
    grid_launch_dependents();  // the GEMM may start its setup and weight loads beside this grid
    const int64_t wid = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (wid >= (int64_t)M_pad * nsb) return;
    const int m = (int)(wid / nsb), sb = (int)(wid % nsb);
    const int64_t K = (int64_t)nsb * 256;
    const int blk = sb * 8 + (lane >> 2);
    uint4 out = make_uint4(0, 0, 0, 0);
    float d = 0.0f;
    if (m < M) {
        const uint8_t *b = xq + ((int64_t)m * nsb * 8 + blk) * kQ81Bytes;
        const uint32_t w0 = *reinterpret_cast<const uint32_t *>(b + 4 + (lane & 3) * 8);
        const uint32_t w1 = *reinterpret_cast<const uint32_t *>(b + 8 + (lane & 3) * 8);
        __half hv[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            hv[i] = __int2half_rn((int)(int8_t)((w0 >> (8 * i)) & 0xff));
            hv[4 + i] = __int2half_rn((int)(int8_t)((w1 >> (8 * i)) & 0xff));
        }
        out = *reinterpret_cast<uint4 *>(hv);
        d = half_bits_to_float(*reinterpret_cast<const uint16_t *>(b));
    }
    *reinterpret_cast<uint4 *>(A + (int64_t)m * K + sb * 256 + lane * 8) = out;
    if ((lane & 3) == 0) D[(int64_t)blk * M_pad + m] = d;
}

// Activation prologue of the folded Q8_0 path: Q8_1 rows -> f16 panel [M_pad][K] of d*q (the f16 block
// scale times the code, exact in fp32 and rounded once to f16); rows past M are zero.  One warp per
// (row, 256 elements): lane l takes elements 8l .. 8l+7 of block l/4.  Also clears the device flag.
__global__ void act_panel_q81_fold_kernel(const uint8_t *__restrict__ xq, int M, int M_pad, int nsb,
                                          __half *__restrict__ A, unsigned long long *__restrict__ err) {
    if (blockIdx.x == 0 && threadIdx.x == 0) *err = 0ull;
    grid_launch_dependents();  // the GEMM may start its setup and weight loads beside this grid
    const int64_t wid = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (wid >= (int64_t)M_pad * nsb) return;
    const int m = (int)(wid / nsb), sb = (int)(wid % nsb);
    const int64_t K = (int64_t)nsb * 256;
    const int blk = sb * 8 + (lane >> 2);
    uint4 out = make_uint4(0, 0, 0, 0);
    if (m < M) {
        const uint8_t *b = xq + ((int64_t)m * nsb * 8 + blk) * kQ81Bytes;
        const uint32_t w0 = *reinterpret_cast<const uint32_t *>(b + 4 + (lane & 3) * 8);
        const uint32_t w1 = *reinterpret_cast<const uint32_t *>(b + 8 + (lane & 3) * 8);
        const float d = half_bits_to_float(*reinterpret_cast<const uint16_t *>(b));
        __half hv[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            hv[i] = __float2half_rn(d * (float)(int8_t)((w0 >> (8 * i)) & 0xff));
            hv[4 + i] = __float2half_rn(d * (float)(int8_t)((w1 >> (8 * i)) & 0xff));
        }
        out = *reinterpret_cast<uint4 *>(hv);
    }
    *reinterpret_cast<uint4 *>(A + (int64_t)m * K + sb * 256 + lane * 8) = out;
}

// Activation prologue of the folded K-quant path: Q8_K rows -> f16 panel [M_pad][K] of d*q (the fp32
// block scale times the code, rounded once to f16); rows past M are zero.  One warp per (row,
// super-block).  Also clears the device flag.
__global__ void act_panel_fold_kernel(const uint8_t *__restrict__ xq, int M, int M_pad, int nsb,
                                      __half *__restrict__ A, unsigned long long *__restrict__ err) {
    if (blockIdx.x == 0 && threadIdx.x == 0) *err = 0ull;
    grid_launch_dependents();  // the GEMM may start its setup and weight loads beside this grid
    const int64_t wid = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (wid >= (int64_t)M_pad * nsb) return;
    const int m = (int)(wid / nsb), sb = (int)(wid % nsb);
    const int64_t K = (int64_t)nsb * 256;
    uint4 out = make_uint4(0, 0, 0, 0);
    if (m < M) {
        const uint8_t *blk = xq + ((int64_t)m * nsb + sb) * kQ8KBytes;
        const uint32_t w0 = *reinterpret_cast<const uint32_t *>(blk + 4 + lane * 8);
        const uint32_t w1 = *reinterpret_cast<const uint32_t *>(blk + 8 + lane * 8);
        const float d = *reinterpret_cast<const float *>(blk);
        __half hv[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            hv[i] = __float2half_rn(d * (float)(int8_t)((w0 >> (8 * i)) & 0xff));
            hv[4 + i] = __float2half_rn(d * (float)(int8_t)((w1 >> (8 * i)) & 0xff));
        }
        out = *reinterpret_cast<uint4 *>(hv);
    }
    *reinterpret_cast<uint4 *>(A + (int64_t)m * K + sb * 256 + lane * 8) = out;
}

// Routed-expert prologue: list entry s (pair lists[s], routed order) goes to panel row prow[s] of the
// f16 code panel, the f16 bsum panel and the f32 scale panel; its activation is Q8_K row pair / top_k
// (one row per token) or row pair (one row per pair).  One warp per (list entry, super-block); only
// the lists' valid entries (offset[E-1] + count[E-1]: pairs with an invalid expert id are in no list)
// are read.  The padding rows between experts are left unwritten: they only feed token columns that
// are discarded.
__global__ void act_panel_grouped_kernel(const uint8_t *__restrict__ xq, int rows_per_token, int top_k, int nsb,
                                         int64_t pairs, const int *__restrict__ lists, const int *__restrict__ prow,
                                         const int *__restrict__ count, const int *__restrict__ offset, int n_experts,
                                         __half *__restrict__ A, __half *__restrict__ E, float *__restrict__ D,
                                         int64_t dstride) {
    const int64_t wid = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (wid >= pairs * nsb) return;
    const int64_t sidx = wid / nsb;
    if (sidx >= (int64_t)offset[n_experts - 1] + count[n_experts - 1]) return;
    const int sb = (int)(wid % nsb);
    const int p = lists[sidx];
    const int64_t r = prow[sidx];
    const int64_t src = rows_per_token == 1 ? p / top_k : p;
    const int64_t K = (int64_t)nsb * 256;
    const uint8_t *blk = xq + (src * nsb + sb) * kQ8KBytes;
    const uint32_t w0 = *reinterpret_cast<const uint32_t *>(blk + 4 + lane * 8);
    const uint32_t w1 = *reinterpret_cast<const uint32_t *>(blk + 8 + lane * 8);
    __half hv[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        hv[k] = __int2half_rn((int)(int8_t)((w0 >> (8 * k)) & 0xff));
        hv[4 + k] = __int2half_rn((int)(int8_t)((w1 >> (8 * k)) & 0xff));
    }
    *reinterpret_cast<uint4 *>(A + r * K + sb * 256 + lane * 8) = *reinterpret_cast<uint4 *>(hv);
    if (lane < 16) E[r * nsb * 16 + sb * 16 + lane] = __int2half_rn((int)reinterpret_cast<const int16_t *>(blk + 260)[lane]);
    if (lane == 0) D[(int64_t)sb * dstride + r] = *reinterpret_cast<const float *>(blk);
}

// Routed-expert prologue for Q8_0 weights: as act_panel_grouped_kernel, from Q8_1 rows -- f16 codes
// and the f32 (widened f16) scale of every 32-element block.  One warp per (list entry, 256 elements):
// lane l takes elements 8l .. 8l+7 of block l/4.
__global__ void act_panel_q81_grouped_kernel(const uint8_t *__restrict__ xq, int rows_per_token, int top_k, int nsb,
                                             int64_t pairs, const int *__restrict__ lists,
                                             const int *__restrict__ prow, const int *__restrict__ count,
                                             const int *__restrict__ offset, int n_experts, __half *__restrict__ A,
                                             float *__restrict__ D, int64_t dstride) {
    const int64_t wid = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (wid >= pairs * nsb) return;
    const int64_t sidx = wid / nsb;
    if (sidx >= (int64_t)offset[n_experts - 1] + count[n_experts - 1]) return;
    const int sb = (int)(wid % nsb);
    const int p = lists[sidx];
    const int64_t r = prow[sidx];
    const int64_t src = rows_per_token == 1 ? p / top_k : p;
    const int64_t K = (int64_t)nsb * 256;
    const int blk = sb * 8 + (lane >> 2);
    const uint8_t *b = xq + (src * nsb * 8 + blk) * kQ81Bytes;
    const uint32_t w0 = *reinterpret_cast<const uint32_t *>(b + 4 + (lane & 3) * 8);
    const uint32_t w1 = *reinterpret_cast<const uint32_t *>(b + 8 + (lane & 3) * 8);
    __half hv[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        hv[i] = __int2half_rn((int)(int8_t)((w0 >> (8 * i)) & 0xff));
        hv[4 + i] = __int2half_rn((int)(int8_t)((w1 >> (8 * i)) & 0xff));
    }
    *reinterpret_cast<uint4 *>(A + r * K + sb * 256 + lane * 8) = *reinterpret_cast<uint4 *>(hv);
    if ((lane & 3) == 0) D[(int64_t)blk * dstride + r] = half_bits_to_float(*reinterpret_cast<const uint16_t *>(b));
}

// ------------------------------------------------------------------ host side
struct TcWs {
    size_t off_flag, off_a, off_e, off_d, total;
    int M_pad;
};

static size_t al256(size_t v) { return (v + 255) & ~(size_t)255; }

// Workspace of the dense tensor-core GEMM: device flag, f16 code panel, (Q4_K/Q6_K) f16 bsum panel,
// f32 scale panel with one row per scale block (256 elements for Q8_K, 32 for Q8_1).
static TcWs tc_ws(kq_dtype wt, int64_t M, int64_t K, int tok = TC_TOK) {
    TcWs w{};
    w.M_pad = (int)((M + tok - 1) / tok * tok);
    const int64_t nsb = K / 256;
    const bool q8 = wt == KQ_Q8_0;
    size_t o = 0;
    w.off_flag = o; o += 256;
    w.off_a = o; o += al256((size_t)w.M_pad * K * 2);
    w.off_e = o; o += q8 ? 0 : al256((size_t)w.M_pad * nsb * 16 * 2);
    w.off_d = o; o += al256((size_t)w.M_pad * nsb * (q8 ? 8 : 1) * 4);
    w.total = o;
    return w;
}

bool tc_eligible(kq_dtype wt, int64_t M, int64_t N, int64_t K) {
    if (wt != KQ_Q4_K && wt != KQ_Q5_K && wt != KQ_Q6_K && wt != KQ_Q8_0) return false;
    // M <= 8 belongs to the batched-decode GEMV; from 9 rows on, a mostly empty 128-token tile still
    // beats the dp4a kernel (measured 3-10x at M = 16..64 on the decode and prefill shapes)
    if (M <= kGemvMaxBatch || N < 128) return false;
    if (K % 256 || K > (1 << 20) || M > (1 << 22) || N > (1 << 22)) return false;
    return true;
}

// Number of SMs of the current device (looked up once per device).
static int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return 152;
    }
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = 152;
        }
        cache[dev] = n;
    }
    return cache[dev];
}

// CTAs of the tensor-core kernel that the current device runs at once when they are launched in
// clusters of S (S = 1: one per SM, the shared-memory budget allows no more).  Clusters fill a GPC
// only in whole multiples of their size, so the count comes from the device's own cluster occupancy;
// without a device it falls back to GB300's 8 GPCs of 19 SMs.  Cached per device and S.
template <int DT>
static int resident_ctas(int S) {
    static int cache[64][4] = {};
    const int si = S == 1 ? 0 : S == 2 ? 1 : S == 4 ? 2 : 3;
    const int fallback = S == 1 ? 152 : 8 * (19 / S) * S;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return fallback;
    }
    if (cache[dev][si]) return cache[dev][si];
    int n = 0;
    if (S == 1) {
        n = sm_count();
    } else {
        auto kern = tc_gemm_kernel<DT, false, false>;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, 1, (unsigned)S);
        cfg.blockDim = dim3(TC_THREADS, 1, 1);
        cfg.dynamicSmemBytes = TcLayout<DT>::ALLOC;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = (unsigned)S;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TcLayout<DT>::ALLOC) ==
                cudaSuccess &&
            cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) == cudaSuccess)
            n = clusters * S;
        else
            cudaGetLastError();  // leave no error behind for the next launch check
    }
    if (n <= 0) n = fallback;
    cache[dev][si] = n;
    return n;
}

static int resident_ctas_dt(kq_dtype wt, int S) {
    switch (wt) {
    case KQ_Q4_K: return resident_ctas<KQ_Q4_K>(S);
    case KQ_Q5_K: return resident_ctas<KQ_Q5_K>(S);
    case KQ_Q6_K: return resident_ctas<KQ_Q6_K>(S);
    default: return resident_ctas<KQ_Q8_0>(S);
    }
}

// Split-K factor: the number of CTAs per output tile (a cluster along z).  Chosen with a small
// cost model measured on GB300: a persistent CTA (S = 1) pays its pipeline fill and drain (~2.5 us)
// once and walks its whole tiles at ~1.3 us (Q4_K), ~1.5 us (Q5_K) or ~1.75 us (Q6_K) per
// super-block; split-K clusters pay the fill in every wave, run their super-blocks ~15% slower
// (measured on the M = 2048, K = 14336 shapes) and add a cluster reduction (~1 us), and only as many
// clusters run at once as the device holds (resident_ctas) -- over power-of-two splits that leave at
// least two super-blocks per CTA.
static int tc_splits(kq_dtype wt, int64_t M, int64_t N, int64_t K) {
    if (wt == KQ_Q8_0) return 1;  // keeps every output's blocks in one ascending sum (bit-exact)
    const int64_t tiles = ((M + TC_TOK - 1) / TC_TOK) * ((N + TC_ROWS - 1) / TC_ROWS);
    const int nsb = (int)(K / 256);
    const double t_sb = wt == KQ_Q4_K ? 1.3 : wt == KQ_Q5_K ? 1.5 : 1.75, t_fill = 2.5, t_red = 1.0;
    int best = 1;
    double best_t = t_fill + (double)((tiles + resident_ctas_dt(wt, 1) - 1) / resident_ctas_dt(wt, 1)) * nsb * t_sb;
    for (int S = 2; S <= 8; S *= 2) {
        const int per = (nsb + S - 1) / S;
        if (per < 2) break;
        if ((nsb + per - 1) / per != S) continue;  // S must be exactly realisable
        const int64_t usable = resident_ctas_dt(wt, S);
        const int64_t waves = (tiles * S + usable - 1) / usable;
        const double t = (double)waves * (t_fill + per * 1.15 * t_sb + t_red);
        if (t < best_t - 1e-9) { best_t = t; best = S; }
    }
    return best;
}

// The split tail: a persistent launch whose last wave would hold R < one wave of tiles runs its whole
// waves persistent and the R leftover tiles as a second launch of split-K clusters (S' CTAs per tile,
// all in one wave of clusters), when the cost model (the same figures, plus ~2 us for the second
// launch) says it saves at least 3%.  tail_split = 1: no tail.
struct TcTail {
    int64_t tiles;
    int split;
};

static TcTail tc_tail(kq_dtype wt, int64_t M, int64_t N, int64_t K) {
    TcTail tl{0, 1};
    if (wt == KQ_Q8_0 || tc_splits(wt, M, N, K) != 1) return tl;
    const int64_t tiles = ((M + TC_TOK - 1) / TC_TOK) * ((N + TC_ROWS - 1) / TC_ROWS);
    const int nsb = (int)(K / 256);
    const double t_sb = wt == KQ_Q4_K ? 1.3 : wt == KQ_Q5_K ? 1.5 : 1.75, t_fill = 2.5, t_red = 1.0, t_launch = 2.0;
    const int64_t G = resident_ctas_dt(wt, 1), W = tiles / G, R = tiles - W * G;
    if (W == 0 || R == 0) return tl;
    double best = t_fill + (double)(W + 1) * nsb * t_sb;
    const double keep = 0.97 * best;
    for (int S = 2; S <= 4; S *= 2) {
        const int per = (nsb + S - 1) / S;
        if (per < 2) break;
        if ((nsb + per - 1) / per != S || R * S > resident_ctas_dt(wt, S)) continue;
        const double t = t_fill + (double)W * nsb * t_sb + (t_fill + per * 1.15 * t_sb + t_red) + t_launch;
        if (t < keep && t < best - 1e-9) { best = t; tl = TcTail{R, S}; }
    }
    return tl;
}

int tc_split_factor(kq_dtype wt, int64_t M, int64_t N, int64_t K) {
    if (!tc_eligible(wt, M, N, K)) return 0;
    return std::max(tc_splits(wt, M, N, K), tc_tail(wt, M, N, K).split);
}

size_t tc_workspace_bytes(kq_dtype wt, int64_t M, int64_t N, int64_t K) {
    if (!tc_eligible(wt, M, N, K)) return 0;
    // room for either form: the exact kernels' 128-token tiles and the folded mode's 256-token tiles
    return std::max(tc_ws(wt, M, K).total, tc_ws(wt, M, K, TcCfg<KQ_Q8_0F>::TOK).total);
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


// One launch of the tensor-core kernel over activation panels built by a prologue.
struct TcLaunch {
    const uint8_t *w;
    float *y;
    int64_t ldy, M, N, K;
    uint8_t *A, *E;       // f16 code panel [rows][K], f16 bsum panel [rows][K/16]
    float *D;             // f32 scale panel [K/256][dstride]
    int64_t rows;         // panel rows (tensor-map extent; tiles past it read zeros)
    int64_t dstride;      // scale-panel row stride: >= any tile's first row + 128, a multiple of 4
    int m_tiles;          // token tiles (dense) or tile-table slots (grouped, an upper bound)
    int nsplit;           // > 1: split-K clusters, one CTA per (tile, split); else persistent CTAs
    unsigned long long *err;
    bool grouped;
    const int *tiles, *tile_count, *count, *offset, *poff, *lists;
    uint8_t *hq;          // non-NULL: fused SwiGLU -> Q8_K output (grouped gate/up only), y unused
    float *scr;           // its scratch: tc_swq_scratch_bytes()
    const TcDebug *dbg;   // NULL, or the debug read-out / wait-limit hooks
    int64_t tail_tiles;   // > 0 (dense, nsplit = 1): the last tail_tiles tiles run as a split-K launch
    int tail_split;       // of tail_split CTAs per tile
    bool pdl;             // the first launch may start while the prologue kernel before it finishes
};

template <int DT>
static kq_status launch_tc(const TcLaunch &a, cudaStream_t st) {
    using Lay = TcLayout<DT>;
    auto encode = get_encode();
    if (!encode) return fail(KQ_ERR_CUDA, "kq_gemm: cuTensorMapEncodeTiled unavailable");
    const int64_t nsb = a.K / 256;
    CUtensorMap tmA, tmE;
    {
        cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.rows};
        cuuint64_t strides[1] = {(cuuint64_t)a.K * 2};
        cuuint32_t box[2] = {TC_KB, (cuuint32_t)TcCfg<DT>::TOK};
        cuuint32_t es[2] = {1, 1};
        CUresult r = encode(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.A, dims, strides, box, es,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(KQ_ERR_CUDA, "kq_gemm: tensor map A encode failed (%d)", (int)r);
    }
    if (!TcCfg<DT>::EXT) {
        tmE = tmA;  // no bsum operand
    } else {
        cuuint64_t dims[2] = {(cuuint64_t)nsb * 16, (cuuint64_t)a.rows};
        cuuint64_t strides[1] = {(cuuint64_t)nsb * 32};
        cuuint32_t box[2] = {16, TC_TOK};
        cuuint32_t es[2] = {1, 1};
        CUresult r = encode(&tmE, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.E, dims, strides, box, es,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(KQ_ERR_CUDA, "kq_gemm: tensor map E encode failed (%d)", (int)r);
    }
    TcParams p{};
    p.w = a.w;
    p.da = a.D;
    p.y = a.y;
    p.ldy = a.ldy;
    p.M = (int)a.M; p.N = (int)a.N; p.K = (int)a.K; p.M_pad = (int)a.dstride;
    const int S = a.nsplit;
    p.nsplit = S;
    p.sb_per_split = (int)((nsb + S - 1) / S);
    p.err = a.err;
    p.grouped = a.grouped ? 1 : 0;
    p.tiles = a.tiles; p.tile_count = a.tile_count; p.count = a.count;
    p.offset = a.offset; p.poff = a.poff; p.lists = a.lists;
    p.n_tiles = (int)((a.N + TC_ROWS - 1) / TC_ROWS);
    p.m_tiles = a.m_tiles;
    p.persistent = S > 1 ? 0 : 1;
    p.swq = a.hq ? 1 : 0;
    p.hq = a.hq;
    p.scr = a.scr;
    p.wait_ns = a.dbg ? a.dbg->wait_ns : kTcWaitNs;
    p.withhold = a.dbg && a.dbg->withhold_act ? 1 : 0;
    const bool dbg_sums = a.dbg && a.dbg->sums;
    p.dbg = dbg_sums ? a.dbg->sums : nullptr;
    p.dbg_nblk = (int)(TcCfg<DT>::Q8 ? a.K / 32 : a.K / 256);
    if (p.swq && (S != 1 || !a.grouped || a.N % 512 || !a.scr))
        return fail(KQ_ERR_INVALID_ARG, "kq_gemm (tensor core): fused SwiGLU needs a routed, unsplit launch");
    if (p.swq && dbg_sums) return fail(KQ_ERR_INVALID_ARG, "kq_gemm (tensor core): no debug read-out with fused SwiGLU");
    const int64_t tiles = (int64_t)p.n_tiles * a.m_tiles;
    const int64_t units = p.swq ? tiles / 4 : tiles;
    if (tiles > 0x7fffffff) return fail(KQ_ERR_INVALID_ARG, "kq_gemm: too many tiles");
    auto kern = p.swq ? tc_gemm_kernel<DT, true, false>
                      : dbg_sums ? tc_gemm_kernel<DT, false, true> : tc_gemm_kernel<DT, false, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::ALLOC);
    if (e != cudaSuccess) return fail(KQ_ERR_CUDA, "kq_gemm: %s", cudaGetErrorString(e));
    const int64_t R = a.tail_tiles;  // > 0: the last R tiles go to a second, split-K launch
    if (R && (S != 1 || a.grouped || p.swq || R >= tiles || a.tail_split < 2))
        return fail(KQ_ERR_INVALID_ARG, "kq_gemm (tensor core): invalid split tail");
    // Dense launches follow their activation prologue in the stream and may start beside its last
    // blocks: the CTAs set up, load and convert their first weights, and wait on the prologue only
    // before the first activation, bsum or scale access.  Routed launches read tile tables that
    // earlier kernels wrote from their first instruction, so they take no such head start.
    bool pdl = a.pdl && !a.grouped;
    auto launch = [&](TcParams q, int split, dim3 grid) -> kq_status {
        q.nsplit = split;
        q.sb_per_split = (int)((nsb + split - 1) / split);
        q.persistent = split > 1 ? 0 : 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(TC_THREADS, 1, 1);
        cfg.dynamicSmemBytes = Lay::ALLOC;
        cfg.stream = st;
        cudaLaunchAttribute attr[2];
        unsigned na = 0;
        if (split > 1) {
            attr[na].id = cudaLaunchAttributeClusterDimension;
            attr[na].val.clusterDim.x = 1;
            attr[na].val.clusterDim.y = 1;
            attr[na].val.clusterDim.z = (unsigned)split;
            ++na;
        }
        if (pdl) {
            attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[na].val.programmaticStreamSerializationAllowed = 1;
            ++na;
        }
        cfg.attrs = attr;
        cfg.numAttrs = na;
        pdl = false;  // a second (split-tail) launch waits for the first in full
        cudaError_t le = cudaLaunchKernelEx(&cfg, kern, tmA, tmE, q);
        if (le != cudaSuccess)
            return fail(KQ_ERR_CUDA, "kq_gemm (tensor core): launch failed: %s", cudaGetErrorString(le));
        return KQ_OK;
    };
    p.unit_base = 0;
    p.unit_limit = 0x7fffffff;
    if (S > 1) return launch(p, S, dim3((unsigned)p.n_tiles, (unsigned)a.m_tiles, (unsigned)S));
    if (!R) return launch(p, 1, dim3((unsigned)std::min<int64_t>(units, sm_count()), 1, 1));  // one CTA per SM
    // whole waves persistent, then the R leftover tiles as split-K clusters (one tile per cluster)
    TcParams q = p;
    q.unit_limit = (int)(tiles - R);
    kq_status ks = launch(q, 1, dim3((unsigned)std::min<int64_t>(tiles - R, sm_count()), 1, 1));
    if (ks != KQ_OK) return ks;
    q.unit_base = (int)(tiles - R);
    q.unit_limit = (int)tiles;
    return launch(q, a.tail_split, dim3((unsigned)R, 1, (unsigned)a.tail_split));
}

static kq_status launch_tc_dt(kq_dtype wt, const TcLaunch &a, cudaStream_t st, bool fold = false, int tok = TC_TOK) {
    if (fold && tok == TC_TOK) {
        switch (wt) {
        case KQ_Q4_K: return launch_tc<KQ_Q4_KF + KQ_FOLD128>(a, st);
        case KQ_Q5_K: return launch_tc<KQ_Q5_KF + KQ_FOLD128>(a, st);
        case KQ_Q6_K: return launch_tc<KQ_Q6_KF + KQ_FOLD128>(a, st);
        default: return launch_tc<KQ_Q8_0F + KQ_FOLD128>(a, st);
        }
    }
    if (fold) {
        switch (wt) {
        case KQ_Q4_K: return launch_tc<KQ_Q4_KF>(a, st);
        case KQ_Q5_K: return launch_tc<KQ_Q5_KF>(a, st);
        case KQ_Q6_K: return launch_tc<KQ_Q6_KF>(a, st);
        default: return launch_tc<KQ_Q8_0F>(a, st);
        }
    }
    switch (wt) {
    case KQ_Q4_K: return launch_tc<KQ_Q4_K>(a, st);
    case KQ_Q5_K: return launch_tc<KQ_Q5_K>(a, st);
    case KQ_Q6_K: return launch_tc<KQ_Q6_K>(a, st);
    default: return launch_tc<KQ_Q8_0>(a, st);
    }
}

// Token-tile width of the folded mode: 256 tokens once they give at least as many tiles as there are
// SMs, else 128 (which may also split K).
static int fold_tok(int64_t M, int64_t N) {
    const int64_t tiles256 = ((M + 255) / 256) * ((N + TC_ROWS - 1) / TC_ROWS);
    return tiles256 >= sm_count() ? 256 : TC_TOK;
}

// The tensor-core GEMM from quantised rows xq, or (xf != NULL, Q4_K/Q5_K/Q6_K) from fp32 rows xf of
// stride ldx quantised to Q8_K inside the prologue.
static kq_status tc_gemm_impl(kq_dtype wt, const uint8_t *w, const uint8_t *xq, const float *xf, int64_t ldx, int64_t M,
                              int64_t N, int64_t K, float *y, int64_t ldy, uint8_t *workspace, cudaStream_t st,
                              const TcDebug *dbg, bool fold = false) {
    const int tok = fold ? fold_tok(M, N) : TC_TOK;
    const TcWs L = tc_ws(wt, M, K, tok);
    if ((N + TC_ROWS - 1) / TC_ROWS > 65535 || L.M_pad / tok > 65535)
        return fail(KQ_ERR_INVALID_ARG, "kq_gemm: shape too large for the tensor-core grid");
    const int64_t nsb = K / 256;
    const int64_t warps = (int64_t)L.M_pad * nsb;
    if (xf && fold) {
        if (wt == KQ_Q8_0) return fail(KQ_ERR_UNSUPPORTED_DTYPE, "kq_gemm_f32: Q8_0 weights take Q8_1 activations");
        const bool vec = (reinterpret_cast<uintptr_t>(xf) & 15) == 0 && ldx % 4 == 0;
        auto kern = vec ? act_panel_f32_fold_kernel<true> : act_panel_f32_fold_kernel<false>;
        kern<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(xf, ldx, (int)M, L.M_pad, (int)nsb,
                                                          reinterpret_cast<__half *>(workspace + L.off_a),
                                                          reinterpret_cast<unsigned long long *>(workspace + L.off_flag));
    } else if (xf) {
        if (wt == KQ_Q8_0) return fail(KQ_ERR_UNSUPPORTED_DTYPE, "kq_gemm_f32: Q8_0 weights take Q8_1 activations");
        const bool vec = (reinterpret_cast<uintptr_t>(xf) & 15) == 0 && ldx % 4 == 0;
        auto kern = vec ? act_panel_f32_kernel<true> : act_panel_f32_kernel<false>;
        kern<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(
            xf, ldx, (int)M, L.M_pad, (int)nsb, reinterpret_cast<__half *>(workspace + L.off_a),
            reinterpret_cast<__half *>(workspace + L.off_e), reinterpret_cast<float *>(workspace + L.off_d),
            reinterpret_cast<unsigned long long *>(workspace + L.off_flag));
    } else if (fold && wt == KQ_Q8_0) {
        act_panel_q81_fold_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(
            xq, (int)M, L.M_pad, (int)nsb, reinterpret_cast<__half *>(workspace + L.off_a),
            reinterpret_cast<unsigned long long *>(workspace + L.off_flag));
    } else if (fold) {
        act_panel_fold_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(
            xq, (int)M, L.M_pad, (int)nsb, reinterpret_cast<__half *>(workspace + L.off_a),
            reinterpret_cast<unsigned long long *>(workspace + L.off_flag));
    } else if (wt == KQ_Q8_0)
        act_panel_q81_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(
            xq, (int)M, L.M_pad, (int)nsb, reinterpret_cast<__half *>(workspace + L.off_a),
            reinterpret_cast<float *>(workspace + L.off_d), reinterpret_cast<unsigned long long *>(workspace + L.off_flag));
    else
        act_panel_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(
            xq, (int)M, L.M_pad, (int)nsb, reinterpret_cast<__half *>(workspace + L.off_a),
            reinterpret_cast<__half *>(workspace + L.off_e), reinterpret_cast<float *>(workspace + L.off_d),
            reinterpret_cast<unsigned long long *>(workspace + L.off_flag));
    kq_status s = check_launch("kq_gemm (activation panel)");
    if (s != KQ_OK) return s;
    TcLaunch a{};
    a.w = w; a.y = y; a.ldy = ldy; a.M = M; a.N = N; a.K = K;
    a.A = workspace + L.off_a; a.E = workspace + L.off_e; a.D = reinterpret_cast<float *>(workspace + L.off_d);
    a.rows = L.M_pad; a.dstride = L.M_pad; a.m_tiles = (int)(L.M_pad / tok);
    // the 256-token folded tiles are never split (their epilogue writes y); the 128-token ones split as
    // the exact kernels do, with the Q4_K cost model (their steps cost alike)
    a.nsplit = !fold ? tc_splits(wt, M, N, K) : tok == TC_TOK ? tc_splits(KQ_Q4_K, M, N, K) : 1;
    if (!fold) {
        const TcTail tl = tc_tail(wt, M, N, K);
        a.tail_tiles = tl.tiles;
        a.tail_split = tl.split;
    }
    a.err = reinterpret_cast<unsigned long long *>(workspace + L.off_flag);
    a.dbg = dbg;
    a.pdl = true;
    if (fold && dbg && dbg->sums) return fail(KQ_ERR_INVALID_ARG, "kq_gemm_ex: no integer sums with folded scales");
    s = launch_tc_dt(wt, a, st, fold, tok);
    if (s == KQ_OK) count_launch(R_MMQ_TC, a.tail_tiles ? 3 : 2);  // prologue, GEMM (and its split tail)
    return s;
}

kq_status tc_gemm(kq_dtype wt, const uint8_t *w, const uint8_t *xq, int64_t M, int64_t N, int64_t K, float *y,
                  int64_t ldy, uint8_t *workspace, cudaStream_t st, const TcDebug *dbg) {
    return tc_gemm_impl(wt, w, xq, nullptr, 0, M, N, K, y, ldy, workspace, st, dbg);
}

kq_status tc_gemm_folded(kq_dtype wt, const uint8_t *w, const uint8_t *xq, int64_t M, int64_t N, int64_t K, float *y,
                         int64_t ldy, uint8_t *workspace, cudaStream_t st, const TcDebug *dbg) {
    return tc_gemm_impl(wt, w, xq, nullptr, 0, M, N, K, y, ldy, workspace, st, dbg, true);
}

kq_status tc_gemm_f32(kq_dtype wt, const uint8_t *w, const float *x, int64_t ldx, int64_t M, int64_t N, int64_t K,
                      float *y, int64_t ldy, uint8_t *workspace, cudaStream_t st, bool fold) {
    return tc_gemm_impl(wt, w, nullptr, x, ldx, M, N, K, y, ldy, workspace, st, nullptr, fold);
}

// ---- routed experts on the tensor cores
bool tc_grouped_eligible(kq_dtype wt, int64_t N, int64_t K) {
    return (wt == KQ_Q4_K || wt == KQ_Q5_K || wt == KQ_Q6_K || wt == KQ_Q8_0) && N % 16 == 0 && K % 256 == 0 &&
           K <= (1 << 20) &&
           N <= (1 << 22);
}

// Fused SwiGLU scratch: two 128-token x 256-column fp32 tiles per persistent CTA.
size_t tc_swq_scratch_bytes() { return (size_t)sm_count() * 2 * TC_TOK * 256 * sizeof(float); }

// Panels of the routed rows: f16 codes, (Q4_K/Q6_K) f16 bsums, f32 scales with one row per scale block
// (256 elements for Q8_K activations, 32 for Q8_1).
TcGroupedPanels tc_grouped_panels(kq_dtype wt, int64_t pairs, int64_t E, int64_t K) {
    TcGroupedPanels g{};
    const int64_t nsb = K / 256;
    const bool q8 = wt == KQ_Q8_0;
    g.rows = pairs + 3 * E;                      // every expert's rows padded to a multiple of 4
    g.dstride = ((g.rows + TC_TOK) + 3) & ~(int64_t)3;
    size_t o = 0;
    g.off_a = o; o += al256((size_t)g.rows * K * 2);
    g.off_e = o; o += q8 ? 0 : al256((size_t)g.rows * nsb * 32);
    g.off_d = o; o += al256((size_t)nsb * (q8 ? 8 : 1) * g.dstride * 4);
    g.bytes = o;
    return g;
}

kq_status tc_gemm_grouped(kq_dtype wt, const uint8_t *w, const uint8_t *xq, int rows_per_token, int top_k,
                          int64_t pairs, int64_t E, int64_t N, int64_t K, float *y, uint8_t *panels,
                          const int *tiles, const int *tile_count, int64_t max_tiles, const int *count,
                          const int *offset, const int *poff, const int *lists, const int *prow,
                          unsigned long long *err, uint8_t *hq, float *scr, cudaStream_t st, const TcDebug *dbg) {
    const TcGroupedPanels G = tc_grouped_panels(wt, pairs, E, K);
    if ((N + TC_ROWS - 1) / TC_ROWS > 65535 || max_tiles > 65535)
        return fail(KQ_ERR_INVALID_ARG, "kq_gemm_grouped: shape too large for the tensor-core grid");
    const int64_t nsb = K / 256;
    const int64_t warps = pairs * nsb;
    if (wt == KQ_Q8_0)
        act_panel_q81_grouped_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(
            xq, rows_per_token, top_k, (int)nsb, pairs, lists, prow, count, offset, (int)E,
            reinterpret_cast<__half *>(panels + G.off_a), reinterpret_cast<float *>(panels + G.off_d), G.dstride);
    else
        act_panel_grouped_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(
            xq, rows_per_token, top_k, (int)nsb, pairs, lists, prow, count, offset, (int)E,
            reinterpret_cast<__half *>(panels + G.off_a),
            reinterpret_cast<__half *>(panels + G.off_e), reinterpret_cast<float *>(panels + G.off_d), G.dstride);
    kq_status s = check_launch("kq_gemm_grouped (activation panel)");
    if (s != KQ_OK) return s;
    TcLaunch a{};
    a.w = w; a.y = y; a.ldy = N; a.M = pairs; a.N = N; a.K = K;
    a.A = panels + G.off_a; a.E = panels + G.off_e; a.D = reinterpret_cast<float *>(panels + G.off_d);
    a.rows = G.rows; a.dstride = G.dstride; a.m_tiles = (int)max_tiles;
    a.nsplit = 1;
    a.err = err;
    a.grouped = true;
    a.tiles = tiles; a.tile_count = tile_count; a.count = count; a.offset = offset; a.poff = poff; a.lists = lists;
    a.hq = hq; a.scr = scr;
    a.dbg = dbg;
    s = launch_tc_dt(wt, a, st);
    if (s == KQ_OK) count_launch(R_MMQ_TC, 2);
    return s;
}

}  // namespace kq
