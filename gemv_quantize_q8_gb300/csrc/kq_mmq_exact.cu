// kq_mmq_exact.cu -- exact integer MMQ tile kernel (dp4a), its debug-partials mode, and the
// routed-expert (MUL_MAT_ID) variant.
//
// Each 64x64 output tile loops over 256-element super-blocks.  Per super-block the block stages
// ONE activation tile (64 token rows of Q8_K / Q8_1) and one weight tile (64 rows, unpacked to
// int8 codes) in shared memory, and all eight warps read the same activation rows from it -- the
// cooperative activation share that vllm.cpp PR #3035 ("scope a cooperative activation share for
// the WMMA kernels") identifies as the mechanism its per-warp kernel lacked.
//
// The arithmetic is the CPU oracle's, term for term: integer sub-block dots P_j (dp4a), integer
// scale/min sums, one fp32 expression per super-block (Q8_0: per 32-block) built from separately
// rounded multiplies, accumulated in ascending K order per output.  Results are bit-identical to
// the sequential CPU order (vllm.cpp PR #2890, keep-quant provider: "integer dots ... in the CPU
// accumulation order").  This kernel serves kq_debug_partials, the routed-expert GEMM and the
// small-M shapes of kq_gemm; the tensor-core kernel serves large prefill shapes.
#include "kq_internal.cuh"
#include "kq_mmq_exact.cuh"

namespace kq {

constexpr int BM = 64, BN = 64, kRowPad = 272;  // 256 codes + 16 pad bytes per row

struct ExactSmem {
    int8_t aq[BM][kRowPad];
    int8_t wq[BN][kRowPad];
    float ad[BM][8];          // Q8_K: [m][0]; Q8_1: per 32-block
    int16_t abs_[BM][16];     // Q8_K bsums
    int wsc[BN][16];          // Q4_K: 8 scales; Q6_K: 16 scales
    int wmn[BN][8];           // Q4_K mins
    float wd[BN][8];          // Q4_K: d, dmin; Q6_K: d; Q8_0: 8 block scales
};

template <int DT>
__device__ __forceinline__ void stage_weights(ExactSmem &s, const uint8_t *__restrict__ wtile, int64_t nchunk,
                                              int c, int rows_valid) {
    // wtile points at the tile's first row group; the 4 row groups are nchunk chunks apart.
    // Rows at or past rows_valid (a multiple of 16) do not exist in memory and stage as zeros.
    const int tid = threadIdx.x;
    const int cb = chunk_bytes(DT);
    if (rows_valid < BN) {
        for (int u = tid; u < (BN - rows_valid) * (kRowPad / 16); u += 256) {
            const int row = rows_valid + u / (kRowPad / 16), seg = u % (kRowPad / 16);
            *reinterpret_cast<uint4 *>(&s.wq[row][seg * 16]) = make_uint4(0, 0, 0, 0);
        }
        for (int row = rows_valid + tid; row < BN; row += 256) {
#pragma unroll
            for (int j = 0; j < 16; ++j) s.wsc[row][j] = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) { s.wmn[row][j] = 0; s.wd[row][j] = 0.0f; }
        }
    }
    if (DT == KQ_Q4_K || DT == KQ_Q5_K || DT == KQ_Q6_K) {
        // unit = (row, kblock kb, 16-byte half seg): low nibbles -> elements 64kb+16seg+i,
        // high nibbles -> 64kb+32+16seg+i; Q5_K adds one high bit per element (bits 2kb / 2kb+1 of the
        // row's high-bit bytes), Q6_K two high bits and the -32 offset.
        for (int u = tid; u < rows_valid * 8; u += 256) {
            const int row = u >> 3, kb = (u >> 1) & 3, seg = u & 1;
            const uint8_t *ch = wtile + ((row >> 4) * nchunk + c) * (int64_t)cb;
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(ch + kb * 512 + (row & 15) * 32 + seg * 16));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t lo[4], hi[4];
            if (DT == KQ_Q6_K) {
                const uint4 h = __ldg(reinterpret_cast<const uint4 *>(ch + 2048 + kb * 256 + (row & 15) * 16));
                const uint32_t hb[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    lo[i] = __vsub4((w[i] & 0x0f0f0f0fu) | (((hb[i] >> (2 * seg)) & 0x03030303u) << 4), 0x20202020u);
                    hi[i] = __vsub4(((w[i] >> 4) & 0x0f0f0f0fu) | (((hb[i] >> (4 + 2 * seg)) & 0x03030303u) << 4),
                                    0x20202020u);
                }
            } else {
                uint32_t hq[4] = {0u, 0u, 0u, 0u};
                if (DT == KQ_Q5_K) {
                    const uint4 h = __ldg(reinterpret_cast<const uint4 *>(ch + 2304 + (row & 15) * 32 + seg * 16));
                    hq[0] = h.x; hq[1] = h.y; hq[2] = h.z; hq[3] = h.w;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    lo[i] = (w[i] & 0x0f0f0f0fu) | (((hq[i] >> (2 * kb)) & 0x01010101u) << 4);
                    hi[i] = ((w[i] >> 4) & 0x0f0f0f0fu) | (((hq[i] >> (2 * kb + 1)) & 0x01010101u) << 4);
                }
            }
            *reinterpret_cast<uint4 *>(&s.wq[row][64 * kb + 16 * seg]) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            *reinterpret_cast<uint4 *>(&s.wq[row][64 * kb + 32 + 16 * seg]) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        }
        if (tid < rows_valid) {
            const uint8_t *ch = wtile + ((tid >> 4) * nchunk + c) * (int64_t)cb;
            if (DT == KQ_Q4_K || DT == KQ_Q5_K) {
                const uint8_t *h = ch + 2048 + (tid & 15) * 16;
                s.wd[tid][0] = half_bits_to_float(*reinterpret_cast<const uint16_t *>(h));
                s.wd[tid][1] = half_bits_to_float(*reinterpret_cast<const uint16_t *>(h + 2));
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    int sc, mn;
                    q4k_scale_min(h + 4, j, sc, mn);
                    s.wsc[tid][j] = sc;
                    s.wmn[tid][j] = mn;
                }
            } else {
                const int8_t *sc = reinterpret_cast<const int8_t *>(ch + 3072 + (tid & 15) * 16);
#pragma unroll
                for (int j = 0; j < 16; ++j) s.wsc[tid][j] = sc[j];
                s.wd[tid][0] = half_bits_to_float(*reinterpret_cast<const uint16_t *>(ch + 3328 + (tid & 15) * 2));
            }
        }
    } else {
        for (int u = tid; u < rows_valid * 16; u += 256) {
            const int row = u >> 4, seg = u & 15;
            const uint8_t *ch = wtile + ((row >> 4) * nchunk + c) * (int64_t)cb;
            *reinterpret_cast<uint4 *>(&s.wq[row][seg * 16]) =
                __ldg(reinterpret_cast<const uint4 *>(ch + (seg >> 2) * 1024 + (row & 15) * 64 + (seg & 3) * 16));
        }
        for (int u = tid; u < rows_valid * 8; u += 256) {
            const int row = u >> 3, b = u & 7;
            const uint8_t *ch = wtile + ((row >> 4) * nchunk + c) * (int64_t)cb;
            s.wd[row][b] = half_bits_to_float(*reinterpret_cast<const uint16_t *>(ch + 4096 + (row & 15) * 16 + 2 * b));
        }
    }
}

// Stage the activation tile of chunk c.  arow[mi] = source activation row or -1 (zero row).
template <int DT>
__device__ __forceinline__ void stage_acts(ExactSmem &s, const uint8_t *__restrict__ xq, const int64_t *arow,
                                           int64_t nchunk, int c) {
    const int tid = threadIdx.x;
    if (DT != KQ_Q8_0) {
        for (int u = tid; u < BM * 16; u += 256) {
            const int mi = u >> 4, seg = u & 15;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (arow[mi] >= 0) {
                const uint32_t *src =
                    reinterpret_cast<const uint32_t *>(xq + (arow[mi] * nchunk + c) * kQ8KBytes + 4 + seg * 16);
                v = make_uint4(src[0], src[1], src[2], src[3]);
            }
            *reinterpret_cast<uint4 *>(&s.aq[mi][seg * 16]) = v;
        }
        for (int u = tid; u < BM * 17; u += 256) {
            const int mi = u / 17, k = u % 17;
            const uint8_t *blk = arow[mi] >= 0 ? xq + (arow[mi] * nchunk + c) * kQ8KBytes : nullptr;
            if (k == 16) s.ad[mi][0] = blk ? *reinterpret_cast<const float *>(blk) : 0.0f;
            else s.abs_[mi][k] = blk ? reinterpret_cast<const int16_t *>(blk + 260)[k] : (int16_t)0;
        }
    } else {
        for (int u = tid; u < BM * 8; u += 256) {
            const int mi = u >> 3, b = u & 7;
            uint32_t *dst = reinterpret_cast<uint32_t *>(&s.aq[mi][32 * b]);
            if (arow[mi] >= 0) {
                const uint8_t *blk = xq + (arow[mi] * nchunk * 8 + (int64_t)c * 8 + b) * kQ81Bytes;
                const uint32_t *src = reinterpret_cast<const uint32_t *>(blk + 4);
#pragma unroll
                for (int i = 0; i < 8; ++i) dst[i] = src[i];
                s.ad[mi][b] = half_bits_to_float(*reinterpret_cast<const uint16_t *>(blk));
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) dst[i] = 0u;
                s.ad[mi][b] = 0.0f;
            }
        }
    }
}

// MODE 0: fp32 output.  MODE 1: int32 partials.
// GROUPED: blockIdx.y indexes the routed tile table instead of a dense M tile.
template <int DT, int MODE, bool GROUPED>
__global__ void __launch_bounds__(256) mmq_exact_kernel(MmqExactArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    ExactSmem &s = *reinterpret_cast<ExactSmem *>(smem_raw);
    __shared__ int64_t arow[BM];
    __shared__ int64_t yrow[BM];
    __shared__ int64_t wrow_base;

    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const int64_t n0 = (int64_t)blockIdx.x * BN;
    if (tid < BM) {
        int64_t ar = -1, yr = -1;
        if (!GROUPED) {
            const int64_t m = (int64_t)blockIdx.y * BM + tid;
            if (m < a.M) { ar = m; yr = m; }
        } else {
            const int ntile = a.tile_count[0];
            if ((int)blockIdx.y < ntile) {
                const int e = a.tiles[2 * blockIdx.y], start = a.tiles[2 * blockIdx.y + 1];
                const int cnt_e = a.expert_count[e];
                const int idx = start + tid;
                if (idx < cnt_e) {
                    const int p = a.lists[a.expert_offset[e] + idx];
                    yr = p;
                    ar = a.rows_per_token == 1 ? p / a.top_k : p;
                }
            }
        }
        arow[tid] = ar;
        yrow[tid] = yr;
    }
    if (tid == 0) {
        int64_t base = 0;
        if (GROUPED && (int)blockIdx.y < a.tile_count[0]) base = (int64_t)a.tiles[2 * blockIdx.y] * a.N;
        wrow_base = base;
    }
    __syncthreads();
    if (GROUPED && (int)blockIdx.y >= a.tile_count[0]) return;
    if (n0 >= a.N) return;

    const int64_t nchunk = a.K / 256;
    const int cb = chunk_bytes(DT);
    const uint8_t *wtile = a.w + ((wrow_base + n0) / 16) * nchunk * (int64_t)cb;

    constexpr int nsub = DT == KQ_Q6_K ? 16 : 8;
    constexpr int L = 256 / nsub;  // sub-block length: 32 or 16
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

    const int64_t groups_left = (a.N + 15) / 16 - n0 / 16;
    const int rows_valid = groups_left >= 4 ? BN : (int)groups_left * 16;
    for (int c = 0; c < (int)nchunk; ++c) {
        stage_weights<DT>(s, wtile, nchunk, c, rows_valid);
        stage_acts<DT>(s, a.xq, arow, nchunk, c);
        __syncthreads();
        int sumi[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) sumi[i][j] = 0;
#pragma unroll 1
        for (int sb = 0; sb < nsub; ++sb) {
            int P[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) P[i][j] = 0;
#pragma unroll
            for (int k4 = 0; k4 < L / 16; ++k4) {
                int4 av[4], wv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) av[i] = *reinterpret_cast<const int4 *>(&s.aq[ty + 16 * i][sb * L + 16 * k4]);
#pragma unroll
                for (int j = 0; j < 4; ++j) wv[j] = *reinterpret_cast<const int4 *>(&s.wq[tx + 16 * j][sb * L + 16 * k4]);
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        P[i][j] = dp4a(wv[j].x, av[i].x, P[i][j]);
                        P[i][j] = dp4a(wv[j].y, av[i].y, P[i][j]);
                        P[i][j] = dp4a(wv[j].z, av[i].z, P[i][j]);
                        P[i][j] = dp4a(wv[j].w, av[i].w, P[i][j]);
                    }
            }
            if (MODE == 1) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int64_t m = (int64_t)blockIdx.y * BM + ty + 16 * i, n = n0 + tx + 16 * j;
                        if (m < a.M && n < a.N)
                            a.partials[(m * a.N + n) * (nchunk * nsub) + (int64_t)c * nsub + sb] = P[i][j];
                    }
            } else if (DT == KQ_Q8_0) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float t1 = __fmul_rn(s.wd[tx + 16 * j][sb], s.ad[ty + 16 * i][sb]);
                        acc[i][j] = __fadd_rn(acc[i][j], __fmul_rn(t1, (float)P[i][j]));
                    }
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) sumi[i][j] += s.wsc[tx + 16 * j][sb] * P[i][j];
            }
        }
        if (MODE == 0 && DT != KQ_Q8_0) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int mi = ty + 16 * i;
                const float da = s.ad[mi][0];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int ni = tx + 16 * j;
                    const float t1 = __fmul_rn(da, s.wd[ni][0]);
                    float term = __fmul_rn(t1, (float)sumi[i][j]);
                    if (DT == KQ_Q4_K || DT == KQ_Q5_K) {
                        int summ = 0;
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) summ += s.wmn[ni][jj] * (s.abs_[mi][2 * jj] + s.abs_[mi][2 * jj + 1]);
                        const float t3 = __fmul_rn(da, s.wd[ni][1]);
                        term = __fsub_rn(term, __fmul_rn(t3, (float)summ));
                    }
                    acc[i][j] = __fadd_rn(acc[i][j], term);
                }
            }
        }
        __syncthreads();
    }
    if (MODE == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t yr = yrow[ty + 16 * i];
            if (yr < 0) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t n = n0 + tx + 16 * j;
                if (n < a.N) a.y[yr * a.ldy + n] = acc[i][j];
            }
        }
    }
}

size_t mmq_exact_smem() { return sizeof(ExactSmem); }

template <int DT, int MODE, bool GROUPED>
static kq_status launch_one(const MmqExactArgs &a, unsigned grid_y, cudaStream_t st) {
    auto kern = mmq_exact_kernel<DT, MODE, GROUPED>;
    const size_t smem = sizeof(ExactSmem);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(KQ_ERR_CUDA, "mmq_exact: %s", cudaGetErrorString(e));
    dim3 grid((unsigned)((a.N + BN - 1) / BN), grid_y, 1);
    kern<<<grid, 256, smem, st>>>(a);
    kq_status s = check_launch("mmq_exact");
    if (s == KQ_OK) count_launch(R_MMQ_EXACT);
    return s;
}

kq_status launch_mmq_exact(int dt, int mode, bool grouped, const MmqExactArgs &a, unsigned grid_y, cudaStream_t st) {
    if (grid_y == 0) return KQ_OK;
#define KQ_DISPATCH(DTV)                                                                       \
    if (dt == DTV) {                                                                           \
        if (grouped) return launch_one<DTV, 0, true>(a, grid_y, st);                           \
        return mode == 1 ? launch_one<DTV, 1, false>(a, grid_y, st) : launch_one<DTV, 0, false>(a, grid_y, st); \
    }
    KQ_DISPATCH(KQ_Q4_K)
    KQ_DISPATCH(KQ_Q5_K)
    KQ_DISPATCH(KQ_Q6_K)
    KQ_DISPATCH(KQ_Q8_0)
#undef KQ_DISPATCH
    return fail(KQ_ERR_UNSUPPORTED_DTYPE, "mmq_exact: dtype %d", dt);
}

}  // namespace kq
