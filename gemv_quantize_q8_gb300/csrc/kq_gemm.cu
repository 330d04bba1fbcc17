// kq_gemm.cu -- C ABI of the matmul entry points: dense GEMM dispatch, debug partials, routed-expert
// GEMM (routing compaction + per-expert tiles), device flag, weighted expert sum.
//
// Routed experts follow strix-llama.cpp PR #18 ("Optimize ROCM Prefill and Decode"): the
// (token, slot) pairs are compacted per expert and each expert gets as many tiles as ITS row count
// needs, not a tiling chosen from the total number of pairs (the routed-compact commit's lesson: a
// tile chosen from the total left 50-87% of every tile as padding).  The tile width is the
// tensor-core tile's for every expert.  The compaction is a stable per-expert scan, so the row order
// -- and the result -- is deterministic.
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "kq_internal.cuh"
#include "kq_mmq_exact.cuh"
#include "kq_tc.cuh"

namespace kq {

constexpr int kTileM = 64;
constexpr int kRouteChunk = 1024;   // chunked routing: pairs per block, 8 warps x 4 rows of 32
constexpr int kRouteThreads = 256;
constexpr int kRouteMaxE = 2048;    // chunked routing's shared counters: 8 warps x n_experts ints

static bool chunked_routing(int64_t E) { return E <= kRouteMaxE; }

static size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

struct GroupedWs {
    size_t off_flag, off_tile_count, off_count, off_offset, off_tiles, off_lists, total;
    int64_t max_tiles;
};

// Regions the tensor-core grouped path appends to the routing workspace.
struct GroupedTcWs {
    size_t off_poff, off_prow, off_tile_count, off_tiles, off_panels, total;
    int64_t max_tiles;
};

static GroupedTcWs grouped_tc_ws(kq_dtype wt, size_t base, int64_t pairs, int64_t E, int64_t K) {
    GroupedTcWs w{};
    w.max_tiles = (pairs + kTcTileRows - 1) / kTcTileRows + E;
    size_t o = base;
    w.off_poff = o; o += align256(sizeof(int) * E);
    w.off_prow = o; o += align256(sizeof(int) * pairs);
    w.off_tile_count = o; o += align256(sizeof(int));
    w.off_tiles = o; o += align256(sizeof(int) * 2 * w.max_tiles);
    w.off_panels = o; o += tc_grouped_panels(wt, pairs, E, K).bytes;
    w.total = o;
    return w;
}

// Chunked-routing region the workspace path appends after the routing base (n_experts <= kRouteMaxE).
struct RouteHistWs {
    size_t off_hist, off_bad, total;
    int nchunks;
};

static RouteHistWs route_hist_ws(size_t base, int64_t pairs, int64_t E) {
    RouteHistWs w{};
    w.nchunks = chunked_routing(E) ? (int)((pairs + kRouteChunk - 1) / kRouteChunk) : 0;
    size_t o = base;
    w.off_hist = o; o += align256(sizeof(int) * (size_t)w.nchunks * E);
    w.off_bad = o; o += align256(sizeof(int) * (size_t)w.nchunks);
    w.total = o;
    return w;
}

static GroupedWs grouped_ws(int64_t M, int64_t top_k, int64_t E) {
    GroupedWs w{};
    const int64_t pairs = M * top_k;
    w.max_tiles = (pairs + kTileM - 1) / kTileM + E;
    size_t o = 0;
    w.off_flag = o; o += align256(sizeof(long long));
    w.off_tile_count = o; o += align256(sizeof(int));
    w.off_count = o; o += align256(sizeof(int) * E);
    w.off_offset = o; o += align256(sizeof(int) * E);
    w.off_tiles = o; o += align256(sizeof(int) * 2 * w.max_tiles);
    w.off_lists = o; o += align256(sizeof(int) * pairs);
    w.total = o;
    return w;
}

// One block per expert: number of pairs routed to it.  Block 0 also counts invalid ids.
__global__ void route_count_kernel(const int32_t *__restrict__ ids, int64_t pairs, int E, int *__restrict__ count,
                                   long long *__restrict__ flag) {
    __shared__ int red[256];
    __shared__ int bad_red[256];
    const int e = blockIdx.x;
    int c = 0, bad = 0;
    for (int64_t p = threadIdx.x; p < pairs; p += blockDim.x) {
        const int id = ids[p];
        c += id == e;
        bad += (id < 0 || id >= E);
    }
    red[threadIdx.x] = c;
    bad_red[threadIdx.x] = bad;
    __syncthreads();
    for (int s = 128; s > 0; s >>= 1) {
        if (threadIdx.x < s) {
            red[threadIdx.x] += red[threadIdx.x + s];
            bad_red[threadIdx.x] += bad_red[threadIdx.x + s];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        count[e] = red[0];
        if (e == 0) *flag = bad_red[0];
    }
}

// Inclusive scan over the 1024 threads of a block (warp shuffles, then the 32 warp totals).
__device__ __forceinline__ int block_scan_incl(int v, int *warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, v, s);
        if (lane >= s) v += o;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int t = warp_tot[lane];
#pragma unroll
        for (int s = 1; s < 32; s <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, t, s);
            if (lane >= s) t += o;
        }
        warp_tot[lane] = t;
    }
    __syncthreads();
    const int r = v + (warp > 0 ? warp_tot[warp - 1] : 0);
    __syncthreads();
    return r;
}

// One block of 1024 threads: exclusive scan of the expert counts (offset), the dp4a tile table of
// 64-row tiles (expert, first row) and, when poff != NULL, the tensor-core table: expert rows padded
// to a multiple of 4 (poff) and one (expert, 128-row tile index) entry per tile.
// With hist != NULL (chunked routing) the counts are first summed from the per-chunk histograms and
// written to count, the histograms are turned into per-chunk list bases (offset[e] + pairs of expert e
// in earlier chunks), and the device flag gets the number of invalid ids.
__global__ void __launch_bounds__(1024) route_scan_kernel(int *__restrict__ count, int E, int *__restrict__ offset,
                                                          int *__restrict__ tiles, int *__restrict__ tile_count,
                                                          int *__restrict__ poff, int *__restrict__ tc_tiles,
                                                          int *__restrict__ tc_tile_count, int *__restrict__ hist,
                                                          int nchunks, const int *__restrict__ bad,
                                                          long long *__restrict__ flag) {
    __shared__ int wt[32];
    __shared__ int tot[4];
    int carry_off = 0, carry_t = 0, carry_p = 0, carry_tc = 0;
    for (int e0 = 0; e0 < E; e0 += 1024) {
        const int e = e0 + threadIdx.x;
        int c = 0;
        if (e < E) {
            if (hist) {
                for (int k = 0; k < nchunks; ++k) c += hist[(int64_t)k * E + e];
                count[e] = c;
            } else {
                c = count[e];
            }
        }
        const int nt = (c + kTileM - 1) / kTileM, ntc = (c + kTcTileRows - 1) / kTcTileRows, cp = (c + 3) & ~3;
        const int i_off = block_scan_incl(c, wt);
        const int i_t = block_scan_incl(nt, wt);
        const int i_p = block_scan_incl(cp, wt);
        const int i_tc = block_scan_incl(ntc, wt);
        if (e < E) {
            offset[e] = carry_off + i_off - c;
            if (hist) {
                int run = carry_off + i_off - c;
                for (int k = 0; k < nchunks; ++k) {
                    const int h = hist[(int64_t)k * E + e];
                    hist[(int64_t)k * E + e] = run;
                    run += h;
                }
            }
            const int t0 = carry_t + i_t - nt;
            for (int j = 0; j < nt; ++j) { tiles[2 * (t0 + j)] = e; tiles[2 * (t0 + j) + 1] = j * kTileM; }
            if (poff) {
                poff[e] = carry_p + i_p - cp;
                const int u0 = carry_tc + i_tc - ntc;
                for (int j = 0; j < ntc; ++j) { tc_tiles[2 * (u0 + j)] = e; tc_tiles[2 * (u0 + j) + 1] = j; }
            }
        }
        // block totals: the last thread's inclusive values
        if (threadIdx.x == 1023) { tot[0] = i_off; tot[1] = i_t; tot[2] = i_p; tot[3] = i_tc; }
        __syncthreads();
        carry_off += tot[0]; carry_t += tot[1]; carry_p += tot[2]; carry_tc += tot[3];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        *tile_count = carry_t;
        if (poff) *tc_tile_count = carry_tc;
        if (hist) {
            long long nb = 0;
            for (int k = 0; k < nchunks; ++k) nb += bad[k];
            *flag = nb;
        }
    }
}

// One warp per expert: stable compaction of its pairs, in ascending pair order.  A step covers 256
// pairs: lane l holds pairs 8l .. 8l+7 of the step, an exclusive warp scan of the per-lane match
// counts places them.  With prow != NULL also the tensor-core panel row of every list entry.
__global__ void route_fill_kernel(const int32_t *__restrict__ ids, int64_t pairs, int E, const int *__restrict__ offset,
                                  int *__restrict__ lists, const int *__restrict__ poff, int *__restrict__ prow) {
    const int e = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (e >= E) return;
    const int base0 = offset[e];
    const int pbase = poff ? poff[e] : 0;
    const bool vec = (reinterpret_cast<uintptr_t>(ids) & 15) == 0;
    int n = 0;
    for (int64_t p0 = 0; p0 < pairs; p0 += 256) {
        const int64_t q = p0 + 8 * lane;
        int v[8];
        if (vec && q + 8 <= pairs) {
            const int4 a = *reinterpret_cast<const int4 *>(ids + q);
            const int4 b = *reinterpret_cast<const int4 *>(ids + q + 4);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = q + k < pairs ? ids[q + k] : -1;
        }
        int c = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) c += v[k] == e;
        int incl = c;
#pragma unroll
        for (int s2 = 1; s2 < 32; s2 <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, s2);
            if (lane >= s2) incl += o;
        }
        int i = n + incl - c;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (v[k] == e) {
                lists[base0 + i] = (int)(q + k);
                if (prow) prow[base0 + i] = pbase + i;
                ++i;
            }
        }
        n += __shfl_sync(0xffffffffu, incl, 31);
    }
}

// ---- chunked routing (workspace path, n_experts <= kRouteMaxE): a stable counting sort of the pairs by
// expert.  Pairs are cut into chunks of kRouteChunk; route_hist_kernel counts each chunk's pairs per
// expert, route_scan_kernel sums the chunk counts and turns them into per-chunk list bases, and
// route_fill_chunk_kernel writes every pair at base + its rank among the chunk's pairs of the same
// expert (ascending pair order), so the lists equal those of route_fill_kernel.
// hist[chunk][e] = pairs of the chunk routed to expert e; bad[chunk] = ids outside [0, E).
__global__ void __launch_bounds__(kRouteThreads) route_hist_kernel(const int32_t *__restrict__ ids, int64_t pairs,
                                                                   int E, int *__restrict__ hist, int *__restrict__ bad) {
    extern __shared__ int cnt[];  // E
    __shared__ int nbad;
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    if (threadIdx.x == 0) nbad = 0;
    __syncthreads();
    const int64_t p0 = (int64_t)blockIdx.x * kRouteChunk;
    int b = 0;
    for (int i = threadIdx.x; i < kRouteChunk; i += blockDim.x) {
        const int64_t p = p0 + i;
        if (p < pairs) {
            const int id = ids[p];
            if (id >= 0 && id < E) atomicAdd(&cnt[id], 1);
            else ++b;
        }
    }
    if (b) atomicAdd(&nbad, b);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(int64_t)blockIdx.x * E + e] = cnt[e];
    if (threadIdx.x == 0) bad[blockIdx.x] = nbad;
}

// One block per chunk.  Warp w takes the chunk's pairs w*128 .. w*128+127 in four rows of 32 (row k:
// pairs w*128 + 32k + lane).  Within a row, lanes holding the same expert find each other with
// __match_any_sync and rank by lane; a per-warp counter per expert carries the rank across rows; an
// exclusive prefix over the warps carries it across warps.  base (= hist after the scan) carries it
// across chunks.  With prow != NULL also the tensor-core panel row of every list entry.
__global__ void __launch_bounds__(kRouteThreads) route_fill_chunk_kernel(
    const int32_t *__restrict__ ids, int64_t pairs, int E, const int *__restrict__ base,
    const int *__restrict__ offset, int *__restrict__ lists, const int *__restrict__ poff, int *__restrict__ prow) {
    extern __shared__ int wcnt[];  // [8][E]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < 8 * E; i += blockDim.x) wcnt[i] = 0;
    __syncthreads();
    const int64_t p0 = (int64_t)blockIdx.x * kRouteChunk + warp * 128;
    const unsigned below = (1u << lane) - 1u;
    int ev[4], rk[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int64_t p = p0 + k * 32 + lane;
        int e = p < pairs ? ids[p] : -1;
        if (e < 0 || e >= E) e = -1;
        const unsigned m = __match_any_sync(0xffffffffu, e);
        const int before = e >= 0 ? wcnt[warp * E + e] : 0;
        rk[k] = before + __popc(m & below);
        ev[k] = e;
        __syncwarp();
        if (e >= 0 && (m & below) == 0) wcnt[warp * E + e] = before + __popc(m);  // the group's lowest lane
        __syncwarp();
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
        for (int w = 0; w < 8; ++w) {
            const int c = wcnt[w * E + e];
            wcnt[w * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int e = ev[k];
        if (e < 0) continue;
        const int pos = base[(int64_t)blockIdx.x * E + e] + wcnt[warp * E + e] + rk[k];
        lists[pos] = (int)(p0 + k * 32 + lane);
        if (prow) prow[pos] = poff[e] + (pos - offset[e]);
    }
}

// out[t][n] = w[t][0]*y[t][0][n] + ... in slot order, products rounded before each add.
template <bool VEC>
__global__ void weighted_sum_kernel(const float *__restrict__ ys, const float *__restrict__ w, int64_t M, int top_k,
                                    int64_t N, float *__restrict__ out) {
    const int64_t per_row = VEC ? N / 4 : N;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= M * per_row) return;
    const int64_t t = i / per_row, j = i % per_row;
    const float *wt = w + t * top_k;
    if (VEC) {
        const float4 *y4 = reinterpret_cast<const float4 *>(ys + t * top_k * N) + j;
        float4 v = y4[0];
        const float w0 = wt[0];
        float4 acc = make_float4(__fmul_rn(w0, v.x), __fmul_rn(w0, v.y), __fmul_rn(w0, v.z), __fmul_rn(w0, v.w));
        for (int k = 1; k < top_k; ++k) {
            v = y4[k * (N / 4)];
            const float wk = wt[k];
            acc.x = __fadd_rn(acc.x, __fmul_rn(wk, v.x));
            acc.y = __fadd_rn(acc.y, __fmul_rn(wk, v.y));
            acc.z = __fadd_rn(acc.z, __fmul_rn(wk, v.z));
            acc.w = __fadd_rn(acc.w, __fmul_rn(wk, v.w));
        }
        reinterpret_cast<float4 *>(out + t * N)[j] = acc;
    } else {
        const float *yr = ys + t * top_k * N + j;
        float acc = __fmul_rn(wt[0], yr[0]);
        for (int k = 1; k < top_k; ++k) acc = __fadd_rn(acc, __fmul_rn(wt[k], yr[k * N]));
        out[t * N + j] = acc;
    }
}

static kq_status check_matmul_args(const char *name, kq_dtype wt, const void *w, const void *xq, int64_t M, int64_t N,
                                   int64_t K) {
    if (wt != KQ_Q4_K && wt != KQ_Q5_K && wt != KQ_Q6_K && wt != KQ_Q8_0)
        return fail(KQ_ERR_UNSUPPORTED_DTYPE, "%s: weight dtype %s is not Q4_K, Q5_K, Q6_K or Q8_0", name,
                    dtype_name(wt));
    if (!w || !xq) return fail(KQ_ERR_INVALID_ARG, "%s: null pointer", name);
    if (M <= 0 || N <= 0 || K <= 0 || K % 256)
        return fail(KQ_ERR_INVALID_ARG, "%s: need M, N > 0 and K a positive multiple of 256 (M=%lld N=%lld K=%lld)",
                    name, (long long)M, (long long)N, (long long)K);
    if (!aligned(w, 16)) return fail(KQ_ERR_ALIGNMENT, "%s: w must be 16-byte aligned", name);
    if (!aligned(xq, 4)) return fail(KQ_ERR_ALIGNMENT, "%s: xq must be 4-byte aligned", name);
    return KQ_OK;
}

// Argument checks shared by kq_gemm and its debug twins: matmul arguments, output, workspace.
static kq_status check_gemm_call(const char *name, kq_dtype wt, const void *w, const void *xq, int64_t M, int64_t N,
                                 int64_t K, const float *y, int64_t ldy, const void *workspace, size_t ws_bytes) {
    kq_status s = check_matmul_args(name, wt, w, xq, M, N, K);
    if (s != KQ_OK) return s;
    if (!y) return fail(KQ_ERR_INVALID_ARG, "%s: null y", name);
    if (ldy < N) return fail(KQ_ERR_INVALID_ARG, "%s: ldy %lld < N %lld", name, (long long)ldy, (long long)N);
    if (!aligned(y, 4)) return fail(KQ_ERR_ALIGNMENT, "%s: y must be 4-byte aligned", name);
    const size_t need = kq_gemm_workspace_bytes(wt, M, N, K, 0, 0);
    if (need > 0 && (!workspace || ws_bytes < need))
        return fail(KQ_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", name, need,
                    workspace ? ws_bytes : 0);
    if (workspace && !aligned(workspace, 256))
        return fail(KQ_ERR_ALIGNMENT, "%s: workspace must be 256-byte aligned", name);
    return KQ_OK;
}

}  // namespace kq

using namespace kq;

extern "C" {

size_t kq_gemm_workspace_bytes(kq_dtype wt, int64_t M, int64_t N, int64_t K, int64_t n_experts, int64_t top_k) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    if (n_experts > 0) {
        const int64_t tk = top_k > 0 ? top_k : 1;
        const size_t base = route_hist_ws(grouped_ws(M, tk, n_experts).total, M * tk, n_experts).total;
        return tc_grouped_eligible(wt, N, K) ? grouped_tc_ws(wt, base, M * tk, n_experts, K).total : base;
    }
    return tc_workspace_bytes(wt, M, N, K);
}

kq_status kq_gemm(kq_dtype wt, const void *w, const void *xq, int64_t M, int64_t N, int64_t K, float *y, int64_t ldy,
                  void *workspace, size_t ws_bytes, kq_stream_t stream) {
    kq_status s = check_gemm_call("kq_gemm", wt, w, xq, M, N, K, y, ldy, workspace, ws_bytes);
    if (s != KQ_OK) return s;
    cudaStream_t st = (cudaStream_t)stream;
    if (tc_eligible(wt, M, N, K))
        return tc_gemm(wt, static_cast<const uint8_t *>(w), static_cast<const uint8_t *>(xq), M, N, K, y, ldy,
                       static_cast<uint8_t *>(workspace), st);
    // batched decode: the weight-streaming GEMV kernel serves up to kGemvMaxBatch activation rows
    if (M <= kGemvMaxBatch && aligned(w, 16) &&
        gemv_batched(wt, static_cast<const uint8_t *>(w), static_cast<const uint8_t *>(xq), M, N, K, y, ldy, st) ==
            KQ_OK)
        return KQ_OK;
    MmqExactArgs a{};
    a.w = static_cast<const uint8_t *>(w);
    a.xq = static_cast<const uint8_t *>(xq);
    a.M = M; a.N = N; a.K = K; a.y = y; a.ldy = ldy;
    const int64_t gy = (M + kTileM - 1) / kTileM;
    if (gy > 65535) return fail(KQ_ERR_INVALID_ARG, "kq_gemm: M=%lld too large", (long long)M);
    return launch_mmq_exact(wt, 0, false, a, (unsigned)gy, st);
}

kq_status kq_gemm_ex(kq_dtype wt, const void *w, const void *xq, int64_t M, int64_t N, int64_t K, float *y,
                     int64_t ldy, unsigned flags, void *workspace, size_t ws_bytes, kq_stream_t stream) {
    if (flags & ~(unsigned)KQ_GEMM_FOLD_SCALES)
        return fail(KQ_ERR_INVALID_ARG, "kq_gemm_ex: unknown flags 0x%x", flags & ~(unsigned)KQ_GEMM_FOLD_SCALES);
    if (!(flags & KQ_GEMM_FOLD_SCALES)) return kq_gemm(wt, w, xq, M, N, K, y, ldy, workspace, ws_bytes, stream);
    kq_status s = check_gemm_call("kq_gemm_ex", wt, w, xq, M, N, K, y, ldy, workspace, ws_bytes);
    if (s != KQ_OK) return s;
    if (wt != KQ_Q4_K && wt != KQ_Q5_K && wt != KQ_Q6_K && wt != KQ_Q8_0)
        return fail(KQ_ERR_UNSUPPORTED_DTYPE, "kq_gemm_ex: KQ_GEMM_FOLD_SCALES takes Q4_K, Q5_K, Q6_K or Q8_0 "
                    "weights, not %s", dtype_name(wt));
    // shapes off the tensor-core path have no folded form: the exact kernels serve them
    if (!tc_eligible(wt, M, N, K)) return kq_gemm(wt, w, xq, M, N, K, y, ldy, workspace, ws_bytes, stream);
    return tc_gemm_folded(wt, static_cast<const uint8_t *>(w), static_cast<const uint8_t *>(xq), M, N, K, y, ldy,
                          static_cast<uint8_t *>(workspace), (cudaStream_t)stream);
}

size_t kq_gemm_f32_workspace_bytes(kq_dtype wt, int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0 || K % 256) return 0;
    // kq_gemm's workspace first (at least the 256-byte header holding the device flag, so
    // kq_read_device_flag applies), then room for the quantised rows, which the paths other than the
    // tensor-core prologue need
    const size_t g = std::max<size_t>(256, (kq_gemm_workspace_bytes(wt, M, N, K, 0, 0) + 255) & ~(size_t)255);
    const size_t xq = wt == KQ_Q8_0 ? (size_t)M * (K / 32) * kQ81Bytes : (size_t)M * (K / 256) * kQ8KBytes;
    return g + xq;
}

kq_status kq_gemm_f32(kq_dtype wt, const void *w, const float *x, int64_t ldx, int64_t M, int64_t N, int64_t K,
                      float *y, int64_t ldy, void *workspace, size_t ws_bytes, kq_stream_t stream) {
    return kq_gemm_f32_ex(wt, w, x, ldx, M, N, K, y, ldy, 0u, workspace, ws_bytes, stream);
}

kq_status kq_gemm_f32_ex(kq_dtype wt, const void *w, const float *x, int64_t ldx, int64_t M, int64_t N, int64_t K,
                         float *y, int64_t ldy, unsigned flags, void *workspace, size_t ws_bytes, kq_stream_t stream) {
    if (flags & ~(unsigned)KQ_GEMM_FOLD_SCALES)
        return fail(KQ_ERR_INVALID_ARG, "kq_gemm_f32_ex: unknown flags 0x%x", flags & ~(unsigned)KQ_GEMM_FOLD_SCALES);
    const bool fold = (flags & KQ_GEMM_FOLD_SCALES) != 0;
    kq_status s = check_matmul_args("kq_gemm_f32", wt, w, x, M, N, K);
    if (s != KQ_OK) return s;
    if (!y) return fail(KQ_ERR_INVALID_ARG, "kq_gemm_f32: null y");
    if (ldy < N || ldx < K)
        return fail(KQ_ERR_INVALID_ARG, "kq_gemm_f32: ldy %lld < N %lld or ldx %lld < K %lld", (long long)ldy,
                    (long long)N, (long long)ldx, (long long)K);
    if (!aligned(y, 4)) return fail(KQ_ERR_ALIGNMENT, "kq_gemm_f32: y must be 4-byte aligned");
    const size_t need = kq_gemm_f32_workspace_bytes(wt, M, N, K);
    if (!workspace || ws_bytes < need)
        return fail(KQ_ERR_WORKSPACE, "kq_gemm_f32: workspace of %zu bytes needed, %zu given", need,
                    workspace ? ws_bytes : 0);
    if (!aligned(workspace, 256)) return fail(KQ_ERR_ALIGNMENT, "kq_gemm_f32: workspace must be 256-byte aligned");
    cudaStream_t st = (cudaStream_t)stream;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    if (wt != KQ_Q8_0 && tc_eligible(wt, M, N, K))
        return tc_gemm_f32(wt, static_cast<const uint8_t *>(w), x, ldx, M, N, K, y, ldy, ws, st, fold);
    // other paths: quantise into the workspace's tail, then the GEMM
    const size_t gneed = kq_gemm_workspace_bytes(wt, M, N, K, 0, 0);
    const size_t g = std::max<size_t>(256, (gneed + 255) & ~(size_t)255);
    uint8_t *xq = ws + g;
    s = wt == KQ_Q8_0 ? kq_quantize_q8_1(x, M, K, ldx, xq, stream) : kq_quantize_q8k(x, M, K, ldx, xq, stream);
    if (s != KQ_OK) return s;
    return kq_gemm_ex(wt, w, xq, M, N, K, y, ldy, flags, gneed ? workspace : nullptr, gneed, stream);
}

kq_status kq_debug_partials(kq_dtype wt, const void *w, const void *xq, int64_t M, int64_t N, int64_t K,
                            int32_t *partials, kq_stream_t stream) {
    kq_status s = check_matmul_args("kq_debug_partials", wt, w, xq, M, N, K);
    if (s != KQ_OK) return s;
    if (!partials) return fail(KQ_ERR_INVALID_ARG, "kq_debug_partials: null partials");
    MmqExactArgs a{};
    a.w = static_cast<const uint8_t *>(w);
    a.xq = static_cast<const uint8_t *>(xq);
    a.M = M; a.N = N; a.K = K; a.partials = partials;
    const int64_t gy = (M + kTileM - 1) / kTileM;
    if (gy > 65535) return fail(KQ_ERR_INVALID_ARG, "kq_debug_partials: M=%lld too large", (long long)M);
    return launch_mmq_exact(wt, 1, false, a, (unsigned)gy, (cudaStream_t)stream);
}

int kq_debug_tc_splits(kq_dtype wt, int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0 || K % 256) return 0;
    return tc_split_factor(wt, M, N, K);
}

kq_status kq_debug_tc_sums(kq_dtype wt, const void *w, const void *xq, int64_t M, int64_t N, int64_t K, float *y,
                           int64_t ldy, int32_t *sums, void *workspace, size_t ws_bytes, kq_stream_t stream) {
    kq_status s = check_gemm_call("kq_debug_tc_sums", wt, w, xq, M, N, K, y, ldy, workspace, ws_bytes);
    if (s != KQ_OK) return s;
    if (!sums || !aligned(sums, 4)) return fail(KQ_ERR_INVALID_ARG, "kq_debug_tc_sums: null or misaligned sums");
    if (!tc_eligible(wt, M, N, K))
        return fail(KQ_ERR_INVALID_ARG, "kq_debug_tc_sums: %s M=%lld N=%lld K=%lld does not take the tensor-core path",
                    dtype_name(wt), (long long)M, (long long)N, (long long)K);
    TcDebug d;
    d.sums = sums;
    return tc_gemm(wt, static_cast<const uint8_t *>(w), static_cast<const uint8_t *>(xq), M, N, K, y, ldy,
                   static_cast<uint8_t *>(workspace), (cudaStream_t)stream, &d);
}

kq_status kq_debug_tc_wait_timeout(kq_dtype wt, const void *w, const void *xq, int64_t M, int64_t N, int64_t K,
                                   float *y, int64_t ldy, int64_t wait_limit_ns, void *workspace, size_t ws_bytes,
                                   kq_stream_t stream) {
    kq_status s = check_gemm_call("kq_debug_tc_wait_timeout", wt, w, xq, M, N, K, y, ldy, workspace, ws_bytes);
    if (s != KQ_OK) return s;
    if (wait_limit_ns < 1000 || wait_limit_ns > 1000000000)
        return fail(KQ_ERR_INVALID_ARG, "kq_debug_tc_wait_timeout: wait_limit_ns must be in [1e3, 1e9]");
    if (!tc_eligible(wt, M, N, K))
        return fail(KQ_ERR_INVALID_ARG, "kq_debug_tc_wait_timeout: %s M=%lld N=%lld K=%lld does not take the "
                    "tensor-core path", dtype_name(wt), (long long)M, (long long)N, (long long)K);
    TcDebug d;
    d.wait_ns = (unsigned long long)wait_limit_ns;
    d.withhold_act = true;
    return tc_gemm(wt, static_cast<const uint8_t *>(w), static_cast<const uint8_t *>(xq), M, N, K, y, ldy,
                   static_cast<uint8_t *>(workspace), (cudaStream_t)stream, &d);
}

}  // extern "C"

namespace kq {

static size_t swq_scratch_offset(size_t base) { return (base + 255) & ~(size_t)255; }

// The routed GEMM behind kq_gemm_grouped (hq == NULL: fp32 rows to y) and kq_gemm_grouped_swiglu_q8k
// (hq != NULL: N = 2F gate/up rows, Q8_K rows of silu(gate)*up to hq; the caller has checked the
// fused preconditions and sized the workspace with the scratch after need_base bytes).
static kq_status grouped_run(kq_dtype wt, const void *w, int64_t n_experts, const void *xq, int64_t xq_rows_per_token,
                             const int32_t *ids, int64_t M, int64_t top_k, int64_t N, int64_t K, float *y, uint8_t *hq,
                             void *workspace, size_t ws_bytes, kq_stream_t stream, const TcDebug *dbg = nullptr) {
    kq_status s = check_matmul_args("kq_gemm_grouped", wt, w, xq, M, N, K);
    if (s != KQ_OK) return s;
    if (!ids || (!y && !hq)) return fail(KQ_ERR_INVALID_ARG, "kq_gemm_grouped: null ids or y");
    if (n_experts <= 0 || top_k <= 0 || n_experts > 65535)
        return fail(KQ_ERR_INVALID_ARG, "kq_gemm_grouped: need 0 < n_experts <= 65535 and top_k > 0");
    if (xq_rows_per_token != 1 && xq_rows_per_token != top_k)
        return fail(KQ_ERR_INVALID_ARG, "kq_gemm_grouped: xq_rows_per_token must be 1 or top_k");
    if (N % 16) return fail(KQ_ERR_INVALID_ARG, "kq_gemm_grouped: N=%lld must be a multiple of 16", (long long)N);
    if (M * top_k > (int64_t)1 << 30) return fail(KQ_ERR_INVALID_ARG, "kq_gemm_grouped: too many (token, slot) pairs");
    if (!aligned(ids, 4) || !aligned(y, 4) || !aligned(hq, 4))
        return fail(KQ_ERR_ALIGNMENT, "kq_gemm_grouped: ids/y must be 4-byte aligned");
    const GroupedWs L = grouped_ws(M, top_k, n_experts);
    const size_t need_base = kq_gemm_workspace_bytes(wt, M, N, K, n_experts, top_k);
    const size_t need = hq ? swq_scratch_offset(need_base) + tc_swq_scratch_bytes() : need_base;
    if (!workspace || ws_bytes < need)
        return fail(KQ_ERR_WORKSPACE, "kq_gemm_grouped: workspace of %zu bytes needed, %zu given", need,
                    workspace ? ws_bytes : 0);
    if (!aligned(workspace, 256)) return fail(KQ_ERR_ALIGNMENT, "kq_gemm_grouped: workspace must be 256-byte aligned");
    if (L.max_tiles > 65535) return fail(KQ_ERR_INVALID_ARG, "kq_gemm_grouped: too many tiles");
    cudaStream_t st = (cudaStream_t)stream;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    long long *flag = reinterpret_cast<long long *>(ws + L.off_flag);
    int *tile_count = reinterpret_cast<int *>(ws + L.off_tile_count);
    int *count = reinterpret_cast<int *>(ws + L.off_count);
    int *offset = reinterpret_cast<int *>(ws + L.off_offset);
    int *tiles = reinterpret_cast<int *>(ws + L.off_tiles);
    int *lists = reinterpret_cast<int *>(ws + L.off_lists);
    const int64_t pairs = M * top_k;
    const RouteHistWs H = route_hist_ws(L.total, pairs, n_experts);
    const bool tc = tc_grouped_eligible(wt, N, K);
    if (dbg && !tc) return fail(KQ_ERR_INVALID_ARG, "kq_debug_tc_sums_grouped: shape not served by the tensor cores");
    const GroupedTcWs T = grouped_tc_ws(wt, H.total, pairs, n_experts, K);
    int *poff = tc ? reinterpret_cast<int *>(ws + T.off_poff) : nullptr;
    int *prow = tc ? reinterpret_cast<int *>(ws + T.off_prow) : nullptr;
    int *tc_tiles = tc ? reinterpret_cast<int *>(ws + T.off_tiles) : nullptr;
    int *tc_count = tc ? reinterpret_cast<int *>(ws + T.off_tile_count) : nullptr;
    if (H.nchunks > 0) {
        int *hist = reinterpret_cast<int *>(ws + H.off_hist);
        int *bad = reinterpret_cast<int *>(ws + H.off_bad);
        const size_t fill_smem = sizeof(int) * 8 * (size_t)n_experts;
        if (fill_smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(route_fill_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)fill_smem);
            if (e != cudaSuccess) return fail(KQ_ERR_CUDA, "kq_gemm_grouped: %s", cudaGetErrorString(e));
        }
        route_hist_kernel<<<(unsigned)H.nchunks, kRouteThreads, sizeof(int) * n_experts, st>>>(ids, pairs, (int)n_experts,
                                                                                              hist, bad);
        route_scan_kernel<<<1, 1024, 0, st>>>(count, (int)n_experts, offset, tiles, tile_count, poff, tc_tiles, tc_count,
                                              hist, H.nchunks, bad, flag);
        route_fill_chunk_kernel<<<(unsigned)H.nchunks, kRouteThreads, fill_smem, st>>>(ids, pairs, (int)n_experts, hist,
                                                                                       offset, lists, poff, prow);
    } else {
        route_count_kernel<<<(unsigned)n_experts, 256, 0, st>>>(ids, pairs, (int)n_experts, count, flag);
        route_scan_kernel<<<1, 1024, 0, st>>>(count, (int)n_experts, offset, tiles, tile_count, poff, tc_tiles, tc_count,
                                              nullptr, 0, nullptr, nullptr);
        route_fill_kernel<<<(unsigned)((n_experts + 7) / 8), 256, 0, st>>>(ids, pairs, (int)n_experts, offset, lists,
                                                                          poff, prow);
    }
    s = check_launch("kq_gemm_grouped routing");
    if (s != KQ_OK) return s;
    count_launch(R_ROUTE, 3);
    if (tc)
        return tc_gemm_grouped(wt, static_cast<const uint8_t *>(w), static_cast<const uint8_t *>(xq),
                               (int)xq_rows_per_token, (int)top_k, pairs, n_experts, N, K, y, ws + T.off_panels,
                               tc_tiles, tc_count, T.max_tiles, count, offset, poff, lists, prow,
                               reinterpret_cast<unsigned long long *>(flag), hq,
                               hq ? reinterpret_cast<float *>(ws + swq_scratch_offset(need_base)) : nullptr, st, dbg);
    if (hq) return fail(KQ_ERR_INVALID_ARG, "kq_gemm_grouped_swiglu_q8k: shape not served by the tensor cores");
    MmqExactArgs a{};
    a.w = static_cast<const uint8_t *>(w);
    a.xq = static_cast<const uint8_t *>(xq);
    a.M = M; a.N = N; a.K = K; a.y = y; a.ldy = N;
    a.tile_count = tile_count; a.tiles = tiles; a.expert_count = count; a.expert_offset = offset; a.lists = lists;
    a.rows_per_token = (int)xq_rows_per_token;
    a.top_k = (int)top_k;
    return launch_mmq_exact(wt, 0, true, a, (unsigned)L.max_tiles, st);
}

}  // namespace kq

extern "C" {

kq_status kq_gemm_grouped(kq_dtype wt, const void *w, int64_t n_experts, const void *xq, int64_t xq_rows_per_token,
                          const int32_t *ids, int64_t M, int64_t top_k, int64_t N, int64_t K, float *y, void *workspace,
                          size_t ws_bytes, kq_stream_t stream) {
    if (!y) return fail(KQ_ERR_INVALID_ARG, "kq_gemm_grouped: null ids or y");
    return grouped_run(wt, w, n_experts, xq, xq_rows_per_token, ids, M, top_k, N, K, y, nullptr, workspace, ws_bytes,
                       stream);
}

kq_status kq_debug_tc_sums_grouped(kq_dtype wt, const void *w, int64_t n_experts, const void *xq,
                                   int64_t xq_rows_per_token, const int32_t *ids, int64_t M, int64_t top_k, int64_t N,
                                   int64_t K, float *y, int32_t *sums, void *workspace, size_t ws_bytes,
                                   kq_stream_t stream) {
    if (!sums || !aligned(sums, 4)) return fail(KQ_ERR_INVALID_ARG, "kq_debug_tc_sums_grouped: null or misaligned sums");
    TcDebug d;
    d.sums = sums;
    return grouped_run(wt, w, n_experts, xq, xq_rows_per_token, ids, M, top_k, N, K, y, nullptr, workspace, ws_bytes,
                       stream, &d);
}

size_t kq_gemm_grouped_swiglu_workspace_bytes(kq_dtype wt, int64_t M, int64_t F, int64_t K, int64_t n_experts,
                                              int64_t top_k) {
    if (M <= 0 || F <= 0 || K <= 0 || n_experts <= 0) return 0;
    return swq_scratch_offset(kq_gemm_workspace_bytes(wt, M, 2 * F, K, n_experts, top_k)) + tc_swq_scratch_bytes();
}

kq_status kq_gemm_grouped_swiglu_q8k(kq_dtype wt, const void *w, int64_t n_experts, const void *xq,
                                     int64_t xq_rows_per_token, const int32_t *ids, int64_t M, int64_t top_k, int64_t F,
                                     int64_t K, void *hq, void *workspace, size_t ws_bytes, kq_stream_t stream) {
    const char *name = "kq_gemm_grouped_swiglu_q8k";
    if (!hq) return fail(KQ_ERR_INVALID_ARG, "%s: null hq", name);
    if (F <= 0 || F % 256 || F > (1 << 21))
        return fail(KQ_ERR_INVALID_ARG, "%s: F=%lld must be a positive multiple of 256 (at most 2^21)", name,
                    (long long)F);
    if (!tc_grouped_eligible(wt, 2 * F, K) || K % 256)
        return fail(KQ_ERR_INVALID_ARG, "%s: weight type %s with K=%lld is not served by the tensor cores", name,
                    dtype_name(wt), (long long)K);
    return grouped_run(wt, w, n_experts, xq, xq_rows_per_token, ids, M, top_k, 2 * F, K, nullptr,
                       static_cast<uint8_t *>(hq), workspace, ws_bytes, stream);
}

kq_status kq_read_device_flag(void *workspace, int64_t *n_bad, kq_stream_t stream) {
    if (!workspace) return fail(KQ_ERR_INVALID_ARG, "kq_read_device_flag: null workspace");
    long long v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return fail(KQ_ERR_CUDA, "kq_read_device_flag: %s", cudaGetErrorString(e));
    if (n_bad) *n_bad = v;
    if (v != 0) {
        long long zero = 0;
        e = cudaMemcpyAsync(workspace, &zero, sizeof(zero), cudaMemcpyHostToDevice, (cudaStream_t)stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
        if (e != cudaSuccess) return fail(KQ_ERR_CUDA, "kq_read_device_flag: %s", cudaGetErrorString(e));
        return fail(KQ_ERR_DEVICE_FLAG,
                    "kq_read_device_flag: device flag %lld (expert ids out of range, or tensor-core pipeline timeouts)", v);
    }
    return KQ_OK;
}

kq_status kq_moe_weighted_sum(const float *y_slots, const float *w, int64_t M, int64_t top_k, int64_t N, float *out,
                              kq_stream_t stream) {
    if (!y_slots || !w || !out) return fail(KQ_ERR_INVALID_ARG, "kq_moe_weighted_sum: null pointer");
    if (M <= 0 || top_k <= 0 || N <= 0 || top_k > 1024)
        return fail(KQ_ERR_INVALID_ARG, "kq_moe_weighted_sum: need M, N > 0 and 0 < top_k <= 1024");
    if (!aligned(y_slots, 4) || !aligned(w, 4) || !aligned(out, 4))
        return fail(KQ_ERR_ALIGNMENT, "kq_moe_weighted_sum: pointers must be 4-byte aligned");
    cudaStream_t st = (cudaStream_t)stream;
    const bool vec = N % 4 == 0 && aligned(y_slots, 16) && aligned(out, 16);
    const int64_t items = vec ? M * (N / 4) : M * N;
    const int64_t grid = (items + 255) / 256;
    if (vec) weighted_sum_kernel<true><<<(unsigned)grid, 256, 0, st>>>(y_slots, w, M, (int)top_k, N, out);
    else weighted_sum_kernel<false><<<(unsigned)grid, 256, 0, st>>>(y_slots, w, M, (int)top_k, N, out);
    kq_status s = check_launch("kq_moe_weighted_sum");
    if (s == KQ_OK) count_launch(R_WSUM);
    return s;
}

}  // extern "C"

// ---------------------------------------------------------------------------------------------
// Routed-expert GEMM without a caller workspace.
//
// Some callers cannot allocate device memory at the point where they run the MoE layer: code that
// runs under a memory pool it does not own, plug-ins whose host framework hands them only the
// input and output buffers, or code that must not call cudaMalloc after start-up.  For them the
// routing scratch (expert counts, offsets, tile table and per-expert row lists) lives in one
// fixed array in this library's device memory instead of a workspace.
namespace kq {

constexpr size_t kStaticScratchBytes = (size_t)1 << 20;  // 1 MiB: up to ~250k (token, slot) pairs
static __device__ __align__(256) uint8_t g_grouped_scratch[kStaticScratchBytes];

static std::mutex g_scratch_mu;
// Device address of g_grouped_scratch per device ordinal, with the id of the CUDA context it was
// looked up in: the address belongs to the module loaded into that context, and a reset of the device
// (cudaDeviceReset, or any teardown of its primary context) unloads the module, so a cached address
// whose context id differs from the current one is looked up again.
static void *g_scratch_addr[256];
static unsigned long long g_scratch_ctx[256];

// Unique id of the current thread's CUDA context (driver cuCtxGetCurrent + cuCtxGetId, reached through
// the runtime's entry-point query, so no driver library is linked); 0 if it cannot be read.
static unsigned long long current_ctx_id() {
    static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static bool looked_up = false;
    if (!looked_up) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
        cudaGetLastError();
        looked_up = true;
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_cur || !get_id || get_cur(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of the static scratch on the current device, looked up once per device (with that
// device current, the first call does cudaGetSymbolAddress) and again after the device's context
// changed.
static kq_status static_scratch(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(KQ_ERR_CUDA, "kq_gemm_grouped_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 256) return fail(KQ_ERR_CUDA, "kq_gemm_grouped_noalloc: device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    // cudaGetSymbolAddress makes the device's primary context current if none is; the context id is
    // read after it, so the first lookup records the context the address belongs to
    const unsigned long long ctx = current_ctx_id();
    if (!g_scratch_addr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_grouped_scratch);
        if (e != cudaSuccess || !p)
            return fail(KQ_ERR_CUDA, "kq_gemm_grouped_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = current_ctx_id();
    }
    *out = g_scratch_addr[dev];
    return KQ_OK;
}

}  // namespace kq

extern "C" kq_status kq_gemm_grouped_noalloc(kq_dtype wt, const void *w, int64_t n_experts, const void *xq,
                                             int64_t xq_rows_per_token, const int32_t *ids, int64_t M, int64_t top_k,
                                             int64_t N, int64_t K, float *y, kq_stream_t stream) {
    kq_status s = check_matmul_args("kq_gemm_grouped_noalloc", wt, w, xq, M, N, K);
    if (s != KQ_OK) return s;
    if (!ids || !y) return fail(KQ_ERR_INVALID_ARG, "kq_gemm_grouped_noalloc: null ids or y");
    if (n_experts <= 0 || top_k <= 0 || n_experts > 65535)
        return fail(KQ_ERR_INVALID_ARG, "kq_gemm_grouped_noalloc: need 0 < n_experts <= 65535 and top_k > 0");
    if (xq_rows_per_token != 1 && xq_rows_per_token != top_k)
        return fail(KQ_ERR_INVALID_ARG, "kq_gemm_grouped_noalloc: xq_rows_per_token must be 1 or top_k");
    if (N % 16) return fail(KQ_ERR_INVALID_ARG, "kq_gemm_grouped_noalloc: N=%lld must be a multiple of 16", (long long)N);
    if (M > ((int64_t)1 << 30) / top_k)
        return fail(KQ_ERR_INVALID_ARG, "kq_gemm_grouped_noalloc: too many (token, slot) pairs");
    if (!aligned(ids, 4) || !aligned(y, 4))
        return fail(KQ_ERR_ALIGNMENT, "kq_gemm_grouped_noalloc: ids/y must be 4-byte aligned");
    const GroupedWs L = grouped_ws(M, top_k, n_experts);
    if (L.total > kStaticScratchBytes)
        return fail(KQ_ERR_INVALID_ARG,
                    "kq_gemm_grouped_noalloc: M*top_k=%lld pairs with %lld experts need %zu bytes of routing scratch, "
                    "more than the fixed %zu; use kq_gemm_grouped with a workspace",
                    (long long)(M * top_k), (long long)n_experts, L.total, kStaticScratchBytes);
    if (L.max_tiles > 65535) return fail(KQ_ERR_INVALID_ARG, "kq_gemm_grouped_noalloc: too many tiles");
    void *scratch = nullptr;
    s = static_scratch(&scratch);
    if (s != KQ_OK) return s;
    cudaStream_t st = (cudaStream_t)stream;
    uint8_t *ws = static_cast<uint8_t *>(scratch);
    long long *flag = reinterpret_cast<long long *>(ws + L.off_flag);
    int *tile_count = reinterpret_cast<int *>(ws + L.off_tile_count);
    int *count = reinterpret_cast<int *>(ws + L.off_count);
    int *offset = reinterpret_cast<int *>(ws + L.off_offset);
    int *tiles = reinterpret_cast<int *>(ws + L.off_tiles);
    int *lists = reinterpret_cast<int *>(ws + L.off_lists);
    const int64_t pairs = M * top_k;
    // Every scratch field is fully rewritten below before it is read, so nothing left by an earlier
    // call needs clearing.
    route_count_kernel<<<(unsigned)n_experts, 256, 0, st>>>(ids, pairs, (int)n_experts, count, flag);
    route_scan_kernel<<<1, 1024, 0, st>>>(count, (int)n_experts, offset, tiles, tile_count, nullptr, nullptr, nullptr,
                                          nullptr, 0, nullptr, nullptr);
    route_fill_kernel<<<(unsigned)((n_experts + 7) / 8), 256, 0, st>>>(ids, pairs, (int)n_experts, offset, lists,
                                                                      nullptr, nullptr);
    s = check_launch("kq_gemm_grouped_noalloc routing");
    if (s != KQ_OK) return s;
    count_launch(R_ROUTE, 3);
    MmqExactArgs a{};
    a.w = static_cast<const uint8_t *>(w);
    a.xq = static_cast<const uint8_t *>(xq);
    a.M = M; a.N = N; a.K = K; a.y = y; a.ldy = N;
    a.tile_count = tile_count; a.tiles = tiles; a.expert_count = count; a.expert_offset = offset; a.lists = lists;
    a.rows_per_token = (int)xq_rows_per_token;
    a.top_k = (int)top_k;
    return launch_mmq_exact(wt, 0, true, a, (unsigned)L.max_tiles, st);
}
