// kq_tc.cuh -- tensor-core (tcgen05) prefill GEMM interface (internal).
#pragma once
#include "kq_internal.cuh"

namespace kq {

// Wall-time limit of every wait of the tensor-core pipeline: past it the CTA records an error in the
// workspace's device flag, drains its own copies and MMAs, and leaves.
constexpr unsigned long long kTcWaitNs = 2000000000ull;

// Debug hooks of the tensor-core kernel (NULL everywhere on the product path).
struct TcDebug {
    int32_t *sums = nullptr;               // read-out of the integer block sums: [rows][N][nblk][2] int32
    unsigned long long wait_ns = kTcWaitNs;  // limit of every pipeline wait
    bool withhold_act = false;             // keep the activation producer idle (the first wait times out)
};

// True when the tensor-core kernel handles this shape (large-M prefill of a supported dtype).
bool tc_eligible(kq_dtype wt, int64_t M, int64_t N, int64_t K);
// Workspace bytes the tensor-core path needs for this shape (0 when it is not eligible).
size_t tc_workspace_bytes(kq_dtype wt, int64_t M, int64_t N, int64_t K);
kq_status tc_gemm(kq_dtype wt, const uint8_t *w, const uint8_t *xq, int64_t M, int64_t N, int64_t K, float *y,
                  int64_t ldy, uint8_t *workspace, cudaStream_t st, const TcDebug *dbg = nullptr);
// The GEMM with the block scales folded into the f16 operands (dequantised weights times f16(d_a*q), one
// fp32 accumulator per 128 x 256 tile over the whole of K): not bit-exact; Q4_K, Q5_K, Q6_K (Q8_K rows)
// and Q8_0 (Q8_1 rows); shape and workspace as tc_gemm.
kq_status tc_gemm_folded(kq_dtype wt, const uint8_t *w, const uint8_t *xq, int64_t M, int64_t N, int64_t K, float *y,
                         int64_t ldy, uint8_t *workspace, cudaStream_t st, const TcDebug *dbg = nullptr);
// Split-K factor (CTAs per output tile) the tensor-core path takes for this shape on the current
// device; 0 when the shape does not take the tensor-core path.
int tc_split_factor(kq_dtype wt, int64_t M, int64_t N, int64_t K);
// The same GEMM from fp32 activation rows (stride ldx), quantised to Q8_K inside the prologue with the
// standalone quantizer's arithmetic (Q4_K, Q5_K, Q6_K weights).
kq_status tc_gemm_f32(kq_dtype wt, const uint8_t *w, const float *x, int64_t ldx, int64_t M, int64_t N, int64_t K,
                      float *y, int64_t ldy, uint8_t *workspace, cudaStream_t st, bool fold = false);

// Routed experts on the tensor cores: 128-row tiles of each expert's routed rows (a tile table built
// by the routing pass), activation panels gathered in routed order, outputs scattered back to their
// (token, slot) rows.
constexpr int kTcTileRows = 128;
bool tc_grouped_eligible(kq_dtype wt, int64_t N, int64_t K);
struct TcGroupedPanels {
    int64_t rows, dstride;
    size_t off_a, off_e, off_d, bytes;
};
TcGroupedPanels tc_grouped_panels(kq_dtype wt, int64_t pairs, int64_t E, int64_t K);
kq_status tc_gemm_grouped(kq_dtype wt, const uint8_t *w, const uint8_t *xq, int rows_per_token, int top_k,
                          int64_t pairs, int64_t E, int64_t N, int64_t K, float *y, uint8_t *panels,
                          const int *tiles, const int *tile_count, int64_t max_tiles, const int *count,
                          const int *offset, const int *poff, const int *lists, const int *prow,
                          unsigned long long *err, uint8_t *hq, float *scr, cudaStream_t st,
                          const TcDebug *dbg = nullptr);
// Scratch bytes of the fused SwiGLU -> Q8_K epilogue (hq != NULL above, N = 2F, F % 256 == 0): one
// pair of 128 KB tiles per SM of the current device.
size_t tc_swq_scratch_bytes();

}  // namespace kq
