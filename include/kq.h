/*
 * kq.h -- C ABI of the keep-quant int8 matmul library for GB300 (sm_103a).
 *
 * Block-quantised weights (Q4_K, Q5_K, Q6_K, Q8_0) stay packed in device memory;
 * activations are quantised on the fly to Q8_K (256-element blocks) or Q8_1
 * (32-element blocks) and multiplied with integer dot products, scaled into
 * fp32.  Sources of the operations (prose descriptions on three pages):
 *   [vllm-2890]  vllm.cpp PR #2890 "fuse silu-mul with Q8_K quant epilogue
 *                (VT_SILU_QUANT_FUSED)" -- Q8_K quantizer, keep-quant provider,
 *                MMVQ decode GEMV, fused SiLU-mul + quant.
 *   [vllm-3035]  vllm.cpp PR #3035 "scope a cooperative activation share for
 *                the WMMA kernels" -- prefill GEMM with one activation tile
 *                staged once per block and shared by all warps.
 *   [llama-18]   strix-llama.cpp PR #18 "Optimize ROCM Prefill and Decode" --
 *                Q8_1 quantizer, fused-quant MMVQ, routed-expert MMQ
 *                (MUL_MAT_ID), weighted expert sum.
 *
 * Conventions (every entry point):
 *   - All pointers named w, x, xq, y, g, u, ids, workspace... are DEVICE
 *     pointers unless stated; the caller owns every buffer.  The library
 *     allocates nothing and keeps no state between calls.
 *   - Work is enqueued on `stream` (NULL = legacy default stream) and is
 *     asynchronous: no entry point synchronises, except kq_read_device_flag.
 *   - Return value: KQ_OK, or an error status without launching anything;
 *     kq_last_error() then holds a one-line, thread-local description that
 *     names the offending argument or dtype.  A CUDA launch failure returns
 *     KQ_ERR_CUDA.  Unsupported dtypes are rejected, never routed elsewhere.
 *   - Results are deterministic: no atomics in any reduction.
 *   - Sizes are elements unless named *_bytes.  K must be a multiple of 256
 *     for every path (all K-quant super-blocks, and Q8_0 rows are grouped in
 *     256-element chunks in the native layout).
 *
 * Canonical (GGUF-style) block layouts, little-endian:
 *   Q4_K (144 B / 256): f16 d, f16 dmin, 12 bytes of packed 6-bit sub-block
 *        scales and mins (8 each), 128 bytes of 4-bit codes; element 64c+l is
 *        the low nibble and 64c+32+l the high nibble of code byte 32c+l.
 *        x = d*sc_j*c - dmin*m_j, j = sub-block of 32.
 *   Q5_K (176 B / 256): f16 d, f16 dmin, the 12 Q4_K scale/min bytes, qh[32]
 *        (high code bits), 128 bytes of 4-bit codes in the Q4_K arrangement;
 *        element 64c+l takes bit 2c of qh[l] and 64c+32+l bit 2c+1 as its
 *        fifth bit (c = 0..31); x = d*sc_j*c - dmin*m_j.
 *   Q6_K (210 B / 256): ql[128], qh[64], int8 scales[16], f16 d;
 *        x = d*sc_j*(c - 32), j = sub-block of 16.
 *   Q8_0 (34 B / 32):   f16 d, int8 w[32]; x = d*w.
 *   Q8_K (292 B / 256): f32 d, int8 q[256], int16 bsums[16] (sums of 16 q).
 *   Q8_1 (36 B / 32):   f16 d, f16 s (block sum of the input), int8 q[32].
 *
 * Native weight layout (what the matmul entry points consume; produced by
 * kq_repack_weights): rows are taken in groups of 16 (the last group is
 * padded with zero rows) and each group is stored as consecutive chunks of
 * 256 elements along K.  Inside a chunk, the codes of each 64-element
 * "kblock" kb (0..3) are stored for the 16 rows together, so one kblock of a
 * row group is one contiguous run:
 *   Q4_K chunk (2304 B): codes [kb][16 rows][32 B] -- byte l holds element
 *        64kb+l (low nibble) and 64kb+32+l (high nibble); then headers
 *        [16][16 B] (d, dmin, 12 scale/min bytes: the canonical first 16).
 *   Q6_K chunk (3360 B): low 4 code bits [kb][16][32 B] (nibble order as
 *        Q4_K); high 2 code bits [kb][16][16 B] (byte j: elements 64kb+j,
 *        +16+j, +32+j, +48+j in bits 0-1, 2-3, 4-5, 6-7); int8 scales
 *        [16][16]; f16 d [16].
 *   Q5_K chunk (2816 B): the Q4_K chunk, then each row's 32 high-bit bytes
 *        [16][32 B] (canonical order).
 *   Q8_0 chunk (4352 B): codes [kb][16][64 B]; f16 d [16][8].
 * Every chunk starts on a 16-byte boundary when the buffer does.
 */
#ifndef KQ_H
#define KQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KQ_API __attribute__((visibility("default")))
#else
#define KQ_API
#endif

struct CUstream_st;
typedef struct CUstream_st *kq_stream_t; /* same handle as cudaStream_t */

typedef enum { KQ_Q4_K = 1, KQ_Q6_K = 2, KQ_Q8_0 = 3, KQ_Q8_K = 4, KQ_Q8_1 = 5, KQ_Q5_K = 6 } kq_dtype;

typedef enum {
    KQ_OK = 0,
    KQ_ERR_INVALID_ARG = 1,       /* null pointer, negative/zero size, K not a multiple of 256, bad ld */
    KQ_ERR_UNSUPPORTED_DTYPE = 2, /* dtype not handled by this entry point (named in kq_last_error) */
    KQ_ERR_ALIGNMENT = 3,         /* a pointer or leading dimension breaks the stated alignment */
    KQ_ERR_WORKSPACE = 4,         /* workspace missing or smaller than *_workspace_bytes */
    KQ_ERR_CUDA = 5,              /* a CUDA call failed (message in kq_last_error) */
    KQ_ERR_DEVICE_FLAG = 6        /* a kernel recorded an invalid input (e.g. an expert id out of range) */
} kq_status;

/* Static description of a status.  Never NULL. */
KQ_API const char *kq_status_string(kq_status s);

/* Thread-local detail of the last failing call on this host thread ("" if none). */
KQ_API const char *kq_last_error(void);

/* Library ABI version (major*100 + minor). */
KQ_API int kq_version(void);

/* Elements per canonical block (256 or 32) and bytes per canonical block; 0 for an unknown dtype. */
KQ_API int64_t kq_block_elems(kq_dtype dtype);
KQ_API int64_t kq_block_bytes(kq_dtype dtype);

/* Bytes of one canonical row of K elements (K/block_elems * block_bytes); 0 if K is not a block multiple. */
KQ_API int64_t kq_row_bytes(kq_dtype dtype, int64_t K);

/* Bytes of the native layout for an [N, K] weight (N padded to a multiple of 16). 0 if unsupported. */
KQ_API int64_t kq_native_bytes(kq_dtype dtype, int64_t N, int64_t K);

/* Repack canonical weight rows [N][K] (w_canon, N*kq_row_bytes bytes) into the native layout
 * (w_native, kq_native_bytes bytes, 16-byte aligned).  This is the stage-once step of the keep-quant
 * provider ([vllm-2890], keep-quant provider commit: weights are staged once and dispatched many
 * times).  For routed experts, repack [E*N][K] at once: with N a multiple of 16 each expert's rows
 * stay in their own row groups.  Padding rows are written as zeros.  Dtypes: Q4_K, Q5_K, Q6_K, Q8_0. */
KQ_API kq_status kq_repack_weights(kq_dtype dtype, const void *w_canon, void *w_native, int64_t N, int64_t K,
                            kq_stream_t stream);

/* Q8_K quantizer ([vllm-2890], warp-cooperative quantizer commit and the NaN/amax-seeding fix).
 * x: fp32 [M][ldx] (row m starts at x + m*ldx; ldx >= K); xq: M*(K/256) Q8_K blocks, row-major.
 * Per 256-element block: amax = largest |x| (strict >, so the first occurrence wins; NaN never
 * wins), mx = that element's signed value, iscale = -127/mx, q = clamp(nearest-even(iscale*x),
 * -127, 127) with NaN -> 0, d = 1/iscale, bsums[j] = sum of q[16j..16j+15].  A block with amax = 0
 * (all zeros, or only NaN/zeros) is the zero block.  x and xq need 4-byte alignment. */
KQ_API kq_status kq_quantize_q8k(const float *x, int64_t M, int64_t K, int64_t ldx, void *xq, kq_stream_t stream);

/* Q8_1 quantizer ([llama-18], fused-quant MMVQ commit).  Per 32 elements: amax = max|x| (NaN
 * ignored), d = amax/127 (IEEE division), q = roundf(x/d) (0 if amax = 0 or the quotient is not
 * finite), s = sum of the 32 inputs in xor-butterfly order (strides 16, 8, 4, 2, 1); d and s are
 * stored as f16 (round to nearest even).  Layout as kq_quantize_q8k with 36-byte blocks. */
KQ_API kq_status kq_quantize_q8_1(const float *x, int64_t M, int64_t K, int64_t ldx, void *xq, kq_stream_t stream);

/* Fused SwiGLU + Q8_1 ([vllm-2890] fused SiLU-mul quant epilogue; [llama-18] "SwiGLU
 * quantization"): h = (g / (1 + expf(-g))) * u in fp32 (no bf16 round trip), then Q8_1 of h as
 * kq_quantize_q8_1.  g and u: fp32 [M][ld] (they may be two column ranges of one buffer).
 * h_out: optional fp32 [M][K] copy of h (NULL to skip). */
KQ_API kq_status kq_swiglu_quantize_q8_1(const float *g, const float *u, int64_t M, int64_t K, int64_t ld, void *xq,
                                  float *h_out, kq_stream_t stream);

/* Fused RMSNorm + Q8_K producer ([vllm-2890], fused norm-quant epilogue): per row,
 *   r = 1 / sqrt(sum_i x_i^2 / K + eps),  y_i = (x_i * r) * gamma_i   (fp32, each operation rounded),
 * with the sum in a fixed order (256 partial sums: thread t takes x[t], x[t+256], ...; groups of 32
 * combined in xor-butterfly order; the 8 group sums added in order), then y quantised exactly as
 * kq_quantize_q8k does (byte-identical).  x: fp32 [M][ldx]; gamma: fp32 [K]; xq: Q8_K [M][K/256];
 * y_out: optional fp32 [M][K] copy of y (NULL to skip).  One launch replaces norm + quantize; its
 * output feeds kq_gemv (xq) or kq_gemm. */
KQ_API kq_status kq_rmsnorm_quantize_q8k(const float *x, const float *gamma, float eps, int64_t M, int64_t K,
                                         int64_t ldx, void *xq, float *y_out, kq_stream_t stream);

/* Fused SwiGLU + Q8_K: as kq_swiglu_quantize_q8_1 but the quantizer is kq_quantize_q8k's
 * (used between the routed gate/up and down projections). */
KQ_API kq_status kq_swiglu_quantize_q8k(const float *g, const float *u, int64_t M, int64_t K, int64_t ld, void *xq,
                                 float *h_out, kq_stream_t stream);

/* Decode GEMV, one activation column (MMVQ; [vllm-2890] MMVQ arm, [llama-18] fused-quant MMVQ).
 * Launched with programmatic dependent launch: the kernel may start, and start streaming w, while the
 * kernel issued just before it on `stream` is still running; it waits for that kernel before it
 * reads x/xq or writes y.  So w must already be in place when that earlier kernel runs: stage the
 * weights once (kq_repack_weights, then any synchronisation) as the keep-quant provider does.
 * w: native [N][K] of dtype wt (Q4_K, Q5_K or Q6_K: activation Q8_K; Q8_0: activation Q8_1).
 * Exactly one of x (fp32 [K]: quantised inside the kernel, no separate launch) and xq (pre-quantised
 * activation row, K/256 Q8_K or K/32 Q8_1 blocks) must be non-NULL.  y: fp32 [N].
 * y[n] = sum over blocks of the scaled integer block dots (the kq_gemm formula); the reduction
 * order is fixed, so results are deterministic.  Pointers: w 16-byte aligned, x/xq/y 4-byte.
 * K is at most 65536 (Q4_K, Q5_K), 55296 (Q6_K) or 26624 (Q8_0): a thread block stages its share of
 * every row's weights in shared memory; a larger K returns KQ_ERR_INVALID_ARG ("too large") without
 * launching (kq_gemm with M = 1 takes a larger K through its other kernels). */
KQ_API kq_status kq_gemv(kq_dtype wt, const void *w, const float *x, const void *xq, int64_t N, int64_t K, float *y,
                  kq_stream_t stream);

/* Workspace bytes needed by kq_gemm (n_experts = 0, top_k = 0) or by kq_gemm_grouped for the
 * same arguments.  0 means no workspace is needed. */
KQ_API size_t kq_gemm_workspace_bytes(kq_dtype wt, int64_t M, int64_t N, int64_t K, int64_t n_experts, int64_t top_k);

/* Prefill GEMM (MMQ; [vllm-3035]: one activation tile staged in shared memory per block and shared
 * by every warp).  Y[m][n] = sum_sb blockdot(W row n, X row m):
 *   Q4_K x Q8_K: per super-block d_a*(d_w*sum_j sc_j*P_j - dmin*sum_j m_j*(bs_2j + bs_2j+1)),
 *                P_j = sum of c*q over sub-block j (32 elements)
 *   Q5_K x Q8_K: the Q4_K formula over the 5-bit codes c
 *   Q6_K x Q8_K: per super-block d_a*d_w*sum_j sc_j*P_j, P_j = sum of (c-32)*q over 16 elements
 *   Q8_0 x Q8_1: per 32-block d_w*d_a*P_b
 * w: native [N][K]; xq: M activation rows (Q8_K or Q8_1 per wt); y: fp32 rows of stride ldy >= N.
 * Paths: M <= 8 (batched decode) the weight-streaming GEMV kernel, bit-exact with the sequential CPU
 * order; M >= 9 with N >= 128 the tensor-core kernel (Q8_0 bit-exact; Q4_K/Q5_K/Q6_K integer parts exact,
 * fp32 promotion fused, NMSE ~1e-14); otherwise, or when a shape does not fit the GEMV kernel, the
 * exact dp4a kernel.
 * workspace: device buffer of at least kq_gemm_workspace_bytes(wt, M, N, K, 0, 0) bytes (may be
 * NULL when that is 0), 256-byte aligned. */
KQ_API kq_status kq_gemm(kq_dtype wt, const void *w, const void *xq, int64_t M, int64_t N, int64_t K, float *y,
                  int64_t ldy, void *workspace, size_t ws_bytes, kq_stream_t stream);

/* kq_gemm with options.  flags = 0 is kq_gemm itself.
 * KQ_GEMM_FOLD_SCALES -- an opt-in throughput mode for the tensor-core shapes (M >= 9, N >= 128) of
 * Q4_K, Q5_K, Q6_K (Q8_K rows) and Q8_0 (Q8_1 rows) weights: the block scales are folded into the
 * tensor-core operands instead of being applied to integer block sums.  The weights enter the MMA as
 * their dequantised f16 values -- f16(c*f16(d*sc) + f16(-dmin*m)) (Q4_K, Q5_K), f16((c-32)*f16(d*sc))
 * (Q6_K), f16(d_w*w) (Q8_0) -- and the activations as f16(d_a*q), so a 128 x 256 output tile
 * accumulates over the whole of K in one fp32 tensor-memory buffer read out once per tile: no per-block
 * read-out, no min-term tile, one MMA per 16 K for Q6_K, and every converted weight serves 256 tokens.
 * The weights stay packed in device memory ([vllm-2890] keep-quant: staged once, never expanded);
 * only the integer dots give way to f16 products.  Not bit-exact: each operand is rounded to f16, so
 * |y - y_exact| <= (3*2^-11 + (K + K/32 + 4)*2^-24) * sum_i (|d*sc*c_i| + |dmin*m_i|)*|x_i| (plus f16
 * subnormal terms); NMSE against the exact result is ~1e-7 on N(0,1) data.  Deterministic.  Other
 * shapes take kq_gemm's exact kernels; other weight types: KQ_ERR_UNSUPPORTED_DTYPE.  Workspace:
 * kq_gemm_workspace_bytes (sized for both tile widths). */
#define KQ_GEMM_FOLD_SCALES 1u
KQ_API kq_status kq_gemm_ex(kq_dtype wt, const void *w, const void *xq, int64_t M, int64_t N, int64_t K, float *y,
                            int64_t ldy, unsigned flags, void *workspace, size_t ws_bytes, kq_stream_t stream);

/* kq_gemm from fp32 activations, with the activation quantizer moved into the GEMM that consumes it
 * ([vllm-2890]: a standalone quantizer launch costs a noticeable share of a step, so it belongs in its
 * consumer): x is fp32 [M][ldx] (ldx >= K, 4-byte aligned).  On the tensor-core
 * path (Q4_K/Q5_K/Q6_K weights, M >= 9, N >= 128) the prologue quantises each 256-element block with
 * the Q8_K quantizer's own arithmetic and writes the codes, bsums and scale straight into the GEMM's
 * f16 panels, so the Q8_K rows never travel through memory and one launch is saved; on the other paths
 * x is quantised into the workspace (Q8_K, or Q8_1 for Q8_0 weights) and kq_gemm runs on it.  Either
 * way y is bit-identical to kq_quantize_q8k (or kq_quantize_q8_1) followed by kq_gemm.
 * workspace: kq_gemm_f32_workspace_bytes(wt, M, N, K) bytes, 256-byte aligned; it begins with
 * kq_gemm's workspace, so kq_read_device_flag applies to it. */
KQ_API size_t kq_gemm_f32_workspace_bytes(kq_dtype wt, int64_t M, int64_t N, int64_t K);
KQ_API kq_status kq_gemm_f32(kq_dtype wt, const void *w, const float *x, int64_t ldx, int64_t M, int64_t N, int64_t K,
                             float *y, int64_t ldy, void *workspace, size_t ws_bytes, kq_stream_t stream);

/* kq_gemm_f32 with kq_gemm_ex's flags: with KQ_GEMM_FOLD_SCALES on the tensor-core path the prologue
 * quantises each 256-element block with the Q8_K quantizer's arithmetic and writes f16(d*q) straight
 * into the folded mode's activation panel (same result as kq_quantize_q8k followed by kq_gemm_ex). */
KQ_API kq_status kq_gemm_f32_ex(kq_dtype wt, const void *w, const float *x, int64_t ldx, int64_t M, int64_t N,
                                int64_t K, float *y, int64_t ldy, unsigned flags, void *workspace, size_t ws_bytes,
                                kq_stream_t stream);

/* Routed-expert GEMM (MUL_MAT_ID; [llama-18] routed-compact MMQ: each expert's tiles cover only the
 * rows routed to it, never a width chosen from the total number of pairs).  The tile width itself is
 * the tensor-core tile's 128 rows for every expert; the pages' narrower per-expert widths (J by rows
 * per expert) are not applied, since here a tile's cost is set by its weight conversion, which a
 * narrower tile does not reduce.
 * w: n_experts native weights, repacked together as one [n_experts*N][K] matrix (N % 16 == 0).
 * ids: int32 [M][top_k] expert of each (token, slot).  xq: activation rows; xq_rows_per_token = 1
 * ("broadcast": slot (t,k) reads row t) or top_k ("per-row": slot (t,k) reads row t*top_k+k).
 * y: fp32 [M][top_k][N]; y[t][k] = W_{ids[t][k]} . X_row.  Rows are gathered per expert in
 * (token, slot) order, so the result is deterministic.  All four weight types run on the tensor
 * cores in 128-row tiles of each expert's rows with exact integer parts; Q4_K, Q5_K and Q6_K promote to fp32
 * with fused multiply-adds (outputs match the sequential CPU order to within rounding, not bit for
 * bit), Q8_0 adds every 32-block's scaled dot in the CPU order (bit-exact).  An id outside
 * [0, n_experts) is skipped
 * (its y row is not written) and recorded in the workspace's device flag: kq_read_device_flag
 * then returns KQ_ERR_DEVICE_FLAG.  workspace: kq_gemm_workspace_bytes(wt, M, N, K, n_experts,
 * top_k) bytes, 256-byte aligned. */
KQ_API kq_status kq_gemm_grouped(kq_dtype wt, const void *w, int64_t n_experts, const void *xq, int64_t xq_rows_per_token,
                          const int32_t *ids, int64_t M, int64_t top_k, int64_t N, int64_t K, float *y,
                          void *workspace, size_t ws_bytes, kq_stream_t stream);

/* Routed gate/up GEMM with SwiGLU and Q8_K quantisation fused into its epilogue ([vllm-2890] "fuse
 * silu-mul with Q8_K quant epilogue", moved from the quantizer into the routed GEMM).
 * w: n_experts native gate/up weights repacked together as [n_experts*2F][K], each expert's gate rows
 * [0, F) followed by its up rows [F, 2F).  ids, xq, xq_rows_per_token, M, top_k, K: as for
 * kq_gemm_grouped.  hq: Q8_K [M][top_k][F/256] blocks of h = silu(gate)*up, where gate and up are the
 * rows kq_gemm_grouped would write to y (N = 2F).  The result is byte-identical to kq_gemm_grouped
 * followed by kq_swiglu_quantize_q8k(y, y + F, M*top_k, F, 2F, hq): each 128-token tile's gate and up
 * values meet in an L2-resident scratch tile of the workspace and never reach device memory as fp32.
 * F: a positive multiple of 256 (at most 2^21); K: a multiple of 256 up to 2^20; all four weight types.
 * An id outside [0, n_experts) is skipped (its hq row is not written) and recorded in the workspace's
 * device flag (kq_read_device_flag).  workspace: kq_gemm_grouped_swiglu_workspace_bytes(wt, M, F, K,
 * n_experts, top_k) bytes, 256-byte aligned; the size depends on the current device's SM count. */
KQ_API size_t kq_gemm_grouped_swiglu_workspace_bytes(kq_dtype wt, int64_t M, int64_t F, int64_t K, int64_t n_experts,
                                                     int64_t top_k);
KQ_API kq_status kq_gemm_grouped_swiglu_q8k(kq_dtype wt, const void *w, int64_t n_experts, const void *xq,
                                            int64_t xq_rows_per_token, const int32_t *ids, int64_t M, int64_t top_k,
                                            int64_t F, int64_t K, void *hq, void *workspace, size_t ws_bytes,
                                            kq_stream_t stream);

/* kq_gemm_grouped without a workspace, for callers that cannot allocate device memory when they
 * run this layer (for example a plug-in that is handed only its input and output buffers, or code
 * that must not call cudaMalloc after start-up).  The pages have no counterpart to this entry
 * point; it exists only for such callers.
 * Arguments, layouts, results and determinism are those of kq_gemm_grouped.  The routing scratch
 * lives in one fixed 1 MiB array in this library's device memory (every GPU that loads the library
 * holds it until the process exits), which allows about 250k (token, slot) pairs; larger
 * M*top_k (or n_experts) is rejected with KQ_ERR_INVALID_ARG before anything is launched.
 * The first call on a device looks the array's address up (cudaGetSymbolAddress, once per
 * device, with that device current); make that first call before any stream capture.  The address
 * belongs to the device's CUDA context: after a reset of the device (cudaDeviceReset) the next call
 * sees a new context and looks the address up again, so make that call outside a capture too.  The call
 * allocates nothing.  All calls share the one array, so calls that overlap on the GPU (other
 * streams, other host threads) race: serialise them.  Ids outside [0, n_experts) are skipped (their
 * y rows are not written) but, unlike kq_gemm_grouped, their number is not reported. */
KQ_API kq_status kq_gemm_grouped_noalloc(kq_dtype wt, const void *w, int64_t n_experts, const void *xq,
                                         int64_t xq_rows_per_token, const int32_t *ids, int64_t M, int64_t top_k,
                                         int64_t N, int64_t K, float *y, kq_stream_t stream);

/* Measurement aid, not on the hot path: the throughput ceiling of the warp-level int8 tensor path
 * (mma.sync m16n8k32 s8 x s8 -> s32), the only integer MMA sm_103a code can issue.  Launches one kernel
 * on `stream` in which every warp of 32 per SM issues `iters` x 4 independent MMAs on register
 * operands; the caller times it (CUDA events around the call).  *ops (host) receives the int8 ops
 * issued (2*16*8*32 per MMA).  sink: one int32 of device memory the kernel may write (keeps the work
 * live).  Returns KQ_ERR_INVALID_ARG for iters <= 0 or NULL pointers. */
KQ_API kq_status kq_probe_int8_mma_sync(int64_t iters, int32_t *sink, double *ops, kq_stream_t stream);

/* Read (and clear) the device flag of a kq_gemm / kq_gemm_grouped workspace.  Synchronises `stream`.
 * Returns KQ_OK, KQ_ERR_DEVICE_FLAG (an invalid expert id was seen, or a tensor-core pipeline wait
 * timed out; the count is in *n_bad if non-NULL), or KQ_ERR_CUDA. */
KQ_API kq_status kq_read_device_flag(void *workspace, int64_t *n_bad, kq_stream_t stream);

/* Weighted expert sum ([llama-18] weighted_expert_sum commit): out[t][n] = w[t][0]*y[t][0][n] +
 * w[t][1]*y[t][1][n] + ... in slot order, each product rounded before its add (no fused
 * multiply-add).  y_slots: fp32 [M][top_k][N]; w: fp32 [M][top_k]; out: fp32 [M][N]. */
KQ_API kq_status kq_moe_weighted_sum(const float *y_slots, const float *w, int64_t M, int64_t top_k, int64_t N, float *out,
                              kq_stream_t stream);

/* Routing witness (host-side dispatch counters): number of kernel launches made by this library
 * since load, in total (route = NULL) or for one route: "quantize", "repack", "gemv", "mmq_exact",
 * "mmq_tc", "route", "weighted_sum".  Unknown route names return -1.  Thread-safe. */
KQ_API int64_t kq_launch_count(const char *route);

/* Debug: the integer sub-block dots of kq_gemm, partials[m][n][j] (int32)
 * ([vllm-2890] keep-quant provider commit: the integer dots are taken in the CPU accumulation order and
 * gated bit-exact against the CPU tier):
 * Q4_K/Q5_K: K/32 per (m,n), P_j = sum c*q; Q6_K: K/16, P_j = sum (c-32)*q; Q8_0: K/32, P_b = sum w*q.
 * Computed by the exact dp4a kernel, one integer dot per sub-block; bit-exact by contract. */
KQ_API kq_status kq_debug_partials(kq_dtype wt, const void *w, const void *xq, int64_t M, int64_t N, int64_t K,
                            int32_t *partials, kq_stream_t stream);

/* Debug: the split-K factor (CTAs of a thread-block cluster per 128 x 128 output tile, 1 = no split)
 * that kq_gemm's tensor-core path takes for this shape on the current device -- the most CTAs any output
 * tile's K is shared between: the cluster split, or the split of the tail launch (a persistent launch
 * whose last wave would leave most SMs idle runs its whole waves and then the leftover tiles as split-K
 * clusters) -- or 0 when the shape does not take the tensor-core path.  Host only; launches nothing. */
KQ_API int kq_debug_tc_splits(kq_dtype wt, int64_t M, int64_t N, int64_t K);

/* Debug twin of kq_gemm's tensor-core path ([vllm-2890] keep-quant provider commit: integer dots
 * bit-exact against the CPU tier).  Runs the very kernel kq_gemm runs for this shape (same tiles, same
 * split-K clusters, same TMEM accumulation), with a debug epilogue that also writes, before the fp32
 * promotion, the integer sums each scale block accumulated in tensor memory:
 *   sums[m][n][b][0] = sum_j sc_j*P_j over block b (Q4_K, Q5_K, Q6_K: 256 elements), P_b (Q8_0: 32)
 *   sums[m][n][b][1] = sum_j m_j*(bs_2j + bs_2j+1) (Q4_K, Q5_K min term), else 0
 * as int32 [M][N][nblk][2], nblk = K/256 (K/32 for Q8_0).  y is written as by kq_gemm.  Arguments and
 * workspace as kq_gemm; KQ_ERR_INVALID_ARG when the shape does not take the tensor-core path (M <= 8 or
 * N < 128). */
KQ_API kq_status kq_debug_tc_sums(kq_dtype wt, const void *w, const void *xq, int64_t M, int64_t N, int64_t K,
                                  float *y, int64_t ldy, int32_t *sums, void *workspace, size_t ws_bytes,
                                  kq_stream_t stream);

/* Debug twin of kq_gemm_grouped's tensor-core path: sums as kq_debug_tc_sums, one row per (token, slot)
 * pair, int32 [M*top_k][N][nblk][2]; rows of invalid ids are not written.  Arguments and workspace as
 * kq_gemm_grouped. */
KQ_API kq_status kq_debug_tc_sums_grouped(kq_dtype wt, const void *w, int64_t n_experts, const void *xq,
                                          int64_t xq_rows_per_token, const int32_t *ids, int64_t M, int64_t top_k,
                                          int64_t N, int64_t K, float *y, int32_t *sums, void *workspace,
                                          size_t ws_bytes, kq_stream_t stream);

/* Test hook of the tensor-core pipeline's bounded waits: runs kq_gemm's tensor-core kernel with its
 * activation-tile producer kept idle, so the first wait for an activation tile can never complete,
 * and with every pipeline wait limited to wait_limit_ns (1e3 .. 1e9; kq_gemm uses 2 s).  The waits
 * run out, each CTA records the timeout in the workspace's device flag, waits (bounded) for its own
 * copies and MMAs in flight, frees its tensor memory and returns: the call itself returns KQ_OK, y is
 * left incomplete, and kq_read_device_flag then reports KQ_ERR_DEVICE_FLAG.  Nothing faults or hangs;
 * the stream stays usable for the next call. */
KQ_API kq_status kq_debug_tc_wait_timeout(kq_dtype wt, const void *w, const void *xq, int64_t M, int64_t N, int64_t K,
                                          float *y, int64_t ldy, int64_t wait_limit_ns, void *workspace,
                                          size_t ws_bytes, kq_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* KQ_H */
