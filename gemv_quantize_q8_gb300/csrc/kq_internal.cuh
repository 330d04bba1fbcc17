// kq_internal.cuh -- shared internals of the kq CUDA library (not part of the ABI).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kq.h"

namespace kq {

// ---------------------------------------------------------------- error reporting (host)
void set_error(const char *fmt, ...);
kq_status fail(kq_status s, const char *fmt, ...);
kq_status check_launch(const char *what);
const char *dtype_name(kq_dtype d);

// Host-side routing witness: counts kernel launches per route.
enum Route { R_QUANT = 0, R_REPACK, R_GEMV, R_MMQ_EXACT, R_MMQ_TC, R_ROUTE, R_WSUM, R_COUNT };
void count_launch(Route r, int kernels = 1);

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---------------------------------------------------------------- native layout geometry
constexpr int kRowGroup = 16;   // rows per native row group
constexpr int kChunkK = 256;    // elements per native chunk along K

constexpr int kQ4KCodeBytes = 128, kQ4KHdrBytes = 16;
constexpr int kQ4KChunk = kRowGroup * (kQ4KCodeBytes + kQ4KHdrBytes);        // 2304
constexpr int kQ6KCodeBytes = 192, kQ6KScaleBytes = 16;
constexpr int kQ6KChunk = kRowGroup * (kQ6KCodeBytes + kQ6KScaleBytes + 2);  // 3360
constexpr int kQ80Chunk = kRowGroup * (256 + 8 * 2);                          // 4352
// Q5_K: the Q4_K chunk (nibbles of 4 kblocks, then 16-byte row headers) followed by each row's 32
// high-bit bytes: 2048 + 256 + 512
constexpr int kQ5KChunk = kRowGroup * (kQ4KCodeBytes + kQ4KHdrBytes + 32);     // 2816

__host__ __device__ constexpr int chunk_bytes(int dtype) {
    return dtype == KQ_Q4_K ? kQ4KChunk : dtype == KQ_Q5_K ? kQ5KChunk : dtype == KQ_Q6_K ? kQ6KChunk
           : dtype == KQ_Q8_0 ? kQ80Chunk : 0;
}

// Byte offset of chunk (row group g, K-chunk c) for a weight with nchunk chunks per row.
__host__ __device__ inline int64_t chunk_offset(int dtype, int64_t g, int64_t c, int64_t nchunk) {
    return (g * nchunk + c) * (int64_t)chunk_bytes(dtype);
}

// ---------------------------------------------------------------- activation block geometry
constexpr int kQ8KBytes = 292;  // f32 d, int8 q[256], int16 bsums[16]
constexpr int kQ81Bytes = 36;   // f16 d, f16 s, int8 q[32]

// ---------------------------------------------------------------- batched decode (kq_gemv.cu)
constexpr int kGemvMaxBatch = 8;
// y[m*ldy + n] for m < M <= kGemvMaxBatch quantised activation rows, bit-identical to the CPU order;
// KQ_ERR_INVALID_ARG when the shape does not fit (the caller then takes the general path).
kq_status gemv_batched(kq_dtype wt, const uint8_t *w, const uint8_t *xq, int64_t M, int64_t N, int64_t K, float *y,
                       int64_t ldy, cudaStream_t st);

// ---------------------------------------------------------------- device helpers
__device__ __forceinline__ int dp4a(int a, int b, int c) { return __dp4a(a, b, c); }

__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
    return __half2float(__ushort_as_half(h));
}

// Q4_K 6-bit scale and min of sub-block j from the 12 packed bytes (canonical GGUF packing).
__device__ __forceinline__ void q4k_scale_min(const uint8_t *s12, int j, int &sc, int &mn) {
    if (j < 4) {
        sc = s12[j] & 63;
        mn = s12[j + 4] & 63;
    } else {
        sc = (s12[j + 4] & 0x0f) | ((s12[j - 4] >> 6) << 4);
        mn = (s12[j + 4] >> 4) | ((s12[j] >> 6) << 4);
    }
}

}  // namespace kq
