// kq_api.cu -- status strings, thread-local error detail, geometry queries, weight repack.
#include <atomic>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "kq_internal.cuh"

namespace kq {

static thread_local char g_last_error[512] = "";
static std::atomic<int64_t> g_launches[R_COUNT];
static const char *kRouteNames[R_COUNT] = {"quantize", "repack", "gemv", "mmq_exact", "mmq_tc", "route", "weighted_sum"};

void count_launch(Route r, int kernels) { g_launches[r].fetch_add(kernels, std::memory_order_relaxed); }

void set_error(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
}

kq_status fail(kq_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return s;
}

kq_status check_launch(const char *what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(KQ_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
    return KQ_OK;
}

const char *dtype_name(kq_dtype d) {
    switch (d) {
    case KQ_Q4_K: return "Q4_K";
    case KQ_Q5_K: return "Q5_K";
    case KQ_Q6_K: return "Q6_K";
    case KQ_Q8_0: return "Q8_0";
    case KQ_Q8_K: return "Q8_K";
    case KQ_Q8_1: return "Q8_1";
    default: return "unknown";
    }
}

// One thread block per (row group, K-chunk).  Each thread owns one (row, 64-element kblock) slice of
// the chunk and writes that slice's planes; rows past N are written as zeros.
__global__ void repack_kernel(int dtype, const uint8_t *__restrict__ src, uint8_t *__restrict__ dst, int64_t N,
                              int64_t K) {
    const int64_t g = blockIdx.y, c = blockIdx.x;
    const int64_t nchunk = K / kChunkK;
    uint8_t *out = dst + chunk_offset(dtype, g, c, nchunk);
    const int tid = threadIdx.x;
    if (tid >= kRowGroup * 4) return;
    const int r = tid >> 2, kb = tid & 3;
    const int64_t n = g * kRowGroup + r;
    const bool valid = n < N;
    if (dtype == KQ_Q4_K || dtype == KQ_Q5_K) {
        // Q5_K canonical block: header 16 | high bits 32 | nibbles 128; the native chunk keeps the Q4_K
        // arrangement and appends each row's 32 high-bit bytes at 2304 + r*32
        const int bb = dtype == KQ_Q4_K ? 144 : 176, qs = dtype == KQ_Q4_K ? 16 : 48;
        const uint8_t *blk = src + n * (nchunk * bb) + c * bb;
        uint8_t *codes = out + kb * 512 + r * 32;
        for (int l = 0; l < 32; ++l) codes[l] = valid ? blk[qs + 32 * kb + l] : 0;
        if (kb == 0)
            for (int i = 0; i < 16; ++i) out[2048 + r * 16 + i] = valid ? blk[i] : 0;
        if (dtype == KQ_Q5_K && kb == 1)
            for (int i = 0; i < 32; ++i) out[2304 + r * 32 + i] = valid ? blk[16 + i] : 0;
    } else if (dtype == KQ_Q6_K) {
        const uint8_t *blk = src + n * (nchunk * 210) + c * 210;
        uint8_t code[64];
        for (int e = 0; e < 64; ++e) {
            const int el = 64 * kb + e;            // element within the super-block
            uint8_t v = 0;
            if (valid) {
                const uint8_t *ql = blk + 64 * (el / 128);
                const uint8_t *qh = blk + 128 + 32 * (el / 128);
                const int rr = el % 128, quarter = rr / 32, l = rr % 32;
                int lo = (quarter & 1) ? ql[l + 32] : ql[l];
                lo = (quarter & 2) ? (lo >> 4) : (lo & 15);
                const int hi = (qh[l] >> (2 * quarter)) & 3;
                v = (uint8_t)(lo | (hi << 4));
            }
            code[e] = v;
        }
        uint8_t *nib = out + kb * 512 + r * 32;
        for (int l = 0; l < 32; ++l) nib[l] = (code[l] & 15) | ((code[l + 32] & 15) << 4);
        uint8_t *hb = out + 2048 + kb * 256 + r * 16;
        for (int j = 0; j < 16; ++j)
            hb[j] = (code[j] >> 4) | ((code[j + 16] >> 4) << 2) | ((code[j + 32] >> 4) << 4) | ((code[j + 48] >> 4) << 6);
        if (kb == 0) {
            for (int i = 0; i < 16; ++i) out[3072 + r * 16 + i] = valid ? blk[192 + i] : 0;
            out[3328 + r * 2] = valid ? blk[208] : 0;
            out[3328 + r * 2 + 1] = valid ? blk[209] : 0;
        }
    } else {  // Q8_0: 8 canonical 34-byte blocks per chunk, two per kblock
        const int64_t rowb = (K / 32) * 34;
        uint8_t *codes = out + kb * 1024 + r * 64;
        for (int h = 0; h < 2; ++h) {
            const uint8_t *blk = src + n * rowb + (c * 8 + 2 * kb + h) * 34;
            for (int i = 0; i < 32; ++i) codes[32 * h + i] = valid ? blk[2 + i] : 0;
            out[4096 + r * 16 + 2 * (2 * kb + h)] = valid ? blk[0] : 0;
            out[4096 + r * 16 + 2 * (2 * kb + h) + 1] = valid ? blk[1] : 0;
        }
    }
}

}  // namespace kq

using namespace kq;

extern "C" {

const char *kq_status_string(kq_status s) {
    switch (s) {
    case KQ_OK: return "ok";
    case KQ_ERR_INVALID_ARG: return "invalid argument";
    case KQ_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
    case KQ_ERR_ALIGNMENT: return "misaligned pointer or stride";
    case KQ_ERR_WORKSPACE: return "workspace missing or too small";
    case KQ_ERR_CUDA: return "CUDA error";
    case KQ_ERR_DEVICE_FLAG: return "device reported invalid input";
    default: return "unknown status";
    }
}

const char *kq_last_error(void) { return g_last_error; }

int kq_version(void) { return 100; }

int64_t kq_launch_count(const char *route) {
    if (!route) {
        int64_t t = 0;
        for (int i = 0; i < R_COUNT; ++i) t += g_launches[i].load(std::memory_order_relaxed);
        return t;
    }
    for (int i = 0; i < R_COUNT; ++i)
        if (strcmp(route, kRouteNames[i]) == 0) return g_launches[i].load(std::memory_order_relaxed);
    return -1;
}

int64_t kq_block_elems(kq_dtype d) {
    switch (d) {
    case KQ_Q4_K: case KQ_Q5_K: case KQ_Q6_K: case KQ_Q8_K: return 256;
    case KQ_Q8_0: case KQ_Q8_1: return 32;
    default: return 0;
    }
}

int64_t kq_block_bytes(kq_dtype d) {
    switch (d) {
    case KQ_Q4_K: return 144;
    case KQ_Q5_K: return 176;
    case KQ_Q6_K: return 210;
    case KQ_Q8_0: return 34;
    case KQ_Q8_K: return 292;
    case KQ_Q8_1: return 36;
    default: return 0;
    }
}

int64_t kq_row_bytes(kq_dtype d, int64_t K) {
    int64_t be = kq_block_elems(d);
    if (be == 0 || K <= 0 || K % be) return 0;
    return K / be * kq_block_bytes(d);
}

int64_t kq_native_bytes(kq_dtype d, int64_t N, int64_t K) {
    if (chunk_bytes(d) == 0 || N <= 0 || K <= 0 || K % kChunkK) return 0;
    int64_t groups = (N + kRowGroup - 1) / kRowGroup;
    return groups * (K / kChunkK) * chunk_bytes(d);
}

kq_status kq_repack_weights(kq_dtype dtype, const void *w_canon, void *w_native, int64_t N, int64_t K,
                            kq_stream_t stream) {
    if (dtype != KQ_Q4_K && dtype != KQ_Q5_K && dtype != KQ_Q6_K && dtype != KQ_Q8_0)
        return fail(KQ_ERR_UNSUPPORTED_DTYPE, "kq_repack_weights: weight dtype %s is not Q4_K, Q5_K, Q6_K or Q8_0",
                    dtype_name(dtype));
    if (!w_canon || !w_native) return fail(KQ_ERR_INVALID_ARG, "kq_repack_weights: null pointer");
    if (N <= 0 || K <= 0 || K % kChunkK)
        return fail(KQ_ERR_INVALID_ARG, "kq_repack_weights: need N > 0 and K a positive multiple of 256 (N=%lld K=%lld)",
                    (long long)N, (long long)K);
    if (!aligned(w_native, 16)) return fail(KQ_ERR_ALIGNMENT, "kq_repack_weights: w_native must be 16-byte aligned");
    int64_t groups = (N + kRowGroup - 1) / kRowGroup;
    if (groups > 65535 * 64)
        return fail(KQ_ERR_INVALID_ARG, "kq_repack_weights: N=%lld too large", (long long)N);
    dim3 grid((unsigned)(K / kChunkK), 1, 1);
    // grid.y is limited to 65535: loop over row-group slabs.
    for (int64_t g0 = 0; g0 < groups; g0 += 65535) {
        int64_t gn = groups - g0 < 65535 ? groups - g0 : 65535;
        grid.y = (unsigned)gn;
        const uint8_t *src = static_cast<const uint8_t *>(w_canon) + g0 * kRowGroup * kq_row_bytes(dtype, K);
        uint8_t *dst = static_cast<uint8_t *>(w_native) + chunk_offset(dtype, g0, 0, K / kChunkK);
        repack_kernel<<<grid, 64, 0, (cudaStream_t)stream>>>(dtype, src, dst, N - g0 * kRowGroup, K);
        kq_status s = check_launch("kq_repack_weights");
        if (s != KQ_OK) return s;
        count_launch(R_REPACK);
    }
    return KQ_OK;
}

}  // extern "C"
