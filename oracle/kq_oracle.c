/*
 * kq_oracle.c -- plain, slow CPU oracle for the keep-quant matmul path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file.  Only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table
 * or constant with the CUDA library.
 *
 * What it follows (the pages print prose only; no listing is restated):
 *  - vllm.cpp PR #2890 "fuse silu-mul with Q8_K quant epilogue", commit
 *    "QuantizeQ8KKWarpCoop": Q8_K quantizer semantics (first max-|x| element
 *    mx, iscale = -127/mx, nearest integer, clamp 127, d = 1/iscale, bsums
 *    of 16), and the commit that seeds amax at 0 so a NaN/zero block gives
 *    the zero block.
 *  - same page, commit "register MatmulBTQuant ... kROCM": integer dots in a
 *    fixed CPU accumulation order, f64 dequant band 5e-4, NMSE 1e-6.
 *  - strix-llama.cpp PR #18 "Optimize ROCM Prefill and Decode", commits
 *    "mul_mat_vec_q_fq" (Q8_1: amax, d = amax/127, IEEE division, roundf,
 *    block sum in xor-butterfly order) and "weighted_expert_sum_f32"
 *    (explicit multiply then add, fixed slot order), and the MUL_MAT_ID
 *    commits (per-expert row lists from routing ids).
 *  - the public GGUF block layouts (Q4_K, Q6_K, Q8_0, Q8_K, Q8_1), which the
 *    pages name but do not print.
 *
 * Floating point: every fp32 operation below is a single IEEE operation in
 * round-to-nearest-even; the build uses -ffp-contract=off so no multiply and
 * add fuse.  f64 is used only where a function says so (dequantisation for
 * the f64 reference band).
 *
 * Parity status per function: see the header comment of each.  Functions
 * whose results are pinned only by self-consistency say "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_API __attribute__((visibility("default")))

enum { ORC_Q4_K = 1, ORC_Q6_K = 2, ORC_Q8_0 = 3, ORC_Q8_K = 4, ORC_Q8_1 = 5, ORC_Q5_K = 6 };

/* ------------------------------------------------------------------------ */
/* IEEE binary16 <-> binary32, written from the IEEE 754 definition.         */
/* ------------------------------------------------------------------------ */

ORC_API float orc_half_to_float(uint16_t h) {
    uint32_t sign = (uint32_t)(h >> 15) & 1u;
    uint32_t expo = (uint32_t)(h >> 10) & 0x1fu;
    uint32_t mant = (uint32_t)h & 0x3ffu;
    float mag;
    if (expo == 0) {
        mag = ldexpf((float)mant, -24);            /* subnormal: mant * 2^-24 */
    } else if (expo == 31) {
        mag = mant ? NAN : INFINITY;
    } else {
        mag = ldexpf((float)(mant | 0x400u), (int)expo - 25);
    }
    return sign ? -mag : mag;
}

/* Round-to-nearest-even conversion, overflow to infinity.  Any NaN becomes the
 * one quiet NaN 0x7e00 (IEEE arithmetic does not fix the sign or payload of a
 * NaN result, so no sign is carried). */
ORC_API uint16_t orc_float_to_half(float f) {
    uint32_t bits;
    memcpy(&bits, &f, 4);
    uint16_t sign = (uint16_t)((bits >> 16) & 0x8000u);
    if (isnan(f)) return (uint16_t)0x7e00u;
    double a = fabs((double)f);               /* exact copy of |f| */
    if (a == 0.0) return sign;
    /* find the binary16 exponent: value = m * 2^(e-10), 1024 <= m < 2048 */
    int e;
    (void)frexp(a, &e);                        /* a = fr * 2^e, 0.5 <= fr < 1 */
    int ue = e - 1;                            /* a in [2^ue, 2^(ue+1)) */
    if (ue < -14) ue = -14;                    /* subnormal range: fixed quantum 2^-24 */
    double quantum = ldexp(1.0, ue - 10);
    double q = a / quantum;                    /* exact: power-of-two scaling */
    double r = nearbyint(q);                   /* ties to even in default mode */
    /* r may have rounded up to 2048 -> next binade, handled by re-encoding */
    double val = r * quantum;
    if (val >= 65520.0 || val > 65504.0) return (uint16_t)(sign | 0x7c00u);
    if (val == 0.0) return sign;
    int e2;
    (void)frexp(val, &e2);
    int ue2 = e2 - 1;
    if (ue2 < -14) {
        uint32_t m = (uint32_t)(val / ldexp(1.0, -24));
        return (uint16_t)(sign | m);
    }
    uint32_t m = (uint32_t)(val / ldexp(1.0, ue2 - 10)) - 1024u;
    return (uint16_t)(sign | ((uint32_t)(ue2 + 15) << 10) | m);
}

static void wr_half(uint8_t *p, uint16_t h) {
    p[0] = (uint8_t)(h & 0xff);
    p[1] = (uint8_t)(h >> 8);
}
static float rd_f32(const uint8_t *p) {
    float f;
    memcpy(&f, p, 4);
    return f;
}
static int16_t rd_i16(const uint8_t *p) {
    int16_t v;
    memcpy(&v, p, 2);
    return v;
}

/* ------------------------------------------------------------------------ */
/* Block geometry of the GGUF-style canonical layouts.                      */
/* ------------------------------------------------------------------------ */

ORC_API int64_t orc_block_elems(int dtype) {
    switch (dtype) {
    case ORC_Q4_K: case ORC_Q5_K: case ORC_Q6_K: case ORC_Q8_K: return 256;
    case ORC_Q8_0: case ORC_Q8_1: return 32;
    default: return 0;
    }
}
ORC_API int64_t orc_block_bytes(int dtype) {
    switch (dtype) {
    case ORC_Q4_K: return 144;  /* d, dmin, 12 scale bytes, 128 nibble bytes */
    case ORC_Q5_K: return 176;  /* d, dmin, 12 scale bytes, 32 high-bit bytes, 128 nibble bytes */
    case ORC_Q6_K: return 210;  /* ql[128], qh[64], int8 scales[16], d */
    case ORC_Q8_0: return 34;   /* d, int8[32] */
    case ORC_Q8_K: return 292;  /* f32 d, int8[256], int16 bsums[16] */
    case ORC_Q8_1: return 36;   /* d, s, int8[32] */
    default: return 0;
    }
}

/* Q4_K: 6-bit scale and min of sub-block j (0..7) from the 12 packed bytes.
 * Bytes 0..3: low 6 bits = scale j, top 2 bits = high bits of scale j+4.
 * Bytes 4..7: same for the mins.  Bytes 8..11: low nibble = low 4 bits of
 * scale j+4, high nibble = low 4 bits of min j+4. */
static void q4k_scale_min(const uint8_t *s12, int j, int *sc, int *mn) {
    if (j < 4) {
        *sc = s12[j] & 63;
        *mn = s12[j + 4] & 63;
    } else {
        *sc = (s12[j + 4] & 0x0f) | ((s12[j - 4] >> 6) << 4);
        *mn = (s12[j + 4] >> 4) | ((s12[j] >> 6) << 4);
    }
}

/* Q4_K: 4-bit code of element i (0..255).  Codes come in 64-element chunks;
 * byte l of chunk c holds element 64c+l (low nibble) and 64c+32+l (high). */
static int q4k_code(const uint8_t *qs, int i) {
    int c = i / 64, r = i % 64;
    uint8_t b = qs[32 * c + (r % 32)];
    return r < 32 ? (b & 0x0f) : (b >> 4);
}

/* Q5_K: 5-bit code (0..31) of element i: the Q4_K nibble (same 64-element chunk layout, nibbles at
 * byte 48 of the block) plus 16 times a high bit from qh[32] (byte 16 of the block): for element
 * 64c + l (l < 32) bit 2c of qh[l], for element 64c + 32 + l bit 2c+1 of qh[l]. */
static int q5k_code(const uint8_t *blk, int i) {
    int c = i / 64, r = i % 64, l = r % 32;
    int hb = (blk[16 + l] >> (2 * c + (r >= 32))) & 1;
    return q4k_code(blk + 48, i) | (hb << 4);
}

/* Q6_K: 6-bit code (0..63, stored with an offset of 32) of element i.
 * Two 128-element halves; in half h, for l < 32:
 *   element l    : ql[l]    low nibble, qh[l] bits 0-1
 *   element l+32 : ql[l+32] low nibble, qh[l] bits 2-3
 *   element l+64 : ql[l]    high nibble, qh[l] bits 4-5
 *   element l+96 : ql[l+32] high nibble, qh[l] bits 6-7          */
static int q6k_code(const uint8_t *blk, int i) {
    const uint8_t *ql = blk + 64 * (i / 128);
    const uint8_t *qh = blk + 128 + 32 * (i / 128);
    int r = i % 128, quarter = r / 32, l = r % 32;
    int lo = (quarter & 1) ? ql[l + 32] : ql[l];
    lo = (quarter & 2) ? (lo >> 4) : (lo & 0x0f);
    int hi = (qh[l] >> (2 * quarter)) & 3;
    return lo | (hi << 4);
}

/* ------------------------------------------------------------------------ */
/* Dequantisation into f64 (for the f64 reference band and the pins).       */
/* ------------------------------------------------------------------------ */

/* Q4_K: x = d*sc*c - dmin*m.  Parity pinned by hand-built blocks. */
ORC_API void orc_dequant_q4_k(const uint8_t *blk, double *out) {
    double d = orc_half_to_float((uint16_t)(blk[0] | (blk[1] << 8)));
    double dmin = orc_half_to_float((uint16_t)(blk[2] | (blk[3] << 8)));
    const uint8_t *s12 = blk + 4, *qs = blk + 16;
    for (int i = 0; i < 256; ++i) {
        int sc, mn;
        q4k_scale_min(s12, i / 32, &sc, &mn);
        out[i] = d * sc * q4k_code(qs, i) - dmin * mn;
    }
}

/* Q5_K: x = d*sc*c - dmin*m with the 5-bit code c.  Pinned by single-element position sweeps and the
 * unit-scale integer reduction. */
ORC_API void orc_dequant_q5_k(const uint8_t *blk, double *out) {
    double d = orc_half_to_float((uint16_t)(blk[0] | (blk[1] << 8)));
    double dmin = orc_half_to_float((uint16_t)(blk[2] | (blk[3] << 8)));
    const uint8_t *s12 = blk + 4;
    for (int i = 0; i < 256; ++i) {
        int sc, mn;
        q4k_scale_min(s12, i / 32, &sc, &mn);
        out[i] = d * sc * q5k_code(blk, i) - dmin * mn;
    }
}

/* Q6_K: x = d*sc*(c-32), sub-blocks of 16.  Pinned by hand-built blocks. */
ORC_API void orc_dequant_q6_k(const uint8_t *blk, double *out) {
    double d = orc_half_to_float((uint16_t)(blk[208] | (blk[209] << 8)));
    const int8_t *sc = (const int8_t *)(blk + 192);
    for (int i = 0; i < 256; ++i) out[i] = d * sc[i / 16] * (q6k_code(blk, i) - 32);
}

/* Q8_0: x = d*w. */
ORC_API void orc_dequant_q8_0(const uint8_t *blk, double *out) {
    double d = orc_half_to_float((uint16_t)(blk[0] | (blk[1] << 8)));
    const int8_t *w = (const int8_t *)(blk + 2);
    for (int i = 0; i < 32; ++i) out[i] = d * w[i];
}

/* Q8_K activation: x = d*q (d is f32). */
ORC_API void orc_dequant_q8_k(const uint8_t *blk, double *out) {
    double d = rd_f32(blk);
    const int8_t *q = (const int8_t *)(blk + 4);
    for (int i = 0; i < 256; ++i) out[i] = d * q[i];
}

/* Q8_1 activation: x = d*q (d stored as f16). */
ORC_API void orc_dequant_q8_1(const uint8_t *blk, double *out) {
    double d = orc_half_to_float((uint16_t)(blk[0] | (blk[1] << 8)));
    const int8_t *q = (const int8_t *)(blk + 4);
    for (int i = 0; i < 32; ++i) out[i] = d * q[i];
}

/* ------------------------------------------------------------------------ */
/* Activation quantisers.                                                   */
/* ------------------------------------------------------------------------ */

/* Nearest integer, ties to even (the "DNearestInt" of the warp-cooperative
 * quantizer commit, read as round-half-even), with the code clamped to
 * [-127, 127] and a NaN product mapped to 0.  For finite inputs the product
 * never leaves [-127, 127] by more than rounding, so the clamp is the
 * "clamp 127" of the page and the lower side never binds. */
static int q8k_code(float p) {
    if (isnan(p)) return 0;
    if (p >= 127.0f) return 127;
    if (p <= -127.0f) return -127;
    return (int)rintf(p);
}

/* Q8_K quantizer, one 256-element block.
 * Parity pinned: closed forms (spike, zero block, tie, ramp, half-way tie),
 * the |x - d*q| <= |d|/2 rounding bound, bsums recomputed independently. */
static void quantize_block_q8_k(const float *x, uint8_t *blk) {
    float amax = 0.0f, mx = 0.0f;
    for (int i = 0; i < 256; ++i) {            /* first occurrence wins: strict > */
        float ax = fabsf(x[i]);
        if (ax > amax) { amax = ax; mx = x[i]; }
    }
    int8_t *q = (int8_t *)(blk + 4);
    if (amax == 0.0f) {                        /* zero block: d = 0, q = 0, bsums = 0 */
        memset(blk, 0, 292);
        return;
    }
    float iscale = -127.0f / mx;
    for (int i = 0; i < 256; ++i) q[i] = (int8_t)q8k_code(iscale * x[i]);
    for (int j = 0; j < 16; ++j) {
        int s = 0;
        for (int i = 0; i < 16; ++i) s += q[16 * j + i];
        int16_t s16 = (int16_t)s;
        memcpy(blk + 260 + 2 * j, &s16, 2);
    }
    float d = 1.0f / iscale;
    memcpy(blk, &d, 4);
}

ORC_API void orc_quantize_q8_k(const float *x, int64_t M, int64_t K, int64_t ldx, uint8_t *out) {
    int64_t nb = K / 256;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t b = 0; b < nb; ++b)
            quantize_block_q8_k(x + m * ldx + 256 * b, out + (m * nb + b) * 292);
}

/* Sum of 32 values in xor-butterfly order: at each stride (16, 8, 4, 2, 1)
 * every slot i becomes p[i] + p[i ^ stride]; the result is slot 0.
 * Parity pinned: bounded against an exact sum, and the stride order by inputs
 * whose large parts cancel exactly only at the right stage (the sum is then a
 * closed-form exact value that a differently ordered tree misses). */
static float butterfly_sum32(const float *v) {
    float p[32], t[32];
    for (int i = 0; i < 32; ++i) p[i] = v[i];
    for (int stride = 16; stride >= 1; stride /= 2) {
        for (int i = 0; i < 32; ++i) t[i] = p[i] + p[i ^ stride];
        for (int i = 0; i < 32; ++i) p[i] = t[i];
    }
    return p[0];
}

/* Q8_1 quantizer, one 32-element block: amax = max|x| (NaN ignored),
 * d = amax/127 (IEEE), q = roundf(x/d) (0 when amax == 0 or the quotient is
 * not finite), s = butterfly sum of x; d and s are stored as f16 (RNE).
 * Parity pinned: rounding bound |x - d*q| <= d/2, zero block, s against an
 * exact sum within the fp32 error bound of a 32-term tree. */
static void quantize_block_q8_1(const float *x, uint8_t *blk) {
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
    float d = amax / 127.0f;
    int8_t *q = (int8_t *)(blk + 4);
    for (int i = 0; i < 32; ++i) {
        float r = amax == 0.0f ? 0.0f : roundf(x[i] / d);
        if (!isfinite(r)) r = 0.0f;            /* NaN input, or d underflowed to 0 */
        if (r > 127.0f) r = 127.0f;            /* never binds for finite input */
        if (r < -127.0f) r = -127.0f;
        q[i] = (int8_t)(int)r;
    }
    float s = butterfly_sum32(x);
    wr_half(blk, orc_float_to_half(d));
    wr_half(blk + 2, orc_float_to_half(s));
}

ORC_API void orc_quantize_q8_1(const float *x, int64_t M, int64_t K, int64_t ldx, uint8_t *out) {
    int64_t nb = K / 32;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t b = 0; b < nb; ++b)
            quantize_block_q8_1(x + m * ldx + 32 * b, out + (m * nb + b) * 36);
}

/* SwiGLU: h = silu(g) * u with silu(g) = g / (1 + exp(-g)), all fp32.
 * (Parity vs a GPU exp is ulp-bounded, not bit-exact: parity unpinned for
 * exact equality; the tests bound the difference.) */
ORC_API void orc_swiglu(const float *g, const float *u, int64_t M, int64_t K, int64_t ld, float *h, int64_t ldh) {
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) {
            float gv = g[m * ld + k];
            float e = expf(-gv);
            float den = 1.0f + e;
            float s = gv / den;
            h[m * ldh + k] = s * u[m * ld + k];
        }
}

/* RMSNorm producer (vllm.cpp PR #2890, the fused norm-quant epilogue commit: the norm row kernel
 * emits the row's Q8_K blocks beside its normalized output, byte-identical to quantizing that output
 * with the standalone quantizer).  The pages give no formula; the reading is the usual definition:
 *   ss = sum_i x_i^2,  r = 1 / sqrt(ss / K + eps),  y_i = (x_i * r) * gamma_i        (all fp32)
 * with the sum of squares taken in plain ascending order (i = 0, 1, ..., K-1), each square and each
 * add rounded on its own.  Division and square root are the IEEE ones (sqrtf, /).  A GPU row
 * reduction sums in another order, so its ss differs from this one within the error bound of
 * recursive summation; the tests bound y by that, and check the Q8_K bytes on the GPU's own y.
 * Parity pinned: f64 RMSNorm within the fp32 error bound, a constant row (exact), the zero row,
 * invariance under scaling x by a power of two, position independence of x_i*gamma_i, and the
 * ascending order itself by rows whose total is a closed form only in that order. */
ORC_API void orc_rmsnorm(const float *x, const float *gamma, float eps, int64_t M, int64_t K, int64_t ldx, float *y,
                         int64_t ldy) {
    for (int64_t m = 0; m < M; ++m) {
        const float *xr = x + m * ldx;
        float total = 0.0f;
        for (int64_t i = 0; i < K; ++i) {
            float sq = xr[i] * xr[i];
            total = total + sq;
        }
        float mean = total / (float)K;
        float r = 1.0f / sqrtf(mean + eps);
        for (int64_t i = 0; i < K; ++i) {
            float a = xr[i] * r;
            y[m * ldy + i] = a * gamma[i];
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Integer block dots.                                                       */
/* ------------------------------------------------------------------------ */

/* Partial integer dots of one weight block row against one activation row.
 * Q4_K x Q8_K: P_j = sum_{i<32} c*q over sub-block j (8 per super-block).
 * Q5_K x Q8_K: the same over the 5-bit codes.
 * Q6_K x Q8_K: P_j = sum_{i<16} (c-32)*q over sub-block j (16 per super-block).
 * Q8_0 x Q8_1: P_b = sum_{i<32} w*q over block b.
 * Output: K/32 (Q4_K, Q5_K, Q8_0) or K/16 (Q6_K) int32 values. */
ORC_API void orc_partials_row(int dtype, const uint8_t *wrow, const uint8_t *xrow, int64_t K, int32_t *out) {
    if (dtype == ORC_Q4_K) {
        for (int64_t b = 0; b < K / 256; ++b) {
            const uint8_t *wb = wrow + 144 * b;
            const int8_t *q = (const int8_t *)(xrow + 292 * b + 4);
            for (int j = 0; j < 8; ++j) {
                int32_t acc = 0;
                for (int i = 32 * j; i < 32 * j + 32; ++i) acc += q4k_code(wb + 16, i) * q[i];
                out[8 * b + j] = acc;
            }
        }
    } else if (dtype == ORC_Q5_K) {
        for (int64_t b = 0; b < K / 256; ++b) {
            const uint8_t *wb = wrow + 176 * b;
            const int8_t *q = (const int8_t *)(xrow + 292 * b + 4);
            for (int j = 0; j < 8; ++j) {
                int32_t acc = 0;
                for (int i = 32 * j; i < 32 * j + 32; ++i) acc += q5k_code(wb, i) * q[i];
                out[8 * b + j] = acc;
            }
        }
    } else if (dtype == ORC_Q6_K) {
        for (int64_t b = 0; b < K / 256; ++b) {
            const uint8_t *wb = wrow + 210 * b;
            const int8_t *q = (const int8_t *)(xrow + 292 * b + 4);
            for (int j = 0; j < 16; ++j) {
                int32_t acc = 0;
                for (int i = 16 * j; i < 16 * j + 16; ++i) acc += (q6k_code(wb, i) - 32) * q[i];
                out[16 * b + j] = acc;
            }
        }
    } else if (dtype == ORC_Q8_0) {
        for (int64_t b = 0; b < K / 32; ++b) {
            const int8_t *w = (const int8_t *)(wrow + 34 * b + 2);
            const int8_t *q = (const int8_t *)(xrow + 36 * b + 4);
            int32_t acc = 0;
            for (int i = 0; i < 32; ++i) acc += w[i] * q[i];
            out[b] = acc;
        }
    }
}

/* The integer sums of one scale block, built from the partial dots and the block's integer scales:
 *   Q4_K, Q5_K (per 256): sumi = sum_j sc_j*P_j,  summ = sum_j m_j*(bs_2j + bs_2j+1)  (j < 8)
 *   Q6_K (per 256):       sumi = sum_j sc_j*P_j (j < 16),  summ = 0
 *   Q8_0 (per 32):        sumi = P_b,  summ = 0
 * wb / xb point at the weight and activation block.  These are the integers the keep-quant formula
 * scales: y = sum over blocks of d_a*(d_w*sumi - dmin*summ) (vllm.cpp PR #2890, keep-quant
 * provider commit: integer dots in the CPU accumulation order). */
static void block_sums(int dtype, const uint8_t *wb, const uint8_t *xb, int64_t *sumi, int64_t *summ) {
    *sumi = 0;
    *summ = 0;
    if (dtype == ORC_Q4_K || dtype == ORC_Q5_K) {
        int32_t P[8];
        orc_partials_row(dtype, wb, xb, 256, P);
        for (int j = 0; j < 8; ++j) {
            int sc, mn;
            q4k_scale_min(wb + 4, j, &sc, &mn);
            *sumi += (int64_t)sc * P[j];
            *summ += (int64_t)mn * (rd_i16(xb + 260 + 4 * j) + rd_i16(xb + 262 + 4 * j));
        }
    } else if (dtype == ORC_Q6_K) {
        int32_t P[16];
        orc_partials_row(ORC_Q6_K, wb, xb, 256, P);
        const int8_t *sc = (const int8_t *)(wb + 192);
        for (int j = 0; j < 16; ++j) *sumi += (int64_t)sc[j] * P[j];
    } else if (dtype == ORC_Q8_0) {
        int32_t P;
        orc_partials_row(ORC_Q8_0, wb, xb, 32, &P);
        *sumi = P;
    }
}

/* One output y = sum over blocks of the scaled integer dots, in ascending
 * block order, fp32, no fused multiply-add:
 *   Q4_K: acc += (d_a*d_w)*(float)sumi - (d_a*dmin)*(float)summ,
 *         sumi = sum_j sc_j*P_j, summ = sum_j m_j*(bs_2j + bs_2j+1)
 *   Q6_K: acc += (d_a*d_w)*(float)sumi,  sumi = sum_j sc_j*P_j
 *   Q8_0: acc += (d_w*d_a)*(float)P_b
 * absterms (may be NULL) receives, in f64, the sum over blocks of |(d_a*d_w)*sumi| + |(d_a*dmin)*summ|:
 * the scale of the rounding errors of any order of these fp32 operations.
 * Parity pinned: f64 dequant band, integer-matmul special cases, zero input,
 * independent brute force on tiny inputs. */
static float dot_row(int dtype, const uint8_t *wrow, const uint8_t *xrow, int64_t K, double *absterms) {
    float acc = 0.0f;
    double mag = 0.0;
    if (dtype == ORC_Q4_K || dtype == ORC_Q5_K) {
        /* Q5_K: the Q4_K formula over 5-bit codes (same header: d, dmin, packed scales and mins) */
        const int64_t bb = dtype == ORC_Q4_K ? 144 : 176;
        for (int64_t b = 0; b < K / 256; ++b) {
            const uint8_t *wb = wrow + bb * b;
            const uint8_t *xb = xrow + 292 * b;
            int64_t sumi, summ;
            block_sums(dtype, wb, xb, &sumi, &summ);
            float da = rd_f32(xb);
            float dw = orc_half_to_float((uint16_t)(wb[0] | (wb[1] << 8)));
            float dmin = orc_half_to_float((uint16_t)(wb[2] | (wb[3] << 8)));
            float t1 = da * dw;
            float t2 = t1 * (float)(int32_t)sumi;
            float t3 = da * dmin;
            float t4 = t3 * (float)(int32_t)summ;
            float t5 = t2 - t4;
            acc = acc + t5;
            mag += fabs((double)t2) + fabs((double)t4);
        }
    } else if (dtype == ORC_Q6_K) {
        for (int64_t b = 0; b < K / 256; ++b) {
            const uint8_t *wb = wrow + 210 * b;
            const uint8_t *xb = xrow + 292 * b;
            int64_t sumi, summ;
            block_sums(ORC_Q6_K, wb, xb, &sumi, &summ);
            float da = rd_f32(xb);
            float dw = orc_half_to_float((uint16_t)(wb[208] | (wb[209] << 8)));
            float t1 = da * dw;
            float t2 = t1 * (float)(int32_t)sumi;
            acc = acc + t2;
            mag += fabs((double)t2);
        }
    } else if (dtype == ORC_Q8_0) {
        for (int64_t b = 0; b < K / 32; ++b) {
            const uint8_t *wb = wrow + 34 * b;
            const uint8_t *xb = xrow + 36 * b;
            int64_t P, unused;
            block_sums(ORC_Q8_0, wb, xb, &P, &unused);
            float dw = orc_half_to_float((uint16_t)(wb[0] | (wb[1] << 8)));
            float da = orc_half_to_float((uint16_t)(xb[0] | (xb[1] << 8)));
            float t1 = dw * da;
            float t2 = t1 * (float)(int32_t)P;
            acc = acc + t2;
            mag += fabs((double)t2);
        }
    }
    if (absterms) *absterms = mag;
    return acc;
}

ORC_API float orc_dot_row(int dtype, const uint8_t *wrow, const uint8_t *xrow, int64_t K) {
    return dot_row(dtype, wrow, xrow, K, NULL);
}

static int64_t act_row_bytes(int wdtype, int64_t K) {
    return wdtype == ORC_Q8_0 ? (K / 32) * 36 : (K / 256) * 292;
}
static int64_t w_row_bytes(int wdtype, int64_t K) {
    return (K / orc_block_elems(wdtype)) * orc_block_bytes(wdtype);
}

/* Dense GEMM: y[m, n] = orc_dot_row(W row n, X row m); rows are independent,
 * so the threads only split the (m, n) loop, never a sum. */
ORC_API void orc_gemm(int dtype, const uint8_t *w, const uint8_t *xq, int64_t M, int64_t N, int64_t K,
                      float *y, int64_t ldy, int nthreads) {
    int64_t wrb = w_row_bytes(dtype, K), xrb = act_row_bytes(dtype, K);
    int64_t total = M * N;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads > 0 ? nthreads : 1)
#endif
    for (int64_t t = 0; t < total; ++t) {
        int64_t m = t / N, n = t % N;
        y[m * ldy + n] = orc_dot_row(dtype, w + n * wrb, xq + m * xrb, K);
    }
    (void)nthreads;
}

/* Sampled outputs y[m_idx[s], n_idx[s]] for large shapes. */
ORC_API void orc_gemm_sampled(int dtype, const uint8_t *w, const uint8_t *xq, int64_t K, int64_t S,
                              const int64_t *m_idx, const int64_t *n_idx, float *out) {
    int64_t wrb = w_row_bytes(dtype, K), xrb = act_row_bytes(dtype, K);
    for (int64_t s = 0; s < S; ++s) out[s] = orc_dot_row(dtype, w + n_idx[s] * wrb, xq + m_idx[s] * xrb, K);
}

/* Sampled outputs together with their error scale (dot_row's absterms), for elementwise bounds. */
ORC_API void orc_gemm_sampled_terms(int dtype, const uint8_t *w, const uint8_t *xq, int64_t K, int64_t S,
                                    const int64_t *m_idx, const int64_t *n_idx, float *out, double *absterms) {
    int64_t wrb = w_row_bytes(dtype, K), xrb = act_row_bytes(dtype, K);
    for (int64_t s = 0; s < S; ++s)
        out[s] = dot_row(dtype, w + n_idx[s] * wrb, xq + m_idx[s] * xrb, K, absterms + s);
}

/* The integer sums (block_sums) of every scale block of a whole GEMM: out[m][n][nblk][2] holds
 * (sumi, summ) as int64, nblk = K/256 (Q4_K, Q5_K, Q6_K) or K/32 (Q8_0).  Rows are independent. */
ORC_API void orc_block_sums(int dtype, const uint8_t *w, const uint8_t *xq, int64_t M, int64_t N, int64_t K,
                            int64_t *out, int nthreads) {
    int64_t wrb = w_row_bytes(dtype, K), xrb = act_row_bytes(dtype, K);
    int64_t be = orc_block_elems(dtype), bb = orc_block_bytes(dtype);
    int64_t ab = dtype == ORC_Q8_0 ? 36 : 292;
    int64_t nblk = K / be;
    int64_t total = M * N;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads > 0 ? nthreads : 1)
#endif
    for (int64_t t = 0; t < total; ++t) {
        int64_t m = t / N, n = t % N;
        for (int64_t b = 0; b < nblk; ++b) {
            int64_t *o = out + (t * nblk + b) * 2;
            block_sums(dtype, w + n * wrb + b * bb, xq + m * xrb + b * ab, o, o + 1);
        }
    }
    (void)nthreads;
}

/* Magnitudes of the two parts of a dequantised weight: |d*sc*c| and |dmin*m| (Q4_K, Q5_K), |x| and 0
 * (Q6_K, Q8_0), for the 256 (Q8_0: 32) elements of one block. */
static void weight_parts(int dtype, const uint8_t *blk, double *t1, double *t2) {
    if (dtype == ORC_Q4_K || dtype == ORC_Q5_K) {
        double d = orc_half_to_float((uint16_t)(blk[0] | (blk[1] << 8)));
        double dmin = orc_half_to_float((uint16_t)(blk[2] | (blk[3] << 8)));
        for (int i = 0; i < 256; ++i) {
            int sc, mn;
            q4k_scale_min(blk + 4, i / 32, &sc, &mn);
            int c = dtype == ORC_Q4_K ? q4k_code(blk + 16, i) : q5k_code(blk, i);
            t1[i] = fabs(d * sc * c);
            t2[i] = fabs(dmin * mn);
        }
    } else {
        int n = dtype == ORC_Q8_0 ? 32 : 256;
        if (dtype == ORC_Q6_K) orc_dequant_q6_k(blk, t1);
        else orc_dequant_q8_0(blk, t1);
        for (int i = 0; i < n; ++i) {
            t1[i] = fabs(t1[i]);
            t2[i] = 0.0;
        }
    }
}

/* Magnitudes of a sampled dot product, from the dequantised values a_i (weight row n) and b_i
 * (activation row m), in f64: out[4s] = sum |a_i*b_i|, out[4s+1] = sum |a_i|, out[4s+2] = sum |b_i|,
 * out[4s+3] = sum (|d*sc*c_i| + |dmin*m_i|)*|b_i| (the weight's two parts apart; equal to the first
 * sum for Q6_K and Q8_0).  The scale of the rounding error of any computation that rounds the
 * operands, or the parts of a weight, themselves. */
ORC_API void orc_absdot_sampled(int dtype, const uint8_t *w, const uint8_t *xq, int64_t K, int64_t S,
                                const int64_t *m_idx, const int64_t *n_idx, double *out) {
    int64_t wrb = w_row_bytes(dtype, K), xrb = act_row_bytes(dtype, K);
    int64_t we = orc_block_elems(dtype), wb = orc_block_bytes(dtype);
    int adt = dtype == ORC_Q8_0 ? ORC_Q8_1 : ORC_Q8_K;
    int64_t ae = orc_block_elems(adt), ab = orc_block_bytes(adt);
    double wv[256], av[256], p1[256], p2[256];
    for (int64_t s = 0; s < S; ++s) {
        const uint8_t *wr = w + n_idx[s] * wrb, *xr = xq + m_idx[s] * xrb;
        double sab = 0.0, sa = 0.0, sb = 0.0, sm = 0.0;
        for (int64_t k0 = 0; k0 < K; k0 += 256) {
            for (int64_t k = k0; k < k0 + 256; k += we) {
                const uint8_t *blk = wr + (k / we) * wb;
                switch (dtype) {
                case ORC_Q4_K: orc_dequant_q4_k(blk, wv + (k - k0)); break;
                case ORC_Q5_K: orc_dequant_q5_k(blk, wv + (k - k0)); break;
                case ORC_Q6_K: orc_dequant_q6_k(blk, wv + (k - k0)); break;
                default: orc_dequant_q8_0(blk, wv + (k - k0)); break;
                }
                weight_parts(dtype, blk, p1 + (k - k0), p2 + (k - k0));
            }
            for (int64_t k = k0; k < k0 + 256; k += ae) {
                const uint8_t *blk = xr + (k / ae) * ab;
                if (adt == ORC_Q8_1) orc_dequant_q8_1(blk, av + (k - k0));
                else orc_dequant_q8_k(blk, av + (k - k0));
            }
            for (int i = 0; i < 256; ++i) {
                sab += fabs(wv[i] * av[i]);
                sa += fabs(wv[i]);
                sb += fabs(av[i]);
                sm += (p1[i] + p2[i]) * fabs(av[i]);
            }
        }
        out[4 * s] = sab;
        out[4 * s + 1] = sa;
        out[4 * s + 2] = sb;
        out[4 * s + 3] = sm;
    }
}

/* Partials for a whole GEMM: out[m][n][K/subblock]. */
ORC_API void orc_partials(int dtype, const uint8_t *w, const uint8_t *xq, int64_t M, int64_t N, int64_t K,
                          int32_t *out) {
    int64_t wrb = w_row_bytes(dtype, K), xrb = act_row_bytes(dtype, K);
    int64_t per = dtype == ORC_Q6_K ? K / 16 : K / 32;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) orc_partials_row(dtype, w + n * wrb, xq + m * xrb, K, out + (m * N + n) * per);
}

/* Routed-expert GEMM (MUL_MAT_ID): for token t and slot k,
 *   y[t][k][:] = W_{ids[t][k]} . X_r   with r = t (broadcast, one activation
 *   row per token) or r = t*top_k + k (per-row, one activation row per slot).
 * w holds n_experts consecutive [N][K] weight matrices. Ids outside
 * [0, n_experts) leave the slot's outputs untouched and are counted. */
ORC_API int64_t orc_gemm_grouped(int dtype, const uint8_t *w, int64_t n_experts, const uint8_t *xq,
                                 int64_t xq_rows_per_token, const int32_t *ids, int64_t M, int64_t top_k,
                                 int64_t N, int64_t K, float *y, int nthreads) {
    int64_t wrb = w_row_bytes(dtype, K), xrb = act_row_bytes(dtype, K);
    int64_t bad = 0;
    for (int64_t p = 0; p < M * top_k; ++p)
        if (ids[p] < 0 || ids[p] >= n_experts) bad++;
    int64_t total = M * top_k * N;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads > 0 ? nthreads : 1)
#endif
    for (int64_t t3 = 0; t3 < total; ++t3) {
        int64_t p = t3 / N, n = t3 % N;
        int64_t t = p / top_k;
        int32_t e = ids[p];
        if (e < 0 || e >= n_experts) continue;
        int64_t r = xq_rows_per_token == 1 ? t : p;
        y[p * N + n] = orc_dot_row(dtype, w + ((int64_t)e * N + n) * wrb, xq + r * xrb, K);
    }
    (void)nthreads;
    return bad;
}

/* Weighted expert sum: out[t][n] = w[t][0]*y[t][0][n] + w[t][1]*y[t][1][n] + ...
 * in slot order, each product rounded before its add (no fused multiply-add). */
ORC_API void orc_moe_weighted_sum(const float *y_slots, const float *wts, int64_t M, int64_t top_k, int64_t N,
                                  float *out) {
    for (int64_t t = 0; t < M; ++t)
        for (int64_t n = 0; n < N; ++n) {
            float acc = wts[t * top_k] * y_slots[(t * top_k) * N + n];
            for (int64_t k = 1; k < top_k; ++k) {
                float prod = wts[t * top_k + k] * y_slots[(t * top_k + k) * N + n];
                acc = acc + prod;
            }
            out[t * N + n] = acc;
        }
}

ORC_API int orc_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
