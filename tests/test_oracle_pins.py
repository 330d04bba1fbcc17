"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks the oracle against something it cannot agree with by
construction: hand-derived fixtures, exact rational arithmetic, closed forms,
numpy/IEEE conversions, exact integer matmuls, or the rounding bounds of the
quantizers.  A plausible mistake (a dropped term, a wrong sign, a swapped
nibble, a wrong tie-break) fails at least one of them.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from gemv_quantize_q8_gb300 import synth
from tests.blockpack import pack_q4_k, pack_q5_k, pack_q6_k, pack_q8_0, parse_fixture

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------- f16


def test_half_to_float_matches_ieee_all_codes():
    h = np.arange(65536, dtype=np.uint16)
    ref = h.view(np.float16).astype(np.float32)
    got = np.array([oracle.half_to_float(int(v)) for v in h], dtype=np.float32)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_float_to_half_round_to_nearest_even():
    g = np.random.default_rng(3)
    finite = np.arange(65536, dtype=np.uint16).view(np.float16)
    finite = finite[np.isfinite(finite)].astype(np.float64)
    finite = np.unique(finite)
    mids = (finite[:-1] + finite[1:]) / 2                     # exact midpoints (f64)
    mids = mids[np.abs(mids) < 3e38]
    mids32 = mids.astype(np.float32)
    mids32 = mids32[mids32.astype(np.float64) == mids]        # keep those exact in fp32
    rnd = (g.standard_normal(20000) * 10.0 ** g.integers(-9, 6, 20000)).astype(np.float32)
    big = np.array([65504, 65519, 65520, 65536, 1e9, -65520, 6e-8, 3e-8, 2.9802322e-08, 1e-10], dtype=np.float32)
    xs = np.concatenate([rnd, mids32, big])
    ref = xs.astype(np.float16).view(np.uint16)
    got = np.array([oracle.float_to_half(float(v)) for v in xs], dtype=np.uint16)
    assert (got == ref).all()


# --------------------------------------------------------------------------- layouts


@pytest.mark.parametrize("fname,dtype,nbytes,nelem", [("q4_k_blocks.txt", oracle.Q4_K, 144, 256),
                                                      ("q5_k_blocks.txt", oracle.Q5_K, 176, 256),
                                                      ("q6_k_blocks.txt", oracle.Q6_K, 210, 256),
                                                      ("q8_0_blocks.txt", oracle.Q8_0, 34, 32)])
def test_hand_derived_blocks(fname, dtype, nbytes, nelem):
    cases = list(parse_fixture(os.path.join(GOLDEN, fname), nbytes))
    assert cases
    for name, blk, exp in cases:
        x = oracle.dequant(dtype, blk)
        want = np.zeros(nelem)
        for i, v in exp.items():
            want[i] = v
        assert np.array_equal(x, want), name


def test_q4_k_every_element_position():
    """A single nonzero code at element i must dequantise at i and nowhere else."""
    for i in range(256):
        codes = [0] * 256
        codes[i] = 1 + (i % 15)
        sc = [j + 1 for j in range(8)]
        blk = pack_q4_k(1.0, 0.0, sc, [0] * 8, codes)
        x = oracle.dequant(oracle.Q4_K, blk)
        want = np.zeros(256)
        want[i] = sc[i // 32] * codes[i]
        assert np.array_equal(x, want), i


def test_q4_k_scale_min_fields():
    g = np.random.default_rng(5)
    for _ in range(50):
        sc = g.integers(0, 64, 8)
        mn = g.integers(0, 64, 8)
        codes = g.integers(0, 16, 256)
        d, dmin = 0.5, 0.25
        blk = pack_q4_k(d, dmin, sc, mn, codes)
        x = oracle.dequant(oracle.Q4_K, blk)
        want = np.array([d * sc[i // 32] * codes[i] - dmin * mn[i // 32] for i in range(256)])
        assert np.array_equal(x, want)


def test_q5_k_every_element_position_and_high_bit():
    """A single nonzero 5-bit code at element i dequantises at i only; codes >= 16 exercise the high
    bit's byte and bit position (byte i % 32, bit 2*(i // 64) + (i % 64 >= 32))."""
    for i in range(256):
        codes = [0] * 256
        codes[i] = 16 + (i % 16) if i % 2 else 1 + (i % 15)
        sc = [j + 1 for j in range(8)]
        blk = pack_q5_k(1.0, 0.0, sc, [0] * 8, codes)
        x = oracle.dequant(oracle.Q5_K, blk)
        want = np.zeros(256)
        want[i] = sc[i // 32] * codes[i]
        assert np.array_equal(x, want), i


def test_q5_k_all_codes_and_fields():
    g = np.random.default_rng(6)
    for _ in range(40):
        sc = g.integers(0, 64, 8)
        mn = g.integers(0, 64, 8)
        codes = g.integers(0, 32, 256)
        blk = pack_q5_k(0.5, 0.25, sc, mn, codes)
        x = oracle.dequant(oracle.Q5_K, blk)
        want = np.array([0.5 * sc[i // 32] * codes[i] - 0.25 * mn[i // 32] for i in range(256)])
        assert np.array_equal(x, want)


def test_q5_k_unit_scales_is_integer_matmul():
    g = np.random.default_rng(11)
    M, N, K = 3, 4, 512
    codes = g.integers(0, 32, size=(N, K))
    wb = np.concatenate([np.concatenate([pack_q5_k(1.0, 0.0, [1] * 8, [0] * 8, codes[n, 256 * b:256 * b + 256])
                                         for b in range(K // 256)]) for n in range(N)])
    x = _integer_acts(M, K, g)
    y = oracle.gemm(oracle.Q5_K, wb, oracle.quantize_q8_k(x), M, N, K)
    assert np.array_equal(y.astype(np.int64), x.astype(np.int64) @ codes.T)


def test_q5_k_min_term_sign():
    """d = 0, dmin = 1, every min 1: y = -sum(q) over the row."""
    g = np.random.default_rng(12)
    M, N, K = 2, 3, 256
    wb = np.concatenate([pack_q5_k(0.0, 1.0, [5] * 8, [1] * 8, g.integers(0, 32, 256)) for _ in range(N)])
    x = _integer_acts(M, K, g)
    y = oracle.gemm(oracle.Q5_K, wb, oracle.quantize_q8_k(x), M, N, K)
    assert np.array_equal(y, np.repeat(-x.sum(axis=1, keepdims=True), N, axis=1).astype(np.float32))


def test_q6_k_every_element_position():
    for i in range(256):
        codes = [32] * 256                 # 32 is the zero of the offset code
        codes[i] = 32 + 1 + (i % 31)
        sc = [(-1) ** j * (j + 1) for j in range(16)]
        blk = pack_q6_k(1.0, sc, codes)
        x = oracle.dequant(oracle.Q6_K, blk)
        want = np.zeros(256)
        want[i] = sc[i // 16] * (codes[i] - 32)
        assert np.array_equal(x, want), i


def test_q6_k_all_codes_roundtrip():
    g = np.random.default_rng(6)
    codes = g.permutation(np.tile(np.arange(64), 4))
    sc = g.integers(-128, 128, 16)
    blk = pack_q6_k(2.0, sc, codes)
    x = oracle.dequant(oracle.Q6_K, blk)
    want = np.array([2.0 * sc[i // 16] * (codes[i] - 32) for i in range(256)])
    assert np.array_equal(x, want)


# --------------------------------------------------------------------------- Q8_K quantizer


def _q8k_fields(blk):
    d = np.frombuffer(blk[0:4].tobytes(), dtype=np.float32)[0]
    q = blk[4:260].view(np.int8).astype(np.int64)
    bs = np.frombuffer(blk[260:292].tobytes(), dtype=np.int16).astype(np.int64)
    return d, q, bs


def test_q8_k_spike():
    x = np.zeros((1, 256), dtype=np.float32)
    x[0, 37] = 3.5
    d, q, bs = _q8k_fields(oracle.quantize_q8_k(x)[0])
    want = np.zeros(256, dtype=np.int64)
    want[37] = -127                               # the max element maps to -127 (iscale = -127/mx)
    assert np.array_equal(q, want)
    assert d < 0 and abs(d * -127 - 3.5) <= 4 * np.spacing(np.float32(3.5))
    assert bs[2] == -127 and np.count_nonzero(bs) == 1


def test_q8_k_negative_spike_and_sign_of_d():
    x = np.zeros((1, 256), dtype=np.float32)
    x[0, 200] = -2.0
    d, q, _ = _q8k_fields(oracle.quantize_q8_k(x)[0])
    assert q[200] == -127 and d == np.float32(1.0) / np.float32(63.5)


def test_q8_k_first_occurrence_tie():
    x = np.zeros((1, 256), dtype=np.float32)
    x[0, 5], x[0, 9] = -1.5, 1.5
    d, q, _ = _q8k_fields(oracle.quantize_q8_k(x)[0])
    assert q[5] == -127 and q[9] == 127 and d > 0


def test_q8_k_zero_block():
    out = oracle.quantize_q8_k(np.zeros((2, 512), dtype=np.float32))
    assert not out.any()


def test_q8_k_ramp_exact_rational():
    """x_i = i - 128: mx = -128, iscale = 127/128 exactly; codes are the
    round-half-even of the exact rationals k*127/128 (k = -128..127)."""
    k = np.arange(256) - 128
    x = k.astype(np.float32)[None, :]
    d, q, bs = _q8k_fields(oracle.quantize_q8_k(x)[0])
    want = []
    for kk in k:
        v = Fraction(int(kk) * 127, 128)
        fl = math.floor(v)
        r = v - fl
        want.append(fl + (1 if (r > Fraction(1, 2) or (r == Fraction(1, 2) and fl % 2 == 1)) else 0))
    assert np.array_equal(q, np.array(want))
    assert q[128 + 64] == 64 and q[128 - 64] == -64    # the two exact half-way ties went to even
    assert np.array_equal(bs, np.array(want).reshape(16, 16).sum(1))
    assert d == np.float32(1.0) / np.float32(np.float32(127.0) / np.float32(128.0))


def test_q8_k_rounding_bound_and_bsums():
    g = np.random.default_rng(7)
    x = synth.activations(16, 1024, g, outliers=True)
    out = oracle.quantize_q8_k(x).reshape(16, 4, 292)
    for m in range(16):
        for b in range(4):
            d, q, bs = _q8k_fields(out[m, b])
            xb = x[m, 256 * b:256 * b + 256].astype(np.float64)
            assert np.all(np.abs(q) <= 127)
            err = np.abs(xb - float(d) * q)
            assert err.max() <= abs(float(d)) * 0.5 * (1 + 1e-5)
            assert np.array_equal(bs, q.reshape(16, 16).sum(1))
            i = int(np.argmax(np.abs(xb)))             # first occurrence of the max
            assert q[i] == -127


def test_q8_k_nan_is_ignored_in_amax_and_coded_zero():
    x = np.linspace(-1, 1, 256, dtype=np.float32)[None, :].copy()
    x[0, 10] = np.nan
    d, q, _ = _q8k_fields(oracle.quantize_q8_k(x)[0])
    assert q[10] == 0 and np.isfinite(d) and q[0] == -127


# --------------------------------------------------------------------------- Q8_1 quantizer


def test_q8_1_bounds_zero_block_and_sum():
    g = np.random.default_rng(8)
    x = synth.activations(8, 256, g, outliers=True)
    x[3, 32:64] = 0.0
    out = oracle.quantize_q8_1(x).reshape(8, 8, 36)
    for m in range(8):
        for b in range(8):
            blk = out[m, b]
            xb = x[m, 32 * b:32 * b + 32]
            d16 = blk[0:2].view(np.float16)[0]
            s16 = blk[2:4].view(np.float16)[0]
            q = blk[4:36].view(np.int8).astype(np.int64)
            amax = np.float32(np.abs(xb).max())
            dfull = np.float32(amax / np.float32(127.0))
            assert d16 == np.float16(dfull)
            if amax == 0:
                assert not q.any() and float(s16) == 0.0
                continue
            err = np.abs(xb.astype(np.float64) - float(dfull) * q)
            assert err.max() <= float(dfull) * 0.5 * (1 + 1e-5)
            exact = math.fsum(float(v) for v in xb)
            bound = 5 * 2.0 ** -24 * float(np.abs(xb).sum()) + abs(exact) * 2.0 ** -11 + 2.0 ** -24
            assert abs(float(s16) - exact) <= bound + abs(float(s16)) * 2.0 ** -11


def test_q8_1_block_sum_follows_the_butterfly_order():
    """Pins the order of the Q8_1 block sum s without restating it.  x_i = B*sign_i + r_i with the sign
    taken from one index bit and B = 2**(21 - k): in the xor-butterfly order (strides 16, 8, 4, 2, 1)
    the slots paired before stage k share a sign, so their large parts stay at or below 2**21 (every
    partial sum exact), and stage k cancels them exactly; s is then exactly the sum of the small parts
    r_i (multiples of 1/4), known in closed form.  An order that pairs one more same-sign bit first has
    to hold 2**22 and loses the quarter bits: the butterfly with stages k and k+1 swapped misses the
    exact value, checked below so the pin can fail.  The GPU quantizer is compared with the oracle byte
    for byte, so this pins its order too."""
    g = np.random.default_rng(81)
    strides = [16, 8, 4, 2, 1]

    def xor_tree(x, order):  # a differently ordered tree, only to show the construction separates orders
        p = x.astype(np.float32)
        for st in order:
            p = (p + p[np.arange(32) ^ st]).astype(np.float32)
        return float(p[0])

    wrong = [0] * 4
    for k, st in enumerate(strides):                  # stage k of the butterfly pairs indices i, i ^ st
        B = 2.0 ** (21 - k)
        sign = np.array([-1.0 if i & st else 1.0 for i in range(32)])
        for _ in range(16):
            r = g.integers(-8, 9, 32) * 0.25
            x64 = B * sign + r
            x = x64.astype(np.float32)
            assert np.array_equal(x.astype(np.float64), x64)        # every input exactly representable
            s16 = oracle.quantize_q8_1(x[None, :])[0][2:4].view(np.float16)[0]
            assert float(s16) == r.sum(), (k, float(s16), r.sum())  # exact: large parts cancel at stage k
            if k < 4:
                swapped = strides[:k] + [strides[k + 1], strides[k]] + strides[k + 2:]
                wrong[k] += xor_tree(x, swapped) != r.sum()
    assert all(w > 0 for w in wrong), wrong


def test_q8_1_roundf_half_away():
    # amax = 127 -> d = 1 exactly; x = 2.5 -> roundf gives 3 (half away from zero), -0.5 -> -1
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, 0], x[0, 1], x[0, 2] = 127.0, 2.5, -0.5
    blk = oracle.quantize_q8_1(x)[0]
    q = blk[4:36].view(np.int8)
    assert q[0] == 127 and q[1] == 3 and q[2] == -1


# --------------------------------------------------------------------------- block dots


def _integer_acts(M, K, g):
    """Integer activations in [-127, 127] whose first max per 256 block is -127
    (so Q8_K has iscale = 1, q = x, d = 1) -- also amax = 127 per 32 (Q8_1 d = 1)."""
    x = g.integers(-126, 127, size=(M, K)).astype(np.float32)
    x[:, ::32] = -127.0
    return x


def test_q8_0_unit_scales_is_integer_matmul():
    g = np.random.default_rng(9)
    M, N, K = 3, 5, 128
    w = g.integers(-127, 128, size=(N, K))
    wb = np.concatenate([np.concatenate([pack_q8_0(1.0, w[n, 32 * b:32 * b + 32]) for b in range(K // 32)])
                         for n in range(N)])
    x = _integer_acts(M, K, g)
    xq = oracle.quantize_q8_1(x)
    assert np.array_equal(xq.reshape(M, -1, 36)[:, :, 4:].view(np.int8).reshape(M, K), x.astype(np.int8))
    y = oracle.gemm(oracle.Q8_0, wb, xq, M, N, K)
    assert np.array_equal(y.astype(np.int64), x.astype(np.int64) @ w.T)


def test_q4_k_unit_scales_is_integer_matmul():
    g = np.random.default_rng(10)
    M, N, K = 3, 4, 512
    codes = g.integers(0, 16, size=(N, K))
    wb = np.concatenate([np.concatenate([pack_q4_k(1.0, 0.0, [1] * 8, [0] * 8, codes[n, 256 * b:256 * b + 256])
                                         for b in range(K // 256)]) for n in range(N)])
    x = _integer_acts(M, K, g)
    xq = oracle.quantize_q8_k(x)
    y = oracle.gemm(oracle.Q4_K, wb, xq, M, N, K)
    assert np.array_equal(y.astype(np.int64), x.astype(np.int64) @ codes.T)


def test_q4_k_min_term_sign_and_bsums():
    """d = 0, dmin = 1, m_j = 1: y = -sum(q), which exercises bsums and the minus sign."""
    g = np.random.default_rng(11)
    M, N, K = 2, 3, 256
    wb = np.concatenate([pack_q4_k(0.0, 1.0, [5] * 8, [1] * 8, g.integers(0, 16, 256)) for _ in range(N)])
    x = _integer_acts(M, K, g)
    y = oracle.gemm(oracle.Q4_K, wb, oracle.quantize_q8_k(x), M, N, K)
    want = -x.astype(np.int64).sum(1)
    assert np.array_equal(y.astype(np.int64), np.repeat(want[:, None], N, 1))


def test_q6_k_unit_scales_is_integer_matmul():
    g = np.random.default_rng(12)
    M, N, K = 3, 4, 512
    codes = g.integers(0, 64, size=(N, K))
    wb = np.concatenate([np.concatenate([pack_q6_k(1.0, [1] * 16, codes[n, 256 * b:256 * b + 256])
                                         for b in range(K // 256)]) for n in range(N)])
    x = _integer_acts(M, K, g)
    y = oracle.gemm(oracle.Q6_K, wb, oracle.quantize_q8_k(x), M, N, K)
    assert np.array_equal(y.astype(np.int64), x.astype(np.int64) @ (codes - 32).T)


@pytest.mark.parametrize("dtype", [oracle.Q4_K, oracle.Q6_K, oracle.Q8_0])
def test_partials_identity_against_f64_dequant(dtype):
    """sum_i deq_w(i) * deq_a(i) in f64 equals the scaled-integer identity built
    from the oracle's int32 partials, to 1e-12 relative."""
    g = np.random.default_rng(13 + dtype)
    M, N, K = 2, 3, 512
    w = synth.weights(dtype, N, K, g)
    x = synth.activations(M, K, g, outliers=True)
    xq = oracle.quantize_q8_1(x) if dtype == oracle.Q8_0 else oracle.quantize_q8_k(x)
    P = oracle.partials(dtype, w, xq, M, N, K)
    ad = oracle.ACT_DTYPE[dtype]
    wd = oracle.dequant(dtype, w).reshape(N, K)
    xd = oracle.dequant(ad, xq).reshape(M, K)
    for m in range(M):
        for n in range(N):
            ref = float(np.dot(wd[n], xd[m]))
            tot = 0.0
            if dtype == oracle.Q8_0:
                for b in range(K // 32):
                    dw = float(w[n, 34 * b:34 * b + 2].view(np.float16)[0])
                    da = float(xq[m, 36 * b:36 * b + 2].view(np.float16)[0])
                    tot += dw * da * P[m, n, b]
            else:
                bb = 144 if dtype == oracle.Q4_K else 210
                for b in range(K // 256):
                    blk = w[n, bb * b:bb * b + bb]
                    xb = xq[m, 292 * b:292 * b + 292]
                    da = float(np.frombuffer(xb[0:4].tobytes(), np.float32)[0])
                    bs = np.frombuffer(xb[260:292].tobytes(), np.int16).astype(np.int64)
                    if dtype == oracle.Q4_K:
                        s = blk[4:16].astype(np.int64)
                        sc = [s[j] & 63 if j < 4 else (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4) for j in range(8)]
                        mn = [s[j + 4] & 63 if j < 4 else (s[j + 4] >> 4) | ((s[j] >> 6) << 4) for j in range(8)]
                        dw = float(blk[0:2].view(np.float16)[0])
                        dmin = float(blk[2:4].view(np.float16)[0])
                        sumi = sum(sc[j] * int(P[m, n, 8 * b + j]) for j in range(8))
                        summ = sum(mn[j] * int(bs[2 * j] + bs[2 * j + 1]) for j in range(8))
                        tot += da * (dw * sumi - dmin * summ)
                    else:
                        sc = blk[192:208].view(np.int8).astype(np.int64)
                        dw = float(blk[208:210].view(np.float16)[0])
                        tot += da * dw * sum(int(sc[j]) * int(P[m, n, 16 * b + j]) for j in range(16))
            assert abs(tot - ref) <= 1e-12 * max(1.0, abs(ref)), (m, n, tot, ref)


def _brute_force_f64(dtype, w, x_blocks, M, N, K):
    """Independent pure-Python f64 evaluation from the canonical bytes."""
    def unpack_w(row):
        vals = []
        if dtype == oracle.Q8_0:
            for b in range(K // 32):
                blk = row[34 * b:34 * b + 34]
                d = float(blk[0:2].view(np.float16)[0])
                vals += [d * int(v) for v in blk[2:34].view(np.int8)]
            return vals
        bb = {oracle.Q4_K: 144, oracle.Q5_K: 176, oracle.Q6_K: 210}[dtype]
        for b in range(K // 256):
            blk = row[bb * b:bb * b + bb]
            if dtype in (oracle.Q4_K, oracle.Q5_K):
                d = float(blk[0:2].view(np.float16)[0]); dm = float(blk[2:4].view(np.float16)[0])
                s = [int(v) for v in blk[4:16]]
                qs = 16 if dtype == oracle.Q4_K else 48
                for i in range(256):
                    j, c, r = i // 32, i // 64, i % 64
                    sc = s[j] & 63 if j < 4 else (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4)
                    mn = s[j + 4] & 63 if j < 4 else (s[j + 4] >> 4) | ((s[j] >> 6) << 4)
                    byte = int(blk[qs + 32 * c + r % 32])
                    code = byte & 15 if r < 32 else byte >> 4
                    if dtype == oracle.Q5_K:
                        code += 16 * ((int(blk[16 + r % 32]) >> (2 * c + (r >= 32))) & 1)
                    vals.append(d * sc * code - dm * mn)
            else:
                d = float(blk[208:210].view(np.float16)[0])
                for i in range(256):
                    h, r = i // 128, i % 128
                    qtr, l = r // 32, r % 32
                    lo = int(blk[64 * h + l + (32 if qtr & 1 else 0)])
                    lo = lo >> 4 if qtr & 2 else lo & 15
                    hi = (int(blk[128 + 32 * h + l]) >> (2 * qtr)) & 3
                    vals.append(d * int(blk[192:208].view(np.int8)[i // 16]) * ((lo | hi << 4) - 32))
        return vals

    def unpack_x(row):
        vals = []
        if dtype == oracle.Q8_0:
            for b in range(K // 32):
                blk = row[36 * b:36 * b + 36]
                d = float(blk[0:2].view(np.float16)[0])
                vals += [d * int(v) for v in blk[4:36].view(np.int8)]
        else:
            for b in range(K // 256):
                blk = row[292 * b:292 * b + 292]
                d = float(np.frombuffer(blk[0:4].tobytes(), np.float32)[0])
                vals += [d * int(v) for v in blk[4:260].view(np.int8)]
        return vals

    W = [unpack_w(w[n]) for n in range(N)]
    X = [unpack_x(x_blocks[m]) for m in range(M)]
    return np.array([[math.fsum(a * b for a, b in zip(X[m], W[n])) for n in range(N)] for m in range(M)])


@pytest.mark.parametrize("dtype", [oracle.Q4_K, oracle.Q5_K, oracle.Q6_K, oracle.Q8_0])
def test_block_sums_against_brute_force(dtype):
    """The integer sums per scale block (sum_j sc_j*P_j and the min term), scaled in f64 as
    d_a*(d_w*sumi - dmin*summ) and added over blocks, equal the independent pure-Python f64 brute force
    to 1e-12 relative; their error scale (sum of |scaled terms|) bounds |y| from above."""
    g = np.random.default_rng(23 + dtype)
    M, N, K = 2, 3, 512
    w = synth.weights(dtype, N, K, g)
    x = synth.activations(M, K, g, outliers=True)
    xq = oracle.quantize_q8_1(x) if dtype == oracle.Q8_0 else oracle.quantize_q8_k(x)
    S = oracle.block_sums(dtype, w, xq, M, N, K)
    ref = _brute_force_f64(dtype, w, xq, M, N, K)
    for m in range(M):
        for n in range(N):
            tot = 0.0
            if dtype == oracle.Q8_0:
                for b in range(K // 32):
                    dw = float(w[n, 34 * b:34 * b + 2].view(np.float16)[0])
                    da = float(xq[m, 36 * b:36 * b + 2].view(np.float16)[0])
                    assert S[m, n, b, 1] == 0
                    tot += dw * da * int(S[m, n, b, 0])
            else:
                bb = {oracle.Q4_K: 144, oracle.Q5_K: 176, oracle.Q6_K: 210}[dtype]
                for b in range(K // 256):
                    blk = w[n, bb * b:bb * b + bb]
                    da = float(np.frombuffer(xq[m, 292 * b:292 * b + 4].tobytes(), np.float32)[0])
                    if dtype == oracle.Q6_K:
                        dw, dmin = float(blk[208:210].view(np.float16)[0]), 0.0
                        assert S[m, n, b, 1] == 0
                    else:
                        dw, dmin = (float(v) for v in blk[0:4].view(np.float16))
                    tot += da * (dw * int(S[m, n, b, 0]) - dmin * int(S[m, n, b, 1]))
            assert abs(tot - ref[m, n]) <= 1e-12 * max(1.0, abs(ref[m, n])), (m, n, tot, ref[m, n])
    mi, ni = np.repeat(np.arange(M), N), np.tile(np.arange(N), M)
    y, terms = oracle.gemm_sampled_terms(dtype, w, xq, K, mi, ni)
    assert np.array_equal(y, oracle.gemm(dtype, w, xq, M, N, K).reshape(-1))
    assert np.all(terms >= np.abs(ref.reshape(-1)) * (1 - 1e-6))


@pytest.mark.parametrize("dtype", [oracle.Q4_K, oracle.Q5_K, oracle.Q6_K, oracle.Q8_0])
def test_absdot_magnitudes(dtype):
    """The error-scale helper: sum |a_i*b_i|, sum |a_i|, sum |b_i| over the dequantised weight row a and
    activation row b, against numpy on the dequantised blocks (whose values the fixtures pin); and the
    two-part magnitude sum (|d*sc*c_i| + |dmin*m_i|)*|b_i|: equal to the first sum for Q6_K and Q8_0;
    for Q4_K/Q5_K at least the first sum and at most it plus 2*sum |dmin*m_i|*|b_i|, where dmin*m_i is
    read off a copy of the weights with every code 0 (its dequantised values are exactly -dmin*m_i)."""
    g = np.random.default_rng(31 + dtype)
    N, K, M = 3, 512, 2
    w = synth.weights(dtype, N, K, g)
    x = synth.activations(M, K, g, outliers=True)
    xq = oracle.quantize_q8_1(x) if dtype == oracle.Q8_0 else oracle.quantize_q8_k(x)
    a = oracle.dequant(dtype, w).reshape(N, K)
    b = oracle.dequant(oracle.ACT_DTYPE[dtype], xq).reshape(M, K)
    pairs = [(0, 2), (1, 0), (1, 1)]
    r = oracle.absdot_sampled(dtype, w, xq, K, [p[0] for p in pairs], [p[1] for p in pairs])
    for s, (m, n) in enumerate(pairs):
        want = [np.abs(a[n] * b[m]).sum(), np.abs(a[n]).sum(), np.abs(b[m]).sum()]
        assert np.allclose(r[s, :3], want, rtol=1e-12, atol=0)
    if dtype in (oracle.Q6_K, oracle.Q8_0):
        assert np.allclose(r[:, 3], r[:, 0], rtol=1e-12, atol=0)
    else:
        bb = {oracle.Q4_K: 144, oracle.Q5_K: 176}[dtype]
        w0 = w.reshape(N, K // 256, bb).copy()
        w0[:, :, bb - 128:] = 0                  # every 4-bit code 0
        if dtype == oracle.Q5_K:
            w0[:, :, 16:48] = 0                  # and every fifth bit
        mins = -oracle.dequant(dtype, w0.reshape(N, -1)).reshape(N, K)   # dmin*m_i
        assert (mins >= 0).all()
        for s, (m, n) in enumerate(pairs):
            assert r[s, 3] >= r[s, 0] * (1 - 1e-12)
            assert r[s, 3] <= (r[s, 0] + 2 * (mins[n] * np.abs(b[m])).sum()) * (1 + 1e-12)


@pytest.mark.parametrize("dtype", [oracle.Q4_K, oracle.Q5_K, oracle.Q6_K, oracle.Q8_0])
def test_brute_force_tiny(dtype):
    g = np.random.default_rng(20 + dtype)
    M, N, K = 3, 4, 512
    w = synth.weights(dtype, N, K, g)
    x = synth.activations(M, K, g)
    xq = oracle.quantize_q8_1(x) if dtype == oracle.Q8_0 else oracle.quantize_q8_k(x)
    y = oracle.gemm(dtype, w, xq, M, N, K).astype(np.float64)
    ref = _brute_force_f64(dtype, w, xq, M, N, K)
    scale = np.abs(ref).max()
    assert np.abs(y - ref).max() <= 1e-5 * scale


@pytest.mark.parametrize("dtype", [oracle.Q4_K, oracle.Q5_K, oracle.Q6_K, oracle.Q8_0])
def test_f64_band_and_zero_input(dtype):
    g = np.random.default_rng(30 + dtype)
    M, N, K = 8, 64, 1024
    w = synth.weights(dtype, N, K, g)
    x = synth.activations(M, K, g, outliers=True)
    qf = oracle.quantize_q8_1 if dtype == oracle.Q8_0 else oracle.quantize_q8_k
    xq = qf(x)
    y = oracle.gemm(dtype, w, xq, M, N, K).astype(np.float64)
    wd = oracle.dequant(dtype, w).reshape(N, K)
    xd = oracle.dequant(oracle.ACT_DTYPE[dtype], xq).reshape(M, K)
    y64 = xd @ wd.T
    rel = np.linalg.norm(y - y64) / np.linalg.norm(y64)
    assert rel <= 5e-4          # the pages' f64 dequant band
    assert rel <= 1e-6          # what exact integer dots + fp32 scaling actually give
    yz = oracle.gemm(dtype, w, qf(np.zeros((M, K), np.float32)), M, N, K)
    assert np.all(yz == 0.0)


# --------------------------------------------------------------------------- grouped + weighted sum


def test_grouped_reduces_to_dense_and_per_row_arm():
    g = np.random.default_rng(40)
    E, M, N, K = 3, 5, 16, 512
    w = synth.weights(oracle.Q4_K, E * N, K, g)
    x = synth.activations(M, K, g)
    xq = oracle.quantize_q8_k(x)
    ids = np.zeros((M, 1), np.int32)
    y, bad = oracle.gemm_grouped(oracle.Q4_K, w, E, xq, 1, ids, M, 1, N, K)
    dense = oracle.gemm(oracle.Q4_K, w[:N], xq, M, N, K)
    assert bad == 0 and np.array_equal(y[:, 0, :], dense)
    # per-row arm: slot (t, k) reads activation row t*top_k + k
    top_k = 2
    ids = np.array([[t % E, (t + 1) % E] for t in range(M)], np.int32)
    xr = synth.activations(M * top_k, K, g)
    xrq = oracle.quantize_q8_k(xr)
    y2, _ = oracle.gemm_grouped(oracle.Q4_K, w, E, xrq, top_k, ids, M, top_k, N, K)
    for t in range(M):
        for k in range(top_k):
            e = ids[t, k]
            ref = oracle.gemm(oracle.Q4_K, w[e * N:(e + 1) * N], xrq[t * top_k + k:t * top_k + k + 1], 1, N, K)
            assert np.array_equal(y2[t, k], ref[0])


def test_grouped_invalid_ids_counted_and_untouched():
    g = np.random.default_rng(41)
    E, M, N, K = 2, 3, 8, 256
    w = synth.weights(oracle.Q6_K, E * N, K, g)
    xq = oracle.quantize_q8_k(synth.activations(M, K, g))
    ids = np.array([[0, 5], [-1, 1], [1, 0]], np.int32)
    y, bad = oracle.gemm_grouped(oracle.Q6_K, w, E, xq, 1, ids, M, 2, N, K)
    assert bad == 2
    assert np.isnan(y[0, 1]).all() and np.isnan(y[1, 0]).all() and np.isfinite(y[2]).all()


def test_weighted_sum_one_hot_and_f64_bound():
    g = np.random.default_rng(42)
    M, top_k, N = 4, 8, 64
    ys = g.standard_normal((M, top_k, N)).astype(np.float32)
    onehot = np.zeros((M, top_k), np.float32)
    onehot[np.arange(M), np.arange(M) % top_k] = 1.0
    out = oracle.moe_weighted_sum(ys, onehot)
    assert np.array_equal(out, ys[np.arange(M), np.arange(M) % top_k])
    _, w = synth.routing(M, 16, top_k, g)
    out = oracle.moe_weighted_sum(ys, w).astype(np.float64)
    ref = np.einsum("tk,tkn->tn", w.astype(np.float64), ys.astype(np.float64))
    bound = 2 * top_k * 2.0 ** -24 * np.einsum("tk,tkn->tn", np.abs(w), np.abs(ys)).astype(np.float64)
    assert np.all(np.abs(out - ref) <= bound)


def test_swiglu_against_f64():
    g = np.random.default_rng(43)
    gg = (g.standard_normal((4, 256)) * 4).astype(np.float32)
    uu = g.standard_normal((4, 256)).astype(np.float32)
    h = oracle.swiglu(gg, uu).astype(np.float64)
    g64, u64 = gg.astype(np.float64), uu.astype(np.float64)
    ref = g64 / (1 + np.exp(-g64)) * u64
    assert np.all(np.abs(h - ref) <= 8 * 2.0 ** -24 * np.abs(ref) + 1e-30)


def test_routing_generator_shapes():
    g = np.random.default_rng(44)
    ids, w = synth.routing(64, 256, 8, g)
    assert ids.shape == (64, 8) and all(len(set(r)) == 8 for r in ids)
    assert np.allclose(w.sum(1), 1.0, atol=1e-6) and (ids >= 0).all() and (ids < 256).all()


def test_input_recipe_is_seeded_and_matches_its_description():
    """The synthetic inputs follow the stated recipe: N(0,1) activations with each element scaled by 10
    with probability 1%, routing draws distinct experts per token uniformly, and a seed fixes every
    byte (weights, activations and routing)."""
    x = synth.activations(512, 1024, np.random.default_rng(0), outliers=True)
    x0 = synth.activations(512, 1024, np.random.default_rng(0))   # the same N(0,1) draws, unscaled
    scaled = x == x0 * np.float32(10.0)
    assert np.all(scaled | (x == x0))                                # each element x1 or x10
    assert 0.008 < float(scaled.mean()) < 0.012                      # with probability 1%
    xn = synth.activations(512, 1024, np.random.default_rng(1))
    assert abs(float(xn.mean())) < 0.01 and abs(float(xn.std()) - 1.0) < 0.01
    ids, _ = synth.routing(2048, 256, 8, np.random.default_rng(2))
    counts = np.bincount(ids.reshape(-1), minlength=256)
    assert counts.sum() == 2048 * 8 and counts.min() > 20 and counts.max() < 120   # mean 64
    for dt in (synth.Q4_K, synth.Q5_K, synth.Q6_K, synth.Q8_0):
        a = synth.weights(dt, 32, 512, synth.rng(7))
        b = synth.weights(dt, 32, 512, synth.rng(7))
        assert np.array_equal(a, b) and a.nbytes == 32 * (512 // oracle.BLOCK_ELEMS[dt]) * oracle.BLOCK_BYTES[dt]
    r1 = synth.routing(16, 64, 4, synth.rng(3))
    r2 = synth.routing(16, 64, 4, synth.rng(3))
    assert np.array_equal(r1[0], r2[0]) and np.array_equal(r1[1], r2[1])


def test_q8_k_half_way_ties_go_to_even():
    """mx = -127 gives iscale = 1 exactly, so x = n + 1/2 is an exact tie:
    the nearest-integer reading is round-half-to-even (2.5 -> 2, 3.5 -> 4)."""
    x = np.zeros((1, 256), dtype=np.float32)
    x[0, 0] = -127.0
    halves = np.arange(-60, 60) + 0.5
    x[0, 1:1 + halves.size] = halves
    d, q, _ = _q8k_fields(oracle.quantize_q8_k(x)[0])
    assert d == 1.0
    want = [math.floor(v) + (math.floor(v) % 2) for v in halves]   # the even neighbour of each tie
    assert list(q[1:1 + halves.size]) == want


# ----------------------------------------------------------------------------- RMSNorm producer


@pytest.mark.parametrize("pos", [(1, 2), (700, 767), (383, 384)])
def test_rmsnorm_sum_of_squares_ascending(pos):
    """Pins the plain ascending sum of squares with a closed form: x[0] = 4096 (square 2^24), two other
    elements 1 at the given positions, the rest 0, K = 768.  Added left to right, 2^24 + 1 is a tie
    that rounds to even (2^24), and so is the second + 1: the total is exactly 2^24.  Any order that
    adds the two 1s together before meeting 2^24 (a tree, a reversed loop, strided partial sums) keeps
    2^24 + 2, which gives another r (checked, so the pin can fail).  Expected y_0 = (4096 * r) * 1 with
    r = 1 / sqrt(2^24 / 768), each an IEEE fp32 step."""
    K = 768
    x = np.zeros((1, K), np.float32)
    x[0, 0] = 4096.0
    x[0, list(pos)] = 1.0
    gamma = np.ones(K, np.float32)
    y = oracle.rmsnorm(x, gamma, 0.0)

    def r_of(total):
        return np.float32(np.float32(1.0) / np.sqrt(np.float32(np.float32(total) / np.float32(K))))

    r = r_of(2.0 ** 24)
    assert y[0, 0] == np.float32(np.float32(4096.0) * r) and y[0, pos[0]] == r and y[0, pos[1]] == r
    assert np.float32(np.float32(4096.0) * r) != np.float32(np.float32(4096.0) * r_of(2.0 ** 24 + 2))


def test_rmsnorm_sum_of_squares_small_first():
    """The other direction of the same pin: ones first, then the large square.  Left to right the ones
    add exactly (1 + 1 = 2), and 2 + 2^24 is exact too, so the total is 2^24 + 2: an order that puts the
    large element first would round the ones away."""
    K = 512
    x = np.zeros((1, K), np.float32)
    x[0, 10], x[0, 20], x[0, 300] = 1.0, 1.0, 4096.0
    y = oracle.rmsnorm(x, np.ones(K, np.float32), 0.0)
    r = np.float32(np.float32(1.0) / np.sqrt(np.float32(np.float32(2.0 ** 24 + 2) / np.float32(K))))
    assert y[0, 10] == r and y[0, 300] == np.float32(np.float32(4096.0) * r)


def test_rmsnorm_against_f64():
    # y = x / sqrt(mean(x^2) + eps) * gamma in f64; the fp32 oracle differs by a few roundings only
    g = synth.rng(700)
    for K in (256, 2560, 9728):
        x = synth.activations(3, K, g, outliers=True)
        gamma = (g.standard_normal(K) * 0.5 + 1.0).astype(np.float32)
        eps = 1e-6
        y = oracle.rmsnorm(x, gamma, eps)
        xd = x.astype(np.float64)
        ref = xd / np.sqrt((xd * xd).mean(axis=1, keepdims=True) + eps) * gamma.astype(np.float64)
        assert np.all(np.abs(y - ref) <= 1e-5 * np.abs(ref) + 1e-30), np.abs((y - ref) / ref).max()


def test_rmsnorm_constant_row_is_exact():
    # x = 3: sum of squares 9K is exact, r = fl(1/3), y = fl(3 * fl(1/3)) = 1 exactly; the Q8_K block of
    # an all-ones row: first maximum at element 0, iscale = -127, every code -127, d = 1/(-127)
    K = 512
    x = np.full((1, K), 3.0, np.float32)
    q, y = oracle.rmsnorm_quantize_q8_k(x, np.ones(K, np.float32), 0.0)
    assert np.array_equal(y, np.ones((1, K), np.float32))
    blk = q[0, :292]
    assert np.frombuffer(blk[:4].tobytes(), np.float32)[0] == np.float32(1.0) / np.float32(-127.0)
    assert (blk[4:260].view(np.int8) == -127).all()
    assert (np.frombuffer(blk[260:292].tobytes(), np.int16) == -127 * 16).all()


def test_rmsnorm_zero_row_gives_zero_block():
    K = 256
    q, y = oracle.rmsnorm_quantize_q8_k(np.zeros((2, K), np.float32), np.ones(K, np.float32), 1e-6)
    assert (y == 0).all() and (q == 0).all()


def test_rmsnorm_scale_invariance_by_powers_of_two():
    # with eps = 0, scaling x by 2^k scales every square and the sum by 4^k exactly and r by 2^-k,
    # so y is unchanged bit for bit -- a misplaced mean, square root or eps would break this
    g = synth.rng(701)
    K = 2560
    x = synth.activations(2, K, g, outliers=True)
    gamma = (g.standard_normal(K) + 1.0).astype(np.float32)
    y = oracle.rmsnorm(x, gamma, 0.0)
    for k in (-3, 2, 5):
        assert np.array_equal(oracle.rmsnorm(x * np.float32(2.0 ** k), gamma, 0.0), y)


def test_rmsnorm_elementwise_positions():
    # y_i = (x_i * r) * gamma_i: with gamma_3 = 1, y_3 is x_3 * r itself; swapping gamma_3 and
    # gamma_700 (r does not depend on gamma) gives y_3 = (x_3 * r) * gamma_700 and leaves every other
    # position unchanged -- an index slip between x, gamma and y breaks this
    g = synth.rng(702)
    K = 1024
    x = synth.activations(1, K, g)
    gamma = (g.standard_normal(K) + 1.0).astype(np.float32)
    gamma[3] = 1.0
    y = oracle.rmsnorm(x, gamma, 1e-5)
    gs = gamma.copy()
    gs[[3, 700]] = gs[[700, 3]]
    ys = oracle.rmsnorm(x, gs, 1e-5)
    assert ys[0, 3] == np.float32(y[0, 3] * gamma[700])
    keep = np.ones(K, bool)
    keep[[3, 700]] = False
    assert np.array_equal(ys[0, keep], y[0, keep])
