"""GPU parity of the activation quantizers against the CPU oracle (bit-exact).

Where fp32 decides an integer code, both sides take the decision in fp32 with
the same IEEE operations (division, multiply, nearest-even or roundf), so
codes, scales and bsums must match byte for byte.  The fused SwiGLU variants
differ only in exp(): CUDA's expf is within 2 ulp and the host's within 1 ulp
of exp, and 1 + e, the division and the product each add at most half an ulp,
so h on the two sides differs by at most 6 ulp; the test bounds h by that and
checks the quantizer bit-exactly on the GPU's own h.
"""
import numpy as np
import pytest
import torch

import gemv_quantize_q8_gb300 as kq
import oracle
from gemv_quantize_q8_gb300 import synth
from tests.gpu_util import DEV, dev, host, q8_1, q8k

pytestmark = pytest.mark.gpu


def _special_rows(K):
    rows = []
    z = np.zeros(K, np.float32); rows.append(z)
    s = np.zeros(K, np.float32); s[37] = 3.5; s[300 % K] = -1e-3; rows.append(s)
    t = np.zeros(K, np.float32); t[5], t[9] = -1.5, 1.5; rows.append(t)
    r = (np.arange(K) % 256 - 128).astype(np.float32); rows.append(r)
    h = np.zeros(K, np.float32); h[0] = -127.0; h[1:121] = np.arange(-60, 60) + 0.5; rows.append(h)
    n = np.linspace(-1, 1, K, dtype=np.float32); n[10] = np.nan; rows.append(n)
    i = np.linspace(-1, 1, K, dtype=np.float32); i[3] = np.inf; rows.append(i)
    tiny = np.full(K, 1e-40, np.float32); tiny[1] = -3e-39; rows.append(tiny)
    big = np.full(K, 3e38, np.float32); big[2] = -3.4e38; rows.append(big)
    return np.stack(rows)


@pytest.mark.parametrize("M,K,outliers", [(8, 1024, False), (3, 2560, True), (1, 9728, False), (64, 4096, True)])
def test_q8k_bit_exact(M, K, outliers):
    g = synth.rng(100 + M)
    x = synth.activations(M, K, g, outliers=outliers)
    got = host(q8k(dev(x), M, K)).reshape(M, -1)
    assert np.array_equal(got, oracle.quantize_q8_k(x))


def test_q8k_special_values_bit_exact():
    x = _special_rows(512)
    M = x.shape[0]
    got = host(q8k(dev(x), M, 512)).reshape(M, -1)
    assert np.array_equal(got, oracle.quantize_q8_k(x))


def test_q8k_strided_rows():
    g = synth.rng(101)
    full = synth.activations(5, 1280, g)
    got = host(q8k(dev(full), 5, 1024, ld=1280)).reshape(5, -1)
    assert np.array_equal(got, oracle.quantize_q8_k(full[:, :1024]))


def test_q8k_full_prefill_size():
    g = synth.rng(102)
    x = synth.activations(2048, 4096, g, outliers=True)
    got = host(q8k(dev(x), 2048, 4096)).reshape(2048, -1)
    assert np.array_equal(got, oracle.quantize_q8_k(x))


@pytest.mark.parametrize("M,K", [(8, 1024), (3, 2560), (7, 96), (2048, 512)])
def test_q8_1_bit_exact(M, K):
    g = synth.rng(110 + M)
    x = synth.activations(M, K, g, outliers=True)
    got = host(q8_1(dev(x), M, K)).reshape(M, -1)
    assert np.array_equal(got, oracle.quantize_q8_1(x))


def test_q8_1_special_values():
    x = _special_rows(512)
    M = x.shape[0]
    got = host(q8_1(dev(x), M, 512)).reshape(M, -1)
    ref = oracle.quantize_q8_1(x)
    assert np.array_equal(got, ref)


def test_q8_1_half_integer_quotients():
    """Values whose quotient v/d lies on or within a few ulps of a half-integer (where the rounding
    is decided by the last bits of the IEEE quotient): blocks with d exactly 1 (amax 127), with
    d = amax/127 of arbitrary amax, and with amax near and below 2^-100; bytes equal the oracle's."""
    rng = np.random.default_rng(7)
    rows = []
    for _ in range(4):
        blocks = []
        for amax in (127.0, 3.7, 0.0123, 1.0e-30, 1.0e-29, 5.0e3, 5.0e-32, 0.5):
            d = np.float32(np.float32(amax) / np.float32(127.0))
            blk = np.zeros(32, np.float32)
            blk[0] = amax
            k = rng.integers(-126, 126, 31).astype(np.float64) + 0.5
            vals = (k * np.float64(d)).astype(np.float32)
            # the half-integer multiple itself and its float neighbours (up to 3 ulps either way)
            for i, st in enumerate(rng.integers(-3, 4, 31)):
                for _ in range(abs(int(st))):
                    vals[i] = np.nextafter(vals[i], np.float32(np.inf if st > 0 else -np.inf), dtype=np.float32)
            blk[1:] = np.clip(vals, -amax, amax)
            blocks.append(blk)
        rows.append(np.concatenate(blocks))
    x = np.stack(rows).astype(np.float32)
    M, K = x.shape
    got = host(q8_1(dev(x), M, K)).reshape(M, -1)
    ref = oracle.quantize_q8_1(x)
    assert np.array_equal(got, ref)


def _swiglu_gpu(fn, g, u, M, K, ld, nbytes):
    xq = torch.full((nbytes,), 0xAB, dtype=torch.uint8, device=DEV)
    h = torch.full((M, K), float("nan"), dtype=torch.float32, device=DEV)
    fn(g, u, M, K, ld, xq, h)
    return host(xq).reshape(M, -1), host(h)


@pytest.mark.parametrize("q81", [True, False])
def test_swiglu_quant(q81):
    gen = synth.rng(120)
    M, K = 64, 1024
    gu = (synth.activations(M, 2 * K, gen) * 3).astype(np.float32)     # g = cols [0, K), u = [K, 2K)
    d = dev(gu)
    fn = kq.kq_swiglu_quantize_q8_1 if q81 else kq.kq_swiglu_quantize_q8k
    nbytes = kq.q8_1_bytes(M, K) if q81 else kq.q8k_bytes(M, K)
    xq, h = _swiglu_gpu(fn, d, d[:, K:], M, K, 2 * K, nbytes)
    h_ref = oracle.swiglu(gu[:, :K], gu[:, K:])
    qf = oracle.quantize_q8_1 if q81 else oracle.quantize_q8_k
    assert np.array_equal(xq, qf(h))                      # quantizer bit-exact on the GPU's own h
    ulp = np.abs(h.view(np.int32).astype(np.int64) - h_ref.view(np.int32).astype(np.int64))
    assert ulp.max() <= 6, ulp.max()                      # exp() implementations differ by a few ulp
    diff = (xq != qf(h_ref)).mean()
    assert diff < 1e-3                                    # codes flip only at rounding boundaries


def test_swiglu_q8_1_full_size_sampled_rows():
    gen = synth.rng(121)
    M, K = 2048, 9728
    gu = synth.activations(M, 2 * K, gen)
    d = dev(gu)
    xq, h = _swiglu_gpu(kq.kq_swiglu_quantize_q8_1, d, d[:, K:], M, K, 2 * K, kq.q8_1_bytes(M, K))
    rows = gen.choice(M, 16, replace=False)
    assert np.array_equal(xq[rows], oracle.quantize_q8_1(h[rows]))
    h_ref = oracle.swiglu(gu[rows, :K], gu[rows, K:])
    ulp = np.abs(h[rows].view(np.int32).astype(np.int64) - h_ref.view(np.int32).astype(np.int64))
    assert ulp.max() <= 6


def test_quantizer_rejects_bad_args():
    x = torch.zeros(300, device=DEV)
    out = torch.zeros(1024, dtype=torch.uint8, device=DEV)
    with pytest.raises(kq.KqError) as e:
        kq.kq_quantize_q8k(x, 1, 300, 300, out)
    assert e.value.status == 1


# ----------------------------------------------------------------------------- RMSNorm -> Q8_K producer


def _rmsnorm_gpu(x, gamma, eps, ld=None, with_y=True):
    M, K = x.shape[0], gamma.shape[0]
    ld = ld or K
    xd = torch.zeros((M, ld), device=DEV)
    xd[:, :K] = dev(np.ascontiguousarray(x[:, :K]))
    xq = torch.full((kq.q8k_bytes(M, K),), 0xAB, dtype=torch.uint8, device=DEV)
    y = torch.full((M, K), float("nan"), device=DEV) if with_y else None
    kq.kq_rmsnorm_quantize_q8k(xd, dev(gamma), eps, M, K, ld, xq, y)
    return host(xq).reshape(M, -1), (host(y) if with_y else None)


_U = 2.0 ** -24   # unit roundoff of fp32


def _gamma(n: int) -> float:
    return n * _U / (1.0 - n * _U)


def _rmsnorm_rel_bound(K: int) -> float:
    """Relative bound on |y_gpu - y_oracle| / |y_oracle| from the two sum-of-squares orders.

    Both sides sum the K squares (each rounded once): the oracle left to right (K - 1 adds, error at
    most gamma_{K-1} of the sum, all terms being >= 0), the kernel in a fixed tree of depth
    K/256 - 1 (a thread's serial sum) + 5 (butterfly) + 7 (the group sums) < K/256 + 12.  So the two
    sums differ by at most (gamma_{K-1} + gamma_{K/256+12} + 2u) of the exact one; r = 1/sqrt(ss/K + eps)
    halves a relative change of its argument (eps >= 0 only shrinks it) and adds at most four roundings
    per side (/K, +eps, sqrt, 1/x), and y = (x*r)*gamma two more per side."""
    return 0.5 * (_gamma(K - 1) + _gamma(K // 256 + 12) + 2 * _U) + 12 * _U


def _dequant_q8k_rows(q: np.ndarray) -> np.ndarray:
    return oracle.dequant(oracle.Q8_K, q.reshape(-1)).reshape(q.shape[0], -1)


def _check_rmsnorm(x, gamma, eps, q, y):
    """The GPU producer against the oracle: y within the summation-order bound of the oracle's y; the
    Q8_K bytes equal the oracle quantizer's on the GPU's own y (bit for bit); the dequantised rows within
    NMSE 1e-6 of the oracle's whole chain (norm, then quantize)."""
    q_ref, y_ref = oracle.rmsnorm_quantize_q8_k(x, gamma, eps)
    rel = _rmsnorm_rel_bound(x.shape[1])
    err = np.abs(y.astype(np.float64) - y_ref.astype(np.float64))
    assert np.all(err <= rel * np.abs(y_ref.astype(np.float64))), (err / np.maximum(np.abs(y_ref), 1e-300)).max()
    assert np.array_equal(q, oracle.quantize_q8_k(y))
    a, b = _dequant_q8k_rows(q), _dequant_q8k_rows(q_ref)
    assert ((a - b) ** 2).sum() <= 1e-6 * max((b ** 2).sum(), 1e-300)


@pytest.mark.parametrize("M,K", [(1, 256), (1, 2560), (1, 9728), (3, 4096), (64, 2048), (5, 16384), (2, 24576),
                                 (65, 1024), (70, 20480)])
def test_rmsnorm_q8k_against_oracle(M, K):
    g = synth.rng(720 + M + K)
    x = synth.activations(M, K, g, outliers=True)
    gamma = (g.standard_normal(K) * 0.3 + 1.0).astype(np.float32)
    q, y = _rmsnorm_gpu(x, gamma, 1e-6)
    _check_rmsnorm(x, gamma, 1e-6, q, y)


def test_rmsnorm_q8k_special_rows_and_stride():
    # zero row (r = 1/sqrt(eps), y = 0: the zero block), a constant row (exact sum in any order), huge and
    # tiny magnitudes, a row stride larger than K (scalar loads), and no y output
    K = 512
    rows = [np.zeros(K, np.float32), np.full(K, 3.0, np.float32), np.full(K, -1e-20, np.float32),
            (np.arange(K) - 256).astype(np.float32) * 1e15]
    x = np.stack(rows)
    gamma = np.linspace(0.5, 1.5, K, dtype=np.float32)
    q, y = _rmsnorm_gpu(x, gamma, 1e-5, ld=K + 3)
    _check_rmsnorm(x, gamma, 1e-5, q, y)
    q_ref, y_ref = oracle.rmsnorm_quantize_q8_k(x, gamma, 1e-5)
    assert (q[0] == 0).all() and (y[0] == 0).all()
    assert np.array_equal(y[1], y_ref[1]) and np.array_equal(q[1], q_ref[1])   # 9K is exact in any order
    q2, _ = _rmsnorm_gpu(x, gamma, 1e-5, with_y=False)
    assert np.array_equal(q2, q)


def test_rmsnorm_q8k_feeds_decode_gemv():
    # the producer's Q8_K row drives the decode GEMV directly (no separate quantize launch): the GEMV's
    # result is the oracle's GEMV on those very bytes, bit for bit, and within NMSE 1e-6 of the oracle's
    # GEMV on the oracle's own normalized-and-quantised row
    g = synth.rng(730)
    N, K = 640, 2560
    x = synth.activations(1, K, g, outliers=True)
    gamma = (g.standard_normal(K) * 0.3 + 1.0).astype(np.float32)
    w = synth.weights(kq.Q4_K, N, K, g)
    wn = torch.empty(kq.native_bytes(kq.Q4_K, N, K), dtype=torch.uint8, device=DEV)
    kq.kq_repack_weights(kq.Q4_K, dev(w.reshape(-1)), wn, N, K)
    xq = torch.empty(kq.q8k_bytes(1, K), dtype=torch.uint8, device=DEV)
    kq.kq_rmsnorm_quantize_q8k(dev(x), dev(gamma), 1e-6, 1, K, K, xq)
    y = torch.full((N,), float("nan"), device=DEV)
    kq.kq_gemv(kq.Q4_K, wn, None, xq, N, K, y)
    got = host(y)
    assert np.array_equal(got, oracle.gemm(kq.Q4_K, w, host(xq).reshape(1, -1), 1, N, K)[0])
    q_ref, _ = oracle.rmsnorm_quantize_q8_k(x, gamma, 1e-6)
    ref = oracle.gemm(kq.Q4_K, w, q_ref, 1, N, K)[0].astype(np.float64)
    assert ((got - ref) ** 2).sum() <= 1e-6 * (ref ** 2).sum()


def test_rmsnorm_q8k_rejects_bad_args():
    K = 256
    x = torch.zeros((1, K), device=DEV)
    gm = torch.ones(K, device=DEV)
    xq = torch.empty(kq.q8k_bytes(1, K), dtype=torch.uint8, device=DEV)
    for args in [(x, gm, 1e-6, 1, 300, K), (x, gm, -1.0, 1, K, K), (x, gm, 1e-6, 1, K, K - 1), (x, gm, 1e-6, 0, K, K)]:
        with pytest.raises(kq.KqError):
            kq.kq_rmsnorm_quantize_q8k(*args, xq)
