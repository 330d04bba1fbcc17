"""GPU parity of kq_gemm_f32: the GEMM from fp32 activations with the Q8_K quantizer in its prologue.

The prologue quantises with the standalone quantizer's own block arithmetic, so the output must equal
kq_quantize_q8k (kq_quantize_q8_1 for Q8_0) followed by kq_gemm bit for bit, on the tensor-core path
and on the others; the oracle checks the result independently (NMSE against its quantizer and GEMM)."""
import numpy as np
import pytest
import torch

import gemv_quantize_q8_gb300 as kq
import oracle
from gemv_quantize_q8_gb300 import synth
from tests.gpu_util import DEV, act_quant, dev, host, nmse, repack

pytestmark = pytest.mark.gpu

DTS = [kq.Q4_K, kq.Q5_K, kq.Q6_K, kq.Q8_0]


def _two_step(dtype, wn, xd, M, N, K, ldx):
    xq = act_quant(dtype, xd[:, :K].contiguous(), M, K)
    y = torch.full((M, N), float("nan"), device=DEV)
    wsb = kq.gemm_workspace_bytes(dtype, M, N, K)
    ws = torch.zeros(max(wsb, 256), dtype=torch.uint8, device=DEV)
    kq.kq_gemm(dtype, wn, xq, M, N, K, y, N, ws if wsb else None, wsb)
    return y


def _fused(dtype, wn, xd, M, N, K, ldx):
    y = torch.full((M, N), float("nan"), device=DEV)
    wsb = kq.kq_gemm_f32_workspace_bytes(dtype, M, N, K)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=DEV)
    kq.kq_gemm_f32(dtype, wn, xd, ldx, M, N, K, y, N, ws, wsb)
    assert kq.kq_read_device_flag(ws) == 0
    return y


@pytest.mark.parametrize("dtype", DTS)
@pytest.mark.parametrize("M,N,K,pad", [(160, 256, 512, 0), (130, 200, 768, 3), (300, 392, 1536, 4), (8, 256, 1024, 0),
                                       (3, 100, 2560, 1), (20, 64, 512, 0)])
def test_gemm_f32_equals_quantize_then_gemm(dtype, M, N, K, pad):
    g = synth.rng(900 + dtype + M + K)
    w = synth.weights(dtype, N, K, g)
    x = synth.activations(M, K, g, outliers=True)
    ldx = K + pad
    xp = np.zeros((M, ldx), np.float32)
    xp[:, :K] = x
    wn = repack(dtype, w, N, K)
    xd = dev(xp)
    a = _fused(dtype, wn, xd.reshape(-1), M, N, K, ldx)
    b = _two_step(dtype, wn, xd, M, N, K, ldx)
    assert torch.equal(a, b), "kq_gemm_f32 differs from kq_quantize + kq_gemm"
    xa = oracle.quantize_q8_1(x) if dtype == kq.Q8_0 else oracle.quantize_q8_k(x)
    ref = oracle.gemm(dtype, w, xa, M, N, K)
    assert nmse(host(a), ref) <= 1e-6


def test_gemm_f32_zero_and_unaligned_rows():
    # all-zero rows give the zero block (exact zeros out); x only 4-byte aligned takes the scalar loads
    dtype, M, N, K = kq.Q4_K, 140, 256, 512
    g = synth.rng(950)
    w = synth.weights(dtype, N, K, g)
    wn = repack(dtype, w, N, K)
    x = synth.activations(M, K, g)
    x[5] = 0.0
    buf = torch.zeros(M * K + 1, device=DEV)
    buf[1:] = dev(x).reshape(-1)
    a = _fused(dtype, wn, buf[1:], M, N, K, K)
    b = _two_step(dtype, wn, dev(x), M, N, K, K)
    assert torch.equal(a, b)
    assert (host(a)[5] == 0).all()


def test_gemm_f32_prefill_full_size_equals_two_step():
    # the largest prefill GEMM shape at M = 2048: bit-equal to the two-step path
    dtype, (N, K), M = kq.Q6_K, synth.PREFILL_SHAPES[2], 2048
    g = synth.rng(960)
    w = synth.weights(dtype, N, K, g)
    x = synth.activations(M, K, g, outliers=True)
    wn = repack(dtype, w, N, K)
    xd = dev(x)
    a = _fused(dtype, wn, xd, M, N, K, K)
    b = _two_step(dtype, wn, xd, M, N, K, K)
    assert torch.equal(a, b)


@pytest.mark.parametrize("dtype", DTS)
@pytest.mark.parametrize("M,N,K,pad", [(160, 256, 512, 0), (300, 392, 1536, 4), (8, 256, 1024, 0), (1100, 4300, 256, 0)])
def test_gemm_f32_folded_equals_quantize_then_folded_gemm(dtype, M, N, K, pad):
    """kq_gemm_f32_ex with KQ_GEMM_FOLD_SCALES: the prologue's f16(d*q) panel from the fp32 rows is the one
    the folded GEMM builds from the quantiser's Q8_K rows, so the result equals kq_quantize_q8k (Q8_0:
    kq_quantize_q8_1) followed by kq_gemm_ex with the same flag, bit for bit -- with 128-token tiles
    (split or not), 256-token tiles (M = 1100) and the exact fallback (M = 8)."""
    g = synth.rng(970 + dtype + M + K)
    w = synth.weights(dtype, N, K, g)
    x = synth.activations(M, K, g, outliers=True)
    ldx = K + pad
    xp = np.zeros((M, ldx), np.float32)
    xp[:, :K] = x
    wn = repack(dtype, w, N, K)
    xd = dev(xp)
    ya = torch.full((M, N), float("nan"), device=DEV)
    wsa = kq.kq_gemm_f32_workspace_bytes(dtype, M, N, K)
    wsa_t = torch.zeros(wsa, dtype=torch.uint8, device=DEV)
    kq.kq_gemm_f32_ex(dtype, wn, xd.reshape(-1), ldx, M, N, K, ya, N, kq.GEMM_FOLD_SCALES, wsa_t, wsa)
    assert kq.kq_read_device_flag(wsa_t) == 0
    xq = act_quant(dtype, xd[:, :K].contiguous(), M, K)
    yb = torch.full((M, N), float("nan"), device=DEV)
    wsb = kq.gemm_workspace_bytes(dtype, M, N, K)
    wsb_t = torch.zeros(max(wsb, 256), dtype=torch.uint8, device=DEV)
    kq.kq_gemm_ex(dtype, wn, xq, M, N, K, yb, N, kq.GEMM_FOLD_SCALES, wsb_t if wsb else None, wsb)
    assert torch.equal(ya, yb), "kq_gemm_f32_ex (folded) differs from quantize + kq_gemm_ex"
    xa = oracle.quantize_q8_1(x) if dtype == kq.Q8_0 else oracle.quantize_q8_k(x)
    mi, ni = g.integers(0, M, 1500), g.integers(0, N, 1500)
    assert nmse(host(ya)[mi, ni], oracle.gemm_sampled(dtype, w, xa, K, mi, ni)) <= 1e-6


def test_gemm_f32_chain_sharing_one_workspace():
    """GEMMs of different shapes and schedules (split-K clusters, persistent CTAs, a split tail) issued
    back to back on one stream with one shared workspace, no synchronisation between them: each GEMM's
    tensor-core launch may start beside its own activation prologue, but the next prologue rewrites the
    shared panels only once the GEMM before it has finished, so every output equals the same GEMM run
    alone, bit for bit."""
    cases = [(kq.Q4_K, 128, 1024, 4096), (kq.Q6_K, 512, 1024, 2048), (kq.Q4_K, 2048, 2560, 2048),
             (kq.Q6_K, 130, 768, 4096), (kq.Q4_K, 300, 392, 1536)]
    g = synth.rng(980)
    prepared = []
    wsb = 0
    for dtype, M, N, K in cases:
        w = synth.weights(dtype, N, K, g)
        x = synth.activations(M, K, g, outliers=True)
        prepared.append((dtype, M, N, K, repack(dtype, w, N, K), dev(x)))
        wsb = max(wsb, kq.kq_gemm_f32_workspace_bytes(dtype, M, N, K))
    ws = torch.zeros(wsb, dtype=torch.uint8, device=DEV)
    chain = []
    for dtype, M, N, K, wn, xd in prepared:
        y = torch.full((M, N), float("nan"), device=DEV)
        kq.kq_gemm_f32(dtype, wn, xd, K, M, N, K, y, N, ws, wsb)
        chain.append(y)
    torch.cuda.synchronize()
    assert kq.kq_read_device_flag(ws) == 0
    for (dtype, M, N, K, wn, xd), y in zip(prepared, chain):
        alone = _fused(dtype, wn, xd, M, N, K, K)
        assert torch.equal(y, alone), (dtype, M, N, K)
