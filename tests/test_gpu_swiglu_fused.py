"""GPU parity of the routed gate/up GEMM with SwiGLU and Q8_K quantisation fused into its epilogue.

The fused call must write the same bytes as the unfused pipeline (routed GEMM to fp32 rows, then the
SwiGLU quantizer over them): both take every step in the same arithmetic, so the comparison is
byte-for-byte.  The oracle pins the result independently: its grouped GEMM, its SwiGLU and its Q8_K
quantizer, compared after dequantisation (exp may differ by an ulp between CPU and GPU, which can move a
code by one at a rounding boundary).
"""
import numpy as np
import pytest
import torch

import gemv_quantize_q8_gb300 as kq
import oracle
from gemv_quantize_q8_gb300 import synth
from tests.gpu_util import DEV, act_quant, dev, host, nmse, repack

pytestmark = pytest.mark.gpu

DTS = [kq.Q4_K, kq.Q5_K, kq.Q6_K, kq.Q8_0]
SENTINEL = 0xAB


def _oracle_act(dtype, x):
    return oracle.quantize_q8_1(x) if dtype == kq.Q8_0 else oracle.quantize_q8_k(x)


def _fused(dtype, wn, E, xq, rpt, ids, M, top_k, F, K):
    hq = torch.full((kq.q8k_bytes(M * top_k, F),), SENTINEL, dtype=torch.uint8, device=DEV)
    wsb = kq.kq_gemm_grouped_swiglu_workspace_bytes(dtype, M, F, K, E, top_k)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=DEV)
    kq.kq_gemm_grouped_swiglu_q8k(dtype, wn, E, xq, rpt, dev(ids), M, top_k, F, K, hq, ws, wsb)
    return hq, ws


def _unfused(dtype, wn, E, xq, rpt, ids, M, top_k, F, K):
    y = torch.full((M * top_k, 2 * F), float("nan"), device=DEV)
    wsb = kq.gemm_workspace_bytes(dtype, M, 2 * F, K, E, top_k)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=DEV)
    kq.kq_gemm_grouped(dtype, wn, E, xq, rpt, dev(ids), M, top_k, 2 * F, K, y, ws, wsb)
    hq = torch.full((kq.q8k_bytes(M * top_k, F),), SENTINEL, dtype=torch.uint8, device=DEV)
    kq.kq_swiglu_quantize_q8k(y, y[:, F:], M * top_k, F, 2 * F, hq)
    return hq, y, ws


def _oracle_h(dtype, w, E, x, rpt, ids, M, top_k, F, K):
    ref_gu, bad = oracle.gemm_grouped(dtype, w, E, _oracle_act(dtype, x), rpt, ids, M, top_k, 2 * F, K)
    flat = ref_gu.reshape(M * top_k, 2 * F)
    return flat, bad


CASES = [
    # E, M, top_k, F, K, rows per token, note
    (5, 300, 2, 512, 1024, "per_row"),    # experts over two 128-token tiles, ragged tails, an empty expert
    (8, 50, 3, 256, 512, "broadcast"),    # one 256-column block per pair, tiles far from full
    (3, 130, 1, 768, 256, "broadcast"),   # three blocks, one super-block of K, a 129-token expert
]


@pytest.mark.parametrize("dtype", DTS)
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"E{c[0]}_M{c[1]}_k{c[2]}_F{c[3]}_K{c[4]}_{c[5]}")
def test_fused_swiglu_equals_unfused_and_oracle(dtype, case):
    E, M, top_k, F, K, mode = case
    g = synth.rng(700 + dtype + 10 * F + K)
    w = synth.weights(dtype, E * 2 * F, K, g)
    ids, _ = synth.routing(M, E, top_k, g)
    if E == 5:
        ids[ids == 4] = 0                      # expert 4 empty, expert 0 over several tiles
    if E == 3:
        ids[:, 0] = 0                          # expert 0: 129 tokens (a full tile and a 1-token tail),
        ids[0, 0] = 1                          # expert 1: one token, expert 2: none
    rpt = 1 if mode == "broadcast" else top_k
    rows = M if rpt == 1 else M * top_k
    x = synth.activations(rows, K, g, outliers=True)
    wn = repack(dtype, w, E * 2 * F, K)
    xq = act_quant(dtype, dev(x), rows, K)
    hq, ws = _fused(dtype, wn, E, xq, rpt, ids, M, top_k, F, K)
    assert kq.kq_read_device_flag(ws) == 0
    hq_u, y_u, ws_u = _unfused(dtype, wn, E, xq, rpt, ids, M, top_k, F, K)
    assert kq.kq_read_device_flag(ws_u) == 0
    got = host(hq)
    assert np.array_equal(got, host(hq_u)), "fused epilogue differs from GEMM + SwiGLU quantizer"
    # the oracle: its GEMM rows, its SwiGLU, its quantizer
    ref_gu, bad = _oracle_h(dtype, w, E, x, rpt, ids, M, top_k, F, K)
    assert bad == 0
    h_ref = oracle.swiglu(ref_gu[:, :F], ref_gu[:, F:])
    hq_ref = oracle.quantize_q8_k(h_ref)
    deq = oracle.dequant(kq.Q8_K, got)
    deq_ref = oracle.dequant(kq.Q8_K, hq_ref.reshape(-1))
    assert nmse(deq, deq_ref) <= 1e-6
    # codes: h differs from the oracle's by ulps (fp32 promotion order, exp), so a code moves by at
    # most one, and only at a rounding boundary
    codes = got.reshape(-1, 292)[:, 4:260].view(np.int8).astype(np.int32)
    codes_ref = hq_ref.reshape(-1, 292)[:, 4:260].view(np.int8).astype(np.int32)
    assert np.abs(codes - codes_ref).max() <= 1
    assert (codes == codes_ref).mean() > 0.999


def test_fused_swiglu_invalid_ids_untouched_rows():
    g = synth.rng(720)
    E, M, top_k, F, K = 4, 40, 2, 256, 512
    w = synth.weights(kq.Q4_K, E * 2 * F, K, g)
    ids, _ = synth.routing(M, E, top_k, g)
    ids[3, 1] = 9
    ids[17, 0] = -1
    x = synth.activations(M, K, g)
    wn = repack(kq.Q4_K, w, E * 2 * F, K)
    xq = act_quant(kq.Q4_K, dev(x), M, K)
    hq, ws = _fused(kq.Q4_K, wn, E, xq, 1, ids, M, top_k, F, K)
    assert kq.kq_read_device_flag(ws) == 2
    rows = host(hq).reshape(M * top_k, -1)
    bad = [3 * top_k + 1, 17 * top_k + 0]
    assert (rows[bad] == SENTINEL).all()
    hq_u, _, _ = _unfused(kq.Q4_K, wn, E, xq, 1, ids, M, top_k, F, K)
    ok = np.ones(M * top_k, bool)
    ok[bad] = False
    assert np.array_equal(rows[ok], host(hq_u).reshape(M * top_k, -1)[ok])


def test_fused_swiglu_zero_rows_are_zero_blocks():
    # all-zero activations: every gate/up value is 0, h = 0, and each block is the zero block
    g = synth.rng(721)
    E, M, top_k, F, K = 2, 20, 2, 256, 256
    w = synth.weights(kq.Q6_K, E * 2 * F, K, g)
    ids, _ = synth.routing(M, E, top_k, g)
    wn = repack(kq.Q6_K, w, E * 2 * F, K)
    xq = act_quant(kq.Q6_K, torch.zeros((M, K), device=DEV), M, K)
    hq, ws = _fused(kq.Q6_K, wn, E, xq, 1, ids, M, top_k, F, K)
    assert kq.kq_read_device_flag(ws) == 0
    assert (host(hq) == 0).all()


def test_fused_swiglu_argument_errors():
    g = synth.rng(722)
    E, M, top_k, F, K = 2, 8, 1, 256, 256
    w = synth.weights(kq.Q4_K, E * 2 * F, K, g)
    ids, _ = synth.routing(M, E, top_k, g)
    wn = repack(kq.Q4_K, w, E * 2 * F, K)
    xq = act_quant(kq.Q4_K, dev(synth.activations(M, K, g)), M, K)
    hq = torch.empty(kq.q8k_bytes(M * top_k, F), dtype=torch.uint8, device=DEV)
    wsb = kq.kq_gemm_grouped_swiglu_workspace_bytes(kq.Q4_K, M, F, K, E, top_k)
    assert wsb > kq.gemm_workspace_bytes(kq.Q4_K, M, 2 * F, K, E, top_k)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=DEV)
    with pytest.raises(kq.KqError):   # F not a multiple of 256
        kq.kq_gemm_grouped_swiglu_q8k(kq.Q4_K, wn, E, xq, 1, dev(ids), M, top_k, 128, K, hq, ws, wsb)
    with pytest.raises(kq.KqError):   # workspace one byte short
        kq.kq_gemm_grouped_swiglu_q8k(kq.Q4_K, wn, E, xq, 1, dev(ids), M, top_k, F, K, hq, ws, wsb - 1)
    with pytest.raises(kq.KqError):   # no output
        kq.kq_gemm_grouped_swiglu_q8k(kq.Q4_K, wn, E, xq, 1, dev(ids), M, top_k, F, K, None, ws, wsb)


def test_fused_moe_block_full_size_equals_unfused():
    """The MoE block's gate/up at its full size (256 experts, top-8, 2048 tokens, hidden 2048, ffn 512):
    every pair's Q8_K row from the fused epilogue equals the unfused pipeline's; sampled tokens are
    checked against the oracle."""
    c = synth.MOE
    E, top_k, M, H, F = c["n_experts"], c["top_k"], c["M"], c["hidden"], c["ffn"]
    g = synth.rng(0)
    w_gu = synth.weights(kq.Q4_K, E * 2 * F, H, g)
    x = synth.activations(M, H, g)
    ids, _ = synth.routing(M, E, top_k, g)
    wn = repack(kq.Q4_K, w_gu, E * 2 * F, H)
    xq = act_quant(kq.Q4_K, dev(x), M, H)
    hq, ws = _fused(kq.Q4_K, wn, E, xq, 1, ids, M, top_k, F, H)
    assert kq.kq_read_device_flag(ws) == 0
    hq_u, _, _ = _unfused(kq.Q4_K, wn, E, xq, 1, ids, M, top_k, F, H)
    got = host(hq).reshape(M, top_k, -1)
    assert np.array_equal(got.reshape(-1), host(hq_u))
    toks = g.choice(M, 8, replace=False)
    ref_gu, _ = oracle.gemm_grouped(kq.Q4_K, w_gu, E, oracle.quantize_q8_k(x[toks]), 1, ids[toks], len(toks), top_k,
                                    2 * F, H)
    flat = ref_gu.reshape(-1, 2 * F)
    hq_ref = oracle.quantize_q8_k(oracle.swiglu(flat[:, :F], flat[:, F:]))
    deq = oracle.dequant(kq.Q8_K, got[toks].reshape(-1))
    assert nmse(deq, oracle.dequant(kq.Q8_K, hq_ref.reshape(-1))) <= 1e-6
