"""The allocation-free routed-expert GEMM, kq_gemm_grouped_noalloc.

It serves callers that cannot allocate device memory when they run the MoE
layer (they are handed only their input and output buffers), so its routing
scratch is a fixed array inside the library instead of a caller workspace.
Checked here through the C ABI on two calls in a row with different routing
and sizes -- the second call must not see anything the first left in the
shared array -- against the oracle (bit for bit: it runs the exact dp4a path)
and against kq_gemm_grouped with a workspace (whose Q4_K/Q6_K tensor-core path
agrees to within rounding), and for its clear refusal of problems too large for
the fixed array.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import gemv_quantize_q8_gb300 as kq
import oracle
from gemv_quantize_q8_gb300 import synth
from tests.gpu_util import DEV, act_quant, dev, host, nmse, repack

pytestmark = pytest.mark.gpu


def _with_workspace(dtype, wn, E, xq, rpt, ids, M, top_k, N, K):
    y = torch.full((M, top_k, N), float("nan"), device=DEV)
    wsb = kq.gemm_workspace_bytes(dtype, M, N, K, E, top_k)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=DEV)
    kq.kq_gemm_grouped(dtype, wn, E, xq, rpt, dev(ids), M, top_k, N, K, y, ws, wsb)
    return host(y)


def _no_alloc(dtype, wn, E, xq, rpt, ids, M, top_k, N, K):
    y = torch.full((M, top_k, N), float("nan"), device=DEV)
    kq.kq_gemm_grouped_noalloc(dtype, wn, E, xq, rpt, dev(ids), M, top_k, N, K, y)
    return host(y)


def _case(dtype, E, M, top_k, N, K, per_row, seed):
    g = synth.rng(seed)
    w = synth.weights(dtype, E * N, K, g)
    ids, _ = synth.routing(M, E, top_k, g)
    rows = M * top_k if per_row else M
    x = synth.activations(rows, K, g)
    wn = repack(dtype, w, E * N, K)
    xq = act_quant(dtype, dev(x), rows, K)
    ref, _ = oracle.gemm_grouped(dtype, w, E, oracle.quantize_q8_k(x), top_k if per_row else 1, ids, M, top_k, N, K)
    return wn, xq, (top_k if per_row else 1), ids, ref


def test_no_alloc_matches_workspace_path_on_two_calls():
    # first call: 256 experts, 512 tokens, top-8, Q4_K gate/up-like shape (broadcast activations)
    E, M, top_k, N, K = 256, 512, 8, 64, 2048
    wn, xq, rpt, ids, ref1 = _case(kq.Q4_K, E, M, top_k, N, K, False, 900)
    got1 = _no_alloc(kq.Q4_K, wn, E, xq, rpt, ids, M, top_k, N, K)
    ws1 = _with_workspace(kq.Q4_K, wn, E, xq, rpt, ids, M, top_k, N, K)
    assert np.isfinite(got1).all()
    assert np.array_equal(got1, ref1)
    assert nmse(ws1, got1) <= 1e-10
    # second call right after: fewer experts, other routing, Q6_K per-row activations
    E2, M2, top_k2, N2, K2 = 12, 40, 3, 48, 512
    wn2, xq2, rpt2, ids2, ref2 = _case(kq.Q6_K, E2, M2, top_k2, N2, K2, True, 901)
    got2 = _no_alloc(kq.Q6_K, wn2, E2, xq2, rpt2, ids2, M2, top_k2, N2, K2)
    ws2 = _with_workspace(kq.Q6_K, wn2, E2, xq2, rpt2, ids2, M2, top_k2, N2, K2)
    assert np.isfinite(got2).all()
    assert np.array_equal(got2, ref2)
    assert nmse(ws2, got2) <= 1e-10


def test_no_alloc_rejects_problems_beyond_its_fixed_scratch():
    t = torch.zeros(1024, dtype=torch.uint8, device=DEV)
    y = torch.zeros(16, device=DEV)
    with pytest.raises(kq.KqError) as e:
        # 1M tokens x top-8 needs far more routing scratch than the fixed 1 MiB
        kq.kq_gemm_grouped_noalloc(kq.Q4_K, t, 256, t, 1, t, 1 << 20, 8, 64, 256, y)
    assert e.value.status == 1 and "routing scratch" in str(e.value)
