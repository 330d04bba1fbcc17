"""The tensor-core GEMM's integer sums, read out of tensor memory, against the oracle (bit-exact), and
its bounded pipeline waits made to run out.

kq_debug_tc_sums runs the very kernel kq_gemm runs for a shape (same tiles, split-K clusters and TMEM
accumulation) with a debug epilogue that also writes, for every (row, token, scale block), the integer
sums held in the fp32 accumulator before the fp32 promotion: sum_j sc_j*P_j and the Q4_K/Q5_K min term
sum_j m_j*(bs_2j + bs_2j+1) (Q8_0: each 32-block's P_b).  The oracle builds the same integers from its
int32 partial dots and the blocks' integer scales (oracle.block_sums); they must be equal.
"""
import ctypes

import numpy as np
import pytest
import torch

import gemv_quantize_q8_gb300 as kq
import oracle
from gemv_quantize_q8_gb300 import synth
from tests.gpu_util import DEV, act_quant, dev, gemm, host, nmse, repack
from tests.test_gpu_matmul import tc_bound

pytestmark = pytest.mark.gpu

SENTINEL = -0x5A5A5A5A


def _oracle_act(dtype, x):
    return oracle.quantize_q8_1(x) if dtype == kq.Q8_0 else oracle.quantize_q8_k(x)


def _nblk(dtype, K):
    return K // 32 if dtype == kq.Q8_0 else K // 256


def _tc_sums(dtype, wn, xq, M, N, K):
    y = torch.full((M, N), float("nan"), device=DEV)
    sums = torch.full((M, N, _nblk(dtype, K), 2), SENTINEL, dtype=torch.int32, device=DEV)
    wsb = kq.gemm_workspace_bytes(dtype, M, N, K)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=DEV)
    kq.kq_debug_tc_sums(dtype, wn, xq, M, N, K, y, N, sums, ws, wsb)
    assert kq.kq_read_device_flag(ws) == 0
    return host(y), host(sums)


@pytest.mark.parametrize("dtype", [kq.Q4_K, kq.Q5_K, kq.Q6_K, kq.Q8_0])
@pytest.mark.parametrize("M,N,K", [(300, 392, 1536), (250, 600, 4096), (129, 1280, 3072), (640, 256, 1024)])
def test_tc_integer_sums_bit_exact(dtype, M, N, K):
    """Multi-tile shapes, ragged in M and N, persistent (S = 1) and split-K (S = 8, 4) launches: every
    integer sum equals the oracle's, and the y the debug twin writes equals kq_gemm's bit for bit."""
    g = synth.rng(950 + M + N + K + dtype)
    w = synth.weights(dtype, N, K, g)
    x = synth.activations(M, K, g, outliers=True)
    wn = repack(dtype, w, N, K)
    xq = act_quant(dtype, dev(x), M, K)
    xq_h = host(xq).reshape(M, -1)
    assert np.array_equal(xq_h, _oracle_act(dtype, x))
    y, sums = _tc_sums(dtype, wn, xq, M, N, K)
    ref = oracle.block_sums(dtype, w, xq_h, M, N, K)
    assert np.abs(ref).max() < 2 ** 24, "inputs of this test keep every sum exact in fp32"
    assert np.array_equal(sums.astype(np.int64), ref)
    assert np.array_equal(y, host(gemm(dtype, wn, xq, M, N, K)))


@pytest.mark.parametrize("dtype", [kq.Q4_K, kq.Q6_K])
@pytest.mark.parametrize("M,N,K", [(128, 4096, 4096), (2048, 2560, 2048)])
def test_tc_integer_sums_full_size_split_k(dtype, M, N, K):
    """The benchmark's M = 128 [4096 x 4096] GEMM, which the tensor-core path splits across clusters of
    CTAs, and a [2560 x 2048] M = 2048 GEMM whose leftover tiles after two whole waves run as a split-K
    launch: the integer sums of 16 token rows (for the second, also 16 rows of the last token tile, in
    the split tail) and every weight row against the oracle."""
    assert kq.kq_debug_tc_splits(dtype, M, N, K) > 1
    g = synth.rng(0)
    w = synth.weights(dtype, N, K, g)
    x = synth.activations(M, K, g, outliers=True)
    wn = repack(dtype, w, N, K)
    xq = act_quant(dtype, dev(x), M, K)
    _, sums = _tc_sums(dtype, wn, xq, M, N, K)
    xq_h = host(xq).reshape(M, -1)
    for r in ([np.arange(16)] + ([np.arange(M - 100, M - 84)] if M > 128 else [])):
        ref = oracle.block_sums(dtype, w, np.ascontiguousarray(xq_h[r]), 16, N, K)
        assert np.array_equal(sums[r].astype(np.int64), ref)


@pytest.mark.parametrize("dtype", [kq.Q4_K, kq.Q5_K, kq.Q6_K, kq.Q8_0])
@pytest.mark.parametrize("rpt", ["broadcast", "per_row"])
def test_tc_integer_sums_routed(dtype, rpt):
    """Routed experts: several 128-row tiles for one expert, a tail tile, an empty expert and two
    invalid ids.  Every valid (token, slot) row's integer sums equal the oracle's on its expert's
    weights; the rows of invalid ids are left untouched."""
    g = synth.rng(970 + dtype)
    E, M, top_k, N, K = 5, 300, 2, 256, 1024
    w = synth.weights(dtype, E * N, K, g)
    ids, _ = synth.routing(M, E, top_k, g)
    ids[ids == 4] = 0
    ids[7, 1], ids[100, 0] = E + 3, -1
    per_row = rpt == "per_row"
    rows = M * top_k if per_row else M
    x = synth.activations(rows, K, g, outliers=True)
    wn = repack(dtype, w, E * N, K)
    xq = act_quant(dtype, dev(x), rows, K)
    xq_h = host(xq).reshape(rows, -1)
    nblk = _nblk(dtype, K)
    y = torch.full((M, top_k, N), float("nan"), device=DEV)
    sums = torch.full((M * top_k, N, nblk, 2), SENTINEL, dtype=torch.int32, device=DEV)
    wsb = kq.gemm_workspace_bytes(dtype, M, N, K, E, top_k)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=DEV)
    kq.kq_debug_tc_sums_grouped(dtype, wn, E, xq, top_k if per_row else 1, dev(ids), M, top_k, N, K, y, sums, ws, wsb)
    assert kq.kq_read_device_flag(ws) == 2
    got = host(sums).astype(np.int64)
    flat = ids.reshape(-1)
    wb = w.reshape(E, N, -1)
    for e in range(E):
        pairs = np.nonzero(flat == e)[0]
        if pairs.size == 0:
            continue
        src = pairs if per_row else pairs // top_k
        ref = oracle.block_sums(dtype, np.ascontiguousarray(wb[e]), np.ascontiguousarray(xq_h[src]), pairs.size, N, K)
        assert np.array_equal(got[pairs], ref), e
    bad = np.nonzero((flat < 0) | (flat >= E))[0]
    assert bad.size == 2 and (got[bad] == SENTINEL).all()


def test_tc_bounded_wait_runs_out_and_recovers():
    """A pipeline wait that can never complete (the activation producer is kept idle) runs into its
    limit: the kernel returns, the device flag reports the timeout, and the next normal call on the
    same stream computes the right result.  Nothing faults or hangs: every CTA drains its own copies
    and MMAs (bounded waits) and frees its tensor memory before it leaves."""
    dtype, M, N, K = kq.Q4_K, 200, 384, 512
    assert kq.kq_debug_tc_splits(dtype, M, N, K) == 1
    g = synth.rng(990)
    w = synth.weights(dtype, N, K, g)
    x = synth.activations(M, K, g)
    wn = repack(dtype, w, N, K)
    xq = act_quant(dtype, dev(x), M, K)
    wsb = kq.gemm_workspace_bytes(dtype, M, N, K)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    y = torch.full((M, N), float("nan"), device=DEV)
    kq.kq_debug_tc_wait_timeout(dtype, wn, xq, M, N, K, y, N, 200_000, ws, wsb)
    torch.cuda.synchronize()
    n_bad = ctypes.c_int64(0)
    st = kq.lib().kq_read_device_flag(ws.data_ptr(), ctypes.byref(n_bad), torch.cuda.current_stream().cuda_stream)
    assert st == 6, kq.lib().kq_status_string(st)          # KQ_ERR_DEVICE_FLAG
    assert n_bad.value >= 1                                 # one count per CTA that timed out
    assert kq.kq_read_device_flag(ws) == 0                  # reading clears it
    # the stream and the context are still usable: a normal call is correct
    y2 = host(gemm(dtype, wn, xq, M, N, K))
    xq_h = host(xq).reshape(M, -1)
    mi, ni = np.repeat(np.arange(M), N), np.tile(np.arange(N), M)
    ref, terms = oracle.gemm_sampled_terms(dtype, w, xq_h, K, mi, ni)
    assert np.all(np.abs(y2.reshape(-1).astype(np.float64) - ref) <= tc_bound(terms, K, 1))
    assert nmse(y2.reshape(-1), ref) <= 1e-6
