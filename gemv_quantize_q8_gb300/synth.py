"""Seeded synthetic inputs for the keep-quant matmul workloads.

This module only draws random numbers and places them into the canonical
(GGUF-style) block byte layouts; it holds none of the method's arithmetic
(no quantisation, no dot products, no dequantisation).  Both the CUDA path's
tests/benchmark and the CPU oracle consume what it produces.

Generator: numpy ``default_rng(seed)`` (PCG64).  Draw order per weight
tensor: the per-super-block f16 fields (d, then dmin), then scale/min bytes,
then code bytes; activations after weights; routing last.

Distributions (the five workloads of this library's benchmark and tests):
  * Q4_K: d, dmin = |N(0,1)| * 0.01 (f16); 6-bit scale and min codes uniform
    in 0..63 and 4-bit codes uniform in 0..15.  Every bit of the 12 scale/min
    bytes and of the 128 code bytes is used by exactly one field, so uniform
    fields are uniform random bytes.
  * Q5_K: as Q4_K, with d, dmin = |N(0,1)| * 0.005 and 32 uniform high-bit bytes (5-bit codes
    uniform in 0..31).
  * Q6_K: d = |N(0,1)| * 0.002 (f16); int8 scales uniform in -128..127;
    6-bit codes uniform in 0..63 (stored with an offset of 32): again uniform
    random ql/qh bytes.
  * Q8_0: d = |N(0,1)| * 0.005 (f16); int8 codes uniform in -127..127.
  * activations: fp32 N(0,1); with ``outliers`` each element independently
    (p = 0.01) is multiplied by 10.
  * routing: per token, ``top_k`` distinct experts drawn uniformly
    (partial Fisher-Yates), logits N(0,1) for the chosen ones, softmax
    weights over them (computed in f64, stored as fp32); slot order is the
    draw order.
"""
from __future__ import annotations

import numpy as np

Q4_K, Q6_K, Q8_0, Q8_K, Q8_1, Q5_K = 1, 2, 3, 4, 5, 6
NAMES = {Q4_K: "q4_k", Q5_K: "q5_k", Q6_K: "q6_k", Q8_0: "q8_0", Q8_K: "q8_k", Q8_1: "q8_1"}
BLOCK_ELEMS = {Q4_K: 256, Q5_K: 256, Q6_K: 256, Q8_0: 32, Q8_K: 256, Q8_1: 32}
BLOCK_BYTES = {Q4_K: 144, Q5_K: 176, Q6_K: 210, Q8_0: 34, Q8_K: 292, Q8_1: 36}


def rng(seed: int = 0) -> np.random.Generator:
    return np.random.default_rng(seed)


def _f16_bytes(v: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(v.astype(np.float16)).view(np.uint8).reshape(v.shape + (2,))


def q4_k_weights(N: int, K: int, g: np.random.Generator) -> np.ndarray:
    """Canonical Q4_K bytes [N, K/256*144]: d, dmin, 12 scale/min bytes, 128 code bytes."""
    assert K % 256 == 0
    nsb = K // 256
    d = np.abs(g.standard_normal((N, nsb))) * 0.01
    dmin = np.abs(g.standard_normal((N, nsb))) * 0.01
    sm = g.integers(0, 256, size=(N, nsb, 12), dtype=np.uint8)
    codes = g.integers(0, 256, size=(N, nsb, 128), dtype=np.uint8)
    blk = np.empty((N, nsb, 144), dtype=np.uint8)
    blk[..., 0:2] = _f16_bytes(d)
    blk[..., 2:4] = _f16_bytes(dmin)
    blk[..., 4:16] = sm
    blk[..., 16:144] = codes
    return blk.reshape(N, nsb * 144)


def q6_k_weights(N: int, K: int, g: np.random.Generator) -> np.ndarray:
    """Canonical Q6_K bytes [N, K/256*210]: ql[128], qh[64], int8 scales[16], d."""
    assert K % 256 == 0
    nsb = K // 256
    d = np.abs(g.standard_normal((N, nsb))) * 0.002
    scales = g.integers(0, 256, size=(N, nsb, 16), dtype=np.uint8)
    codes = g.integers(0, 256, size=(N, nsb, 192), dtype=np.uint8)
    blk = np.empty((N, nsb, 210), dtype=np.uint8)
    blk[..., 0:192] = codes
    blk[..., 192:208] = scales
    blk[..., 208:210] = _f16_bytes(d)
    return blk.reshape(N, nsb * 210)


def q8_0_weights(N: int, K: int, g: np.random.Generator) -> np.ndarray:
    """Canonical Q8_0 bytes [N, K/32*34]: d then int8[32] in -127..127."""
    assert K % 32 == 0
    nb = K // 32
    d = np.abs(g.standard_normal((N, nb))) * 0.005
    w = g.integers(-127, 128, size=(N, nb, 32), dtype=np.int16).astype(np.int8)
    blk = np.empty((N, nb, 34), dtype=np.uint8)
    blk[..., 0:2] = _f16_bytes(d)
    blk[..., 2:34] = w.view(np.uint8)
    return blk.reshape(N, nb * 34)


def q5_k_weights(N: int, K: int, g: np.random.Generator) -> np.ndarray:
    """Canonical Q5_K bytes [N, K/256*176]: d, dmin, 12 scale/min bytes, 32 high-bit bytes, 128 code bytes."""
    assert K % 256 == 0
    nsb = K // 256
    d = np.abs(g.standard_normal((N, nsb))) * 0.005
    dmin = np.abs(g.standard_normal((N, nsb))) * 0.005
    sm = g.integers(0, 256, size=(N, nsb, 12), dtype=np.uint8)
    qh = g.integers(0, 256, size=(N, nsb, 32), dtype=np.uint8)
    codes = g.integers(0, 256, size=(N, nsb, 128), dtype=np.uint8)
    blk = np.empty((N, nsb, 176), dtype=np.uint8)
    blk[..., 0:2] = _f16_bytes(d)
    blk[..., 2:4] = _f16_bytes(dmin)
    blk[..., 4:16] = sm
    blk[..., 16:48] = qh
    blk[..., 48:176] = codes
    return blk.reshape(N, nsb * 176)


def weights(dtype: int, N: int, K: int, g: np.random.Generator) -> np.ndarray:
    return {Q4_K: q4_k_weights, Q5_K: q5_k_weights, Q6_K: q6_k_weights, Q8_0: q8_0_weights}[dtype](N, K, g)


def activations(M: int, K: int, g: np.random.Generator, outliers: bool = False) -> np.ndarray:
    x = g.standard_normal((M, K)).astype(np.float32)
    if outliers:
        mask = g.random((M, K)) < 0.01
        x[mask] *= np.float32(10.0)
    return x


def routing(M: int, n_experts: int, top_k: int, g: np.random.Generator):
    """ids int32 [M, top_k] (distinct per token), weights fp32 [M, top_k] (softmax)."""
    ids = np.empty((M, top_k), dtype=np.int32)
    for t in range(M):
        perm = np.arange(n_experts)
        for k in range(top_k):               # partial Fisher-Yates
            j = int(g.integers(k, n_experts))
            perm[k], perm[j] = perm[j], perm[k]
        ids[t] = perm[:top_k]
    logits = g.standard_normal((M, top_k))
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    w = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, w


# Workload shapes (weight rows N x reduction K, tokens M).
TINY = dict(name="tiny_q4_k_gemm", dtype=Q4_K, N=256, K=1024, M=8)
DECODE = [dict(name="decode_q4_k_9728x2560", dtype=Q4_K, N=9728, K=2560),
          dict(name="decode_q4_k_2560x9728", dtype=Q4_K, N=2560, K=9728),
          dict(name="decode_q6_k_2560x9728", dtype=Q6_K, N=2560, K=9728)]
PREFILL_SHAPES = [(4096, 4096), (14336, 4096), (4096, 14336)]
PREFILL_M = [128, 512, 2048]
SWIGLU_Q8_0 = dict(name="swiglu_q8_0_2048x2560x9728", M=2048, N=2560, K=9728)
MOE = dict(name="moe_256x_top8_2048tok", n_experts=256, top_k=8, M=2048, hidden=2048, ffn=512)
