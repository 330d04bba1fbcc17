"""CPU oracle for the keep-quant matmul path (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, loads or calls it, and it shares no code
with that path: the oracle is plain C (``kq_oracle.c``) compiled with gcc and
``-ffp-contract=off``, wrapped here with ctypes and numpy.

Canonical (GGUF-style) block layouts are used throughout; see ``kq_oracle.c``
for the byte layouts and the passages each function follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kq_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD_DIR, "libkq_oracle.so")

Q4_K, Q6_K, Q8_0, Q8_K, Q8_1, Q5_K = 1, 2, 3, 4, 5, 6
BLOCK_ELEMS = {Q4_K: 256, Q5_K: 256, Q6_K: 256, Q8_0: 32, Q8_K: 256, Q8_1: 32}
BLOCK_BYTES = {Q4_K: 144, Q5_K: 176, Q6_K: 210, Q8_0: 34, Q8_K: 292, Q8_1: 36}
ACT_DTYPE = {Q4_K: Q8_K, Q5_K: Q8_K, Q6_K: Q8_K, Q8_0: Q8_1}
SUBBLOCK = {Q4_K: 32, Q5_K: 32, Q6_K: 16, Q8_0: 32}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available). Returns the .so path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
            "-fvisibility=hidden", SRC, "-o", LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            # KQ_ORACLE_LIB: a differently built copy of this same oracle (the mutation test compiles
            # deliberately broken copies and runs the pins against them)
            path = os.environ.get("KQ_ORACLE_LIB") or build()
            L = ctypes.CDLL(path)
            P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            L.orc_half_to_float.argtypes = [ctypes.c_uint16]
            L.orc_half_to_float.restype = ctypes.c_float
            L.orc_float_to_half.argtypes = [ctypes.c_float]
            L.orc_float_to_half.restype = ctypes.c_uint16
            for name in ("orc_dequant_q4_k", "orc_dequant_q5_k", "orc_dequant_q6_k", "orc_dequant_q8_0",
                         "orc_dequant_q8_k", "orc_dequant_q8_1"):
                getattr(L, name).argtypes = [P, P]
                getattr(L, name).restype = None
            L.orc_quantize_q8_k.argtypes = [P, I64, I64, I64, P]
            L.orc_quantize_q8_1.argtypes = [P, I64, I64, I64, P]
            L.orc_swiglu.argtypes = [P, P, I64, I64, I64, P, I64]
            L.orc_rmsnorm.argtypes = [P, P, ctypes.c_float, I64, I64, I64, P, I64]
            L.orc_partials_row.argtypes = [I32, P, P, I64, P]
            L.orc_dot_row.argtypes = [I32, P, P, I64]
            L.orc_dot_row.restype = ctypes.c_float
            L.orc_gemm.argtypes = [I32, P, P, I64, I64, I64, P, I64, I32]
            L.orc_gemm_sampled.argtypes = [I32, P, P, I64, I64, P, P, P]
            L.orc_partials.argtypes = [I32, P, P, I64, I64, I64, P]
            L.orc_gemm_sampled_terms.argtypes = [I32, P, P, I64, I64, P, P, P, P]
            L.orc_block_sums.argtypes = [I32, P, P, I64, I64, I64, P, I32]
            L.orc_absdot_sampled.argtypes = [I32, P, P, I64, I64, P, P, P]
            L.orc_gemm_grouped.argtypes = [I32, P, I64, P, I64, P, I64, I64, I64, I64, P, I32]
            L.orc_gemm_grouped.restype = I64
            L.orc_moe_weighted_sum.argtypes = [P, P, I64, I64, I64, P]
            L.orc_max_threads.restype = I32
            _lib = L
        return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def max_threads() -> int:
    return int(lib().orc_max_threads())


def half_to_float(h: int) -> float:
    return float(lib().orc_half_to_float(int(h)))


def float_to_half(f: float) -> int:
    return int(lib().orc_float_to_half(float(f)))


def dequant(dtype: int, blocks: np.ndarray) -> np.ndarray:
    """Dequantise a flat byte array of whole blocks into f64 values."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1)
    bb, be = BLOCK_BYTES[dtype], BLOCK_ELEMS[dtype]
    nb = blocks.size // bb
    assert nb * bb == blocks.size
    out = np.empty(nb * be, dtype=np.float64)
    fn = {Q4_K: "orc_dequant_q4_k", Q5_K: "orc_dequant_q5_k", Q6_K: "orc_dequant_q6_k", Q8_0: "orc_dequant_q8_0",
          Q8_K: "orc_dequant_q8_k", Q8_1: "orc_dequant_q8_1"}[dtype]
    f = getattr(lib(), fn)
    base = _ptr(blocks)
    obase = _ptr(out)
    for b in range(nb):
        f(base + b * bb, obase + b * be * 8)
    return out


def quantize_q8_k(x: np.ndarray) -> np.ndarray:
    """fp32 [M, K] -> Q8_K bytes [M, K/256 * 292]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    M, K = x.shape
    assert K % 256 == 0
    out = np.empty((M, K // 256 * 292), dtype=np.uint8)
    lib().orc_quantize_q8_k(_ptr(x), M, K, K, _ptr(out))
    return out


def quantize_q8_1(x: np.ndarray) -> np.ndarray:
    """fp32 [M, K] -> Q8_1 bytes [M, K/32 * 36]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    M, K = x.shape
    assert K % 32 == 0
    out = np.empty((M, K // 32 * 36), dtype=np.uint8)
    lib().orc_quantize_q8_1(_ptr(x), M, K, K, _ptr(out))
    return out


def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """y = (x * r) * gamma, r = 1 / sqrt(sum(x^2) / K + eps), fp32, the sum of squares in ascending order."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    gamma = np.ascontiguousarray(gamma, dtype=np.float32)
    M, K = x.shape
    assert gamma.shape == (K,)
    y = np.empty((M, K), dtype=np.float32)
    lib().orc_rmsnorm(_ptr(x), _ptr(gamma), float(np.float32(eps)), M, K, K, _ptr(y), K)
    return y


def rmsnorm_quantize_q8_k(x: np.ndarray, gamma: np.ndarray, eps: float):
    """The fused norm-quant producer: (Q8_K bytes of the normalized rows, the normalized rows)."""
    y = rmsnorm(x, gamma, eps)
    return quantize_q8_k(y), y


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """h = silu(g) * u in fp32."""
    g = np.ascontiguousarray(g, dtype=np.float32)
    u = np.ascontiguousarray(u, dtype=np.float32)
    M, K = g.shape
    h = np.empty((M, K), dtype=np.float32)
    lib().orc_swiglu(_ptr(g), _ptr(u), M, K, K, _ptr(h), K)
    return h


def _check_gemm_args(dtype, w, xq, N, K):
    w = np.ascontiguousarray(w, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    assert w.size == N * (K // BLOCK_ELEMS[dtype]) * BLOCK_BYTES[dtype], "weight size mismatch"
    return w, xq


def gemm(dtype: int, w: np.ndarray, xq: np.ndarray, M: int, N: int, K: int, threads: int = 0) -> np.ndarray:
    """y[m, n] = dot(W row n, X row m) in the fixed block order; fp32 [M, N]."""
    w, xq = _check_gemm_args(dtype, w, xq, N, K)
    y = np.empty((M, N), dtype=np.float32)
    lib().orc_gemm(dtype, _ptr(w), _ptr(xq), M, N, K, _ptr(y), N, threads or max_threads())
    return y


def gemm_sampled(dtype: int, w: np.ndarray, xq: np.ndarray, K: int, m_idx, n_idx) -> np.ndarray:
    w = np.ascontiguousarray(w, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    mi = np.ascontiguousarray(m_idx, dtype=np.int64)
    ni = np.ascontiguousarray(n_idx, dtype=np.int64)
    out = np.empty(mi.size, dtype=np.float32)
    lib().orc_gemm_sampled(dtype, _ptr(w), _ptr(xq), K, mi.size, _ptr(mi), _ptr(ni), _ptr(out))
    return out


def gemm_sampled_terms(dtype: int, w: np.ndarray, xq: np.ndarray, K: int, m_idx, n_idx):
    """Sampled outputs and, per output, the f64 sum over blocks of |(d_a*d_w)*sumi| + |(d_a*dmin)*summ|
    (the magnitude that any order of the fp32 block scaling rounds against)."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    mi = np.ascontiguousarray(m_idx, dtype=np.int64)
    ni = np.ascontiguousarray(n_idx, dtype=np.int64)
    out = np.empty(mi.size, dtype=np.float32)
    terms = np.empty(mi.size, dtype=np.float64)
    lib().orc_gemm_sampled_terms(dtype, _ptr(w), _ptr(xq), K, mi.size, _ptr(mi), _ptr(ni), _ptr(out), _ptr(terms))
    return out, terms


def absdot_sampled(dtype: int, w: np.ndarray, xq: np.ndarray, K: int, m_idx, n_idx) -> np.ndarray:
    """f64 [S, 4]: for each sampled (m, n) over the dequantised weight row a and activation row b:
    sum |a_i*b_i|, sum |a_i|, sum |b_i|, and sum (|d*sc*c_i| + |dmin*m_i|)*|b_i| (the weight's two parts
    apart; the first sum again for Q6_K and Q8_0)."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    mi = np.ascontiguousarray(m_idx, dtype=np.int64)
    ni = np.ascontiguousarray(n_idx, dtype=np.int64)
    out = np.empty((mi.size, 4), dtype=np.float64)
    lib().orc_absdot_sampled(dtype, _ptr(w), _ptr(xq), K, mi.size, _ptr(mi), _ptr(ni), _ptr(out))
    return out


def block_sums(dtype: int, w: np.ndarray, xq: np.ndarray, M: int, N: int, K: int, threads: int = 0) -> np.ndarray:
    """int64 [M, N, nblk, 2]: per scale block (256 elements; Q8_0: 32) the integer sums the keep-quant
    formula scales -- (sum_j sc_j*P_j, sum_j m_j*(bs_2j + bs_2j+1)) for Q4_K/Q5_K, (sum_j sc_j*P_j, 0)
    for Q6_K, (P_b, 0) for Q8_0."""
    w, xq = _check_gemm_args(dtype, w, xq, N, K)
    nblk = K // BLOCK_ELEMS[dtype]
    out = np.empty((M, N, nblk, 2), dtype=np.int64)
    lib().orc_block_sums(dtype, _ptr(w), _ptr(xq), M, N, K, _ptr(out), threads or max_threads())
    return out


def partials(dtype: int, w: np.ndarray, xq: np.ndarray, M: int, N: int, K: int) -> np.ndarray:
    """int32 [M, N, K/subblock] integer sub-block dots."""
    w, xq = _check_gemm_args(dtype, w, xq, N, K)
    out = np.empty((M, N, K // SUBBLOCK[dtype]), dtype=np.int32)
    lib().orc_partials(dtype, _ptr(w), _ptr(xq), M, N, K, _ptr(out))
    return out


def gemm_grouped(dtype: int, w: np.ndarray, n_experts: int, xq: np.ndarray, rows_per_token: int,
                 ids: np.ndarray, M: int, top_k: int, N: int, K: int, y: np.ndarray | None = None,
                 threads: int = 0):
    """Routed-expert GEMM. Returns (y [M, top_k, N], number of invalid ids)."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    if y is None:
        y = np.full((M, top_k, N), np.nan, dtype=np.float32)
    bad = lib().orc_gemm_grouped(dtype, _ptr(w), n_experts, _ptr(xq), rows_per_token, _ptr(ids), M, top_k, N, K,
                                 _ptr(y), threads or max_threads())
    return y, int(bad)


def moe_weighted_sum(y_slots: np.ndarray, wts: np.ndarray) -> np.ndarray:
    y_slots = np.ascontiguousarray(y_slots, dtype=np.float32)
    wts = np.ascontiguousarray(wts, dtype=np.float32)
    M, top_k, N = y_slots.shape
    out = np.empty((M, N), dtype=np.float32)
    lib().orc_moe_weighted_sum(_ptr(y_slots), _ptr(wts), M, top_k, N, _ptr(out))
    return out
