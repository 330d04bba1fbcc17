"""kq -- keep-quant int8 matmul for GB300 (sm_103a): Python binding of the C ABI in include/kq.h.

This module only marshals arguments: it turns torch tensors into device
pointers and the current torch stream into a ``cudaStream_t``, and calls the
``kq_*`` entry point of the same name in the in-tree CUDA library
(``_build/libkq.so``).  Every step of the computation runs in that library's
kernels; there is no CPU or PyTorch fallback.  If the library is missing the
import of any entry point raises ``KqLibraryMissing``.

Output buffers are allocated by the caller (PyTorch supplies device memory and
streams); sizes come from the geometry helpers (``native_bytes``,
``q8k_bytes``, ``q8_1_bytes``, ``gemm_workspace_bytes``).
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libkq.so")

Q4_K, Q6_K, Q8_0, Q8_K, Q8_1, Q5_K = 1, 2, 3, 4, 5, 6
DTYPES = {"q4_k": Q4_K, "q5_k": Q5_K, "q6_k": Q6_K, "q8_0": Q8_0, "q8_k": Q8_K, "q8_1": Q8_1}
STATUS = {0: "KQ_OK", 1: "KQ_ERR_INVALID_ARG", 2: "KQ_ERR_UNSUPPORTED_DTYPE", 3: "KQ_ERR_ALIGNMENT",
          4: "KQ_ERR_WORKSPACE", 5: "KQ_ERR_CUDA", 6: "KQ_ERR_DEVICE_FLAG"}


class KqLibraryMissing(RuntimeError):
    pass


class KqError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


_lock = threading.Lock()
_lib = None

_P, _I64, _I32, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
_SIGS = {
    "kq_status_string": ([_I32], ctypes.c_char_p),
    "kq_last_error": ([], ctypes.c_char_p),
    "kq_version": ([], _I32),
    "kq_block_elems": ([_I32], _I64),
    "kq_block_bytes": ([_I32], _I64),
    "kq_row_bytes": ([_I32, _I64], _I64),
    "kq_native_bytes": ([_I32, _I64, _I64], _I64),
    "kq_repack_weights": ([_I32, _P, _P, _I64, _I64, _P], _I32),
    "kq_quantize_q8k": ([_P, _I64, _I64, _I64, _P, _P], _I32),
    "kq_quantize_q8_1": ([_P, _I64, _I64, _I64, _P, _P], _I32),
    "kq_swiglu_quantize_q8_1": ([_P, _P, _I64, _I64, _I64, _P, _P, _P], _I32),
    "kq_swiglu_quantize_q8k": ([_P, _P, _I64, _I64, _I64, _P, _P, _P], _I32),
    "kq_rmsnorm_quantize_q8k": ([_P, _P, ctypes.c_float, _I64, _I64, _I64, _P, _P, _P], _I32),
    "kq_gemv": ([_I32, _P, _P, _P, _I64, _I64, _P, _P], _I32),
    "kq_gemm_workspace_bytes": ([_I32, _I64, _I64, _I64, _I64, _I64], _SZ),
    "kq_gemm": ([_I32, _P, _P, _I64, _I64, _I64, _P, _I64, _P, _SZ, _P], _I32),
    "kq_gemm_grouped": ([_I32, _P, _I64, _P, _I64, _P, _I64, _I64, _I64, _I64, _P, _P, _SZ, _P], _I32),
    "kq_read_device_flag": ([_P, ctypes.POINTER(_I64), _P], _I32),
    "kq_moe_weighted_sum": ([_P, _P, _I64, _I64, _I64, _P, _P], _I32),
    "kq_debug_partials": ([_I32, _P, _P, _I64, _I64, _I64, _P, _P], _I32),
    "kq_launch_count": ([ctypes.c_char_p], _I64),
    "kq_gemm_grouped_noalloc": ([_I32, _P, _I64, _P, _I64, _P, _I64, _I64, _I64, _I64, _P, _P], _I32),
    "kq_probe_int8_mma_sync": ([_I64, _P, ctypes.POINTER(ctypes.c_double), _P], _I32),
    "kq_gemm_f32_workspace_bytes": ([_I32, _I64, _I64, _I64], _SZ),
    "kq_gemm_f32": ([_I32, _P, _P, _I64, _I64, _I64, _I64, _P, _I64, _P, _SZ, _P], _I32),
    "kq_gemm_grouped_swiglu_workspace_bytes": ([_I32, _I64, _I64, _I64, _I64, _I64], _SZ),
    "kq_gemm_grouped_swiglu_q8k": ([_I32, _P, _I64, _P, _I64, _P, _I64, _I64, _I64, _I64, _P, _P, _SZ, _P], _I32),
    "kq_debug_tc_splits": ([_I32, _I64, _I64, _I64], _I32),
    "kq_gemm_ex": ([_I32, _P, _P, _I64, _I64, _I64, _P, _I64, ctypes.c_uint, _P, _SZ, _P], _I32),
    "kq_gemm_f32_ex": ([_I32, _P, _P, _I64, _I64, _I64, _I64, _P, _I64, ctypes.c_uint, _P, _SZ, _P], _I32),
    "kq_debug_tc_sums": ([_I32, _P, _P, _I64, _I64, _I64, _P, _I64, _P, _P, _SZ, _P], _I32),
    "kq_debug_tc_sums_grouped": ([_I32, _P, _I64, _P, _I64, _P, _I64, _I64, _I64, _I64, _P, _P, _P, _SZ, _P], _I32),
    "kq_debug_tc_wait_timeout": ([_I32, _P, _P, _I64, _I64, _I64, _P, _I64, _I64, _P, _SZ, _P], _I32),
}


def lib():
    """The loaded CUDA library (ctypes handle).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise KqLibraryMissing(f"{LIB_PATH} is missing: build it with "
                                       "`python -m gemv_quantize_q8_gb300.build` (nvcc, sm_103a)")
            L = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in _SIGS.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
        return _lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check(status: int) -> None:
    if status != 0:
        raise KqError(status, lib().kq_last_error().decode())


# ----------------------------------------------------------------------------- geometry
def block_elems(dtype: int) -> int:
    return int(lib().kq_block_elems(dtype))


def block_bytes(dtype: int) -> int:
    return int(lib().kq_block_bytes(dtype))


def row_bytes(dtype: int, K: int) -> int:
    return int(lib().kq_row_bytes(dtype, K))


def native_bytes(dtype: int, N: int, K: int) -> int:
    return int(lib().kq_native_bytes(dtype, N, K))


def q8k_bytes(M: int, K: int) -> int:
    return M * (K // 256) * 292


def q8_1_bytes(M: int, K: int) -> int:
    return M * (K // 32) * 36


def gemm_workspace_bytes(dtype: int, M: int, N: int, K: int, n_experts: int = 0, top_k: int = 0) -> int:
    return int(lib().kq_gemm_workspace_bytes(dtype, M, N, K, n_experts, top_k))


def version() -> int:
    return int(lib().kq_version())


def launch_count(route: str | None = None) -> int:
    """Kernel launches made by the library since load (all routes, or one route)."""
    return int(lib().kq_launch_count(route.encode() if route else None))


# ----------------------------------------------------------------------------- entry points
def kq_repack_weights(dtype, w_canon, w_native, N, K, stream=None):
    _check(lib().kq_repack_weights(dtype, _ptr(w_canon), _ptr(w_native), N, K, _stream(stream)))


def kq_quantize_q8k(x, M, K, ldx, xq, stream=None):
    _check(lib().kq_quantize_q8k(_ptr(x), M, K, ldx, _ptr(xq), _stream(stream)))


def kq_quantize_q8_1(x, M, K, ldx, xq, stream=None):
    _check(lib().kq_quantize_q8_1(_ptr(x), M, K, ldx, _ptr(xq), _stream(stream)))


def kq_swiglu_quantize_q8_1(g, u, M, K, ld, xq, h_out=None, stream=None):
    _check(lib().kq_swiglu_quantize_q8_1(_ptr(g), _ptr(u), M, K, ld, _ptr(xq), _ptr(h_out), _stream(stream)))


def kq_swiglu_quantize_q8k(g, u, M, K, ld, xq, h_out=None, stream=None):
    _check(lib().kq_swiglu_quantize_q8k(_ptr(g), _ptr(u), M, K, ld, _ptr(xq), _ptr(h_out), _stream(stream)))


def kq_rmsnorm_quantize_q8k(x, gamma, eps, M, K, ldx, xq, y_out=None, stream=None):
    _check(lib().kq_rmsnorm_quantize_q8k(_ptr(x), _ptr(gamma), float(eps), M, K, ldx, _ptr(xq), _ptr(y_out),
                                         _stream(stream)))


def kq_gemv(wt, w, x, xq, N, K, y, stream=None):
    _check(lib().kq_gemv(wt, _ptr(w), _ptr(x), _ptr(xq), N, K, _ptr(y), _stream(stream)))


def kq_gemm(wt, w, xq, M, N, K, y, ldy, workspace=None, ws_bytes=0, stream=None):
    _check(lib().kq_gemm(wt, _ptr(w), _ptr(xq), M, N, K, _ptr(y), ldy, _ptr(workspace), ws_bytes, _stream(stream)))


GEMM_FOLD_SCALES = 1


def kq_gemm_ex(wt, w, xq, M, N, K, y, ldy, flags, workspace=None, ws_bytes=0, stream=None):
    """kq_gemm with options (flags: GEMM_FOLD_SCALES folds the Q8_0 block scales into the f16 operands)."""
    _check(lib().kq_gemm_ex(wt, _ptr(w), _ptr(xq), M, N, K, _ptr(y), ldy, flags, _ptr(workspace), ws_bytes,
                            _stream(stream)))


def kq_gemm_f32_ex(wt, w, x, ldx, M, N, K, y, ldy, flags, workspace, ws_bytes, stream=None):
    """kq_gemm_f32 with kq_gemm_ex's flags (GEMM_FOLD_SCALES: the folded mode, quantised in its prologue)."""
    _check(lib().kq_gemm_f32_ex(wt, _ptr(w), _ptr(x), ldx, M, N, K, _ptr(y), ldy, flags, _ptr(workspace), ws_bytes,
                                _stream(stream)))


def kq_gemm_f32_workspace_bytes(wt, M, N, K) -> int:
    return int(lib().kq_gemm_f32_workspace_bytes(wt, M, N, K))


def kq_gemm_f32(wt, w, x, ldx, M, N, K, y, ldy, workspace, ws_bytes, stream=None):
    """kq_gemm from fp32 rows: the activation quantiser runs inside the GEMM's prologue."""
    _check(lib().kq_gemm_f32(wt, _ptr(w), _ptr(x), ldx, M, N, K, _ptr(y), ldy, _ptr(workspace), ws_bytes,
                             _stream(stream)))


def kq_gemm_grouped(wt, w, n_experts, xq, xq_rows_per_token, ids, M, top_k, N, K, y, workspace, ws_bytes,
                    stream=None):
    _check(lib().kq_gemm_grouped(wt, _ptr(w), n_experts, _ptr(xq), xq_rows_per_token, _ptr(ids), M, top_k, N, K,
                                 _ptr(y), _ptr(workspace), ws_bytes, _stream(stream)))


def kq_gemm_grouped_swiglu_workspace_bytes(wt, M, F, K, n_experts, top_k) -> int:
    return int(lib().kq_gemm_grouped_swiglu_workspace_bytes(wt, M, F, K, n_experts, top_k))


def kq_gemm_grouped_swiglu_q8k(wt, w, n_experts, xq, xq_rows_per_token, ids, M, top_k, F, K, hq, workspace, ws_bytes,
                               stream=None):
    """Routed gate/up GEMM whose epilogue writes Q8_K rows of silu(gate)*up to hq (no fp32 rows)."""
    _check(lib().kq_gemm_grouped_swiglu_q8k(wt, _ptr(w), n_experts, _ptr(xq), xq_rows_per_token, _ptr(ids), M, top_k,
                                            F, K, _ptr(hq), _ptr(workspace), ws_bytes, _stream(stream)))


def kq_gemm_grouped_noalloc(wt, w, n_experts, xq, xq_rows_per_token, ids, M, top_k, N, K, y, stream=None):
    """kq_gemm_grouped for callers that cannot allocate: routing scratch is a fixed array inside the library."""
    _check(lib().kq_gemm_grouped_noalloc(wt, _ptr(w), n_experts, _ptr(xq), xq_rows_per_token, _ptr(ids), M, top_k,
                                         N, K, _ptr(y), _stream(stream)))


def kq_probe_int8_mma_sync(iters, sink, stream=None) -> float:
    """Launch the int8 mma.sync throughput probe; returns the int8 ops it issues (time it with events)."""
    ops = ctypes.c_double(0.0)
    _check(lib().kq_probe_int8_mma_sync(iters, _ptr(sink), ctypes.byref(ops), _stream(stream)))
    return ops.value


def kq_read_device_flag(workspace, stream=None) -> int:
    """Returns the number of invalid (token, slot) ids recorded; raises KqError on KQ_ERR_CUDA."""
    n = _I64(0)
    st = lib().kq_read_device_flag(_ptr(workspace), ctypes.byref(n), _stream(stream))
    if st not in (0, 6):
        _check(st)
    return int(n.value)


def kq_moe_weighted_sum(y_slots, w, M, top_k, N, out, stream=None):
    _check(lib().kq_moe_weighted_sum(_ptr(y_slots), _ptr(w), M, top_k, N, _ptr(out), _stream(stream)))


def kq_debug_partials(wt, w, xq, M, N, K, partials, stream=None):
    _check(lib().kq_debug_partials(wt, _ptr(w), _ptr(xq), M, N, K, _ptr(partials), _stream(stream)))


def kq_debug_tc_splits(wt, M, N, K) -> int:
    """Split-K factor of the tensor-core path for this shape on the current device (0: not that path)."""
    return int(lib().kq_debug_tc_splits(wt, M, N, K))


def kq_debug_tc_sums(wt, w, xq, M, N, K, y, ldy, sums, workspace=None, ws_bytes=0, stream=None):
    """kq_gemm's tensor-core kernel, also writing the integer sums of every scale block (int32 [M][N][nblk][2])."""
    _check(lib().kq_debug_tc_sums(wt, _ptr(w), _ptr(xq), M, N, K, _ptr(y), ldy, _ptr(sums), _ptr(workspace), ws_bytes,
                                  _stream(stream)))


def kq_debug_tc_sums_grouped(wt, w, n_experts, xq, xq_rows_per_token, ids, M, top_k, N, K, y, sums, workspace,
                             ws_bytes, stream=None):
    """kq_gemm_grouped's tensor-core kernel, also writing the integer block sums of every (token, slot) row."""
    _check(lib().kq_debug_tc_sums_grouped(wt, _ptr(w), n_experts, _ptr(xq), xq_rows_per_token, _ptr(ids), M, top_k,
                                          N, K, _ptr(y), _ptr(sums), _ptr(workspace), ws_bytes, _stream(stream)))


def kq_debug_tc_wait_timeout(wt, w, xq, M, N, K, y, ldy, wait_limit_ns, workspace, ws_bytes, stream=None):
    """The tensor-core kernel with its activation producer idle and every wait limited to wait_limit_ns."""
    _check(lib().kq_debug_tc_wait_timeout(wt, _ptr(w), _ptr(xq), M, N, K, _ptr(y), ldy, wait_limit_ns,
                                          _ptr(workspace), ws_bytes, _stream(stream)))
