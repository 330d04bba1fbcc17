"""Helpers for the GPU parity tests: device copies and thin wrappers around the C ABI."""
import numpy as np
import torch

import gemv_quantize_q8_gb300 as kq

DEV = "cuda:0"


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def host(t: torch.Tensor) -> np.ndarray:
    torch.cuda.synchronize()
    return t.cpu().numpy()


def repack(dtype: int, w_canon: np.ndarray, N: int, K: int) -> torch.Tensor:
    src = dev(w_canon.reshape(-1))
    dst = torch.empty(kq.native_bytes(dtype, N, K), dtype=torch.uint8, device=DEV)
    kq.kq_repack_weights(dtype, src, dst, N, K)
    torch.cuda.synchronize()   # weights are staged once, before any matmul reads them
    return dst


def q8k(x: torch.Tensor, M: int, K: int, ld: int | None = None) -> torch.Tensor:
    out = torch.full((kq.q8k_bytes(M, K),), 0xAB, dtype=torch.uint8, device=DEV)
    kq.kq_quantize_q8k(x, M, K, ld or K, out)
    return out


def q8_1(x: torch.Tensor, M: int, K: int, ld: int | None = None) -> torch.Tensor:
    out = torch.full((kq.q8_1_bytes(M, K),), 0xAB, dtype=torch.uint8, device=DEV)
    kq.kq_quantize_q8_1(x, M, K, ld or K, out)
    return out


def act_quant(dtype: int, x: torch.Tensor, M: int, K: int) -> torch.Tensor:
    return q8_1(x, M, K) if dtype == kq.Q8_0 else q8k(x, M, K)


def gemm(dtype: int, w_native: torch.Tensor, xq: torch.Tensor, M: int, N: int, K: int) -> torch.Tensor:
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
    wsb = kq.gemm_workspace_bytes(dtype, M, N, K)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=DEV) if wsb else None
    kq.kq_gemm(dtype, w_native, xq, M, N, K, y, N, ws, wsb)
    if wsb:
        assert kq.kq_read_device_flag(ws) == 0, "tensor-core pipeline reported a timeout"
    return y


def nmse(y: np.ndarray, ref: np.ndarray) -> float:
    y = y.astype(np.float64)
    ref = ref.astype(np.float64)
    return float(((y - ref) ** 2).sum() / max((ref ** 2).sum(), 1e-300))
