"""The C-ABI library loads and exports every symbol include/kq.h declares (no GPU calls)."""
import os
import re
import subprocess

import pytest

import gemv_quantize_q8_gb300 as kq
from gemv_quantize_q8_gb300 import build as kqbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "kq.h")).read()
    return sorted(set(re.findall(r"^KQ_API [^(]*?\b(kq_\w+)\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def built():
    return kqbuild.build()


def test_header_declares_the_boundary():
    names = _declared()
    for fn in ["kq_quantize_q8k", "kq_quantize_q8_1", "kq_gemv", "kq_gemm", "kq_gemm_grouped",
               "kq_repack_weights", "kq_debug_partials", "kq_moe_weighted_sum", "kq_swiglu_quantize_q8_1"]:
        assert fn in names


def test_library_exports_every_declared_symbol(built):
    out = subprocess.run(["nm", "-D", "--defined-only", built], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r" T (kq_\w+)$", out, flags=re.M))
    missing = [n for n in _declared() if n not in exported]
    assert not missing, missing


def test_binding_covers_every_symbol_and_loads(built):
    L = kq.lib()
    for name in _declared():
        assert hasattr(L, name)
        assert name in kq._SIGS, f"binding has no signature for {name}"
    assert kq.version() >= 100
    # pure host queries (no device work)
    assert kq.block_bytes(kq.Q4_K) == 144 and kq.block_bytes(kq.Q6_K) == 210 and kq.block_bytes(kq.Q8_0) == 34
    assert kq.row_bytes(kq.Q4_K, 2560) == 10 * 144
    assert kq.native_bytes(kq.Q4_K, 9728, 2560) == 9728 * 10 * 144
    assert kq.native_bytes(kq.Q6_K, 17, 256) == 2 * 3360          # rows padded to a multiple of 16
    assert kq.block_bytes(kq.Q5_K) == 176 and kq.row_bytes(kq.Q5_K, 512) == 2 * 176
    assert kq.native_bytes(kq.Q5_K, 17, 256) == 2 * 2816          # Q4_K chunk + 32 high-bit bytes per row
    assert kq.native_bytes(kq.Q8_0, 16, 1024) == 4 * 4352
    assert kq.native_bytes(kq.Q8_0, 16, 100) == 0


def test_host_validation_errors_without_gpu(built):
    """Argument errors are returned before any CUDA call, naming the problem."""
    L = kq.lib()
    st = L.kq_gemm(7, 16, 16, 8, 256, 1024, 16, 256, None, 0, None)
    assert st == 2 and b"not Q4_K" in L.kq_last_error()
    st = L.kq_gemv(kq.Q4_K, 16, 16, 16, 256, 1000, 16, None)
    assert st == 1
    st = L.kq_quantize_q8k(None, 1, 256, 256, 16, None)
    assert st == 1
    st = L.kq_gemm(kq.Q4_K, 8, 16, 8, 256, 1024, 16, 256, None, 0, None)   # w not 16-byte aligned
    assert st == 3
    st = L.kq_gemm_grouped(kq.Q4_K, 16, 4, 16, 3, 16, 8, 2, 256, 1024, 16, 256, 1 << 20, None)
    assert st == 1 and b"xq_rows_per_token" in L.kq_last_error()
    st = L.kq_gemm_grouped(kq.Q4_K, 16, 4, 16, 1, 16, 8, 2, 256, 1024, 16, 256, 16, None)
    assert st == 4
    assert L.kq_status_string(6) == b"device reported invalid input"
    # fused SwiGLU epilogue: F must be a positive multiple of 256, hq non-NULL (checked before any launch)
    st = L.kq_gemm_grouped_swiglu_q8k(kq.Q4_K, 16, 4, 16, 1, 16, 8, 2, 128, 1024, 16, 16, 1 << 20, None)
    assert st == 1 and b"multiple of 256" in L.kq_last_error()
    st = L.kq_gemm_grouped_swiglu_q8k(kq.Q4_K, 16, 4, 16, 1, 16, 8, 2, 256, 1024, None, 16, 1 << 20, None)
    assert st == 1 and b"null hq" in L.kq_last_error()
    st = L.kq_gemm_grouped_swiglu_q8k(kq.Q8_K, 16, 4, 16, 1, 16, 8, 2, 256, 1024, 16, 16, 1 << 20, None)
    assert st in (1, 2)
    # RMSNorm producer: K a multiple of 256, eps finite and >= 0
    st = L.kq_rmsnorm_quantize_q8k(16, 16, 1e-6, 1, 300, 300, 16, None, None)
    assert st == 1
    st = L.kq_rmsnorm_quantize_q8k(16, 16, -1.0, 1, 256, 256, 16, None, None)
    assert st == 1 and b"eps" in L.kq_last_error()
    # fp32-input GEMM: ldx >= K, a supported weight type, a workspace of the size it asks for
    st = L.kq_gemm_f32(kq.Q4_K, 16, 16, 1000, 160, 256, 1024, 16, 256, 16, 1 << 30, None)
    assert st == 1 and b"ldx" in L.kq_last_error()
    st = L.kq_gemm_f32(kq.Q8_K, 16, 16, 1024, 160, 256, 1024, 16, 256, 16, 1 << 30, None)
    assert st == 2
    need = L.kq_gemm_f32_workspace_bytes(kq.Q4_K, 160, 256, 1024)
    assert need >= 256 + 160 * 4 * 292
    st = L.kq_gemm_f32(kq.Q4_K, 16, 16, 1024, 160, 256, 1024, 16, 256, 256, need - 1, None)
    assert st == 4
    # int8 probe: iters must be positive
    assert L.kq_probe_int8_mma_sync(0, 16, None, None) == 1
    # debug twins of the tensor-core path: same argument checks, and only tensor-core shapes
    st = L.kq_debug_tc_sums(kq.Q4_K, 16, 16, 8, 256, 1024, 16, 256, 16, 256, 1 << 30, None)
    assert st == 1 and b"tensor-core" in L.kq_last_error()          # M = 8 is the batched-decode path
    st = L.kq_debug_tc_sums(kq.Q4_K, 16, 16, 256, 256, 1024, 16, 256, None, 256, 1 << 30, None)
    assert st == 1 and b"sums" in L.kq_last_error()
    st = L.kq_debug_tc_wait_timeout(kq.Q4_K, 16, 16, 256, 256, 1024, 16, 256, 10, 256, 1 << 30, None)
    assert st == 1 and b"wait_limit_ns" in L.kq_last_error()
    st = L.kq_debug_tc_sums_grouped(kq.Q4_K, 16, 4, 16, 1, 16, 8, 2, 256, 1024, 16, None, 256, 1 << 20, None)
    assert st == 1


def test_split_factor_host_logic(built):
    """The split-K choice is host logic: 0 off the tensor-core path, 1 for Q8_0 (one ascending sum per
    output), a power of two up to 8 that leaves at least two super-blocks per cluster rank, and a split
    for the few-tile long-K shapes (two 128-row tiles over K = 4096: nothing else fills the SMs)."""
    assert kq.kq_debug_tc_splits(kq.Q4_K, 8, 256, 4096) == 0       # batched decode
    assert kq.kq_debug_tc_splits(kq.Q4_K, 256, 64, 4096) == 0      # N < 128
    assert kq.kq_debug_tc_splits(kq.Q8_0, 128, 256, 4096) == 1
    for dt in (kq.Q4_K, kq.Q5_K, kq.Q6_K):
        for (M, N, K) in [(128, 256, 4096), (128, 4096, 4096), (512, 4096, 14336), (2048, 14336, 4096), (130, 200, 768)]:
            S = kq.kq_debug_tc_splits(dt, M, N, K)
            assert S in (1, 2, 4, 8)
            assert S == 1 or -(-(K // 256) // S) >= 2      # at least two super-blocks per rank
        assert kq.kq_debug_tc_splits(dt, 128, 256, 4096) > 1
        assert kq.kq_debug_tc_splits(dt, 2048, 14336, 4096) == 1    # 1792 tiles fill the SMs many times
