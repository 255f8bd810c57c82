"""Host-side checks of the C-ABI library that need no GPU.

The library must load, export every function include/q4k.h declares, and reject
bad arguments with the documented status before it touches a device.
"""
import os
import re

import pytest
import torch

import q4_weight_quantized_gb300 as q4k
from q4_weight_quantized_gb300.build import build_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_library()
    return q4k.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "q4k.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(q4k_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 13
    assert sorted(q4k.EXPORTS) == names
    for n in names:
        assert hasattr(lib, n), n


def test_row_bytes_and_strings(lib):
    assert q4k.q4k_row_bytes(256) == 144
    assert q4k.q4k_row_bytes(5120) == 20 * 144
    assert q4k.q4k_row_bytes(17408) == 68 * 144
    assert q4k.q4k_row_bytes(100) == 0 and q4k.q4k_row_bytes(0) == 0 and q4k.q4k_row_bytes(-256) == 0
    for s in range(0, 10):
        assert isinstance(q4k.status_string(s), str) and q4k.status_string(s)
    # every status the header declares has its own text (9: unknown)
    texts = [q4k.status_string(s) for s in range(0, 9)]
    assert len(set(texts)) == 9 and q4k.status_string(9) == "unknown status"
    src = open(os.path.join(ROOT, "include", "q4k.h")).read()
    assert "Q4K_ERR_ROUTING = 8" in src and q4k.Q4K_ERR_ROUTING == 8
    assert q4k.q4k_version() >= 100


def test_workspace_sizes(lib):
    assert q4k.q4k_moe_workspace_size(0, 768, 2048, 16, 8, 0) == 0          # bad E
    a = q4k.q4k_moe_workspace_size(128, 768, 2048, 16, 8, q4k.Q4K_MOE_Y_PER_SLOT)
    b = q4k.q4k_moe_workspace_size(128, 2048, 768, 16, 8, q4k.Q4K_MOE_Y_COMBINE)
    assert a >= (129 + 128) * 4 and a % 256 == 0
    assert b >= a + 16 * 8 * 2048 * 4
    assert q4k.q4k_gemm_workspace_size(1, 17408, 5120) >= 0
    # expert FFN: routing + g (fp32) + h (bf16) + per-slot outputs (fp32); + sorted x from 32*E items
    assert q4k.q4k_moe_ffn_workspace_size(128, 768, 2000, 16, 8) == 0       # D not a multiple of 256
    assert q4k.q4k_moe_ffn_workspace_size(128, 700, 2048, 16, 8) == 0       # H not a multiple of 256
    f = q4k.q4k_moe_ffn_workspace_size(128, 768, 2048, 16, 8)
    n = 16 * 8
    assert f % 256 == 0 and f >= (129 + n) * 4 + n * 768 * 6 + n * 2048 * 4
    big = q4k.q4k_moe_ffn_workspace_size(128, 768, 2048, 4096, 8)
    n = 4096 * 8
    assert big >= n * 768 * 6 + n * 2048 * 6


A16 = 1 << 20  # a 16-byte aligned fake address; never dereferenced by these calls


@pytest.mark.parametrize("call,status", [
    (lambda L: L.q4k_dequant(None, 4, 256, A16, None), q4k.Q4K_ERR_NULL),
    (lambda L: L.q4k_dequant(A16, 4, 300, A16, None), q4k.Q4K_ERR_SHAPE),
    (lambda L: L.q4k_dequant(A16, 0, 256, A16, None), q4k.Q4K_ERR_SHAPE),
    (lambda L: L.q4k_dequant(A16 + 8, 4, 256, A16, None), q4k.Q4K_ERR_ALIGN),
    (lambda L: L.q4k_dequant_bf16(A16, 4, 256, A16 + 2, None), q4k.Q4K_ERR_ALIGN),
    (lambda L: L.q4k_gemv(A16, 4, 256, None, A16, None), q4k.Q4K_ERR_NULL),
    (lambda L: L.q4k_gemv(A16, 4, 255, A16, A16, None), q4k.Q4K_ERR_SHAPE),
    (lambda L: L.q4k_gemm(A16, 4, 256, A16, 0, 256, A16, 4, None, 0, None), q4k.Q4K_ERR_SHAPE),
    (lambda L: L.q4k_gemm(A16, 4, 256, A16, 2, 128, A16, 4, None, 0, None), q4k.Q4K_ERR_SHAPE),
    (lambda L: L.q4k_gemm(A16, 4, 256, A16, 2, 256, A16, 3, None, 0, None), q4k.Q4K_ERR_SHAPE),
    (lambda L: L.q4k_gemm(A16, 4, 256, A16, 2, 260, A16, 4, None, 0, None), q4k.Q4K_ERR_ALIGN),
    (lambda L: L.q4k_gemm(A16, 4, 256, A16 + 4, 2, 256, A16, 4, None, 0, None), q4k.Q4K_ERR_ALIGN),
    (lambda L: L.q4k_gemm(A16, 4, 256, A16, 32, 256, A16 + 4, 4, None, 0, None), q4k.Q4K_ERR_ALIGN),
    (lambda L: L.q4k_moe_route(None, 4, 2, 8, A16, A16, None), q4k.Q4K_ERR_NULL),
    (lambda L: L.q4k_moe_route(A16, 4, 9, 8, A16, A16, None), q4k.Q4K_ERR_SHAPE),
    (lambda L: L.q4k_moe_route(A16, 4, 2, 2000, A16, A16, None), q4k.Q4K_ERR_SHAPE),
    (lambda L: L.q4k_moe_route(A16 + 1, 4, 2, 8, A16, A16, None), q4k.Q4K_ERR_ALIGN),
    (lambda L: L.q4k_moe_grouped_gemm(A16, 8, 64, 256, A16, 0, A16, None, 4, 2, A16, 1, A16, 1 << 20, None),
     q4k.Q4K_ERR_NULL),
    (lambda L: L.q4k_moe_grouped_gemm(A16, 8, 64, 256, A16, 3, A16, A16, 4, 2, A16, 1, A16, 1 << 20, None),
     q4k.Q4K_ERR_SHAPE),
    (lambda L: L.q4k_moe_grouped_gemm(A16, 8, 62, 256, A16, 0, A16, A16, 4, 2, A16, 1, A16, 1 << 20, None),
     q4k.Q4K_ERR_SHAPE),
    (lambda L: L.q4k_moe_grouped_gemm(A16, 8, 64, 256, A16, 0, A16, A16, 4, 2, A16, 1, A16 + 16, 1 << 20, None),
     q4k.Q4K_ERR_ALIGN),
    (lambda L: L.q4k_moe_grouped_gemm(A16, 8, 64, 256, A16, 0, A16, A16, 4, 2, A16, 1, A16, 64, None),
     q4k.Q4K_ERR_WORKSPACE),
    (lambda L: L.q4k_moe_ffn(A16, A16, None, 8, 256, 512, A16, A16, A16, 4, 2, A16, A16, 1 << 24, None),
     q4k.Q4K_ERR_NULL),
    (lambda L: L.q4k_moe_ffn(A16, A16, A16, 8, 256, 512, A16, A16, None, 4, 2, A16, A16, 1 << 24, None),
     q4k.Q4K_ERR_NULL),
    (lambda L: L.q4k_moe_ffn(A16, A16, A16, 8, 300, 512, A16, A16, A16, 4, 2, A16, A16, 1 << 24, None),
     q4k.Q4K_ERR_SHAPE),
    (lambda L: L.q4k_moe_ffn(A16, A16, A16, 8, 256, 512, A16, A16, A16, 4, 9, A16, A16, 1 << 24, None),
     q4k.Q4K_ERR_SHAPE),
    (lambda L: L.q4k_moe_ffn(A16, A16 + 8, A16, 8, 256, 512, A16, A16, A16, 4, 2, A16, A16, 1 << 24, None),
     q4k.Q4K_ERR_ALIGN),
    (lambda L: L.q4k_moe_ffn(A16, A16, A16, 8, 256, 512, A16, A16, A16, 4, 2, A16, A16 + 64, 1 << 24, None),
     q4k.Q4K_ERR_ALIGN),
    (lambda L: L.q4k_moe_ffn(A16, A16, A16, 8, 256, 512, A16, A16, A16, 4, 2, A16, A16, 1024, None),
     q4k.Q4K_ERR_WORKSPACE),
    (lambda L: L.q4k_quantize_x8(None, 2, 256, 256, A16, A16, None), q4k.Q4K_ERR_NULL),
    (lambda L: L.q4k_quantize_x8(A16, 2, 300, 300, A16, A16, None), q4k.Q4K_ERR_SHAPE),
    (lambda L: L.q4k_quantize_x8(A16, 2, 256, 128, A16, A16, None), q4k.Q4K_ERR_SHAPE),
    (lambda L: L.q4k_quantize_x8(A16, 2, 256, 256, A16 + 8, A16, None), q4k.Q4K_ERR_ALIGN),
    (lambda L: L.q4k_gemm_x8(A16, 4, 256, A16, None, 1, A16, 4, None, 0, None), q4k.Q4K_ERR_NULL),
    (lambda L: L.q4k_gemm_x8(A16, 4, 256, A16, A16, 17, A16, 4, None, 0, None), q4k.Q4K_ERR_WORKSPACE),
    (lambda L: L.q4k_gemm_x8(A16, 4, 256, A16, A16, 17, A16, 4, A16, 17 * 256 * 2 - 1, None), q4k.Q4K_ERR_WORKSPACE),
    (lambda L: L.q4k_gemm_x8(A16, 4, 256, A16, A16, 17, A16, 4, A16 + 16, 1 << 20, None), q4k.Q4K_ERR_ALIGN),
    (lambda L: L.q4k_gemm_x8(A16, 4, 256, A16, A16, 17, A16 + 4, 4, A16, 1 << 20, None), q4k.Q4K_ERR_ALIGN),
    (lambda L: L.q4k_gemm_x8(A16, 4, 256, A16, A16, 0, A16, 4, None, 0, None), q4k.Q4K_ERR_SHAPE),
    (lambda L: L.q4k_gemm_x8(A16, 4, 256, A16, A16 + 4, 1, A16, 4, None, 0, None), q4k.Q4K_ERR_ALIGN),
    (lambda L: L.q4k_nvfp4_dequant(None, 1.0, 4, 256, A16, None), q4k.Q4K_ERR_NULL),
    (lambda L: L.q4k_nvfp4_dequant(A16, 1.0, 4, 200, A16, None), q4k.Q4K_ERR_SHAPE),
    (lambda L: L.q4k_nvfp4_dequant(A16 + 4, 1.0, 4, 256, A16, None), q4k.Q4K_ERR_ALIGN),
    (lambda L: L.q4k_nvfp4_gemm(A16, 1.0, 4, 256, None, 2, 256, A16, 4, None), q4k.Q4K_ERR_NULL),
    (lambda L: L.q4k_nvfp4_gemm(A16, 1.0, 4, 256, A16, 0, 256, A16, 4, None), q4k.Q4K_ERR_SHAPE),
    (lambda L: L.q4k_nvfp4_gemm(A16, 1.0, 4, 256, A16, 2, 128, A16, 4, None), q4k.Q4K_ERR_SHAPE),
    (lambda L: L.q4k_nvfp4_gemm(A16, 1.0, 4, 256, A16 + 8, 2, 256, A16, 4, None), q4k.Q4K_ERR_ALIGN),
])
def test_argument_errors_before_any_device_work(lib, call, status):
    assert call(lib) == status


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device status; a GPU is present")
def test_no_device_status(lib):
    assert lib.q4k_dequant(A16, 4, 256, A16, None) == q4k.Q4K_ERR_DEVICE
    assert lib.q4k_gemv(A16, 4, 256, A16, A16, None) == q4k.Q4K_ERR_DEVICE


def test_static_weights_switch(lib):
    prev = q4k.q4k_set_static_weights(True)
    try:
        assert q4k.q4k_set_static_weights(False) is True
        assert q4k.q4k_set_static_weights(False) is False
        assert lib.q4k_set_static_weights(7) == 0 and lib.q4k_set_static_weights(0) == 1
    finally:
        q4k.q4k_set_static_weights(prev)


def test_binding_raises(lib):
    with pytest.raises(q4k.Q4KError) as ei:
        q4k.q4k_dequant(A16, 4, 300, A16, stream=0)
    assert ei.value.status == q4k.Q4K_ERR_SHAPE
