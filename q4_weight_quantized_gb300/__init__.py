"""Python binding of the q4k C-ABI library (libq4k.so): argument marshalling only.

Every function has the name and argument order of its C entry point in
include/q4k.h.  Pointer arguments take a torch tensor (its data_ptr), a raw int
address or None; `stream` takes a torch.cuda.Stream, a raw cudaStream_t int, or
None for torch's current stream.  A non-OK status raises Q4KError.  All
arithmetic runs in the library's CUDA kernels; there is no Python or CPU path.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libq4k.so")

Q4K_OK, Q4K_ERR_NULL, Q4K_ERR_SHAPE, Q4K_ERR_ALIGN = 0, 1, 2, 3
Q4K_ERR_WORKSPACE, Q4K_ERR_DEVICE, Q4K_ERR_CUDA, Q4K_ERR_TIMEOUT, Q4K_ERR_ROUTING = 4, 5, 6, 7, 8
Q4K_MOE_X_PER_TOKEN, Q4K_MOE_X_PER_SLOT = 0, 1
Q4K_MOE_Y_PER_SLOT, Q4K_MOE_Y_COMBINE = 0, 1

BLOCK_BYTES = 144
QK = 256

# every symbol include/q4k.h declares
EXPORTS = (
    "q4k_status_string", "q4k_last_cuda_error", "q4k_row_bytes", "q4k_version", "q4k_check_device",
    "q4k_set_static_weights", "q4k_set_batch_invariant", "q4k_set_gemv_wait_limit_ns", "q4k_dequant", "q4k_dequant_bf16", "q4k_gemv", "q4k_gemm_workspace_size", "q4k_gemm",
    "q4k_moe_route", "q4k_moe_workspace_size", "q4k_moe_grouped_gemm", "q4k_moe_grouped_gemm_reuse_routing",
    "q4k_moe_grouped_gemm_noalloc", "q4k_moe_ffn_workspace_size", "q4k_moe_ffn", "q4k_quantize_x8", "q4k_gemm_x8_workspace_size", "q4k_gemm_x8",
    "q4k_nvfp4_dequant", "q4k_nvfp4_gemm",
)

# fixed scratch capacity of q4k_moe_grouped_gemm_noalloc (Q4K_MOE_NOALLOC_SCRATCH_BYTES)
MOE_NOALLOC_SCRATCH_BYTES = 8 << 20


class Q4KError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


_lib = None


def load(path: str | None = None):
    """Load libq4k.so (built in-tree by q4_weight_quantized_gb300.build).  Fails
    loudly if it is missing: there is no fallback implementation."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"{p} is missing; build it with q4_weight_quantized_gb300.build.build_library()")
    lib = ctypes.CDLL(p)
    P, i64, i32, sz, st = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t, ctypes.c_int
    sig = {
        "q4k_status_string": ([st], ctypes.c_char_p),
        "q4k_last_cuda_error": ([], st),
        "q4k_row_bytes": ([i64], sz),
        "q4k_version": ([], st),
        "q4k_check_device": ([P], st),
        "q4k_set_static_weights": ([ctypes.c_int], ctypes.c_int),
        "q4k_set_batch_invariant": ([ctypes.c_int], ctypes.c_int),
        "q4k_set_gemv_wait_limit_ns": ([ctypes.c_ulonglong], ctypes.c_ulonglong),
        "q4k_dequant": ([P, i64, i64, P, P], st),
        "q4k_dequant_bf16": ([P, i64, i64, P, P], st),
        "q4k_gemv": ([P, i64, i64, P, P, P], st),
        "q4k_gemm_workspace_size": ([i64, i64, i64], sz),
        "q4k_gemm": ([P, i64, i64, P, i64, i64, P, i64, P, sz, P], st),
        "q4k_moe_route": ([P, i64, i32, i32, P, P, P], st),
        "q4k_moe_workspace_size": ([i32, i64, i64, i64, i32, st], sz),
        "q4k_moe_grouped_gemm": ([P, i32, i64, i64, P, st, P, P, i64, i32, P, st, P, sz, P], st),
        "q4k_moe_grouped_gemm_reuse_routing": ([P, i32, i64, i64, P, st, P, P, i64, i32, P, st, P, sz, P], st),
        "q4k_moe_grouped_gemm_noalloc": ([P, i32, i64, i64, P, st, P, P, i64, i32, P, st, P], st),
        "q4k_moe_ffn_workspace_size": ([i32, i64, i64, i64, i32], sz),
        "q4k_moe_ffn": ([P, P, P, i32, i64, i64, P, P, P, i64, i32, P, P, sz, P], st),
        "q4k_quantize_x8": ([P, i64, i64, i64, P, P, P], st),
        "q4k_gemm_x8_workspace_size": ([i64, i64], sz),
        "q4k_gemm_x8": ([P, i64, i64, P, P, i64, P, i64, P, sz, P], st),
        "q4k_nvfp4_dequant": ([P, ctypes.c_float, i64, i64, P, P], st),
        "q4k_nvfp4_gemm": ([P, ctypes.c_float, i64, i64, P, i64, i64, P, i64, P], st),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    if path is None:
        _lib = lib
    return lib


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, int):
        return a
    return a.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, what: str):
    if status != Q4K_OK:
        raise Q4KError(status, what)


def status_string(status: int) -> str:
    return load().q4k_status_string(status).decode()


def q4k_status_string(status: int) -> str:
    return status_string(status)


def q4k_last_cuda_error() -> int:
    return load().q4k_last_cuda_error()


def q4k_row_bytes(K: int) -> int:
    return load().q4k_row_bytes(K)


def q4k_version() -> int:
    return load().q4k_version()


def q4k_check_device(stream=None) -> None:
    _check(load().q4k_check_device(_stream(stream)), "q4k_check_device")


def q4k_set_static_weights(enable: bool) -> bool:
    """Declare the weights read by the small-M calls static (never written by the
    kernel enqueued just before a call on the same stream); returns the previous
    setting.  See include/q4k.h."""
    return bool(load().q4k_set_static_weights(1 if enable else 0))


def q4k_set_gemv_wait_limit_ns(ns: int) -> int:
    """Test hook: the limit of the decode GEMV's main-loop waits in nanoseconds (0:
    the standard 2 s); returns the previous setting.  See include/q4k.h."""
    return int(load().q4k_set_gemv_wait_limit_ns(int(ns)))


def q4k_set_batch_invariant(enable: bool) -> bool:
    """Batch-invariant mode: one-token calls run the 2..16-token kernel, so rows of
    every call with M <= 16 share their bits; returns the previous setting.  See
    include/q4k.h."""
    return bool(load().q4k_set_batch_invariant(1 if enable else 0))


def q4k_dequant(w, N: int, K: int, out, stream=None) -> None:
    _check(load().q4k_dequant(_ptr(w), N, K, _ptr(out), _stream(stream)), "q4k_dequant")


def q4k_dequant_bf16(w, N: int, K: int, out, stream=None) -> None:
    _check(load().q4k_dequant_bf16(_ptr(w), N, K, _ptr(out), _stream(stream)), "q4k_dequant_bf16")


def q4k_gemv(w, N: int, K: int, x, y, stream=None) -> None:
    _check(load().q4k_gemv(_ptr(w), N, K, _ptr(x), _ptr(y), _stream(stream)), "q4k_gemv")


def q4k_gemm_workspace_size(M: int, N: int, K: int) -> int:
    return load().q4k_gemm_workspace_size(M, N, K)


def q4k_gemm(w, N: int, K: int, x, M: int, ldx: int, y, ldy: int, ws=None, ws_bytes: int = 0, stream=None) -> None:
    _check(load().q4k_gemm(_ptr(w), N, K, _ptr(x), M, ldx, _ptr(y), ldy, _ptr(ws), ws_bytes, _stream(stream)),
           "q4k_gemm")


def q4k_moe_route(topk_ids, T: int, topk: int, n_experts: int, offsets, perm, stream=None) -> None:
    _check(load().q4k_moe_route(_ptr(topk_ids), T, topk, n_experts, _ptr(offsets), _ptr(perm), _stream(stream)),
           "q4k_moe_route")


def q4k_moe_workspace_size(n_experts: int, N: int, K: int, T: int, topk: int, y_mode: int) -> int:
    return load().q4k_moe_workspace_size(n_experts, N, K, T, topk, y_mode)


def q4k_moe_grouped_gemm(w_experts, n_experts: int, N: int, K: int, x, x_mode: int, topk_ids, gates, T: int,
                         topk: int, y, y_mode: int, ws, ws_bytes: int, stream=None) -> None:
    _check(load().q4k_moe_grouped_gemm(_ptr(w_experts), n_experts, N, K, _ptr(x), x_mode, _ptr(topk_ids),
                                       _ptr(gates), T, topk, _ptr(y), y_mode, _ptr(ws), ws_bytes, _stream(stream)),
           "q4k_moe_grouped_gemm")


def q4k_moe_grouped_gemm_reuse_routing(w_experts, n_experts: int, N: int, K: int, x, x_mode: int, topk_ids, gates,
                                       T: int, topk: int, y, y_mode: int, ws, ws_bytes: int, stream=None) -> None:
    """q4k_moe_grouped_gemm reusing the routing that the last q4k_moe_grouped_gemm
    call left in `ws` (same n_experts, T, topk and unchanged topk_ids)."""
    _check(load().q4k_moe_grouped_gemm_reuse_routing(_ptr(w_experts), n_experts, N, K, _ptr(x), x_mode,
                                                     _ptr(topk_ids), _ptr(gates), T, topk, _ptr(y), y_mode, _ptr(ws),
                                                     ws_bytes, _stream(stream)),
           "q4k_moe_grouped_gemm_reuse_routing")


def q4k_moe_grouped_gemm_noalloc(w_experts, n_experts: int, N: int, K: int, x, x_mode: int, topk_ids, gates,
                                 T: int, topk: int, y, y_mode: int, stream=None) -> None:
    """q4k_moe_grouped_gemm without a workspace: for callers that cannot allocate.
    Its scratch is a fixed array inside the library (MOE_NOALLOC_SCRATCH_BYTES per
    GPU); calls that overlap on the GPU share it and race, so keep them on one
    stream, and make the first call on a device before any CUDA graph capture."""
    _check(load().q4k_moe_grouped_gemm_noalloc(_ptr(w_experts), n_experts, N, K, _ptr(x), x_mode, _ptr(topk_ids),
                                               _ptr(gates), T, topk, _ptr(y), y_mode, _stream(stream)),
           "q4k_moe_grouped_gemm_noalloc")


def q4k_moe_ffn_workspace_size(n_experts: int, H: int, D: int, T: int, topk: int) -> int:
    return load().q4k_moe_ffn_workspace_size(n_experts, H, D, T, topk)


def q4k_moe_ffn(w_gate, w_up, w_down, n_experts: int, H: int, D: int, x, topk_ids, gates, T: int, topk: int, y,
                ws, ws_bytes: int, stream=None) -> None:
    """One routed SwiGLU expert layer: y[t] = sum_j gates[t][j] * down_e(bf16(silu(gate_e(x[t])) * up_e(x[t]))),
    e = topk_ids[t][j]; x bf16 [T][D], y fp32 [T][D]."""
    _check(load().q4k_moe_ffn(_ptr(w_gate), _ptr(w_up), _ptr(w_down), n_experts, H, D, _ptr(x), _ptr(topk_ids),
                              _ptr(gates), T, topk, _ptr(y), _ptr(ws), ws_bytes, _stream(stream)),
           "q4k_moe_ffn")


def q4k_quantize_x8(x, M: int, K: int, ldx: int, q, s, stream=None) -> None:
    """Per-32 int8 quantization of bf16 rows: q int8 [M][K], s fp32 [M][K/32]."""
    _check(load().q4k_quantize_x8(_ptr(x), M, K, ldx, _ptr(q), _ptr(s), _stream(stream)), "q4k_quantize_x8")


def q4k_gemm_x8_workspace_size(M: int, K: int) -> int:
    return load().q4k_gemm_x8_workspace_size(M, K)


def q4k_gemm_x8(w, N: int, K: int, q, s, M: int, y, ldy: int, ws=None, ws_bytes: int = 0, stream=None) -> None:
    """y = (s * q) . W^T over int8 activations (M > 16 needs a workspace of
    q4k_gemm_x8_workspace_size(M, K) bytes)."""
    _check(load().q4k_gemm_x8(_ptr(w), N, K, _ptr(q), _ptr(s), M, _ptr(y), ldy, _ptr(ws), ws_bytes,
                              _stream(stream)), "q4k_gemm_x8")


def q4k_nvfp4_dequant(w, g: float, N: int, K: int, out, stream=None) -> None:
    """NVFP4 blocks -> fp32 [N][K], w = g * e4m3 * e2m1."""
    _check(load().q4k_nvfp4_dequant(_ptr(w), g, N, K, _ptr(out), _stream(stream)), "q4k_nvfp4_dequant")


def q4k_nvfp4_gemm(w, g: float, N: int, K: int, x, M: int, ldx: int, y, ldy: int, stream=None) -> None:
    """y = x . W^T with NVFP4 weights (tensor cores, any M >= 1)."""
    _check(load().q4k_nvfp4_gemm(_ptr(w), g, N, K, _ptr(x), M, ldx, _ptr(y), ldy, _stream(stream)), "q4k_nvfp4_gemm")
