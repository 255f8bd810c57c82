"""The Q4_K matmul oracle: plain C (q4k_ref.c), loaded with ctypes.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
benchmark's CPU-baseline leg may import this module.  The product library never
loads it, and it shares no code with the CUDA path.

Every function here is a thin marshalling wrapper; the arithmetic is in
q4k_ref.c, which cites what it computes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4k_ref.c")
_HDR = os.path.join(_HERE, "q4k_ref.h")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libq4k_ref.so")
_lock = threading.Lock()
_lib = None

QK = 256
BLOCK_BYTES = 144


def build(force: bool = False) -> str:
    """Compile the oracle: gcc -std=c99 -O2 -ffp-contract=off (no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < newest:
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-std=c99", "-D_POSIX_C_SOURCE=200809L", "-O2", "-ffp-contract=off",
                               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm", "-lpthread"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # Q4K_ORACLE_SO lets the mutation test load a deliberately broken copy
            lib = ctypes.CDLL(os.environ.get("Q4K_ORACLE_SO") or build())
            P = ctypes.c_void_p
            i64, i32 = ctypes.c_int64, ctypes.c_int32
            lib.q4k_ref_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.q4k_ref_f16_to_f32.restype = ctypes.c_float
            lib.q4k_ref_bf16_to_f32.argtypes = [ctypes.c_uint16]
            lib.q4k_ref_bf16_to_f32.restype = ctypes.c_float
            lib.q4k_ref_f32_to_bf16.argtypes = [ctypes.c_float]
            lib.q4k_ref_f32_to_bf16.restype = ctypes.c_uint16
            lib.q4k_ref_scale_min.argtypes = [P, ctypes.c_int, P, P]
            lib.q4k_ref_scale_min.restype = None
            lib.q4k_ref_dequant_block.argtypes = [P, P]
            lib.q4k_ref_dequant_block.restype = None
            lib.q4k_ref_dequant.argtypes = [P, i64, i64, P]
            lib.q4k_ref_dequant.restype = ctypes.c_int
            lib.q4k_ref_dequant_bf16.argtypes = [P, i64, i64, P]
            lib.q4k_ref_dequant_bf16.restype = ctypes.c_int
            lib.q4k_ref_gemm.argtypes = [P, i64, i64, P, i64, P]
            lib.q4k_ref_gemm.restype = ctypes.c_int
            lib.q4k_ref_gemm_mt.argtypes = [P, i64, i64, P, i64, P, ctypes.c_int]
            lib.q4k_ref_gemm_mt.restype = ctypes.c_int
            lib.q4k_ref_moe_route.argtypes = [P, i64, i32, i32, P, P]
            lib.q4k_ref_moe_route.restype = i64
            lib.q4k_ref_moe_slots.argtypes = [P, i32, i64, i64, P, ctypes.c_int, P, i64, i32, P, ctypes.c_int]
            lib.q4k_ref_moe_slots.restype = ctypes.c_int
            lib.q4k_ref_moe_combine.argtypes = [P, P, i64, i32, i64, P]
            lib.q4k_ref_moe_combine.restype = None
            lib.q4k_ref_f64_to_bf16.argtypes = [ctypes.c_double]
            lib.q4k_ref_f64_to_bf16.restype = ctypes.c_uint16
            lib.q4k_ref_moe_ffn.argtypes = [P, P, P, i32, i64, i64, P, P, P, i64, i32, P, ctypes.c_int]
            lib.q4k_ref_moe_ffn.restype = ctypes.c_int
            lib.q4k_ref_quantize_x8.argtypes = [P, i64, i64, P, P]
            lib.q4k_ref_quantize_x8.restype = None
            lib.q4k_ref_gemm_x8.argtypes = [P, i64, i64, P, P, i64, P]
            lib.q4k_ref_gemm_x8.restype = ctypes.c_int
            lib.q4k_ref_e2m1_to_f32.argtypes = [ctypes.c_uint8]
            lib.q4k_ref_e2m1_to_f32.restype = ctypes.c_float
            lib.q4k_ref_e4m3_to_f32.argtypes = [ctypes.c_uint8]
            lib.q4k_ref_e4m3_to_f32.restype = ctypes.c_float
            lib.q4k_ref_nvfp4_dequant_block.argtypes = [P, ctypes.c_float, P]
            lib.q4k_ref_nvfp4_dequant_block.restype = None
            lib.q4k_ref_nvfp4_dequant.argtypes = [P, ctypes.c_float, i64, i64, P]
            lib.q4k_ref_nvfp4_dequant.restype = ctypes.c_int
            lib.q4k_ref_nvfp4_gemm.argtypes = [P, ctypes.c_float, i64, i64, P, i64, P, ctypes.c_int]
            lib.q4k_ref_nvfp4_gemm.restype = ctypes.c_int
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _blocks(w: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(w, dtype=np.uint8)


def f16_to_f32(h: int) -> float:
    return float(_load().q4k_ref_f16_to_f32(h))


def bf16_to_f32(b: int) -> float:
    return float(_load().q4k_ref_bf16_to_f32(b))


def f32_to_bf16(f: float) -> int:
    return int(_load().q4k_ref_f32_to_bf16(f))


def scale_min(scales: np.ndarray, j: int):
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    sc, m = ctypes.c_int(), ctypes.c_int()
    _load().q4k_ref_scale_min(_p(s), j, ctypes.byref(sc), ctypes.byref(m))
    return sc.value, m.value


def dequant_block(blk: np.ndarray) -> np.ndarray:
    b = _blocks(blk).reshape(-1)
    assert b.size == BLOCK_BYTES
    out = np.empty(QK, dtype=np.float32)
    _load().q4k_ref_dequant_block(_p(b), _p(out))
    return out


def dequant(w: np.ndarray, N: int, K: int) -> np.ndarray:
    """Q4_K blocks of an N x K matrix -> fp32 [N, K]."""
    b = _blocks(w)
    assert b.size == N * (K // QK) * BLOCK_BYTES
    out = np.empty((N, K), dtype=np.float32)
    if _load().q4k_ref_dequant(_p(b), N, K, _p(out)) != 0:
        raise ValueError("bad shape")
    return out


def dequant_bf16(w: np.ndarray, N: int, K: int) -> np.ndarray:
    """Q4_K blocks -> bf16 [N, K] (uint16 bit patterns), RNE of the fp32 weight."""
    b = _blocks(w)
    out = np.empty((N, K), dtype=np.uint16)
    if _load().q4k_ref_dequant_bf16(_p(b), N, K, _p(out)) != 0:
        raise ValueError("bad shape")
    return out


def gemm(w: np.ndarray, N: int, K: int, x_bf16: np.ndarray, threads: int = 1) -> np.ndarray:
    """y [M, N] fp64 = x [M, K] (bf16 bits) @ W^T, fp64 accumulation in increasing k."""
    b = _blocks(w)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16).reshape(-1, K)
    M = x.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    if _load().q4k_ref_gemm_mt(_p(b), N, K, _p(x), M, _p(y), threads) != 0:
        raise ValueError("bad shape")
    return y


def moe_route(ids: np.ndarray, E: int):
    """Stable counting sort of (token, slot) items by expert -> (offsets[E+1], perm[T*topk], n_bad)."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, topk = ids.shape
    offsets = np.zeros(E + 1, dtype=np.int32)
    perm = np.full(T * topk, -1, dtype=np.int32)
    bad = _load().q4k_ref_moe_route(_p(ids), T, topk, E, _p(offsets), _p(perm))
    return offsets, perm, int(bad)


def moe_slots(w_experts: np.ndarray, E: int, N: int, K: int, x_bf16: np.ndarray, x_per_slot: bool,
              ids: np.ndarray, threads: int = 1) -> np.ndarray:
    """Per-slot expert outputs out [T, topk, N] fp64."""
    b = _blocks(w_experts)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, topk = ids.shape
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    out = np.empty((T, topk, N), dtype=np.float64)
    rc = _load().q4k_ref_moe_slots(_p(b), E, N, K, _p(x), int(bool(x_per_slot)), _p(ids), T, topk, _p(out),
                                   threads)
    if rc != 0:
        raise ValueError("bad shape")
    return out


def moe_combine(out: np.ndarray, gates: np.ndarray) -> np.ndarray:
    """y [T, N] = sum_j gates[t, j] * out[t, j, :] in slot order, fp64."""
    out = np.ascontiguousarray(out, dtype=np.float64)
    gates = np.ascontiguousarray(gates, dtype=np.float32)
    T, topk, N = out.shape
    y = np.empty((T, N), dtype=np.float64)
    _load().q4k_ref_moe_combine(_p(out), _p(gates), T, topk, N, _p(y))
    return y


def moe(w_experts, E, N, K, x_bf16, x_per_slot, ids, gates=None, threads: int = 1):
    """Per-slot outputs, or (with gates) their weighted combine [T, N]."""
    out = moe_slots(w_experts, E, N, K, x_bf16, x_per_slot, ids, threads)
    return out if gates is None else moe_combine(out, gates)


def f64_to_bf16(v: float) -> int:
    """The bf16 nearest to a double (ties to even), rounded once; its bits."""
    return int(_load().q4k_ref_f64_to_bf16(float(v)))


def moe_ffn(w_gate, w_up, w_down, E: int, H: int, D: int, x_bf16, ids, gates, threads: int = 1) -> np.ndarray:
    """Routed SwiGLU expert layer y [T, D] fp64 (q4k_ref_moe_ffn)."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, topk = ids.shape
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    gates = np.ascontiguousarray(gates, dtype=np.float32)
    y = np.empty((T, D), dtype=np.float64)
    rc = _load().q4k_ref_moe_ffn(_p(_blocks(w_gate)), _p(_blocks(w_up)), _p(_blocks(w_down)), E, H, D, _p(x),
                                 _p(ids), _p(gates), T, topk, _p(y), threads)
    if rc != 0:
        raise ValueError("bad shape")
    return y


def quantize_x8(x_bf16) -> tuple:
    """Per-32 int8 quantization of bf16 rows [M, K]: (q int8 [M, K], s fp32 [M, K/32])
    (q4k_ref_quantize_x8)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, K = x.shape
    q = np.empty((M, K), dtype=np.int8)
    sc = np.empty((M, K // 32), dtype=np.float32)
    _load().q4k_ref_quantize_x8(_p(x), M, K, _p(q), _p(sc))
    return q, sc


def gemm_x8(w: np.ndarray, N: int, K: int, q, s) -> np.ndarray:
    """y [M, N] fp64 = W . (s * q)^T over the int8 activations (q4k_ref_gemm_x8)."""
    q = np.ascontiguousarray(q, dtype=np.int8)
    s = np.ascontiguousarray(s, dtype=np.float32)
    M = q.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    if _load().q4k_ref_gemm_x8(_p(_blocks(w)), N, K, _p(q), _p(s), M, _p(y)) != 0:
        raise ValueError("bad shape")
    return y


def e2m1_to_f32(code: int) -> float:
    return float(_load().q4k_ref_e2m1_to_f32(code))


def e4m3_to_f32(bits: int) -> float:
    return float(_load().q4k_ref_e4m3_to_f32(bits))


def nvfp4_dequant_block(blk: np.ndarray, g: float) -> np.ndarray:
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    out = np.empty(256, dtype=np.float32)
    _load().q4k_ref_nvfp4_dequant_block(_p(blk), g, _p(out))
    return out


def nvfp4_dequant(w: np.ndarray, g: float, N: int, K: int) -> np.ndarray:
    """NVFP4 blocks [N, K/256*144] -> fp32 [N, K] (q4k_ref_nvfp4_dequant)."""
    out = np.empty((N, K), dtype=np.float32)
    if _load().q4k_ref_nvfp4_dequant(_p(_blocks(w)), g, N, K, _p(out)) != 0:
        raise ValueError("bad shape")
    return out


def nvfp4_gemm(w: np.ndarray, g: float, N: int, K: int, x_bf16, threads: int = 1) -> np.ndarray:
    """y [M, N] fp64 over NVFP4 weights (q4k_ref_nvfp4_gemm)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M = x.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    if _load().q4k_ref_nvfp4_gemm(_p(_blocks(w)), g, N, K, _p(x), M, _p(y), threads) != 0:
        raise ValueError("bad shape")
    return y
