"""Seeded synthetic inputs for the Q4_K matmul workloads (ctypes over q4k_synth.c).

Input generation only: splitmix64 uniforms, Box-Muller normals, bf16 rounding,
outlier injection, top-k routing with Dirichlet(1) gates, and the reference
quantizer that encodes fp32 weights as GGUF Q4_K blocks.  Both the oracle's tests
and the GPU tests/benchmark draw their inputs from here; neither side's
arithmetic lives here.

Seeds follow one rule so that every consumer draws identical inputs:
``seed(config, stream) = 0x5EED0000 + 16 * config + stream`` with stream 0 the
weights, 1 the activations, 2 the routing ids, 3 the gate weights, 4 the outlier
picks (and 5.. for further matrices of one workload).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4k_synth.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libq4k_synth.so")
_lock = threading.Lock()
_lib = None

BLOCK_BYTES = 144
QK = 256


def seed(config: int, stream: int) -> int:
    return 0x5EED0000 + 16 * config + stream


def build(force: bool = False) -> str:
    """Compile q4k_synth.c into a shared library (gcc, -O2, no fp contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, u64, f64 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_double
            lib.q4k_synth_normal_f32.argtypes = [u64, i64, f64, f64, P]
            lib.q4k_synth_normal_f32.restype = None
            lib.q4k_synth_normal_bf16.argtypes = [u64, i64, f64, f64, P]
            lib.q4k_synth_normal_bf16.restype = None
            lib.q4k_synth_f32_to_bf16.argtypes = [P, i64, P]
            lib.q4k_synth_f32_to_bf16.restype = None
            lib.q4k_synth_outliers.argtypes = [u64, P, i64, f64, ctypes.c_float]
            lib.q4k_synth_outliers.restype = i64
            lib.q4k_synth_routing.argtypes = [u64, u64, i64, ctypes.c_int32, ctypes.c_int32, P, P]
            lib.q4k_synth_routing.restype = ctypes.c_int
            lib.q4k_synth_pack_scales.argtypes = [P, P, P]
            lib.q4k_synth_pack_scales.restype = None
            lib.q4k_synth_make_block.argtypes = [ctypes.c_uint16, ctypes.c_uint16, P, P, P, P]
            lib.q4k_synth_make_block.restype = None
            lib.q4k_synth_quantize.argtypes = [P, i64, i64, P]
            lib.q4k_synth_quantize.restype = ctypes.c_int
            lib.q4k_synth_weights.argtypes = [u64, i64, i64, f64, f64, f64, u64, P]
            lib.q4k_synth_weights.restype = ctypes.c_int
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def normal_f32(seed_: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _load().q4k_synth_normal_f32(seed_, n, mean, std, _p(out))
    return out


def normal_bf16(seed_: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """n draws N(mean, std^2) rounded to fp32 then to bf16 (RNE); uint16 bit patterns."""
    out = np.empty(n, dtype=np.uint16)
    _load().q4k_synth_normal_bf16(seed_, n, mean, std, _p(out))
    return out


def f32_to_bf16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().q4k_synth_f32_to_bf16(_p(a), a.size, _p(out))
    return out


def outliers(seed_: int, w: np.ndarray, frac: float = 0.01, factor: float = 10.0) -> int:
    """Scale round(frac*S) of the S 32-weight sub-blocks of w (in place) by factor."""
    assert w.dtype == np.float32 and w.flags["C_CONTIGUOUS"]
    return int(_load().q4k_synth_outliers(seed_, _p(w), w.size, frac, factor))


def routing(seed_ids: int, seed_gates: int, T: int, E: int, topk: int):
    """(ids [T, topk] int32, gates [T, topk] float32): distinct experts, Dirichlet(1) gates."""
    ids = np.empty((T, topk), dtype=np.int32)
    gates = np.empty((T, topk), dtype=np.float32)
    rc = _load().q4k_synth_routing(seed_ids, seed_gates, T, E, topk, _p(ids), _p(gates))
    if rc != 0:
        raise ValueError("bad routing arguments")
    return ids, gates


def pack_scales(sc, mn) -> np.ndarray:
    sc = np.ascontiguousarray(sc, dtype=np.uint8)
    mn = np.ascontiguousarray(mn, dtype=np.uint8)
    out = np.zeros(12, dtype=np.uint8)
    _load().q4k_synth_pack_scales(_p(sc), _p(mn), _p(out))
    return out


def make_block(d_bits: int, dmin_bits: int, sc, mn, q) -> np.ndarray:
    """One 144-byte block from its fields (q: 256 codes 0..15 in weight order)."""
    sc = np.ascontiguousarray(sc, dtype=np.uint8)
    mn = np.ascontiguousarray(mn, dtype=np.uint8)
    q = np.ascontiguousarray(q, dtype=np.uint8)
    out = np.zeros(BLOCK_BYTES, dtype=np.uint8)
    _load().q4k_synth_make_block(d_bits, dmin_bits, _p(sc), _p(mn), _p(q), _p(out))
    return out


def quantize(w: np.ndarray) -> np.ndarray:
    """fp32 [N, K] -> uint8 [N, K/256*144] Q4_K blocks."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    out = np.empty((N, K // QK * BLOCK_BYTES), dtype=np.uint8)
    if _load().q4k_synth_quantize(_p(w), N, K, _p(out)) != 0:
        raise ValueError("K must be a positive multiple of 256")
    return out


def weights(seed_: int, N: int, K: int, std: float = 0.02, outlier_frac: float = 0.0,
            outlier_factor: float = 10.0, seed_outliers: int = 0) -> np.ndarray:
    """Q4_K blocks of an N x K matrix drawn from N(0, std^2) (+ outliers), [N, K/256*144]."""
    out = np.empty((N, K // QK * BLOCK_BYTES), dtype=np.uint8)
    rc = _load().q4k_synth_weights(seed_, N, K, std, outlier_frac, outlier_factor, seed_outliers, _p(out))
    if rc != 0:
        raise ValueError(f"q4k_synth_weights failed ({rc})")
    return out


def row_bytes(K: int) -> int:
    return K // QK * BLOCK_BYTES


# ----------------------------------------------------------------- NVFP4 inputs
# Input generation only: a simple nearest-value NVFP4 quantizer (e2m1 values,
# one e4m3 scale per 16 weights, one fp32 scale per tensor) packed in 144-byte
# blocks of 256 weights: 16 scale bytes, then 128 value bytes (weight 2i in the
# low nibble of byte i).

_E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e4m3_positive_table():
    codes = np.arange(0x7F, dtype=np.int64)  # 0x00 .. 0x7E: every finite non-negative value
    e, m = (codes >> 3) & 15, codes & 7
    vals = np.where(e == 0, m * 2.0 ** -9, (8 + m) * np.exp2(e - 10.0))
    order = np.argsort(vals, kind="stable")
    return vals[order], codes[order].astype(np.uint8)


def nvfp4_quantize(w: np.ndarray) -> tuple:
    """fp32 [N, K] -> (NVFP4 blocks [N, K/256*144] uint8, per-tensor fp32 scale g)."""
    w = np.asarray(w, dtype=np.float64)
    N, K = w.shape
    amax = float(np.abs(w).max()) if w.size else 0.0
    g = np.float32(amax / (6.0 * 448.0) if amax > 0 else 1.0)
    grp = w.reshape(N, K // 16, 16) / float(g)
    tv, tc = _e4m3_positive_table()
    want = np.abs(grp).max(axis=2) / 6.0                    # scale that maps the group's max to 6
    idx = np.clip(np.searchsorted(tv, want), 0, len(tv) - 1)  # smallest table value >= want
    sval, scode = tv[idx], tc[idx]
    r = np.abs(grp) / np.where(sval > 0, sval, 1.0)[..., None]
    mid = (_E2M1_MAG[1:] + _E2M1_MAG[:-1]) / 2
    mag = np.searchsorted(mid, np.minimum(r, 6.0))          # nearest e2m1 magnitude
    code = (mag | np.where(grp < 0, 8, 0)).astype(np.uint8).reshape(N, K)
    out = np.empty((N, K // 256, 144), dtype=np.uint8)
    out[:, :, :16] = scode.reshape(N, K // 256, 16)
    pairs = code.reshape(N, K // 256, 128, 2)
    out[:, :, 16:] = pairs[..., 0] | (pairs[..., 1] << 4)
    return out.reshape(N, K // 256 * 144), g


def nvfp4_weights(seed_: int, N: int, K: int, std: float = 0.02) -> tuple:
    """NVFP4 blocks of an N x K matrix drawn from N(0, std^2), and its tensor scale g."""
    return nvfp4_quantize(normal_f32(seed_, N * K, 0.0, std).reshape(N, K))
