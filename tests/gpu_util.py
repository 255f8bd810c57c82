"""Helpers for the GPU parity tests: seeded workload inputs and device transfer.

Inputs come from the shared seeded generators (synth); expected values come from
the oracle only.  The workload shapes are those of the decode, speculative
verify, prefill and MoE configurations (names below state their sizes).
"""
from __future__ import annotations

import functools

import numpy as np
import torch

import synth

# name -> (config index for seeding, N, K)
DECODE_UP = (1, 17408, 5120)      # gate/up projection K 5120 -> N 17408
DECODE_DOWN = (1, 5120, 17408)    # down projection K 17408 -> N 5120
TINY = (0, 256, 1024)             # dequant + GEMV tiny case
MOE_E, MOE_TOPK = 128, 8
MOE_UP = (768, 2048)              # gate and up: K 2048 -> N 768
MOE_DOWN = (2048, 768)            # down: K 768 -> N 2048


def dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def rel_err(y: np.ndarray, ref: np.ndarray) -> float:
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    m = np.abs(ref).max()
    if m == 0:
        return float(np.abs(y).max())
    return float(np.abs(y - ref).max() / m)


@functools.lru_cache(maxsize=8)
def weights(cfg: int, stream: int, N: int, K: int, outliers: bool = False) -> np.ndarray:
    """Q4_K blocks [N, K/256*144] of N(0, 0.02^2) weights (1% outlier sub-blocks x10 if asked)."""
    return synth.weights(synth.seed(cfg, stream), N, K, 0.02, 0.01 if outliers else 0.0, 10.0,
                         synth.seed(cfg, 4 + stream))


def activations(cfg: int, stream: int, M: int, K: int) -> np.ndarray:
    """bf16 bit patterns [M, K] drawn from N(0, 1)."""
    return synth.normal_bf16(synth.seed(cfg, stream), M * K).reshape(M, K)


def rows_of(blocks: np.ndarray, rows) -> np.ndarray:
    """The Q4_K rows `rows` of a weight matrix, as a smaller matrix."""
    return np.ascontiguousarray(blocks[np.asarray(rows)])


def sample_rows(N: int, n: int = 96, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    r = np.unique(np.concatenate([[0, N - 1], rng.choice(N, size=min(n, N), replace=False)]))
    return np.sort(r)


@functools.lru_cache(maxsize=4)
def moe_experts(cfg: int, stream: int, N: int, K: int, E: int = MOE_E) -> np.ndarray:
    """E stacked expert matrices [E*N, K/256*144] (expert e seeded by stream 16 + e)."""
    return np.concatenate([synth.weights(synth.seed(cfg, stream) + 1000 * (e + 1), N, K, 0.02) for e in range(E)])


def _bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even), back as float64."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float64).numpy()


def tc_weights(blocks: np.ndarray, N: int, K: int) -> np.ndarray:
    """Model of the tensor-core kernels' bf16 weight operand, float64 [N, K].

    Those kernels feed each weight as the round-to-nearest-even bf16 of its fp32
    dequantized value: w = bf16(fl32(q * d*sc - dmin*m)), where d*sc, dmin*m and
    q * d*sc are exact in fp32.  The field layout follows the Q4_K
    block (fp16 d and dmin, twelve bytes of 6-bit scale/offset pairs, 128 bytes
    of codes: sub-blocks 2g and 2g+1 are the low and high nibbles of bytes
    32g..32g+31).  Used only to separate that rounding from other errors."""
    nb = K // 256
    b = np.ascontiguousarray(blocks).reshape(N, nb, 144)
    d = b[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float32)
    dmin = b[..., 2:4].copy().view(np.float16)[..., 0].astype(np.float32)
    s = b[..., 4:16].astype(np.int32)
    sc = np.empty((N, nb, 8), np.int32)
    mm = np.empty((N, nb, 8), np.int32)
    sc[..., :4], mm[..., :4] = s[..., 0:4] & 63, s[..., 4:8] & 63
    sc[..., 4:] = (s[..., 8:12] & 15) | ((s[..., 0:4] >> 6) << 4)
    mm[..., 4:] = (s[..., 8:12] >> 4) | ((s[..., 4:8] >> 6) << 4)
    codes = b[..., 16:].astype(np.int32).reshape(N, nb, 4, 32)
    q = np.stack([codes & 15, codes >> 4], axis=3).reshape(N, nb, 8, 32)
    dsc = (d[..., None] * sc.astype(np.float32)).astype(np.float32)
    dm = (dmin[..., None] * mm.astype(np.float32)).astype(np.float32)
    w = q.astype(np.float32) * dsc[..., None] - dm[..., None]   # float32: one rounding
    return _bf16(w.astype(np.float32)).reshape(N, K)
