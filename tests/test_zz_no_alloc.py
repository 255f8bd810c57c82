"""The allocation-free MoE entry point against the workspace one.

q4k_moe_grouped_gemm_noalloc is for callers that cannot allocate device memory
(no cudaMalloc on their path, or all memory already handed to their own pools);
it keeps its scratch in a fixed array inside the library.  This test calls it
through the C ABI twice in a row - the second call reuses the array the first
one left behind - and checks each result against q4k_moe_grouped_gemm given a
caller-owned workspace: both run the same kernels, so the bits must agree.  The
shapes cover the small-M expert kernels and the tensor-core path (32 or more
items per expert), whose expert-sorted copy of the activations also lives in
the array.  It also checks that a request too large for the array is refused
before anything runs.

The file name sorts last so that a run stopping at its first failure has run
every other test first; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import q4_weight_quantized_gb300 as q4k
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from q4_weight_quantized_gb300.build import build_library
    build_library()
    return q4k.load()


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


@pytest.mark.parametrize("E,T,x_mode,y_mode", [
    (32, 16, q4k.Q4K_MOE_X_PER_SLOT, q4k.Q4K_MOE_Y_COMBINE),   # small-M expert kernels
    (32, 16, q4k.Q4K_MOE_X_PER_TOKEN, q4k.Q4K_MOE_Y_PER_SLOT),
    (8, 32, q4k.Q4K_MOE_X_PER_SLOT, q4k.Q4K_MOE_Y_COMBINE),    # 32 items per expert: tensor cores
    (8, 32, q4k.Q4K_MOE_X_PER_TOKEN, q4k.Q4K_MOE_Y_PER_SLOT)])
def test_noalloc_matches_workspace_entry_point(lib, syn, E, T, x_mode, y_mode):
    N, K, topk = 256, 512, 8
    w = G.dev(np.concatenate([G.weights(4, 40 + e, N, K) for e in range(E)]))
    ids_np, gates_np = syn.routing(901, 902, T, E, topk)
    rows = T * topk if x_mode == q4k.Q4K_MOE_X_PER_SLOT else T
    x = G.dev(G.activations(4, 9, rows, K))
    ids, gates = G.dev(ids_np), G.dev(gates_np)
    shape = (T, N) if y_mode == q4k.Q4K_MOE_Y_COMBINE else (T, topk, N)
    stream = torch.cuda.current_stream().cuda_stream

    ws_bytes = q4k.q4k_moe_workspace_size(E, N, K, T, topk, y_mode)
    assert 0 < ws_bytes <= q4k.MOE_NOALLOC_SCRATCH_BYTES
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    ref = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
    st = lib.q4k_moe_grouped_gemm(_p(w), E, N, K, _p(x), x_mode, _p(ids), _p(gates), T, topk, _p(ref), y_mode,
                                  _p(ws), ws_bytes, stream)
    assert st == q4k.Q4K_OK
    torch.cuda.synchronize()
    want = G.host(ref)
    assert np.isfinite(want).all()

    for call in range(2):
        y = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
        st = lib.q4k_moe_grouped_gemm_noalloc(_p(w), E, N, K, _p(x), x_mode, _p(ids), _p(gates), T, topk, _p(y),
                                              y_mode, stream)
        assert st == q4k.Q4K_OK, q4k.status_string(st)
        torch.cuda.synchronize()
        got = G.host(y)
        assert np.isfinite(got).all(), f"call {call}: rows left unwritten"
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), f"call {call}"
    q4k.q4k_check_device()


def test_noalloc_rejects_requests_beyond_its_scratch(lib):
    # T = 2048, top-8, N = 2048 with the combine needs 128 MiB of per-slot rows
    E, N, K, T, topk = 128, 2048, 768, 2048, 8
    need = q4k.q4k_moe_workspace_size(E, N, K, T, topk, q4k.Q4K_MOE_Y_COMBINE)
    assert need > q4k.MOE_NOALLOC_SCRATCH_BYTES
    a16 = ctypes.c_void_p(1 << 20)  # never dereferenced: the call must fail before any launch
    st = lib.q4k_moe_grouped_gemm_noalloc(a16, E, N, K, a16, q4k.Q4K_MOE_X_PER_SLOT, a16, a16, T, topk, a16,
                                          q4k.Q4K_MOE_Y_COMBINE, torch.cuda.current_stream().cuda_stream)
    assert st == q4k.Q4K_ERR_WORKSPACE
