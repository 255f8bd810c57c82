"""Failure detection on the device: a bounded wait that runs out.

Every wait inside the kernels has a time limit.  When one runs out, the kernel
abandons its work, waits (with the full limit) for its own copies still in
flight, reaches all of its barriers and sets the device status word, which
q4k_check_device reports as Q4K_ERR_TIMEOUT.  These tests shorten the limit of
the decode GEMV's main-loop waits to a few nanoseconds, so that the waits give
up while weight copies are still landing - no fault, no hang, no flag that is
never set - and then check that the status is reported and cleared, and that the
next call with the standard limit matches the oracle.
"""
import numpy as np
import pytest
import torch

import q4_weight_quantized_gb300 as q4k
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

TOL_SMALL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from q4_weight_quantized_gb300.build import build_library
    build_library()
    q4k.load()
    assert torch.cuda.is_available()
    yield
    q4k.q4k_set_gemv_wait_limit_ns(0)


@pytest.mark.parametrize("N,K,static", [(17408, 5120, False), (5120, 17408, False), (5120, 17408, True)],
                         ids=["wide", "k_split", "k_split_static_weights"])
def test_gemv_wait_runs_out_then_recovers(ref, N, K, static):
    b = G.weights(1, 0, N, K)
    x = G.activations(1, 1, 1, K)
    w = G.dev(b)
    xd = G.dev(x)
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")
    q4k.q4k_check_device()  # nothing pending
    prev_static = q4k.q4k_set_static_weights(static)
    try:
        assert q4k.q4k_set_gemv_wait_limit_ns(2) == 0
        for _ in range(3):
            q4k.q4k_gemv(w, N, K, xd, y)
        with pytest.raises(q4k.Q4KError) as err:
            q4k.q4k_check_device()
        assert err.value.status == q4k.Q4K_ERR_TIMEOUT
        q4k.q4k_check_device()  # reading the status cleared it
    finally:
        q4k.q4k_set_gemv_wait_limit_ns(0)
        q4k.q4k_set_static_weights(prev_static)
    # the context is intact: the same call with the standard limit is right
    q4k.q4k_gemv(w, N, K, xd, y)
    q4k.q4k_check_device()
    rows = G.sample_rows(N, 128, seed=9)
    want = ref.gemm(G.rows_of(b, rows), len(rows), K, x, threads=8)
    assert G.rel_err(G.host(y)[:, rows], want) <= TOL_SMALL
