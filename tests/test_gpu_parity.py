"""GPU parity: the CUDA path (through the C-ABI) against the oracle.

Bars: dequantization is bit-exact; the small-M path (M <= 16) is within
max|y - y_ref| / max|y_ref| <= 2e-3; the prefill and MoE tensor-core paths are
within 1e-2; routing is bit-exact.  Full-size workloads are checked on sampled
output rows (the oracle computes those rows one by one), in the launch
configuration the benchmark times.
"""
import functools

import numpy as np
import pytest
import torch

import q4_weight_quantized_gb300 as q4k
from tests import gpu_util as G
from tests.golden import load_blocks

pytestmark = pytest.mark.gpu

TOL_SMALL = 2e-3
TOL_TC = 1e-2
# the routed SwiGLU layer chains three tensor-core GEMMs; with every weight the
# nearest bf16 of its fp32 value, the layer holds the single-GEMM bar
TOL_FFN_TC = TOL_TC
# int8 activations: the sub-block dot products are exact integers on both sides;
# only the fp32 scaling and the fp32 sum over K/32 terms differ from the oracle's
# fp64 (at most ~(K/32) * 2^-24 of the sum of |terms|, typically far less)
TOL_X8 = TOL_SMALL / 10
# NVFP4: every weight enters the MMA as its exact bf16 value (e2m1 * e4m3), so
# only the fp32 accumulation order and the final multiplication by g differ
TOL_FP4 = TOL_SMALL / 10


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from q4_weight_quantized_gb300.build import build_library
    build_library()
    q4k.load()
    assert torch.cuda.is_available()
    yield
    q4k.q4k_check_device()


class batch_invariant:
    """q4k_set_batch_invariant(1) for the duration of a with-block (one-token calls
    then run the 2..16-token kernel)."""

    def __enter__(self):
        self.prev = q4k.q4k_set_batch_invariant(True)
        return self

    def __exit__(self, *a):
        q4k.q4k_set_batch_invariant(self.prev)


def gpu_dequant(blocks, N, K, bf16=False):
    w = G.dev(blocks)
    out = torch.empty((N, K), dtype=torch.int16 if bf16 else torch.float32, device="cuda")
    (q4k.q4k_dequant_bf16 if bf16 else q4k.q4k_dequant)(w, N, K, out)
    torch.cuda.synchronize()
    o = G.host(out)
    return o.view(np.uint16) if bf16 else o


def gpu_gemm(blocks, N, K, x, ldx=None, ldy=None, w_dev=None):
    M = x.shape[0]
    ldx = ldx or K
    ldy = ldy or N
    xp = np.zeros((M, ldx), np.uint16)
    xp[:, :K] = x
    w = w_dev if w_dev is not None else G.dev(blocks)
    xd = G.dev(xp)
    y = torch.full((M, ldy), float("nan"), dtype=torch.float32, device="cuda")
    ws_bytes = q4k.q4k_gemm_workspace_size(M, N, K)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda") if ws_bytes else None
    q4k.q4k_gemm(w, N, K, xd, M, ldx, y, ldy, ws, ws_bytes)
    torch.cuda.synchronize()
    out = G.host(y)
    if ldy > N:
        assert np.all(np.isnan(out[:, N:])), "wrote past N in the padded rows"
    return out[:, :N]


# ----------------------------------------------------------------- dequant

def test_dequant_tiny_bitexact(ref):
    cfg, N, K = G.TINY
    b = G.weights(cfg, 0, N, K)
    got = gpu_dequant(b, N, K)
    want = ref.dequant(b, N, K)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    got16 = gpu_dequant(b, N, K, bf16=True)
    assert np.array_equal(got16, ref.dequant_bf16(b, N, K))


def test_dequant_outliers_ragged_bitexact(ref):
    N, K = 37, 2304
    b = G.weights(3, 0, N, K, outliers=True)
    assert np.array_equal(gpu_dequant(b, N, K).view(np.uint32), ref.dequant(b, N, K).view(np.uint32))
    assert np.array_equal(gpu_dequant(b, N, K, True), ref.dequant_bf16(b, N, K))


def test_dequant_golden_blocks(ref):
    blocks = np.stack([f["block"] for f in load_blocks()])
    N = blocks.shape[0]
    got = gpu_dequant(blocks, N, 256)
    want = ref.dequant(blocks, N, 256)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_dequant_nan_inf_headers(ref):
    blk = load_blocks()[1]["block"].copy()
    nan_blk, inf_blk = blk.copy(), blk.copy()
    nan_blk[0:2] = [0x00, 0x7E]
    inf_blk[2:4] = [0x00, 0x7C]
    blocks = np.stack([nan_blk, inf_blk])
    got = gpu_dequant(blocks, 2, 256)
    want = ref.dequant(blocks, 2, 256)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


def test_dequant_full_size_bitexact(ref):
    cfg, N, K = G.DECODE_DOWN
    b = G.weights(cfg, 0, N, K)
    got = gpu_dequant(b, N, K)
    rows = G.sample_rows(N, 64)
    want = ref.dequant(G.rows_of(b, rows), len(rows), K)
    assert np.array_equal(got[rows].view(np.uint32), want.view(np.uint32))


# ------------------------------------------------------------- GEMV / small-M

def test_gemv_tiny(ref):
    cfg, N, K = G.TINY
    b = G.weights(cfg, 0, N, K)
    x = G.activations(cfg, 1, 1, K)
    w, xd = G.dev(b), G.dev(x)
    y = torch.empty(N, dtype=torch.float32, device="cuda")
    q4k.q4k_gemv(w, N, K, xd, y)
    torch.cuda.synchronize()
    assert G.rel_err(G.host(y), ref.gemm(b, N, K, x)[0]) <= TOL_SMALL


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 9, 15, 16])
def test_smallm_ragged(ref, M):
    N, K = 200, 1280          # N: 6 full 32-row tiles + a tail of 8; K: 5 blocks (ragged last stage)
    b = G.weights(2, 0, N, K, outliers=True)
    x = G.activations(2, 1, M, K)
    assert G.rel_err(gpu_gemm(b, N, K, x), ref.gemm(b, N, K, x)) <= TOL_SMALL


def test_smallm_strided_and_edges(ref):
    for (N, K, M) in [(1, 256, 1), (3, 256, 16), (33, 768, 7), (64, 512, 16)]:
        b = G.weights(2, 2, N, K)
        x = G.activations(2, 3, M, K)
        assert G.rel_err(gpu_gemm(b, N, K, x, ldx=K + 8, ldy=N + 5), ref.gemm(b, N, K, x)) <= TOL_SMALL


def test_one_hot_column_exact(ref):
    N, K = 64, 512
    b = G.weights(2, 4, N, K)
    w = ref.dequant(b, N, K)
    for k in (0, 37, 300, 511):
        x = np.zeros((1, K), np.uint16)
        x[0, k] = 0x3F80
        y = gpu_gemm(b, N, K, x)[0]
        assert np.array_equal(y, w[:, k]), k


def test_prefill_deterministic():
    M, N, K = 128, 5120, 17408   # the cluster split-K path
    b = G.weights(3, 0, N, K, outliers=True)
    w = G.dev(b)
    x = G.activations(3, 1, M, K)
    a = gpu_gemm(b, N, K, x, w_dev=w)
    c = gpu_gemm(b, N, K, x, w_dev=w)
    assert np.array_equal(a.view(np.uint32), c.view(np.uint32))


def test_batch_invariance_and_determinism():
    N, K = 17408, 5120
    b = G.weights(2, 0, N, K)
    w = G.dev(b)
    x = G.activations(2, 1, 16, K)
    y16 = gpu_gemm(b, N, K, x, w_dev=w)
    y16b = gpu_gemm(b, N, K, x, w_dev=w)
    assert np.array_equal(y16.view(np.uint32), y16b.view(np.uint32)), "not run-to-run deterministic"
    y4 = gpu_gemm(b, N, K, x[:4], w_dev=w)
    assert np.array_equal(y4.view(np.uint32), y16[:4].view(np.uint32))
    y2 = gpu_gemm(b, N, K, x[5:7], w_dev=w)
    assert np.array_equal(y2.view(np.uint32), y16[5:7].view(np.uint32))
    with batch_invariant():
        for m in (0, 5, 15):
            y1 = gpu_gemm(b, N, K, x[m:m + 1], w_dev=w)
            assert np.array_equal(y1[0].view(np.uint32), y16[m].view(np.uint32)), m


@pytest.mark.parametrize("KB", [1, 2, 3, 6, 7, 9, 11, 13])
def test_smallm_uneven_warp_blocks(ref, KB):
    # K blocks per split not divisible by the 4 warps (some warps take one block
    # more, or none), N 5120 over a cluster K split; batch invariance on the same shapes
    N, K = 5120, 256 * KB
    b = G.weights(2, 5, N, K, outliers=True)
    x = G.activations(2, 6, 16, K)
    w = G.dev(b)
    y16 = gpu_gemm(b, N, K, x, w_dev=w)
    rows = G.sample_rows(N, 256)
    want = ref.gemm(G.rows_of(b, rows), len(rows), K, x)
    assert G.rel_err(y16[:, rows], want) <= TOL_SMALL
    with batch_invariant():
        for m in (0, 9):
            y1 = gpu_gemm(b, N, K, x[m:m + 1], w_dev=w)
            assert np.array_equal(y1[0].view(np.uint32), y16[m].view(np.uint32)), m
    # the decode GEMV kernel on the same uneven splits
    y1 = gpu_gemm(b, N, K, x[9:10], w_dev=w)
    assert G.rel_err(y1[:, rows], want[9:10]) <= TOL_SMALL


@pytest.mark.parametrize("N,K", [(600, 16384), (1000, 17408)])
def test_smallm_cluster_split_of_eight(ref, N, K):
    # few row tiles and long K: clusters of 8 split K, so ranks 1..7 push their
    # partials (16 tokens: the largest landing buffer) into rank 0
    b = G.weights(2, 8, N, K)
    x = G.activations(2, 9, 16, K)
    w = G.dev(b)
    y16 = gpu_gemm(b, N, K, x, w_dev=w)
    rows = np.unique(np.concatenate([G.sample_rows(N, 96, seed=5), np.arange(N - 8, N)]))
    want = ref.gemm(G.rows_of(b, rows), len(rows), K, x, threads=8)
    assert G.rel_err(y16[:, rows], want) <= TOL_SMALL
    with batch_invariant():
        for m in (0, 13):
            y1 = gpu_gemm(b, N, K, x[m:m + 1], w_dev=w)
            assert np.array_equal(y1[0].view(np.uint32), y16[m].view(np.uint32)), m
    # the decode GEMV kernel: clusters of 8 as well (its landing buffer: one token)
    y1 = gpu_gemm(b, N, K, x[13:14], w_dev=w)
    assert G.rel_err(y1[:, rows], want[13:14]) <= TOL_SMALL


def test_batch_invariance_down_shape():
    # K 17408 over a 4-way cluster split: 17 blocks per CTA, so one warp takes 5 of them
    cfg, N, K = G.DECODE_DOWN
    b = G.weights(cfg, 0, N, K)
    w = G.dev(b)
    x = G.activations(cfg, 7, 16, K)
    y16 = gpu_gemm(b, N, K, x, w_dev=w)
    y4 = gpu_gemm(b, N, K, x[:4], w_dev=w)
    assert np.array_equal(y4.view(np.uint32), y16[:4].view(np.uint32))
    with batch_invariant():
        for m in (0, 7, 15):
            y1 = gpu_gemm(b, N, K, x[m:m + 1], w_dev=w)
            assert np.array_equal(y1[0].view(np.uint32), y16[m].view(np.uint32)), m


@pytest.mark.parametrize("N,K", [(1, 256), (3, 512), (200, 1280), (33, 2304), (1000, 3328), (5120, 17408),
                                 (600, 16384), (17408, 5120)])
def test_decode_gemv_kernel(ref, N, K):
    # the one-token kernel on ragged row tiles, K of 1..68 blocks (warps with no
    # block, uneven warps, cluster K splits of 2..8): against the oracle, run to
    # run, and against the small-M kernel (batch-invariant mode) within the bar
    b = G.weights(2, 11, N, K, outliers=True)
    x = G.activations(2, 12, 1, K)
    w = G.dev(b)
    y = gpu_gemm(b, N, K, x, w_dev=w)
    y2 = gpu_gemm(b, N, K, x, w_dev=w)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32)), "not run-to-run deterministic"
    rows = np.unique(np.concatenate([G.sample_rows(N, min(N, 128), seed=4), np.arange(max(0, N - 40), N)]))
    want = ref.gemm(G.rows_of(b, rows), len(rows), K, x, threads=8)
    assert G.rel_err(y[:, rows], want) <= TOL_SMALL
    with batch_invariant():
        yi = gpu_gemm(b, N, K, x, w_dev=w)
    assert G.rel_err(y, yi.astype(np.float64)) <= TOL_SMALL


def test_decode_gemv_activation_scale_exact():
    # the kernel scales the activations by a power of two inside its operands; so
    # does this test: 2^k x gives exactly 2^k y wherever no intermediate leaves the
    # normal range (|x| from 2^-56 to 2^63)
    N, K = 5120, 17408
    b = G.weights(2, 13, N, K)
    w = G.dev(b)
    x = G.activations(2, 14, 1, K)
    y = gpu_gemm(b, N, K, x, w_dev=w)
    for k in (-20, -7, 9, 40):
        xs = (x.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** k)
        xk = (xs.view(np.uint32) >> 16).astype(np.uint16)
        assert np.array_equal(((xk.astype(np.uint32) << 16).view(np.float32)), xs)  # exact in bf16
        yk = gpu_gemm(b, N, K, xk, w_dev=w)
        assert np.array_equal(yk.view(np.uint32), (y * np.float32(2.0 ** k)).view(np.uint32)), k


@pytest.mark.parametrize("shape", [G.DECODE_UP, G.DECODE_DOWN], ids=["gate_up", "down"])
def test_decode_gemv_full_size(ref, shape):
    cfg, N, K = shape
    b = G.weights(cfg, 0, N, K)
    x = G.activations(cfg, 1, 1, K)
    y = gpu_gemm(b, N, K, x)
    # sampled rows plus the last 64, which lie in the ragged last row tile
    rows = np.unique(np.concatenate([G.sample_rows(N, 256), np.arange(N - 64, N)]))
    want = ref.gemm(G.rows_of(b, rows), len(rows), K, x)
    assert G.rel_err(y[:, rows], want) <= TOL_SMALL


@pytest.mark.parametrize("M,N,K", [(1, 17408, 5120), (2, 17408, 5120), (4, 17408, 5120), (8, 17408, 5120),
                                   (16, 17408, 5120), (4, 5120, 17408), (16, 5120, 17408)])
def test_verify_gemm_full_size(ref, M, N, K):
    cfg = 2
    b = G.weights(cfg, 0, N, K)
    x = G.activations(cfg, 1, M, K)
    y = gpu_gemm(b, N, K, x)
    rows = np.unique(np.concatenate([G.sample_rows(N, 128), np.arange(N - 48, N)]))
    want = ref.gemm(G.rows_of(b, rows), len(rows), K, x, threads=8)
    assert G.rel_err(y[:, rows], want) <= TOL_SMALL



@pytest.mark.parametrize("N,K", [(2000, 5120), (5120, 17408)], ids=["ragged", "split_k"])
def test_static_weights_same_bits(ref, N, K):
    # the early weight copies change when the weights arrive, not what is computed
    b = G.weights(2, 3, N, K)
    w = G.dev(b)
    x = G.activations(2, 4, 16, K)
    off = {m: gpu_gemm(b, N, K, x[:m], w_dev=w) for m in (1, 4, 16)}
    prev = q4k.q4k_set_static_weights(True)
    try:
        assert q4k.q4k_set_static_weights(True) is True
        on = {m: gpu_gemm(b, N, K, x[:m], w_dev=w) for m in (1, 4, 16)}
    finally:
        q4k.q4k_set_static_weights(prev)
    for m in off:
        assert np.array_equal(off[m].view(np.uint32), on[m].view(np.uint32)), m
    rows = np.unique(np.concatenate([G.sample_rows(N, 48, seed=3), np.arange(N - 16, N)]))
    assert G.rel_err(on[16][:, rows], ref.gemm(G.rows_of(b, rows), len(rows), K, x, threads=8)) <= TOL_SMALL


def test_weights_written_by_the_previous_kernel(ref):
    # static weights off (the default): a kernel that writes the weight buffer
    # right before the call finishes before the GEMV reads it, every time
    assert q4k.q4k_set_static_weights(False) is False
    N, K = 4096, 5120
    b = G.weights(2, 5, N, K)
    src = G.dev(b)
    x = G.activations(2, 6, 1, K)
    xd = G.dev(x)
    key = torch.full_like(src, 0x5A)
    scrambled = torch.bitwise_xor(src, key)
    w = torch.empty_like(src)
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")
    outs = []
    for i in range(6):
        # alternate the buffer between garbage and the real weights with kernels
        torch.bitwise_xor(scrambled, key if i % 2 == 0 else torch.zeros_like(key), out=w)
        if i % 2 == 1:
            torch.bitwise_xor(w, key, out=w)
        q4k.q4k_gemv(w, N, K, xd, y)
        outs.append(G.host(y).copy())
    torch.cuda.synchronize()
    rows = G.sample_rows(N, 64, seed=9)
    want = ref.gemm(G.rows_of(b, rows), len(rows), K, x)
    for o in outs:
        assert G.rel_err(o[:, rows], want) <= TOL_SMALL


# ------------------------------------------------------------------ prefill

@pytest.mark.parametrize("M", [17, 40, 128])
def test_prefill_small(ref, M):
    N, K = 320, 2048
    b = G.weights(3, 0, N, K, outliers=True)
    x = G.activations(3, 1, M, K)
    assert G.rel_err(gpu_gemm(b, N, K, x), ref.gemm(b, N, K, x, threads=8)) <= TOL_TC


@pytest.mark.parametrize("M,N,K", [(200, 1000, 4096), (33, 640, 4096)])
def test_prefill_split_k_ragged(ref, M, N, K):
    # few output tiles: K is split over a thread-block cluster; ragged M and N
    b = G.weights(3, 2, N, K, outliers=True)
    x = G.activations(3, 3, M, K)
    assert G.rel_err(gpu_gemm(b, N, K, x), ref.gemm(b, N, K, x, threads=16)) <= TOL_TC


def test_prefill_last_wave_split(ref):
    # 160 tiles of 128 x 256 on 152 SMs: the last token tile (ragged, 232 tokens) becomes
    # a second launch with a cluster K split, which finishes after the main launch
    M, N, K = 1000, 5120, 2048
    b = G.weights(3, 7, N, K, outliers=True)
    x = G.activations(3, 8, M, K)
    y = gpu_gemm(b, N, K, x)
    rows = np.unique(np.concatenate([G.sample_rows(N, 24, seed=7), np.arange(N - 8, N)]))
    want = ref.gemm(G.rows_of(b, rows), len(rows), K, x, threads=16)
    assert G.rel_err(y[:, rows], want) <= TOL_TC


def test_prefill_many_tiles_ragged(ref):
    # more 128 x 256 tiles than SMs, ragged in M (600 = 2*256 + 88) and N (6600 = 51*128 + 72)
    M, N, K = 600, 6600, 1024
    b = G.weights(3, 5, N, K, outliers=True)
    x = G.activations(3, 6, M, K)
    y = gpu_gemm(b, N, K, x)
    rows = np.unique(np.concatenate([G.sample_rows(N, 40, seed=5), np.arange(N - 72, N)]))
    want = ref.gemm(G.rows_of(b, rows), len(rows), K, x, threads=16)
    assert G.rel_err(y[:, rows], want) <= TOL_TC


@pytest.mark.parametrize("M,N,K", [(128, 17408, 5120), (128, 5120, 17408), (1024, 17408, 5120),
                                   (1024, 5120, 17408), (4096, 17408, 5120), (4096, 5120, 17408)])
def test_prefill_full_size(ref, M, N, K):
    # (4096, 5120, 17408) runs as the benchmark's two launches: 15 token tiles, then
    # the last one with the cluster K split
    b = G.weights(3, 0, N, K, outliers=True)
    x = G.activations(3, 1, M, K)
    y = gpu_gemm(b, N, K, x)
    rows = G.sample_rows(N, 24)
    want = ref.gemm(G.rows_of(b, rows), len(rows), K, x, threads=16)
    assert G.rel_err(y[:, rows], want) <= TOL_TC


@pytest.mark.parametrize("N,K", [(17408, 5120), (5120, 17408)], ids=["up", "down"])
def test_prefill_batch_invariant_mode(ref, N, K):
    # q4k_set_batch_invariant(1) on the tensor-core path (M > 16): the K split is
    # chosen from the weight shape alone and no last-wave launch is split off, so a
    # token's output row has the same bits in calls of 17 to 4096 tokens at any
    # offset in the batch.  On the down projection's shape the split is 2-way over a
    # cluster pair at every M (17, 128 and 129 tokens take 128-token tiles, the
    # longer calls 256-token tiles)
    b = G.weights(3, 0, N, K, outliers=True)
    w = G.dev(b)
    x = G.activations(3, 1, 4096, K)
    with batch_invariant():
        yfull = gpu_gemm(b, N, K, x, w_dev=w)
        for m0, M in ((0, 128), (0, 1000), (1000, 17), (2900, 1000), (4096 - 300, 300), (77, 129)):
            y = gpu_gemm(b, N, K, x[m0:m0 + M], w_dev=w)
            assert np.array_equal(y.view(np.uint32), yfull[m0:m0 + M].view(np.uint32)), (m0, M)
    rows = G.sample_rows(N, 16)
    toks = G.sample_rows(4096, 24, seed=5)
    want = ref.gemm(G.rows_of(b, rows), len(rows), K, x[toks], threads=16)
    assert G.rel_err(yfull[np.ix_(toks, rows)], want) <= TOL_TC


# ---------------------------------------------------------------------- MoE

def test_moe_route_bitexact(ref, syn):
    for T in (1, 16, 2048):
        ids, _ = syn.routing(syn.seed(4, 2) + T, syn.seed(4, 3), T, G.MOE_E, G.MOE_TOPK)
        off, perm = torch.empty(G.MOE_E + 1, dtype=torch.int32, device="cuda"), \
            torch.empty(T * G.MOE_TOPK, dtype=torch.int32, device="cuda")
        q4k.q4k_moe_route(G.dev(ids), T, G.MOE_TOPK, G.MOE_E, off, perm)
        torch.cuda.synchronize()
        want_off, want_perm, bad = ref.moe_route(ids, G.MOE_E)
        assert bad == 0
        assert np.array_equal(G.host(off), want_off)
        assert np.array_equal(G.host(perm), want_perm)


def test_moe_route_invalid_ids(ref):
    rng = np.random.default_rng(1)
    T, topk, E = 300, 4, 37
    ids = rng.integers(-3, E + 3, (T, topk)).astype(np.int32)
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * topk, dtype=torch.int32, device="cuda")
    q4k.q4k_moe_route(G.dev(ids), T, topk, E, off, perm)
    torch.cuda.synchronize()
    want_off, want_perm, _ = ref.moe_route(ids, E)
    assert np.array_equal(G.host(off), want_off) and np.array_equal(G.host(perm), want_perm)



@pytest.mark.parametrize("T,topk,E,skew", [(5000, 3, 1024, False), (4000, 2, 8, True), (70000, 8, 128, False)],
                         ids=["E1024", "skewed", "560k_items"])
def test_moe_route_many_ctas(ref, T, topk, E, skew):
    # the routing spreads its items over up to 128 CTAs (ranges of a multiple of 512):
    # positions must still be the stable order across range boundaries, invalid ids included
    rng = np.random.default_rng(T)
    if skew:
        ids = np.where(rng.random((T, topk)) < 0.9, 3, rng.integers(-1, E + 1, (T, topk))).astype(np.int32)
    else:
        ids = rng.integers(-2, E + 2, (T, topk)).astype(np.int32)
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * topk, dtype=torch.int32, device="cuda")
    q4k.q4k_moe_route(G.dev(ids), T, topk, E, off, perm)
    torch.cuda.synchronize()
    want_off, want_perm, _ = ref.moe_route(ids, E)
    assert np.array_equal(G.host(off), want_off) and np.array_equal(G.host(perm), want_perm)


def run_moe(w_blocks, E, N, K, x, x_mode, ids, gates, y_mode, w_dev=None):
    T, topk = ids.shape
    w = w_dev if w_dev is not None else G.dev(w_blocks)
    ws_bytes = q4k.q4k_moe_workspace_size(E, N, K, T, topk, y_mode)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    shape = (T, N) if y_mode == q4k.Q4K_MOE_Y_COMBINE else (T, topk, N)
    y = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
    q4k.q4k_moe_grouped_gemm(w, E, N, K, G.dev(x), x_mode, G.dev(ids), G.dev(gates), T, topk, y, y_mode, ws,
                             ws_bytes)
    torch.cuda.synchronize()
    return G.host(y)


@pytest.fixture(scope="module")
def moe_up():
    N, K = G.MOE_UP
    return G.moe_experts(4, 0, N, K)


@pytest.fixture(scope="module")
def moe_down():
    N, K = G.MOE_DOWN
    return G.moe_experts(4, 5, N, K)


@pytest.mark.parametrize("T", [1, 2, 3, 16])
def test_moe_gate_up_per_slot(ref, syn, moe_up, T):
    N, K = G.MOE_UP
    ids, gates = syn.routing(syn.seed(4, 2) + T, syn.seed(4, 3) + T, T, G.MOE_E, G.MOE_TOPK)
    x = G.activations(4, 1, T, K)
    y = run_moe(moe_up, G.MOE_E, N, K, x, q4k.Q4K_MOE_X_PER_TOKEN, ids, gates, q4k.Q4K_MOE_Y_PER_SLOT)
    want = ref.moe_slots(moe_up, G.MOE_E, N, K, x, False, ids, threads=8)
    assert G.rel_err(y, want) <= TOL_SMALL


@pytest.mark.parametrize("T", [1, 2, 3, 16])
def test_moe_down_combine(ref, syn, moe_down, T):
    N, K = G.MOE_DOWN
    ids, gates = syn.routing(syn.seed(4, 2) + T, syn.seed(4, 3) + T, T, G.MOE_E, G.MOE_TOPK)
    x = G.activations(4, 6, T * G.MOE_TOPK, K)
    y = run_moe(moe_down, G.MOE_E, N, K, x, q4k.Q4K_MOE_X_PER_SLOT, ids, gates, q4k.Q4K_MOE_Y_COMBINE)
    want = ref.moe(moe_down, G.MOE_E, N, K, x, True, ids, gates, threads=8)
    assert G.rel_err(y, want) <= TOL_SMALL


def test_moe_t2048_sampled(ref, syn, moe_up, moe_down):
    T, E, topk = 2048, G.MOE_E, G.MOE_TOPK
    ids, gates = syn.routing(syn.seed(4, 2) + T, syn.seed(4, 3) + T, T, E, topk)
    tok = G.sample_rows(T, 40, seed=3)
    # gate/up, per-slot rows
    N, K = G.MOE_UP
    x = G.activations(4, 1, T, K)
    y = run_moe(moe_up, E, N, K, x, q4k.Q4K_MOE_X_PER_TOKEN, ids, gates, q4k.Q4K_MOE_Y_PER_SLOT)
    want = ref.moe_slots(moe_up, E, N, K, x[tok], False, ids[tok], threads=16)
    assert G.rel_err(y[tok], want) <= TOL_TC
    # down with the weighted combine
    N, K = G.MOE_DOWN
    xs = G.activations(4, 6, T * topk, K).reshape(T, topk, K)
    y = run_moe(moe_down, E, N, K, xs.reshape(T * topk, K), q4k.Q4K_MOE_X_PER_SLOT, ids, gates,
                q4k.Q4K_MOE_Y_COMBINE)
    want = ref.moe(moe_down, E, N, K, xs[tok].reshape(-1, K), True, ids[tok], gates[tok], threads=16)
    assert G.rel_err(y[tok], want) <= TOL_TC


def test_moe_special_cases(ref, syn):
    # every token routed to experts 0..7 in order: per-slot output j equals a dense GEMM with expert j
    E, N, K, T, topk = 12, 96, 512, 5, 8
    w = np.concatenate([G.weights(4, 30 + e, N, K) for e in range(E)])
    ids = np.tile(np.arange(topk, dtype=np.int32), (T, 1))
    gates = np.full((T, topk), 1.0 / topk, np.float32)
    x = G.activations(4, 7, T, K)
    y = run_moe(w, E, N, K, x, q4k.Q4K_MOE_X_PER_TOKEN, ids, gates, q4k.Q4K_MOE_Y_PER_SLOT)
    for j in range(topk):
        dense = gpu_gemm(w[j * N:(j + 1) * N], N, K, x)
        assert G.rel_err(y[:, j], dense) <= TOL_SMALL
    # one-hot gates: the combine returns the chosen slot
    ids2, _ = syn.routing(77, 78, T, E, topk)
    onehot = np.zeros((T, topk), np.float32)
    pick = np.arange(T) % topk
    onehot[np.arange(T), pick] = 1.0
    xs = G.activations(4, 8, T * topk, K)
    yc = run_moe(w, E, N, K, xs, q4k.Q4K_MOE_X_PER_SLOT, ids2, onehot, q4k.Q4K_MOE_Y_COMBINE)
    ys = run_moe(w, E, N, K, xs, q4k.Q4K_MOE_X_PER_SLOT, ids2, onehot, q4k.Q4K_MOE_Y_PER_SLOT)
    assert np.array_equal(yc, ys[np.arange(T), pick])
    # invalid ids: zero per-slot rows, and no contribution to the combine
    ids3 = ids2.copy()
    ids3[0, 0] = -1
    ids3[2, 5] = E
    ys3 = run_moe(w, E, N, K, xs, q4k.Q4K_MOE_X_PER_SLOT, ids3, onehot, q4k.Q4K_MOE_Y_PER_SLOT)
    assert np.all(ys3[0, 0] == 0) and np.all(ys3[2, 5] == 0)
    want = ref.moe(w, E, N, K, xs, True, ids3, onehot)
    yc3 = run_moe(w, E, N, K, xs, q4k.Q4K_MOE_X_PER_SLOT, ids3, onehot, q4k.Q4K_MOE_Y_COMBINE)
    assert G.rel_err(yc3, want) <= TOL_SMALL



@pytest.mark.parametrize("T", [1, 16, 256, 600])
def test_moe_reuse_routing_same_bits(syn, moe_up, moe_down, T):
    # one routing call, then the layer's other projections reuse its sort: the
    # same bits as routing every call, invalid ids included (T = 600: tensor cores)
    E, topk = G.MOE_E, G.MOE_TOPK
    (Nu, Ku), (Nd, Kd) = G.MOE_UP, G.MOE_DOWN
    ids, gates = syn.routing(90 + T, 91 + T, T, E, topk)
    ids[0, 3] = -1
    ids[T - 1, 0] = E + 7
    x = G.dev(G.activations(4, 20, T, Ku))
    xd = G.dev(G.activations(4, 21, T * topk, Kd))
    wu, wd = G.dev(moe_up), G.dev(moe_down)
    wu2 = G.dev(np.ascontiguousarray(moe_up[::-1]))   # another "up" matrix: the experts in reverse order
    idd, gd = G.dev(ids), G.dev(gates)
    P, C = q4k.Q4K_MOE_Y_PER_SLOT, q4k.Q4K_MOE_Y_COMBINE
    calls = [(wu, Nu, Ku, x, q4k.Q4K_MOE_X_PER_TOKEN, P), (wu2, Nu, Ku, x, q4k.Q4K_MOE_X_PER_TOKEN, P),
             (wd, Nd, Kd, xd, q4k.Q4K_MOE_X_PER_SLOT, C)]
    size = max(q4k.q4k_moe_workspace_size(E, N, K, T, topk, ym) for (_, N, K, _, _, ym) in calls)
    ws = torch.empty(size, dtype=torch.uint8, device="cuda")

    def out(N, ym):
        return torch.full((T, N) if ym == C else (T, topk, N), float("nan"), dtype=torch.float32, device="cuda")

    shared, fresh = [], []
    for i, (w, N, K, xx, xm, ym) in enumerate(calls):
        y = out(N, ym)
        fn = q4k.q4k_moe_grouped_gemm if i == 0 else q4k.q4k_moe_grouped_gemm_reuse_routing
        fn(w, E, N, K, xx, xm, idd, gd, T, topk, y, ym, ws, size)
        shared.append(y)
    for (w, N, K, xx, xm, ym) in calls:
        y = out(N, ym)
        wsf = torch.empty(q4k.q4k_moe_workspace_size(E, N, K, T, topk, ym), dtype=torch.uint8, device="cuda")
        q4k.q4k_moe_grouped_gemm(w, E, N, K, xx, xm, idd, gd, T, topk, y, ym, wsf, wsf.numel())
        fresh.append(y)
    torch.cuda.synchronize()
    for a, b in zip(shared, fresh):
        a, b = G.host(a), G.host(b)
        assert not np.isnan(a).any()
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    for y in shared[:2]:
        h = G.host(y)
        assert np.all(h[0, 3] == 0) and np.all(h[T - 1, 0] == 0)



@pytest.mark.parametrize("T,T2", [(16, 20), (600, 601)])
def test_moe_reuse_routing_checks_the_shape(syn, moe_up, T, T2):
    # a routing made for T tokens reused by a call with T2: the kernels find the
    # workspace's routing stamped with another item count, write nothing, and
    # q4k_check_device reports it; a workspace that never held a routing is
    # refused the same way; the next ordinary call is unaffected
    E, topk = G.MOE_E, G.MOE_TOPK
    N, K = G.MOE_UP
    P = q4k.Q4K_MOE_Y_PER_SLOT
    wu = G.dev(moe_up)
    size = max(q4k.q4k_moe_workspace_size(E, N, K, t, topk, P) for t in (T, T2))
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    ids, gates = syn.routing(70 + T, 71 + T, T2, E, topk)
    idd, gd = G.dev(ids), G.dev(gates)
    x = G.dev(G.activations(4, 22, T2, K))

    def call(fn, t):
        y = torch.full((t, topk, N), float("nan"), dtype=torch.float32, device="cuda")
        fn(wu, E, N, K, x, q4k.Q4K_MOE_X_PER_TOKEN, idd, gd, t, topk, y, P, ws, size)
        return y

    y = call(q4k.q4k_moe_grouped_gemm_reuse_routing, T2)  # nothing routed yet
    with pytest.raises(q4k.Q4KError) as err:
        q4k.q4k_check_device()
    assert err.value.status == q4k.Q4K_ERR_ROUTING
    assert np.isnan(G.host(y)).all()
    call(q4k.q4k_moe_grouped_gemm, T)  # a routing for the first T tokens
    y = call(q4k.q4k_moe_grouped_gemm_reuse_routing, T2)
    with pytest.raises(q4k.Q4KError) as err:
        q4k.q4k_check_device()
    assert err.value.status == q4k.Q4K_ERR_ROUTING
    assert np.isnan(G.host(y)).all()
    good = call(q4k.q4k_moe_grouped_gemm, T2)
    again = call(q4k.q4k_moe_grouped_gemm_reuse_routing, T2)
    q4k.q4k_check_device()
    a, b = G.host(good), G.host(again)
    assert not np.isnan(a).any() and np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("K", [768, 2048])
def test_moe_few_items_direct(ref, syn, K):
    # up to 16 items: every item is its own grid layer, its expert read from the ids
    # (no routing); ragged N, invalid ids give zero rows and no combine contribution
    E, N, T, topk = 12, 200, 2, 8
    w = np.concatenate([G.weights(4, 80 + e, N, K) for e in range(E)])
    ids, gates = syn.routing(91, 92, T, E, topk)
    ids[0, 2] = -4
    ids[1, 7] = E
    x = G.activations(4, 13, T, K)
    y = run_moe(w, E, N, K, x, q4k.Q4K_MOE_X_PER_TOKEN, ids, gates, q4k.Q4K_MOE_Y_PER_SLOT)
    assert np.all(y[0, 2] == 0) and np.all(y[1, 7] == 0)
    assert G.rel_err(y, ref.moe_slots(w, E, N, K, x, False, ids)) <= TOL_SMALL
    xs = G.activations(4, 14, T * topk, K)
    yc = run_moe(w, E, N, K, xs, q4k.Q4K_MOE_X_PER_SLOT, ids, gates, q4k.Q4K_MOE_Y_COMBINE)
    assert G.rel_err(yc, ref.moe(w, E, N, K, xs, True, ids, gates)) <= TOL_SMALL


def _fma_f32(a: float, b: float, c: float) -> float:
    """fmaf: a*b + c rounded once to binary32 (nearest, ties to even), exactly."""
    from fractions import Fraction
    v = Fraction(a) * Fraction(b) + Fraction(c)
    if v == 0:
        return 0.0 if (a * b == 0 and c == 0 and not np.signbit(c)) else float(np.float32(float(v)))
    lo = float(np.float32(float(v)))          # a binary32 neighbour of v
    cands = {lo, float(np.nextafter(np.float32(lo), np.float32(np.inf))),
             float(np.nextafter(np.float32(lo), np.float32(-np.inf)))}
    best = min(cands, key=lambda f: (abs(Fraction(f) - v),
                                     int(np.array([f], np.float32).view(np.uint32)[0]) & 1))
    return best


@pytest.mark.parametrize("T,x_mode", [(1, 1), (2, 1), (2, 0)])
def test_moe_combine_in_cta_same_bits(syn, moe_down, T, x_mode):
    # up to 16 items: the down projection sums the slots in the CTA; the result must be
    # the fp32 fma chain over the per-slot rows in slot order, invalid ids skipped
    N, K = G.MOE_DOWN
    E, topk = G.MOE_E, G.MOE_TOPK
    ids, gates = syn.routing(syn.seed(4, 2) + 50 + T, syn.seed(4, 3) + 50 + T, T, E, topk)
    ids[0, 5] = -1
    x = G.activations(4, 9, T * topk if x_mode else T, K)
    w = G.dev(moe_down)
    y = run_moe(None, E, N, K, x, x_mode, ids, gates, q4k.Q4K_MOE_Y_COMBINE, w_dev=w)
    o = run_moe(None, E, N, K, x, x_mode, ids, gates, q4k.Q4K_MOE_Y_PER_SLOT, w_dev=w)
    cols = G.sample_rows(N, 48, seed=T)
    for t in range(T):
        for n in cols:
            acc = 0.0
            for j in range(topk):
                if 0 <= ids[t, j] < E:
                    acc = _fma_f32(float(gates[t, j]), float(o[t, j, n]), acc)
            assert np.float32(acc).view(np.uint32) == np.float32(y[t, n]).view(np.uint32), (t, n)


def test_moe_determinism(syn, moe_up):
    N, K = G.MOE_UP
    T = 16
    ids, gates = syn.routing(5, 6, T, G.MOE_E, G.MOE_TOPK)
    x = G.activations(4, 1, T, K)
    w = G.dev(moe_up)
    a = run_moe(moe_up, G.MOE_E, N, K, x, 0, ids, gates, 0, w_dev=w)
    b = run_moe(moe_up, G.MOE_E, N, K, x, 0, ids, gates, 0, w_dev=w)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("E,T,topk,N,K", [(4, 64, 2, 256, 512), (3, 300, 2, 200, 768)])
def test_moe_tensor_core_path(ref, syn, E, T, topk, N, K):
    # >= 32 items per expert on average: the tcgen05 path with expert-sorted rows;
    # the second case has experts with more than 192 items (several token tiles)
    w = np.concatenate([G.weights(4, 60 + e, N, K, outliers=True) for e in range(E)])
    ids, gates = syn.routing(700 + T, 701 + T, T, E, topk)
    ids[3, 1] = -5                                   # an invalid id: zero row, no contribution
    x = G.activations(4, 11, T, K)
    y = run_moe(w, E, N, K, x, q4k.Q4K_MOE_X_PER_TOKEN, ids, gates, q4k.Q4K_MOE_Y_PER_SLOT)
    want = ref.moe_slots(w, E, N, K, x, False, ids, threads=16)
    assert np.all(y[3, 1] == 0.0)
    assert G.rel_err(y, want) <= TOL_TC
    xs = G.activations(4, 12, T * topk, K)
    yc = run_moe(w, E, N, K, xs, q4k.Q4K_MOE_X_PER_SLOT, ids, gates, q4k.Q4K_MOE_Y_COMBINE)
    yc2 = run_moe(w, E, N, K, xs, q4k.Q4K_MOE_X_PER_SLOT, ids, gates, q4k.Q4K_MOE_Y_COMBINE)
    assert np.array_equal(yc.view(np.uint32), yc2.view(np.uint32))
    want_c = ref.moe(w, E, N, K, xs, True, ids, gates, threads=16)
    assert G.rel_err(yc, want_c) <= TOL_TC


# ------------------------------------------------------- routed expert FFN layer
def run_ffn(wg, wu, wd, E, H, D, x, ids, gates, devs=None):
    T, topk = ids.shape
    if devs is None:
        devs = (G.dev(wg), G.dev(wu), G.dev(wd))
    ws_bytes = q4k.q4k_moe_ffn_workspace_size(E, H, D, T, topk)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    y = torch.full((T, D), float("nan"), dtype=torch.float32, device="cuda")
    q4k.q4k_moe_ffn(*devs, E, H, D, G.dev(x), G.dev(ids), G.dev(gates), T, topk, y, ws, ws_bytes)
    torch.cuda.synchronize()
    return G.host(y)


@pytest.fixture(scope="module")
def ffn_layer():
    # the 128-expert layer: gate and up K 2048 -> H 768, down K 768 -> D 2048
    (H, D), (D2, H2) = G.MOE_UP, G.MOE_DOWN
    assert (H, D) == (H2, D2)
    wg = G.moe_experts(4, 40, H, D)
    wu = G.moe_experts(4, 41, H, D)
    wd = G.moe_experts(4, 42, D, H)
    return wg, wu, wd, (G.dev(wg), G.dev(wu), G.dev(wd))


@pytest.mark.parametrize("T", [1, 2, 3, 16])
def test_moe_ffn_layer(ref, syn, ffn_layer, T):
    # few items (direct and routed small-M paths): gate, up with the SwiGLU
    # epilogue, down on the bf16 h rows, ordered combine; invalid ids add nothing
    wg, wu, wd, devs = ffn_layer
    (H, D), E, topk = G.MOE_UP, G.MOE_E, G.MOE_TOPK
    ids, gates = syn.routing(300 + T, 301 + T, T, E, topk)
    if T > 1:
        ids[1, 4] = -1
    x = G.activations(4, 43, T, D)
    y = run_ffn(wg, wu, wd, E, H, D, x, ids, gates, devs)
    want = ref.moe_ffn(wg, wu, wd, E, H, D, x, ids, gates, threads=16)
    assert not np.isnan(y).any()
    assert G.rel_err(y, want) <= TOL_SMALL


@pytest.mark.parametrize("T", [1, 2])
def test_moe_ffn_static_weights_ids_from_the_previous_kernel(ref, syn, ffn_layer, T):
    # static weights on: the down projection of the fused small layer reads the ids
    # and copies its first expert weight blocks before its own wait.  The ids
    # alternate between two routings, each written by a device copy right before the
    # call, with no host synchronization in between; results match the oracle and
    # the bits of the default mode
    wg, wu, wd, devs = ffn_layer
    (H, D), E, topk = G.MOE_UP, G.MOE_E, G.MOE_TOPK
    routes = [syn.routing(310 + T + 7 * i, 311 + T + 7 * i, T, E, topk) for i in range(2)]
    routes[1][0][0, 2] = -1
    x = G.activations(4, 46, T, D)
    xd = G.dev(x)
    ids_src = [G.dev(r[0]) for r in routes]
    gates_d = [G.dev(r[1]) for r in routes]
    ids_d = torch.empty_like(ids_src[0])
    ws_bytes = q4k.q4k_moe_ffn_workspace_size(E, H, D, T, topk)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    y = torch.empty((T, D), dtype=torch.float32, device="cuda")
    outs = torch.empty((6, T, D), dtype=torch.float32, device="cuda")
    prev = q4k.q4k_set_static_weights(True)
    try:
        for i in range(6):
            ids_d.copy_(ids_src[i % 2])
            q4k.q4k_moe_ffn(*devs, E, H, D, xd, ids_d, gates_d[i % 2], T, topk, y, ws, ws_bytes)
            outs[i].copy_(y)
        torch.cuda.synchronize()
    finally:
        q4k.q4k_set_static_weights(prev)
    got = G.host(outs)
    for j in range(2):
        ids, gates = routes[j]
        want = ref.moe_ffn(wg, wu, wd, E, H, D, x, ids, gates, threads=16)
        off = run_ffn(wg, wu, wd, E, H, D, x, ids, gates, devs)
        for i in range(j, 6, 2):
            assert G.rel_err(got[i], want) <= TOL_SMALL, (i, j)
            assert np.array_equal(got[i].view(np.uint32), off.view(np.uint32)), (i, j)


def test_moe_ffn_t2048_sampled(ref, syn, ffn_layer):
    # the prefill-sized layer (tensor-core path, h stored expert-sorted), in the
    # configuration the benchmark times; the oracle computes sampled tokens
    wg, wu, wd, devs = ffn_layer
    (H, D), E, topk = G.MOE_UP, G.MOE_E, G.MOE_TOPK
    T = 2048
    ids, gates = syn.routing(syn.seed(4, 2) + T, syn.seed(4, 3) + T, T, E, topk)
    x = G.activations(4, 44, T, D)
    y = run_ffn(wg, wu, wd, E, H, D, x, ids, gates, devs)
    assert not np.isnan(y).any()
    tok = G.sample_rows(T, 32, seed=5)
    want = ref.moe_ffn(wg, wu, wd, E, H, D, x[tok], ids[tok], gates[tok], threads=16)
    assert G.rel_err(y[tok], want) <= TOL_FFN_TC
    # the gap to the oracle is the bf16 weight operand's rounding: with that rounding
    # modelled (and nothing else), the kernels agree to fp32 accumulation order
    xb = (x[tok[:6]].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    rb_d, rb_h = D // 256 * 144, H // 256 * 144
    model = np.zeros((len(xb), D))
    for i, t in enumerate(tok[:6]):
        for j in range(topk):
            e = int(ids[t, j])
            g = G.tc_weights(wg.reshape(-1)[e * H * rb_d:(e + 1) * H * rb_d], H, D) @ xb[i]
            u = G.tc_weights(wu.reshape(-1)[e * H * rb_d:(e + 1) * H * rb_d], H, D) @ xb[i]
            h = G._bf16(g / (1.0 + np.exp(-g)) * u)
            model[i] += gates[t, j] * (G.tc_weights(wd.reshape(-1)[e * D * rb_h:(e + 1) * D * rb_h], D, H) @ h)
    assert G.rel_err(y[tok[:6]], model) <= 1e-3


@pytest.mark.parametrize("E,T,topk,H,D", [(4, 64, 2, 256, 512), (3, 300, 2, 512, 768), (6, 40, 3, 256, 256)])
def test_moe_ffn_small_layers(ref, syn, E, T, topk, H, D):
    # the tensor-core path with several token tiles per expert, and the small-M
    # path with row-split CTAs (K = 256); invalid ids, a token with no valid id
    wg = np.concatenate([G.weights(4, 200 + e, H, D, outliers=True) for e in range(E)])
    wu = np.concatenate([G.weights(4, 220 + e, H, D) for e in range(E)])
    wd = np.concatenate([G.weights(4, 240 + e, D, H) for e in range(E)])
    ids, gates = syn.routing(900 + T, 901 + T, T, E, topk)
    ids[3, 1] = -5
    ids[5, :] = E
    x = G.activations(4, 45, T, D)
    y = run_ffn(wg, wu, wd, E, H, D, x, ids, gates)
    want = ref.moe_ffn(wg, wu, wd, E, H, D, x, ids, gates, threads=16)
    assert np.all(y[5] == 0.0)
    tol = TOL_FFN_TC if T * topk >= 32 * E else TOL_SMALL
    assert G.rel_err(y, want) <= tol


@pytest.mark.parametrize("T", [16, 600])
def test_moe_ffn_matches_grouped_calls_and_is_deterministic(syn, ffn_layer, T):
    # same bits on a second call; and the same as the layer written with the
    # grouped-GEMM calls when h is formed the same way (fp32 SwiGLU rounded to bf16)
    wg, wu, wd, devs = ffn_layer
    (H, D), E, topk = G.MOE_UP, G.MOE_E, G.MOE_TOPK
    ids, gates = syn.routing(500 + T, 501 + T, T, E, topk)
    x = G.activations(4, 46, T, D)
    a = run_ffn(wg, wu, wd, E, H, D, x, ids, gates, devs)
    b = run_ffn(wg, wu, wd, E, H, D, x, ids, gates, devs)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    P, C = q4k.Q4K_MOE_Y_PER_SLOT, q4k.Q4K_MOE_Y_COMBINE
    g = run_moe(None, E, H, D, x, q4k.Q4K_MOE_X_PER_TOKEN, ids, gates, P, w_dev=devs[0])
    u = run_moe(None, E, H, D, x, q4k.Q4K_MOE_X_PER_TOKEN, ids, gates, P, w_dev=devs[1])
    gt, ut = torch.from_numpy(g), torch.from_numpy(u)
    h = (gt / (1.0 + torch.exp(-gt)) * ut).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    yc = run_moe(None, E, D, H, h.reshape(T * topk, H), q4k.Q4K_MOE_X_PER_SLOT, ids, gates, C, w_dev=devs[2])
    # h may differ in the last bf16 place where host and device exp differ
    assert G.rel_err(a, yc) <= TOL_SMALL


# ------------------------------------------------------------ int8 activations
def gpu_quantize_x8(x, ldx=None):
    M, K = x.shape
    ldx = ldx or K
    xp = np.zeros((M, ldx), np.uint16)
    xp[:, :K] = x
    q = torch.empty((M, K), dtype=torch.int8, device="cuda")
    sc = torch.full((M, K // 32), float("nan"), dtype=torch.float32, device="cuda")
    q4k.q4k_quantize_x8(G.dev(xp), M, K, ldx, q, sc)
    torch.cuda.synchronize()
    return G.host(q), G.host(sc)


def gpu_gemm_x8(blocks, N, K, q, sc, w_dev=None, ldy=None):
    M = q.shape[0]
    ldy = ldy or N
    y = torch.full((M, ldy), float("nan"), dtype=torch.float32, device="cuda")
    w = w_dev if w_dev is not None else G.dev(blocks)
    wsb = q4k.q4k_gemm_x8_workspace_size(M, K)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda") if wsb else None
    q4k.q4k_gemm_x8(w, N, K, G.dev(np.ascontiguousarray(q)), G.dev(np.ascontiguousarray(sc)), M, y, ldy, ws, wsb)
    torch.cuda.synchronize()
    out = G.host(y)
    if ldy > N:
        assert np.all(np.isnan(out[:, N:]))
    return out[:, :N]


def test_quantize_x8_bitexact(ref):
    M, K = 5, 1024
    x = G.activations(6, 1, M, K).copy()
    x[0, 32:64] = 0                                   # an all-zero block
    x[1, 64:96] = 0
    x[1, 70] = 0x4040                                 # a single non-zero (3.0)
    # exact ties: largest 127/8, then k.5/8
    tie = np.zeros(32)
    tie[0] = 127 / 8
    tie[1:9] = np.array([0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, 126.5]) / 8
    x[2, 0:32] = (np.asarray(tie, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    x[3, :] = 0x0001                                  # tiny subnormal bf16 values
    for ldx in (K, K + 64):
        q, sc = gpu_quantize_x8(x, ldx)
        rq, rs = ref.quantize_x8(x)
        assert np.array_equal(q, rq)
        assert np.array_equal(sc.view(np.uint32), rs.view(np.uint32))
    assert list(q[2, :9]) == [127, 0, 2, 2, 4, 0, -2, -2, 126]


def test_quantize_x8_full_size_bitexact(ref):
    M, K = 16, 17408
    x = G.activations(6, 2, M, K)
    q, sc = gpu_quantize_x8(x)
    rq, rs = ref.quantize_x8(x)
    assert np.array_equal(q, rq) and np.array_equal(sc.view(np.uint32), rs.view(np.uint32))


@pytest.mark.parametrize("M", [1, 2, 3, 8, 9, 16])
def test_gemm_x8_ragged(ref, M):
    N, K = 200, 1024
    w = G.weights(6, 3, N, K, outliers=True)
    x = G.activations(6, 4, M, K)
    q, sc = ref.quantize_x8(x)
    y = gpu_gemm_x8(w, N, K, q, sc, ldy=N + 8)
    assert G.rel_err(y, ref.gemm_x8(w, N, K, q, sc)) <= TOL_X8


@pytest.mark.parametrize("shape", [G.DECODE_UP, G.DECODE_DOWN], ids=["gate_up", "down"])
@pytest.mark.parametrize("M", [1, 4])
def test_gemm_x8_full_size(ref, shape, M):
    # the decode and verify shapes in the benchmark's configuration, sampled rows
    _, N, K = shape
    w = G.weights(1, 0 if N == 17408 else 5, N, K)
    x = G.activations(6, 5, M, K)
    q, sc = gpu_quantize_x8(x)
    y = gpu_gemm_x8(w, N, K, q, sc)
    rows = G.sample_rows(N, 64, seed=M)
    want = ref.gemm_x8(G.rows_of(w, rows), len(rows), K, q, sc)
    assert G.rel_err(y[:, rows], want) <= TOL_X8


@pytest.mark.parametrize("M,N,K", [(17, 200, 1024), (129, 300, 768), (300, 1000, 4096)])
def test_gemm_x8_prefill(ref, M, N, K):
    # M > 16: bf16(s * q) in the workspace, then the tensor-core GEMM (ragged
    # token tiles, the cluster K split at N = 300 and 1000)
    w = G.weights(6, 7, N, K, outliers=True)
    x = G.activations(6, 8, M, K)
    q, sc = ref.quantize_x8(x)
    y = gpu_gemm_x8(w, N, K, q, sc, ldy=N + 4 if N % 4 == 0 else N + 4 - N % 4)
    assert G.rel_err(y, ref.gemm_x8(w, N, K, q, sc)) <= TOL_TC


@pytest.mark.parametrize("M", [128, 4096])
@pytest.mark.parametrize("N,K", [(17408, 5120), (5120, 17408)])
def test_gemm_x8_prefill_full_size(ref, N, K, M):
    # the prefill shapes at 128 and 4096 tokens, sampled output rows and tokens
    w = G.weights(3, 0, N, K, outliers=True)
    x = G.activations(6, 9, M, K)
    q, sc = ref.quantize_x8(x)
    y = gpu_gemm_x8(w, N, K, q, sc)
    rows = G.sample_rows(N, 24, seed=6)
    toks = G.sample_rows(M, 32, seed=7)
    want = ref.gemm_x8(G.rows_of(w, rows), len(rows), K, q[toks], sc[toks])
    assert G.rel_err(y[np.ix_(toks, rows)], want) <= TOL_TC


def test_gemm_x8_batch_invariant_and_close_to_bf16(ref):
    # row m of an M-token call equals the 1-token call, bit for bit; and the int8
    # path stays within the activations' quantization error of the bf16 path
    N, K, M = 640, 4096, 7
    w = G.weights(6, 6, N, K)
    wd = G.dev(w)
    x = G.activations(6, 7, M, K)
    q, sc = ref.quantize_x8(x)
    ym = gpu_gemm_x8(w, N, K, q, sc, w_dev=wd)
    for m in (0, 3, 6):
        y1 = gpu_gemm_x8(w, N, K, q[m:m + 1], sc[m:m + 1], w_dev=wd)
        assert np.array_equal(y1[0].view(np.uint32), ym[m].view(np.uint32))
    yb = ref.gemm(w, N, K, x)
    # |sum w (x - xh)| <= sum |w| * s / 2 per row; checked in aggregate
    assert G.rel_err(ym, yb) <= 2e-2


# ------------------------------------------------------------------- NVFP4
@functools.lru_cache(maxsize=8)
def fp4_weights(stream: int, N: int, K: int):
    import synth
    return synth.nvfp4_weights(synth.seed(7, stream), N, K)


def gpu_nvfp4_dequant(w, g, N, K):
    out = torch.full((N, K), float("nan"), dtype=torch.float32, device="cuda")
    q4k.q4k_nvfp4_dequant(G.dev(w), g, N, K, out)
    torch.cuda.synchronize()
    return G.host(out)


def gpu_nvfp4_gemm(w, g, N, K, x, ldx=None, ldy=None, w_dev=None):
    M = x.shape[0]
    ldx, ldy = ldx or K, ldy or N
    xp = np.zeros((M, ldx), np.uint16)
    xp[:, :K] = x
    y = torch.full((M, ldy), float("nan"), dtype=torch.float32, device="cuda")
    q4k.q4k_nvfp4_gemm(w_dev if w_dev is not None else G.dev(w), g, N, K, G.dev(xp), M, ldx, y, ldy)
    torch.cuda.synchronize()
    out = G.host(y)
    if ldy > N:
        assert np.all(np.isnan(out[:, N:]))
    return out[:, :N]


def _same_bits(a, b):
    a, b = np.asarray(a, np.float32), np.asarray(b, np.float32)
    na, nb = np.isnan(a), np.isnan(b)
    return np.array_equal(na, nb) and np.array_equal(a[~na].view(np.uint32), b[~nb].view(np.uint32))


def test_nvfp4_dequant_bitexact(ref):
    N, K = 64, 512
    w, g = fp4_weights(0, N, K)
    w = w.copy()
    blk = w.reshape(N, K // 256, 144)
    blk[0, 0, :16] = [0x01, 0x07, 0x08, 0x38, 0x7E, 0x7F, 0x00, 0x40] * 2   # subnormal, 1, 448, NaN, 0 scales
    blk[1, 1, 16:] = np.arange(128, dtype=np.uint8) * 2 + 1                   # every code in both nibbles
    got = gpu_nvfp4_dequant(w, float(g), N, K)
    assert _same_bits(got, ref.nvfp4_dequant(w, float(g), N, K))
    rows = G.sample_rows(5120, 48, seed=1)
    wl, gl = fp4_weights(1, 5120, 17408)
    got = gpu_nvfp4_dequant(G.rows_of(wl, rows), float(gl), len(rows), 17408)
    assert _same_bits(got, ref.nvfp4_dequant(G.rows_of(wl, rows), float(gl), len(rows), 17408))


@pytest.mark.parametrize("M,N,K", [(1, 256, 1024), (17, 200, 768), (128, 384, 2048), (200, 1000, 4096),
                                   (33, 640, 4096)])
def test_nvfp4_gemm_parity(ref, M, N, K):
    # M <= 128: 128-token tiles; (33, 640, 4096): few tiles, so the cluster K split runs
    w, g = fp4_weights(2, N, K)
    x = G.activations(7, 3, M, K)
    y = gpu_nvfp4_gemm(w, float(g), N, K, x, ldx=K + 8, ldy=N + 4)
    want = ref.nvfp4_gemm(w, float(g), N, K, x, threads=16)
    err = G.rel_err(y, want)
    assert err <= TOL_FP4, err


@pytest.mark.parametrize("M", [1024, 4096])
@pytest.mark.parametrize("N,K", [(17408, 5120), (5120, 17408)])
def test_nvfp4_gemm_full_size(ref, N, K, M):
    # the prefill shapes, sampled output rows and tokens (M = 4096 is the benchmark's size)
    w, g = fp4_weights(4, N, K)
    x = G.activations(7, 5, M, K)
    y = gpu_nvfp4_gemm(w, float(g), N, K, x)
    rows = G.sample_rows(N, 32, seed=2)
    toks = G.sample_rows(M, 64, seed=3)
    want = ref.nvfp4_gemm(G.rows_of(w, rows), float(g), len(rows), K, x[toks], threads=16)
    err = G.rel_err(y[np.ix_(toks, rows)], want)
    assert err <= TOL_FP4, err


@pytest.mark.parametrize("N,K,M,fp4", [(5120, 17408, 1, False), (2000, 5120, 4, False), (5120, 17408, 1, True)],
                         ids=["split_k_m1", "ragged_m4", "nvfp4_split_k"])
def test_static_weights_activations_from_the_previous_kernel(ref, N, K, M, fp4):
    # static weights on: the first activation blocks are read by plain loads right
    # after the wait on the previous kernel - here the dequantization that writes them,
    # alternating between two sources, with no host synchronization in between
    srcs = [G.weights(2, 20 + i, M, K) for i in range(2)]
    src_d = [G.dev(s) for s in srcs]
    xs = [ref.dequant_bf16(s, M, K).reshape(M, K) for s in srcs]
    if fp4:
        b, g = fp4_weights(6, N, K)
    else:
        b = G.weights(2, 22, N, K)
    w = G.dev(b)
    xd = torch.empty((M, K), dtype=torch.int16, device="cuda")
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    outs = torch.empty((6, M, N), dtype=torch.float32, device="cuda")
    prev = q4k.q4k_set_static_weights(True)
    try:
        for i in range(6):
            q4k.q4k_dequant_bf16(src_d[i % 2], M, K, xd)
            if fp4:
                q4k.q4k_nvfp4_gemm(w, float(g), N, K, xd, M, K, y, N)
            else:
                q4k.q4k_gemm(w, N, K, xd, M, K, y, N, None, 0)
            outs[i].copy_(y)
        torch.cuda.synchronize()
    finally:
        q4k.q4k_set_static_weights(prev)
    got = G.host(outs)
    rows = np.unique(np.concatenate([G.sample_rows(N, 48, seed=4), np.arange(N - 8, N)]))
    for j in range(2):
        if fp4:
            want = ref.nvfp4_gemm(G.rows_of(b, rows), float(g), len(rows), K, xs[j], threads=16)
            tol = TOL_FP4
        else:
            want = ref.gemm(G.rows_of(b, rows), len(rows), K, xs[j], threads=8)
            tol = TOL_SMALL
        for i in range(j, 6, 2):
            assert G.rel_err(got[i][:, rows], want) <= tol, (i, j)


def test_nvfp4_batch_invariant_mode(ref):
    # the NVFP4 tensor-core path in batch-invariant mode: rows independent of M
    # 8 row tiles: every call splits K 2 ways over a cluster pair, from 40 tokens
    # (128-token tiles) to the 2600-token call (11 tiles of 256, more CTAs than SMs)
    N, K = 1000, 4096
    w, g = fp4_weights(2, N, K)
    x = G.activations(7, 9, 2600, K)
    with batch_invariant():
        yfull = gpu_nvfp4_gemm(w, float(g), N, K, x)
        for m0, M in ((0, 40), (300, 300), (2599 - 130, 130), (1000, 1500)):
            y = gpu_nvfp4_gemm(w, float(g), N, K, x[m0:m0 + M])
            assert np.array_equal(y.view(np.uint32), yfull[m0:m0 + M].view(np.uint32)), (m0, M)
    want = ref.nvfp4_gemm(w, float(g), N, K, x[:32], threads=16)
    assert G.rel_err(yfull[:32], want) <= TOL_FP4


def test_nvfp4_gemm_deterministic():
    N, K, M = 640, 4096, 300
    w, g = fp4_weights(5, N, K)
    wd = G.dev(w)
    x = G.activations(7, 6, M, K)
    a = gpu_nvfp4_gemm(w, float(g), N, K, x, w_dev=wd)
    b = gpu_nvfp4_gemm(w, float(g), N, K, x, w_dev=wd)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("M", [1, 2, 5, 9, 16])
def test_nvfp4_small_m_ragged(ref, M):
    # M <= 16: the small-M kernel's NVFP4 mode (exact bf16 operands, no scale table)
    N, K = 200, 1024
    w, g = fp4_weights(6, N, K)
    x = G.activations(7, 7, M, K)
    y = gpu_nvfp4_gemm(w, float(g), N, K, x, ldx=K + 16, ldy=N + 8)
    err = G.rel_err(y, ref.nvfp4_gemm(w, float(g), N, K, x))
    assert err <= TOL_FP4, err


@pytest.mark.parametrize("N,K", [(17408, 5120), (5120, 17408)], ids=["gate_up", "down"])
@pytest.mark.parametrize("M", [1, 4])
def test_nvfp4_decode_full_size(ref, N, K, M):
    # decode and verify shapes (the down projection splits K over a cluster), sampled rows;
    # rows of the M-token call equal the 1-token call bit for bit
    w, g = fp4_weights(8, N, K)
    wd = G.dev(w)
    x = G.activations(7, 8, M, K)
    y = gpu_nvfp4_gemm(w, float(g), N, K, x, w_dev=wd)
    rows = G.sample_rows(N, 64, seed=M + 7)
    want = ref.nvfp4_gemm(G.rows_of(w, rows), float(g), len(rows), K, x, threads=16)
    err = G.rel_err(y[:, rows], want)
    assert err <= TOL_FP4, err
    if M > 1:
        y1 = gpu_nvfp4_gemm(w, float(g), N, K, x[M - 1:M], w_dev=wd)
        assert np.array_equal(y1[0].view(np.uint32), y[M - 1].view(np.uint32))
