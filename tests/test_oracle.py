"""Pins for the oracle, each against something other than the oracle itself.

  - binary16 decode vs numpy's float16 for all 65536 patterns;
  - bf16 rounding vs torch's float32 -> bfloat16 conversion;
  - hand-assembled blocks (tests/golden) vs their closed-form weights;
  - exhaustive 6-bit packing sweep: synth's independent packer -> oracle unpacker;
  - reference-quantizer round trip bounded by each sub-block's step d*sc;
  - GEMM vs exact rational arithmetic (fractions) and vs numpy matmul;
  - one-hot and all-ones activations (closed forms);
  - MoE routing vs Python's stable sort, slots and combine vs numpy;
  - the routed SwiGLU layer vs its pinned pieces, scipy's logistic function and an
    exact-rational bf16 rounding;
  - int8 activations: quantization invariants, exact ties, sign and power-of-two
    symmetries; the int8 GEMM equals the pinned GEMM where the dequantized
    activations are exact in bf16, and exact rationals on a small case;
  - NVFP4: the e2m1 value set, all 256 e4m3 patterns vs torch's float8_e4m3fn,
    block layout (nibble order, scale index) on hand-built blocks, the GEMM vs
    numpy on an independent decode and vs exact rationals.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from tests.golden import fixture_codes, load_blocks

EPS64 = 2.0 ** -53


def f16_value(bits: int) -> float:
    return float(np.array([bits], dtype=np.uint16).view(np.float16)[0])


def bf16_bits_to_f64(x: np.ndarray) -> np.ndarray:
    return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ------------------------------------------------------------ scalar formats

def test_f16_decode_all_patterns(ref):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = pats.view(np.float16).astype(np.float32)
    got = np.array([ref.f16_to_f32(int(h)) for h in pats], dtype=np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def test_bf16_rounding_matches_torch(ref):
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(1000) * 1e-30).astype(np.float32),
        # exact ties: low 16 bits 0x8000 with even and odd upper halves
        (np.arange(2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.4e38, -3.4e38], dtype=np.float32),
    ])
    vals = vals[np.isfinite(vals) | np.isinf(vals)]
    want = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([ref.f32_to_bf16(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, want)
    assert np.isnan(ref.bf16_to_f32(ref.f32_to_bf16(float("nan"))))


# ------------------------------------------------------------ block decode

@pytest.mark.parametrize("fx", load_blocks(), ids=lambda f: f["name"])
def test_golden_block_fields_and_weights(ref, fx):
    blk = fx["block"]
    for j in range(8):
        assert ref.scale_min(blk[4:16], j) == (fx["sc"][j], fx["m"][j]), f"pair {j}"
    d, dmin = Fraction(f16_value(fx["d_bits"])), Fraction(f16_value(fx["dmin_bits"]))
    q = fixture_codes()
    got = ref.dequant_block(blk)
    for s in range(8):
        for l in range(32):
            want = d * fx["sc"][s] * int(q[s, l]) - dmin * fx["m"][s]
            assert Fraction(float(got[32 * s + l])) == want, (fx["name"], s, l)


def test_all_zero_block_is_zero(ref):
    assert np.all(ref.dequant_block(np.zeros(144, np.uint8)) == 0.0)


def test_nan_and_inf_scales_propagate(ref):
    blk = load_blocks()[0]["block"].copy()
    blk[0:2] = [0x00, 0x7E]           # d = NaN
    assert np.isnan(ref.dequant_block(blk)).any()
    blk[0:2] = [0x00, 0x7C]           # d = +inf: weights with sc*q > 0 are inf
    out = ref.dequant_block(blk)
    assert np.isinf(out).any()


def test_scale_packing_sweep(ref, syn):
    """Every 6-bit value in every pair position survives synth's packer -> oracle unpacker."""
    rng = np.random.default_rng(11)
    for field in ("sc", "m"):
        for j in range(8):
            for v in range(64):
                sc = rng.integers(0, 64, 8)
                mn = rng.integers(0, 64, 8)
                (sc if field == "sc" else mn)[j] = v
                packed = syn.pack_scales(sc, mn)
                for jj in range(8):
                    assert ref.scale_min(packed, jj) == (int(sc[jj]), int(mn[jj]))


def test_make_block_codes_in_weight_order(ref, syn):
    """Codes written in weight order by synth come back at the same positions."""
    rng = np.random.default_rng(5)
    q = rng.integers(0, 16, 256)
    blk = syn.make_block(0x3C00, 0x0000, np.ones(8, np.uint8), np.zeros(8, np.uint8), q)
    assert np.array_equal(ref.dequant_block(blk), q.astype(np.float32))


# ------------------------------------------------------- quantizer round trip

def _roundtrip_check(ref, syn, w):
    N, K = w.shape
    blocks = syn.quantize(w)
    deq = ref.dequant(blocks, N, K)
    nb = K // 256
    for n in range(N):
        for b in range(nb):
            blk = blocks[n, b * 144:(b + 1) * 144]
            d = f16_value(int(blk[0]) | int(blk[1]) << 8)
            for s in range(8):
                sc, m = ref.scale_min(blk[4:16], s)
                sl = slice(b * 256 + 32 * s, b * 256 + 32 * s + 32)
                err = np.abs(w[n, sl].astype(np.float64) - deq[n, sl].astype(np.float64)).max()
                step = d * sc
                # within half a step (rounding to the nearest code) plus fp32 rounding
                assert err <= 0.5 * step * (1 + 1e-6) + 4e-7 * np.abs(w[n, sl]).max() + 1e-30, (n, b, s)
                assert err <= step or err == 0.0
    return blocks, deq


def test_quantizer_roundtrip_gaussian(ref, syn):
    w = syn.normal_f32(123, 8 * 1024, 0.0, 0.02).reshape(8, 1024)
    _roundtrip_check(ref, syn, w)


def test_quantizer_roundtrip_outliers(ref, syn):
    w = syn.normal_f32(124, 16 * 512, 0.0, 0.02).reshape(16, 512)
    assert syn.outliers(125, w, 0.05, 10.0) == round(0.05 * w.size / 32)
    _roundtrip_check(ref, syn, w)


def test_quantizer_special_blocks(ref, syn):
    w = np.zeros((4, 256), np.float32)
    w[1] = np.abs(syn.normal_f32(3, 256, 0.0, 1.0))          # all positive
    w[2] = -np.abs(syn.normal_f32(4, 256, 0.0, 1.0))         # all negative
    w[3] = 0.37                                              # constant
    blocks, deq = _roundtrip_check(ref, syn, w)
    assert np.all(deq[0] == 0.0)
    for s in range(8):
        assert ref.scale_min(blocks[1, 4:16], s)[1] == 0     # no min needed
    # fp16 dmin/d stay finite and positive
    for n in range(4):
        for off in (0, 2):
            v = f16_value(int(blocks[n, off]) | int(blocks[n, off + 1]) << 8)
            assert np.isfinite(v) and v >= 0


# ------------------------------------------------------------------- GEMM

def test_gemm_exact_rational(ref, syn):
    """1 x 256 and 1 x 512: fp64 sum within K*eps*sum|w x| of the exact rational sum."""
    for K, sd in ((256, 31), (512, 32)):
        blocks = syn.weights(sd, 1, K)
        x = syn.normal_bf16(sd + 100, K)
        w = ref.dequant(blocks, 1, K)[0]
        xv = bf16_bits_to_f64(x)
        exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(w, xv))
        absum = float(sum(abs(Fraction(float(a)) * Fraction(float(b))) for a, b in zip(w, xv)))
        y = ref.gemm(blocks, 1, K, x.reshape(1, K))[0, 0]
        assert abs(Fraction(y) - exact) <= Fraction(K * EPS64 * absum)


def test_gemm_vs_numpy(ref, syn):
    M, N, K = 3, 5, 768
    blocks = syn.weights(41, N, K)
    x = syn.normal_bf16(42, M * K).reshape(M, K)
    w = ref.dequant(blocks, N, K).astype(np.float64)
    xv = bf16_bits_to_f64(x)
    want = xv @ w.T
    got = ref.gemm(blocks, N, K, x)
    bound = K * EPS64 * (np.abs(xv) @ np.abs(w).T) * 2
    assert got.shape == (M, N)
    assert np.all(np.abs(got - want) <= bound)


def test_gemm_one_hot_column(ref, syn):
    N, K = 7, 512
    blocks = syn.weights(51, N, K)
    w = ref.dequant(blocks, N, K)
    one = 0x3F80  # bf16 1.0
    for k in (0, 31, 32, 255, 256, 300, 511):
        x = np.zeros((1, K), np.uint16)
        x[0, k] = one
        y = ref.gemm(blocks, N, K, x)[0]
        assert np.array_equal(y, w[:, k].astype(np.float64))


@pytest.mark.parametrize("fx", load_blocks()[:2], ids=lambda f: f["name"])
def test_gemm_all_ones_closed_form(ref, fx):
    x = np.full((1, 256), 0x3F80, np.uint16)
    y = ref.gemm(fx["block"], 1, 256, x)[0, 0]
    d, dmin = Fraction(f16_value(fx["d_bits"])), Fraction(f16_value(fx["dmin_bits"]))
    q = fixture_codes()
    want = sum(d * fx["sc"][s] * int(q[s].sum()) - 32 * dmin * fx["m"][s] for s in range(8))
    assert Fraction(y) == want


def test_gemm_threads_agree(ref, syn):
    N, K, M = 33, 512, 2
    blocks = syn.weights(61, N, K)
    x = syn.normal_bf16(62, M * K).reshape(M, K)
    assert np.array_equal(ref.gemm(blocks, N, K, x, threads=1), ref.gemm(blocks, N, K, x, threads=4))


def test_dequant_bf16_is_rne_of_fp32(ref, syn):
    N, K = 4, 512
    blocks = syn.weights(71, N, K, outlier_frac=0.1, seed_outliers=72)
    f32 = ref.dequant(blocks, N, K)
    want = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ref.dequant_bf16(blocks, N, K), want)


# -------------------------------------------------------------------- MoE

def test_moe_route_is_stable_sort(ref):
    rng = np.random.default_rng(3)
    E, T, topk = 16, 40, 4
    ids = rng.integers(-2, E + 2, (T, topk)).astype(np.int32)
    offsets, perm, bad = ref.moe_route(ids, E)
    flat = ids.reshape(-1)
    valid = [i for i in range(flat.size) if 0 <= flat[i] < E]
    want = sorted(valid, key=lambda i: flat[i])          # Python's sort is stable
    assert bad == flat.size - len(valid)
    assert perm[:len(valid)].tolist() == want
    counts = np.bincount(flat[(flat >= 0) & (flat < E)], minlength=E)
    assert offsets.tolist() == [0] + np.cumsum(counts).tolist()


@pytest.mark.parametrize("per_slot", [False, True])
def test_moe_slots_vs_numpy(ref, syn, per_slot):
    E, N, K, T, topk = 6, 16, 512, 5, 3
    w = np.concatenate([syn.weights(80 + e, N, K) for e in range(E)])
    ids, gates = syn.routing(90, 91, T, E, topk)
    ids[1, 2] = E + 3                                  # an invalid id gives a zero slot
    xrows = T * topk if per_slot else T
    x = syn.normal_bf16(92, xrows * K).reshape(xrows, K)
    out = ref.moe_slots(w, E, N, K, x, per_slot, ids)
    deq = [ref.dequant(w[e * N:(e + 1) * N], N, K).astype(np.float64) for e in range(E)]
    xv = bf16_bits_to_f64(x)
    for t in range(T):
        for j in range(topk):
            e = ids[t, j]
            if not 0 <= e < E:
                assert np.all(out[t, j] == 0.0)
                continue
            xr = xv[t * topk + j] if per_slot else xv[t]
            want = deq[e] @ xr
            assert np.allclose(out[t, j], want, rtol=0, atol=K * EPS64 * 4 * (np.abs(deq[e]) @ np.abs(xr)).max())


def test_moe_combine(ref, syn):
    rng = np.random.default_rng(9)
    T, topk, N = 4, 8, 10
    out = rng.standard_normal((T, topk, N))
    gates = rng.dirichlet(np.ones(topk), T).astype(np.float32)
    y = ref.moe_combine(out, gates)
    want = np.einsum("tj,tjn->tn", gates.astype(np.float64), out)
    assert np.allclose(y, want, rtol=1e-14, atol=1e-14)
    onehot = np.zeros((T, topk), np.float32)
    onehot[np.arange(T), [0, 3, 7, 5]] = 1.0
    y1 = ref.moe_combine(out, onehot)
    assert np.array_equal(y1, out[np.arange(T), [0, 3, 7, 5]])



def exact_bf16(v: float) -> int:
    """The bf16 nearest to v (ties to even), in exact rational arithmetic; its bits."""
    if v == 0.0:
        return 0x8000 if np.signbit(v) else 0
    q = Fraction(v)
    sign = 0x8000 if q < 0 else 0
    q = abs(q)
    e = 0
    while q >= 2:
        q /= 2
        e += 1
    while q < 1:
        q *= 2
        e -= 1
    m = q * 128                                        # 128 <= m < 256: 8 significant bits
    fl = m.numerator // m.denominator
    rem = m - fl
    r = fl + (1 if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1) else 0)
    if r == 256:
        r, e = 128, e + 1
    return sign | ((e + 127) << 7) | (r - 128)


def test_f64_to_bf16_exact(ref):
    rng = np.random.default_rng(31)
    vals = list(rng.standard_normal(3000) * np.exp(rng.uniform(-30, 30, 3000)))
    for b in range(0x3F80, 0x3F90):                    # exact ties between neighbours near 1
        lo = bf16_bits_to_f64(np.array([b], np.uint16))[0]
        hi = bf16_bits_to_f64(np.array([b + 1], np.uint16))[0]
        vals += [(lo + hi) / 2, -(lo + hi) / 2, np.nextafter((lo + hi) / 2, 0.0), np.nextafter((lo + hi) / 2, 9.0)]
    vals += [0.0, -0.0, 1.0, 3.0e38, 1.0e-37]
    for v in vals:
        assert ref.f64_to_bf16(v) == exact_bf16(float(v)), v
    # on values exactly representable in fp32 it agrees with the pinned fp32 rounding
    f = rng.standard_normal(500).astype(np.float32)
    assert all(ref.f64_to_bf16(float(a)) == ref.f32_to_bf16(float(a)) for a in f)


def test_moe_ffn_vs_pinned_pieces(ref, syn):
    # the layer = gate and up slots (pinned above), SwiGLU with scipy's logistic
    # function, bf16 rounding (exact rationals), down slots on h, ordered combine
    from scipy.special import expit
    E, H, D, T, topk = 5, 256, 512, 4, 3
    wg = np.concatenate([syn.weights(100 + e, H, D) for e in range(E)])
    wu = np.concatenate([syn.weights(110 + e, H, D) for e in range(E)])
    wd = np.concatenate([syn.weights(120 + e, D, H) for e in range(E)])
    ids, gates = syn.routing(130, 131, T, E, topk)
    ids[2, 1] = -1                                     # an invalid id adds nothing
    x = syn.normal_bf16(132, T * D).reshape(T, D)
    y = ref.moe_ffn(wg, wu, wd, E, H, D, x, ids, gates)
    g = ref.moe_slots(wg, E, H, D, x, False, ids)
    u = ref.moe_slots(wu, E, H, D, x, False, ids)
    hv = g * expit(g) * u
    h = np.array([exact_bf16(float(v)) for v in hv.reshape(-1)], dtype=np.uint16).reshape(T * topk, H)
    out = ref.moe_slots(wd, E, D, H, h, True, ids)
    want = ref.moe_combine(out, gates)
    assert np.allclose(y, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())
    assert np.any(h != 0) and np.abs(y).max() > 0



# ------------------------------------------------------------ int8 activations

def _to_bf16_bits(vals):
    """Exactly bf16-representable float values -> bf16 bits (asserts exactness)."""
    f = np.asarray(vals, dtype=np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0)
    return (u >> 16).astype(np.uint16)


def test_quantize_x8_invariants(ref, syn):
    M, K = 3, 1024
    x = syn.normal_bf16(41, M * K).reshape(M, K).copy()
    x[0, 32:64] = 0                                            # all-zero block
    x[1, 64:96] = _to_bf16_bits(-np.abs(bf16_bits_to_f64(x[1, 64:96])))  # all negative
    x[2, 96:128] = 0
    x[2, 100] = _to_bf16_bits([3.0])[0]                        # a single non-zero
    q, sc = ref.quantize_x8(x)
    xf = bf16_bits_to_f64(x)
    assert q.dtype == np.int8 and np.abs(q.astype(np.int32)).max() <= 127
    for m in range(M):
        for b in range(K // 32):
            blk, qb, s = xf[m, 32 * b:32 * b + 32], q[m, 32 * b:32 * b + 32].astype(np.int64), float(sc[m, b])
            a = np.abs(blk).max()
            if a == 0:
                assert s == 0 and np.all(qb == 0)
                continue
            assert abs(s - a / 127) <= a / 127 * 2.0 ** -23        # the scale is a/127 to fp32 precision
            i = int(np.argmax(np.abs(blk)))
            assert qb[i] == (127 if blk[i] > 0 else -127)           # the largest element maps to +-127
            # nearest integer to x/s, up to the fp32 rounding of x/s (|x/s| <= 127: 127 * 2^-24)
            assert np.all(np.abs(blk - s * qb) <= s * (0.5 + 2.0 ** -16))
            assert np.all(np.sign(qb) * np.sign(blk) >= 0)
    assert np.all(q[2, 96:128][np.arange(32) != 4] == 0) and q[2, 100] == 127


def test_quantize_x8_ties_to_even_and_symmetries(ref, syn):
    # a block whose largest magnitude is 127 * 2^-3: s = 2^-3 exactly, so k.5 * s are exact ties
    vals = np.zeros(32)
    vals[0] = 127 * 0.125
    vals[1:9] = np.array([0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, 126.5]) * 0.125
    x = _to_bf16_bits(vals).reshape(1, 32)
    q, sc = ref.quantize_x8(x)
    assert float(sc[0, 0]) == 0.125
    assert list(q[0, :9]) == [127, 0, 2, 2, 4, 0, -2, -2, 126]
    # q(-x) = -q(x), s(-x) = s(x); q(2x) = q(x), s(2x) = 2 s(x)
    y = syn.normal_bf16(43, 2 * 256).reshape(2, 256)
    q1, s1 = ref.quantize_x8(y)
    q2, s2 = ref.quantize_x8(y ^ np.uint16(0x8000))
    assert np.array_equal(q2, -q1) and np.array_equal(s2, s1)
    y2 = _to_bf16_bits(2.0 * bf16_bits_to_f64(y))
    q3, s3 = ref.quantize_x8(y2)
    assert np.array_equal(q3, q1) and np.array_equal(s3, 2 * s1)


def test_gemm_x8_equals_gemm_on_exact_activations(ref, syn):
    # power-of-two scales make s * q exact in bf16, so the int8 GEMM must give the
    # pinned bf16 GEMM's result on those activations, bit for bit
    N, K, M = 7, 768, 3
    w = syn.weights(44, N, K)
    rng = np.random.default_rng(45)
    q = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    sc = np.ldexp(1.0, rng.integers(-9, 2, size=(M, K // 32))).astype(np.float32)
    xh = np.repeat(sc, 32, axis=1).astype(np.float64) * q
    got = ref.gemm_x8(w, N, K, q, sc)
    want = ref.gemm(w, N, K, _to_bf16_bits(xh))
    assert np.array_equal(got, want)


def test_gemm_x8_exact_rational(ref, syn):
    N, K = 2, 512
    w = syn.weights(46, N, K)
    x = syn.normal_bf16(47, K).reshape(1, K)
    q, sc = ref.quantize_x8(x)
    wd = ref.dequant(w, N, K)
    got = ref.gemm_x8(w, N, K, q, sc)
    for n in range(N):
        exact = sum(Fraction(float(wd[n, k])) * Fraction(float(sc[0, k // 32])) * int(q[0, k]) for k in range(K))
        assert abs(Fraction(float(got[0, n])) - exact) <= abs(exact) * Fraction(1, 2 ** 40) + Fraction(1, 2 ** 60)



# ------------------------------------------------------------------- NVFP4
# the e2m1 value set of the FP4 format: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 for
# codes 0..7, the same negated for codes 8..15
E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_values(ref):
    for c in range(16):
        v = ref.e2m1_to_f32(c)
        assert abs(v) == E2M1[c & 7] and (np.signbit(v) == bool(c & 8))


def test_e4m3_all_patterns_vs_torch(ref):
    import torch
    pats = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    want = pats.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    got = np.array([ref.e4m3_to_f32(b) for b in range(256)], dtype=np.float32)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok].view(np.uint32), want[ok].view(np.uint32))


def _nvfp4_block(scales, codes) -> np.ndarray:
    blk = np.zeros(144, dtype=np.uint8)
    blk[:16] = scales
    codes = np.asarray(codes, dtype=np.uint8)
    blk[16:] = codes[0::2] | (codes[1::2] << 4)
    return blk


def test_nvfp4_block_layout(ref):
    # weight i carries code i % 16 and the scale of group i // 16 (distinct powers of two)
    scales = np.array([0x38 + 8 * (j % 4) - 8 * (j // 4) for j in range(16)], dtype=np.uint8)  # 2^(j%4 - j//4)
    codes = np.arange(256) % 16
    g = 0.75
    out = ref.nvfp4_dequant_block(_nvfp4_block(scales, codes), g)
    for i in range(256):
        j = i // 16
        sv = 2.0 ** (j % 4 - j // 4)
        want = np.float32(g * sv * (E2M1[codes[i] & 7] * (-1 if codes[i] & 8 else 1)))
        assert out[i] == want, i
    # a subnormal and the largest scale; g rounds the product once
    blk = _nvfp4_block([0x01] * 8 + [0x7E] * 8, [7] * 256)
    out = ref.nvfp4_dequant_block(blk, 1.0)
    assert out[0] == 6 * 2.0 ** -9 and out[255] == 6 * 448.0


def _np_nvfp4_decode(w, g, N, K):
    """Independent decode: the byte layout and the pinned value sets, in numpy."""
    b = np.asarray(w, np.uint8).reshape(N, K // 256, 144)
    import torch
    sc = torch.from_numpy(np.ascontiguousarray(b[:, :, :16])).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    v = b[:, :, 16:]
    codes = np.stack([v & 15, v >> 4], axis=-1).reshape(N, K // 256, 256)
    mag = np.array(E2M1)[codes & 7] * np.where(codes & 8, -1.0, 1.0)
    return (float(g) * np.repeat(sc, 16, axis=2) * mag).reshape(N, K)


def test_nvfp4_gemm_vs_numpy(ref, syn):
    N, K, M = 6, 768, 3
    w, g = syn.nvfp4_weights(48, N, K)
    x = syn.normal_bf16(49, M * K).reshape(M, K)
    want = bf16_bits_to_f64(x) @ _np_nvfp4_decode(w, g, N, K).T
    got = ref.nvfp4_gemm(w, float(g), N, K, x)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())
    # the fp32 dequant is the exact value rounded once
    wd = ref.nvfp4_dequant(w, float(g), N, K)
    assert np.array_equal(wd, _np_nvfp4_decode(w, g, N, K).astype(np.float32))


def test_nvfp4_gemm_exact_rational(ref, syn):
    N, K = 2, 256
    w, g = syn.nvfp4_weights(50, N, K)
    x = syn.normal_bf16(51, K).reshape(1, K)
    wd = _np_nvfp4_decode(w, g, N, K)
    got = ref.nvfp4_gemm(w, float(g), N, K, x)
    xf = bf16_bits_to_f64(x)[0]
    for n in range(N):
        exact = sum(Fraction(float(wd[n, k])) * Fraction(float(xf[k])) for k in range(K))
        assert abs(Fraction(float(got[0, n])) - exact) <= abs(exact) * Fraction(1, 2 ** 40) + Fraction(1, 2 ** 70)


# ------------------------------------------------------------ input module

def test_synth_routing_and_gates(syn):
    ids, gates = syn.routing(1, 2, 300, 128, 8)
    assert ids.min() >= 0 and ids.max() < 128
    assert all(len(set(r)) == 8 for r in ids.tolist())
    assert np.allclose(gates.sum(1), 1.0, atol=1e-6) and gates.min() > 0
    # Dirichlet(1,...,1) marginals have mean 1/8
    assert abs(gates.mean() - 0.125) < 0.01


def test_synth_normals(syn):
    x = syn.normal_f32(5, 200000, 0.0, 0.02).astype(np.float64)
    assert abs(x.mean()) < 3e-4 and abs(x.std() - 0.02) < 3e-4
    b = syn.normal_bf16(5, 1001)
    f = syn.normal_f32(5, 1001)
    assert np.array_equal(b, syn.f32_to_bf16(f))
