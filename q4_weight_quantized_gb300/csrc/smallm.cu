// Small-M Q4_K matmul: decode GEMV (M = 1) and speculative-verify GEMM (M <= 16).
//
// The decode projections of the pages run one token per lane, or 1 + accepted
// drafts per lane when a drafter proposes --draft-tokens N (ninfer serving docs,
// "Start the server" and "Determinism"), and carry no floating-point atomics
// (sparkinfer-server README, "Determinism").  At these M the product is bound by
// streaming the 0.5625-byte-per-weight Q4_K matrix from HBM once, so the kernel
// is built around keeping HBM busy and the per-weight instruction count low:
//
//   * A CTA owns 32 consecutive weight rows; its four warps split the K blocks
//     (warp w takes blocks w, w+4, ...).  Every warp streams its own blocks with
//     TMA into a private ring of shared-memory slots: one 2-D bulk-tensor copy of
//     32 rows x 1 block (4.5 KiB) plus one 512-byte copy per token of the
//     matching 256 activations, completed on the slot's mbarrier.  The warp
//     refills a slot as soon as it has consumed it, so the copies of the next
//     slots stay in flight while it computes, and no warp waits for another.
//     Rows past N are zero-filled by the copy and decode to zero weights.
//   * A lane turns one
//     32-bit word of codes into four bf16x2 registers holding 128+q exactly
//     (one byte permute and one LOP3 per pair: 0x4300 is bf16 128.0, whose last
//     seven mantissa bits count units), and feeds them as the A operand of a
//     16x8x16 bf16 tensor-core MMA with fp32 accumulation.  The B operand is the
//     activation, 8 tokens per MMA.  Per 32-weight sub-block s of a row:
//         C_s   = sum_l (128 + q_l) x_l                (exact products, fp32 sum)
//         S_s   = sum_l x_l                            (an MMA against all-ones)
//         y    += (d sc_s) C_s - (128 d sc_s + dmin m_s) S_s
//     which equals sum_l (d sc_s q_l - dmin m_s) x_l.  The (d sc_s, bias) pairs of
//     a block are decoded once per row into a small shared table.
//   * Each warp's partial sums are reduced across the four warps in warp order,
//     and, when narrow N leaves too few row tiles to fill the GPU, across a
//     thread-block cluster that splits K (distributed shared memory, rank
//     order).  No atomics anywhere: the result is run-to-run deterministic, and
//     since neither the split nor the order depends on M, row m of an M-token
//     call equals a 1-token call on row m bit for bit.
//
// The MoE grouped GEMM runs the same kernel with one grid layer per expert: the
// token slots of a chunk are the (token, k-slot) items routed to that expert,
// their activation rows are gathered by the same per-row copies, and each
// output row goes to its item's slot.
#include <cuda.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "q4k_internal.h"
#include "q4k_ptx.cuh"

namespace q4k {
namespace {

constexpr int kWarps = 4;                  // split the CTA's K blocks
constexpr int kThreads = kWarps * 32;
constexpr int kBlkWords = kBlockBytes / 4;       // 36 (TMA box inner dim, uint32)
constexpr int kXBlkBytes = kQK * 2;              // 512: one token's activations for one block
constexpr int kTableRowBytes = 80;  // 8 x (dsc, bias) + 16 pad: conflict-free 16-byte reads

// Shared-memory geometry of a CTA that owns ROWS weight rows (32 or 48).
template <int ROWS>
struct Geo {
    static constexpr int kRowTiles = ROWS / 16;            // 16-row MMA tiles per CTA
    static constexpr int kBlkWBytes = ROWS * kBlockBytes;   // one block column of the CTA's rows
    static constexpr int kTableBytes = ROWS * kTableRowBytes;
    static constexpr int kRedBytes = kWarps * 16 * ROWS * 4 + 16 * ROWS * 4;  // per-warp + final partials
    __host__ __device__ static constexpr int slot_bytes(int nx) {
        return (kBlkWBytes + nx * kXBlkBytes + 127) / 128 * 128;
    }
    // per warp: [ring of `slots` slots][scale table]
    __host__ __device__ static constexpr int warp_bytes(int nx, int slots) { return slots * slot_bytes(nx) + kTableBytes; }
    // CTA: [warp regions][barriers][reduction buffer (MoE only; dense reuses the rings)]
    __host__ __device__ static constexpr int bars_off(int nx, int slots) { return kWarps * warp_bytes(nx, slots); }
    __host__ __device__ static constexpr int red_off(int nx, int slots) {
        return bars_off(nx, slots) + kWarps * slots * 8 + 64;
    }
    // `red`: the MoE K-split mode's reduction buffer (the row-split mode stages its
    // outputs in each warp's scale table, the dense mode reuses the rings)
    __host__ __device__ static constexpr int smem_total(int nx, int slots, bool red) {
        return red_off(nx, slots) + (red ? kRedBytes : 0);
    }
    static_assert(ROWS % 16 == 0 && ROWS <= 64, "rows per CTA");
    static_assert(kRedBytes <= kWarps * 2 * slot_bytes(1), "dense reduction buffers alias the rings");
};

// F16: fp16 pairs 1024 + q (magic 0x6400) instead of bf16 pairs 128 + q (0x4300).
template <bool F16 = false>
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t &lo01, uint32_t &lo23, uint32_t &hi01,
                                            uint32_t &hi23) {
    constexpr uint32_t kMagic = F16 ? 0x64006400u : 0x43004300u;
    const uint32_t t01 = prmt(w, 0u, 0x4140u);  // bytes 0,1 -> 16-bit lanes
    const uint32_t t23 = prmt(w, 0u, 0x4342u);  // bytes 2,3
    lo01 = lop3_and_or(t01, 0x000F000Fu, kMagic);
    lo23 = lop3_and_or(t23, 0x000F000Fu, kMagic);
    hi01 = lop3_and_or(t01 >> 4, 0x000F000Fu, kMagic);
    hi23 = lop3_and_or(t23 >> 4, 0x000F000Fu, kMagic);
}

// byte i of w as an fp32 2^23 + byte (exponent 150, the byte in the low mantissa bits)
__device__ __forceinline__ float byte_magic(uint32_t w, int i) {
    return __uint_as_float(prmt(w, 0x4B000000u, 0x7440u | (uint32_t)i));
}

// Decode one row's block header (d, dmin, 12 scale bytes) into 8 (d*sc, bias)
// pairs, bias = 128*d*sc + dmin*m (MIN: bias = dmin*m).  d*sc and dmin*m are
// exact: fma(2^23+b, d, -2^23*d) rounds d*b, which has at most 17 significant bits.
template <bool MIN = false>
__device__ __forceinline__ void decode_scales(const uint8_t *blk, float *table_row) {
    const uint4 h = *reinterpret_cast<const uint4 *>(blk);
    const float d = __half2float(__ushort_as_half((unsigned short)(h.x & 0xFFFFu)));
    const float dmin = __half2float(__ushort_as_half((unsigned short)(h.x >> 16)));
    const float nd = -8388608.0f * d, ndm = -8388608.0f * dmin;
    const uint32_t sc_lo = h.y & 0x3F3F3F3Fu;
    const uint32_t m_lo = h.z & 0x3F3F3F3Fu;
    const uint32_t sc_hi = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
    const uint32_t m_hi = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
    float v[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float dsc = fmaf(byte_magic(j < 4 ? sc_lo : sc_hi, j & 3), d, nd);
        const float dm = fmaf(byte_magic(j < 4 ? m_lo : m_hi, j & 3), dmin, ndm);
        v[2 * j] = dsc;
        v[2 * j + 1] = MIN ? dm : fmaf(128.0f, dsc, dm);
    }
    float4 *dst = reinterpret_cast<float4 *>(table_row);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

// After a wait gave up: wait (each wait bounded too) for the copies this warp
// still has in flight, ring iterations [from, to), so that none lands after the
// CTA has left.
template <int SLOTS>
__device__ __forceinline__ void drain_ring(uint32_t bar0, int from, int to, unsigned int *status) {
    for (int k = from; k < to; ++k) (void)mbar_wait(bar0 + 8 * (k % SLOTS), (k / SLOTS) & 1, status);
}

// acc += one staged block: the ROWS = 16*RT weight rows of `wst` (144 bytes each),
// the activations of 8*NT token slots in `xs` (512 bytes each; only `live`
// 8-token tiles are read) and the rows' (d*sc, bias) table.  Lane (r, c) of the
// MMA fragment layout.  Per 32-weight sub-block s of a row:
//     acc += (d sc_s) C_s - bias_s S_s,  C_s = sum (128 + q) x,  S_s = sum x.
template <int NT, bool ONE, int RT>
__device__ __forceinline__ void block_mma(const uint8_t *wst, const uint8_t *xs, const float *table,
                                          const bool (&live)[NT], float (&acc)[RT][NT][4], int r, int c) {
    constexpr int kRowTiles = RT;
    const uint32_t ones[4] = {0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u};
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        // activations for sub-blocks 2g (xl) and 2g+1 (xh), per 8-token tile
        uint32_t xl[NT][4], xh[NT][4];
        float sl[NT][4], sh[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
            if (live[nt]) {
                const uint8_t *xp = xs + (nt * 8 + r) * kXBlkBytes + 128 * g + 16 * c;
                a = *reinterpret_cast<const uint4 *>(xp);
                b = *reinterpret_cast<const uint4 *>(xp + 64);
            }
            xl[nt][0] = a.x; xl[nt][1] = a.y; xl[nt][2] = a.z; xl[nt][3] = a.w;
            xh[nt][0] = b.x; xh[nt][1] = b.y; xh[nt][2] = b.z; xh[nt][3] = b.w;
            mma_bf16_16816(sl[nt], ones, xl[nt][0], xl[nt][1], zero4);
            mma_bf16_16816(sl[nt], ones, xl[nt][2], xl[nt][3], sl[nt]);
            mma_bf16_16816(sh[nt], ones, xh[nt][0], xh[nt][1], zero4);
            mma_bf16_16816(sh[nt], ones, xh[nt][2], xh[nt][3], sh[nt]);
        }
#pragma unroll
        for (int rt = 0; rt < kRowTiles; ++rt) {
            const int rA = rt * 16 + r, rB = rA + 8;
            const uint2 wa = *reinterpret_cast<const uint2 *>(wst + rA * kBlockBytes + 16 + 32 * g + 8 * c);
            const uint2 wb = *reinterpret_cast<const uint2 *>(wst + rB * kBlockBytes + 16 + 32 * g + 8 * c);
            uint32_t alo0[4], alo1[4], ahi0[4], ahi1[4];
            // word 0 (elements 8c..8c+3) feeds MMA 0, word 1 (8c+4..8c+7) MMA 1
            unpack_word(wa.x, alo0[0], alo0[2], ahi0[0], ahi0[2]);
            unpack_word(wb.x, alo0[1], alo0[3], ahi0[1], ahi0[3]);
            unpack_word(wa.y, alo1[0], alo1[2], ahi1[0], ahi1[2]);
            unpack_word(wb.y, alo1[1], alo1[3], ahi1[1], ahi1[3]);
            const float4 sa = *reinterpret_cast<const float4 *>(table + rA * (kTableRowBytes / 4) + 4 * g);
            const float4 sb = *reinterpret_cast<const float4 *>(table + rB * (kTableRowBytes / 4) + 4 * g);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float cl[4], chh[4];
                mma_bf16_16816(cl, alo0, xl[nt][0], xl[nt][1], zero4);
                mma_bf16_16816(cl, alo1, xl[nt][2], xl[nt][3], cl);
                mma_bf16_16816(chh, ahi0, xh[nt][0], xh[nt][1], zero4);
                mma_bf16_16816(chh, ahi1, xh[nt][2], xh[nt][3], chh);
                float *a4 = acc[rt][nt];
                // sub-block 2g, then 2g+1; accumulators 1 and 3 hold odd tokens
                a4[0] = fmaf(sa.x, cl[0], a4[0]); a4[0] = fmaf(-sa.y, sl[nt][0], a4[0]);
                a4[2] = fmaf(sb.x, cl[2], a4[2]); a4[2] = fmaf(-sb.y, sl[nt][2], a4[2]);
                a4[0] = fmaf(sa.z, chh[0], a4[0]); a4[0] = fmaf(-sa.w, sh[nt][0], a4[0]);
                a4[2] = fmaf(sb.z, chh[2], a4[2]); a4[2] = fmaf(-sb.w, sh[nt][2], a4[2]);
                if constexpr (!ONE) {
                    a4[1] = fmaf(sa.x, cl[1], a4[1]); a4[1] = fmaf(-sa.y, sl[nt][1], a4[1]);
                    a4[3] = fmaf(sb.x, cl[3], a4[3]); a4[3] = fmaf(-sb.y, sl[nt][3], a4[3]);
                    a4[1] = fmaf(sa.z, chh[1], a4[1]); a4[1] = fmaf(-sa.w, sh[nt][1], a4[1]);
                    a4[3] = fmaf(sb.z, chh[3], a4[3]); a4[3] = fmaf(-sb.w, sh[nt][3], a4[3]);
                }
            }
        }
    }
}

// int8 activations (slot: 256 int8 values, then the block's 8 fp32 scales, per
// token).  The fragment walk of block_mma with fp16 operands: A = 1024 + q and
// B = the int8 values, both exact in fp16, so C = sum (1024 + q) x and S = sum x
// are exact integers (below 2^24) in the fp32 accumulators.  Per 32-weight
// sub-block s: acc += s_x * (d sc_s (C - 1024 S) - dmin m_s S), s_x being the
// activation block's scale; C - 1024 S = sum q x is formed exactly first.
template <int NT, bool ONE, int RT>
__device__ __forceinline__ void block_mma_x8(const uint8_t *wst, const uint8_t *xs, const float *table,
                                             const bool (&live)[NT], int nvalid, float (&acc)[RT][NT][4], int r,
                                             int c) {
    constexpr int kRowTiles = RT;
    const uint32_t ones[4] = {0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u};
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    const __half2 k1152 = __float2half2_rn(1152.0f);
    // int8 pair -> fp16 pair holding the exact value: (b ^ 0x80) = b + 128 in 0..255
    // as the low mantissa byte of 1024.0 (0x64xx), minus 1152
    auto cvt = [&](uint32_t u, uint32_t sel) -> uint32_t {
        const uint32_t h = prmt(u, 0x64646464u, sel);
        const __half2 v = __hsub2(*reinterpret_cast<const __half2 *>(&h), k1152);
        return *reinterpret_cast<const uint32_t *>(&v);
    };
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        uint32_t xl[NT][4], xh[NT][4];
        float sl[NT][4], sh[NT][4];
        float2 s0[NT], s1[NT];  // scales of sub-blocks (2g, 2g+1) for tokens 2c and 2c+1 of the tile
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            uint2 a = make_uint2(0, 0), b = make_uint2(0, 0);
            s0[nt] = make_float2(0.f, 0.f);
            s1[nt] = make_float2(0.f, 0.f);
            if (live[nt]) {
                const uint8_t *xp = xs + (nt * 8 + r) * kXBlkBytes + 64 * g + 8 * c;
                a = *reinterpret_cast<const uint2 *>(xp);       // sub-block 2g, elements 8c..8c+7
                b = *reinterpret_cast<const uint2 *>(xp + 32);  // sub-block 2g+1
            }
            // only the slot's tokens have scales (the others get 0: their x is 0 too)
            const int t0 = nt * 8 + 2 * c;
            const uint8_t *sp = xs + t0 * kXBlkBytes + 256 + 8 * g;
            if (t0 < nvalid) s0[nt] = *reinterpret_cast<const float2 *>(sp);
            if (!ONE && t0 + 1 < nvalid) s1[nt] = *reinterpret_cast<const float2 *>(sp + kXBlkBytes);
            const uint32_t a0 = a.x ^ 0x80808080u, a1 = a.y ^ 0x80808080u;
            const uint32_t b0 = b.x ^ 0x80808080u, b1 = b.y ^ 0x80808080u;
            xl[nt][0] = cvt(a0, 0x5140u); xl[nt][1] = cvt(a0, 0x7362u);
            xl[nt][2] = cvt(a1, 0x5140u); xl[nt][3] = cvt(a1, 0x7362u);
            xh[nt][0] = cvt(b0, 0x5140u); xh[nt][1] = cvt(b0, 0x7362u);
            xh[nt][2] = cvt(b1, 0x5140u); xh[nt][3] = cvt(b1, 0x7362u);
            mma_f16_16816(sl[nt], ones, xl[nt][0], xl[nt][1], zero4);
            mma_f16_16816(sl[nt], ones, xl[nt][2], xl[nt][3], sl[nt]);
            mma_f16_16816(sh[nt], ones, xh[nt][0], xh[nt][1], zero4);
            mma_f16_16816(sh[nt], ones, xh[nt][2], xh[nt][3], sh[nt]);
        }
#pragma unroll
        for (int rt = 0; rt < kRowTiles; ++rt) {
            const int rA = rt * 16 + r, rB = rA + 8;
            const uint2 wa = *reinterpret_cast<const uint2 *>(wst + rA * kBlockBytes + 16 + 32 * g + 8 * c);
            const uint2 wb = *reinterpret_cast<const uint2 *>(wst + rB * kBlockBytes + 16 + 32 * g + 8 * c);
            uint32_t alo0[4], alo1[4], ahi0[4], ahi1[4];
            unpack_word<true>(wa.x, alo0[0], alo0[2], ahi0[0], ahi0[2]);
            unpack_word<true>(wb.x, alo0[1], alo0[3], ahi0[1], ahi0[3]);
            unpack_word<true>(wa.y, alo1[0], alo1[2], ahi1[0], ahi1[2]);
            unpack_word<true>(wb.y, alo1[1], alo1[3], ahi1[1], ahi1[3]);
            // (d sc, dmin m) of sub-blocks 2g and 2g+1
            const float4 sa = *reinterpret_cast<const float4 *>(table + rA * (kTableRowBytes / 4) + 4 * g);
            const float4 sb = *reinterpret_cast<const float4 *>(table + rB * (kTableRowBytes / 4) + 4 * g);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float cl[4], chh[4];
                mma_f16_16816(cl, alo0, xl[nt][0], xl[nt][1], zero4);
                mma_f16_16816(cl, alo1, xl[nt][2], xl[nt][3], cl);
                mma_f16_16816(chh, ahi0, xh[nt][0], xh[nt][1], zero4);
                mma_f16_16816(chh, ahi1, xh[nt][2], xh[nt][3], chh);
                float *a4 = acc[rt][nt];
                // element e: row rA (e < 2) or rB, token 2c + (e & 1)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (ONE && (e & 1)) continue;
                    const float4 &sw = e < 2 ? sa : sb;
                    const float2 &sx = (e & 1) ? s1[nt] : s0[nt];
                    const float dl = fmaf(-1024.0f, sl[nt][e], cl[e]);   // sum q x, sub-block 2g
                    const float dh = fmaf(-1024.0f, sh[nt][e], chh[e]);  // sub-block 2g+1
                    a4[e] = fmaf(sx.x, fmaf(sw.x, dl, -sw.y * sl[nt][e]), a4[e]);
                    a4[e] = fmaf(sx.y, fmaf(sw.z, dh, -sw.w * sh[nt][e]), a4[e]);
                }
            }
        }
    }
}

// NVFP4 weights (144-byte blocks: 16 e4m3 scales, then 128 bytes of e2m1 pairs,
// weight 2i in the low nibble of byte i).  Each operand element is the exact
// bf16 value e4m3 * e2m1, so the MMAs accumulate w . x straight into the fp32
// accumulators (no per-sub-block scaling; the tensor scale is applied by the
// epilogue).  The fragment walk of block_mma: per g, a lane holds x for weights
// 64g + 8c .. +7 (xl) and 64g + 32 + 8c .. +7 (xh); their codes are the value
// words at bytes 32g + 4c and 32g + 16 + 4c, their scales 4g + c/2 and 4g + 2 + c/2.
template <int NT, bool ONE, int RT>
__device__ __forceinline__ void block_mma_fp4(const uint8_t *wst, const uint8_t *xs, const bool (&live)[NT],
                                              float (&acc)[RT][NT][4], int r, int c) {
    constexpr int kRowTiles = RT;
    auto scale2 = [](uint32_t sc4, int i) -> uint32_t {  // e4m3 byte i -> bf16 pair (exact)
        const float f = e4m3_to_f32(sc4 >> (8 * i));
        const __nv_bfloat162 v = __floats2bfloat162_rn(f, f);
        return *reinterpret_cast<const uint32_t *>(&v);
    };
    auto mul2 = [](uint32_t a, uint32_t b) -> uint32_t {
        const __nv_bfloat162 v =
            __hmul2(*reinterpret_cast<const __nv_bfloat162 *>(&a), *reinterpret_cast<const __nv_bfloat162 *>(&b));
        return *reinterpret_cast<const uint32_t *>(&v);
    };
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        uint32_t xl[NT][4], xh[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
            if (live[nt]) {
                const uint8_t *xp = xs + (nt * 8 + r) * kXBlkBytes + 128 * g + 16 * c;
                a = *reinterpret_cast<const uint4 *>(xp);
                b = *reinterpret_cast<const uint4 *>(xp + 64);
            }
            xl[nt][0] = a.x; xl[nt][1] = a.y; xl[nt][2] = a.z; xl[nt][3] = a.w;
            xh[nt][0] = b.x; xh[nt][1] = b.y; xh[nt][2] = b.z; xh[nt][3] = b.w;
        }
#pragma unroll
        for (int rt = 0; rt < kRowTiles; ++rt) {
            const uint8_t *pa = wst + (rt * 16 + r) * kBlockBytes, *pb = pa + 8 * kBlockBytes;
            const uint32_t sa = *reinterpret_cast<const uint32_t *>(pa + 4 * g);
            const uint32_t sb = *reinterpret_cast<const uint32_t *>(pb + 4 * g);
            const uint32_t sal = scale2(sa, c >> 1), sah = scale2(sa, 2 + (c >> 1));
            const uint32_t sbl = scale2(sb, c >> 1), sbh = scale2(sb, 2 + (c >> 1));
            uint32_t a01, a23, a45, a67, b01, b23, b45, b67;
            uint32_t alo0[4], alo1[4], ahi0[4], ahi1[4];
            e2m1x8_to_bf16(*reinterpret_cast<const uint32_t *>(pa + 16 + 32 * g + 4 * c), a01, a23, a45, a67);
            e2m1x8_to_bf16(*reinterpret_cast<const uint32_t *>(pb + 16 + 32 * g + 4 * c), b01, b23, b45, b67);
            alo0[0] = mul2(a01, sal); alo0[1] = mul2(b01, sbl); alo0[2] = mul2(a23, sal); alo0[3] = mul2(b23, sbl);
            alo1[0] = mul2(a45, sal); alo1[1] = mul2(b45, sbl); alo1[2] = mul2(a67, sal); alo1[3] = mul2(b67, sbl);
            e2m1x8_to_bf16(*reinterpret_cast<const uint32_t *>(pa + 32 + 32 * g + 4 * c), a01, a23, a45, a67);
            e2m1x8_to_bf16(*reinterpret_cast<const uint32_t *>(pb + 32 + 32 * g + 4 * c), b01, b23, b45, b67);
            ahi0[0] = mul2(a01, sah); ahi0[1] = mul2(b01, sbh); ahi0[2] = mul2(a23, sah); ahi0[3] = mul2(b23, sbh);
            ahi1[0] = mul2(a45, sah); ahi1[1] = mul2(b45, sbh); ahi1[2] = mul2(a67, sah); ahi1[3] = mul2(b67, sbh);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                mma_bf16_16816(acc[rt][nt], alo0, xl[nt][0], xl[nt][1], acc[rt][nt]);
                mma_bf16_16816(acc[rt][nt], alo1, xl[nt][2], xl[nt][3], acc[rt][nt]);
                mma_bf16_16816(acc[rt][nt], ahi0, xh[nt][0], xh[nt][1], acc[rt][nt]);
                mma_bf16_16816(acc[rt][nt], ahi1, xh[nt][2], xh[nt][3], acc[rt][nt]);
            }
        }
    }
}


// Where each token slot of a chunk reads its activation row and writes its
// output row.  Dense: slot n is token n.  MoE: slot n of a token tile is the
// (token, k-slot) item perm[first + n], first being the tile's first position
// in the expert-sorted order.
struct RowArgs {
    float *y;
    int64_t ldy;          // dense: output row stride; MoE: N
    int M;                // dense: number of tokens (<= 16)
    int x_per_slot;       // MoE: activation row is the item (1) or its token (0)
    int topk;             // MoE
    const int32_t *perm;  // MoE routing permutation
    const int4 *tiles;    // MoE: the routing's token tiles (expert, first item, count)
    const int *n_tiles;
    const int32_t *n_valid;  // MoE: offsets[E]; perm[*n_valid .. n_items) are the invalid items
    int n_items;             // MoE: T * topk
    int zero_invalid;        // MoE: zero the per-slot rows of the invalid items
    int early_w;          // dense: copy the first weight blocks before waiting on the previous kernel
    // MoE with very few items: grid layer z is item z itself (no routing); its
    // expert is ids[z], and an id outside [0, E) zeroes the item's per-slot row
    int direct;
    const int32_t *ids;
    int E;
    GluOut glu;  // MoE with GLU: h (bf16) receives the SwiGLU of the gate and up projections
    float gscale;  // FP4: the weights' tensor scale, applied to the outputs
    const float *gates;  // MoE with DC: the combine weights [T][topk]
    // MoE with DC: the ids may be read, and the first slots' (static) expert weights
    // copied, before waiting on the previous kernel - the expert FFN's down
    // projection, whose previous kernel (gate and up) waited for the ids' writer
    int ids_early;
};

// The (token, k-slot) item at position p of the expert-sorted order (MoE).
__device__ __forceinline__ int item_at(const RowArgs &ra, int p) { return ra.direct ? p : __ldg(ra.perm + p); }


// Activation row and output offset of token slot n (-1 if the slot is empty).
template <bool MOE>
__device__ __forceinline__ void slot_rows(const RowArgs &ra, int off0, int cnt, int n, int &xrow, long long &yoff) {
    xrow = -1;
    yoff = -1;
    if (n < cnt) {
        if constexpr (MOE) {
            const int item = item_at(ra, off0 + n);
            xrow = ra.x_per_slot ? item : item / ra.topk;
            yoff = (long long)item * ra.ldy;
        } else {
            xrow = n;
            yoff = (long long)n * ra.ldy;
        }
    }
}

// NT: 8-token MMA tiles (1 or 2).  ONE: exactly one token (the epilogue keeps
// only the accumulators that hold it).  SLOTS: ring depth per warp.  ROWS:
// weight rows per warp tile (32 or 48).  RS (MoE with few K blocks): the warps
// split rows instead of K - warp w owns rows w*ROWS.. of a 4*ROWS-row CTA over
// all K blocks and stores its own outputs, with no cross-warp reduction.  CH:
// token slots per chunk (at most 8 * NT; fewer shrinks the activation part of a
// slot when experts get few items).  GLU (MoE): the gate (tmW) and up (tmAux)
// projections of an expert FFN in one pass - warps 0-1 take the gate matrix,
// warps 2-3 the up matrix, for the same rows (row split: a 2*ROWS-row CTA, the
// pairs owning ROWS rows each; K split: each pair splits K) - and the epilogue
// stores h = bf16(silu(g) * u) (RowArgs::glu.h) instead of fp32 rows.  DC (MoE
// with very few items, the down projection): grid layer z is token z, warp w
// takes the token's slots w, w+4, ... whole (all K blocks of its expert's rows),
// and the CTA sums g[t][j] * out[t][j] over j in increasing order into y[t]:
// the weighted combine, in the CTA, with the bits of the separate combine pass.
// X8 (dense): int8 activations with per-32 fp32 scales (tmX: the int8 rows,
// tmAux: the scale rows), multiplied through block_mma_x8.
// tmAux: GLU: the up matrix; X8: the activation scales; otherwise unused.
// FP4 (dense): NVFP4 weights in the same 144-byte blocks (block_mma_fp4), the
// outputs multiplied by RowArgs::gscale.
// PUSH (dense, K split over a cluster): ranks 1.. store their CTA partial into a
// landing buffer in rank 0's shared memory and arrive on its barrier, then exit;
// rank 0 adds the partials in rank order.  Without it the K split's ranks meet at
// cluster barriers and rank 0 reads the others' partials (same order, same bits).
template <int NT, bool MOE, bool ONE, int SLOTS, int ROWS, bool RS = false, int CH = 8 * NT, bool GLU = false,
          bool DC = false, bool X8 = false, bool FP4 = false, bool PUSH = false>
__global__ void __launch_bounds__(kThreads) smallm_kernel(const __grid_constant__ CUtensorMap tmW,
                                                          const __grid_constant__ CUtensorMap tmAux,
                                                          const __grid_constant__ CUtensorMap tmX, RowArgs ra, int N,
                                                          int KB, int nx, unsigned int *status) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int abort_flag;
    __shared__ long long yoff_s[16];

    using G = Geo<ROWS>;
    constexpr int kRows = ROWS, kRowTiles = G::kRowTiles, kBlkWBytes = G::kBlkWBytes;
    constexpr int kPerChunk = CH;
    static_assert(CH <= 8 * NT && (CH == 8 * NT || (MOE && RS)), "chunk size");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = lane & 3, r = lane >> 2;
    const int S = gridDim.x;       // K split = cluster size (always 1 for MoE)
    const int split = blockIdx.x;  // == cluster rank
    static_assert(!RS || (MOE && ROWS == 32), "row split is a MoE mode");
    static_assert(!GLU || MOE, "the fused gate and up projections are a MoE mode");
    static_assert(!DC || (MOE && !RS && !GLU && NT == 1 && ONE), "the in-CTA combine is a one-token MoE mode");
    static_assert(!X8 || !MOE, "int8 activations are a dense mode");
    static_assert(!FP4 || (!MOE && !X8), "NVFP4 weights are a dense bf16 mode");
    // activation bytes copied per token slot and block: 512 bf16, or 256 int8 + 32 of scales
    constexpr int kXTx = X8 ? 256 + 32 : kXBlkBytes;
    // GLU: the warp pair of matrix `mat` (0 gate, 1 up); wsub = this warp's index in its pair
    constexpr int kNw = GLU ? 2 : kWarps;  // warps per weight matrix
    const int mat = GLU ? warp >> 1 : 0, wsub = GLU ? warp & 1 : warp;
    const CUtensorMap *tw = mat ? &tmAux : &tmW;
    const int row0 = blockIdx.y * kRows * (RS ? kNw : 1);
    const int wrow0 = row0 + (RS ? wsub * kRows : 0);  // this warp's first row
    // the cluster splits K, except in DC mode, where its ranks split the token's slots
    const int kS = DC ? 1 : S, ksplit = DC ? 0 : split;
    const int kb0 = (int)((int64_t)KB * ksplit / kS), kb1 = (int)((int64_t)KB * (ksplit + 1) / kS);
    // this warp's blocks: all of them (row split), or blocks wsub, wsub+kNw, ... of the split
    const int nblk = RS || DC ? kb1 - kb0 : (kb1 - kb0 > wsub ? (kb1 - kb0 - wsub + kNw - 1) / kNw : 0);
    const int kb_first = RS || DC ? kb0 : kb0 + wsub, kb_step = RS || DC ? 1 : kNw;

    // the routing comes from the previous kernel (DC with ids_early: wait below)
    if constexpr (MOE) {
        if (!DC || !ra.ids_early) pdl_wait();
    }
    int off0 = 0, cnt = ra.M, tma_row = wrow0;
    // DC: bit j of dc_mask marks this warp's j-th slot (slot warp + 4j) as valid;
    // its chunks are the valid ones, in order
    unsigned dc_mask = 0;
    if constexpr (DC) {
        // warp w of cluster rank q takes slots q*4 + w + 4*S*i
        const int j = split * kWarps + warp + kWarps * S * lane;
        bool v = false;
        if (lane < 16 && j < ra.topk) {
            const int e = __ldg(ra.ids + (int)blockIdx.z * ra.topk + j);
            v = e >= 0 && e < ra.E;
        }
        dc_mask = __ballot_sync(0xFFFFFFFFu, v);
        cnt = 1;
    }
    if constexpr (MOE && !DC) if (ra.direct) {
        // grid layer z = item z
        const int item = blockIdx.z, e = __ldg(ra.ids + item);
        if (e < 0 || e >= ra.E) {  // invalid id: zero this CTA's part of the row, leave before any barrier
            if (ra.zero_invalid)
                for (int col = threadIdx.x; col < kRows * (RS ? kNw : 1); col += kThreads)
                    if (row0 + col < N) ra.y[(long long)item * ra.ldy + row0 + col] = 0.0f;
            return;
        }
        off0 = item;
        cnt = 1;
        tma_row = e * N + wrow0;
    }
    if constexpr (MOE && !DC) if (!ra.direct) {
        // grid layer z = token tile z of the routing (only tiles of experts that have items);
        // the layer right after the last tile zeroes the invalid items' rows of this row tile.
        // A routing made for another shape: leave before any barrier, reading none of it
        if (!routing_matches(ra.n_tiles, ra.E, ra.n_items, status)) return;
        const int n_tl = __ldg(ra.n_tiles);
        if ((int)blockIdx.z >= n_tl) {  // leave before any barrier
            if ((int)blockIdx.z == n_tl && ra.zero_invalid)
                for (int p = __ldg(ra.n_valid) + (RS ? 0 : warp); p < ra.n_items; p += (RS ? 1 : kWarps))
                    if (wrow0 + lane < N) ra.y[(long long)__ldg(ra.perm + p) * ra.ldy + wrow0 + lane] = 0.0f;
            return;
        }
        const int4 tl = __ldg(ra.tiles + blockIdx.z);
        const int e = tl.x;
        off0 = tl.y;
        cnt = tl.z;
        if (cnt <= 0) return;  // expert without tokens: the whole CTA leaves before any barrier
        tma_row = e * N + wrow0;
    }
    const int chunks = DC ? __popc(dc_mask) : (cnt + kPerChunk - 1) / kPerChunk;
    const int total = chunks * nblk;  // this warp's (chunk, block) iterations
    // DC: the token slot of chunk ch
    auto dc_slot = [&](int ch) {
        unsigned m = dc_mask;
        for (int i = 0; i < ch; ++i) m &= m - 1;  // drop the ch lowest valid slots
        return split * kWarps + warp + kWarps * S * (__ffs(m) - 1);
    };

    const int sbytes = G::slot_bytes(nx);
    uint8_t *region = smem + warp * G::warp_bytes(nx, SLOTS);
    float *table = reinterpret_cast<float *>(region + SLOTS * sbytes);
    const uint32_t bar0 = smem_u32(smem + G::bars_off(nx, SLOTS)) + warp * SLOTS * 8;
    // PUSH (dense K split): rank 0's landing barrier for the other ranks' partials
    const uint32_t lbar = smem_u32(smem + G::bars_off(nx, SLOTS)) + kWarps * SLOTS * 8;
    if (threadIdx.x == 0) abort_flag = 0;
    if constexpr (PUSH && !MOE) {
        if (threadIdx.x == 0) mbar_init(lbar, (S - 1) * kThreads);
    }
    if (lane == 0) {
        for (int i = 0; i < SLOTS; ++i) mbar_init(bar0 + 8 * i, 1);
        fence_mbar_init();
        prefetch_tmap(tw);
        prefetch_tmap(&tmX);
        if constexpr (!MOE) {
            // static weights: the weight halves of the first slots go out before the
            // wait (the transaction count covers the activations copied after it)
            if (ra.early_w)
                for (int it = 0; it < SLOTS && it < total; ++it) {
                    const uint32_t bar = bar0 + 8 * (it % SLOTS);
                    mbar_arrive_expect_tx(bar, kBlkWBytes + min(kPerChunk, cnt) * kXTx);
                    tma_load_2d(smem_u32(region + (it % SLOTS) * sbytes), tw, (kb_first + kb_step * it) * kBlkWords,
                                tma_row, bar);
                }
        }
        if constexpr (DC) {
            // the same for the first slots' expert weights (one token slot each)
            if (ra.ids_early)
                for (int it = 0; it < SLOTS && it < total; ++it) {
                    const uint32_t bar = bar0 + 8 * (it % SLOTS);
                    const int item = (int)blockIdx.z * ra.topk + dc_slot(it / nblk);
                    mbar_arrive_expect_tx(bar, kBlkWBytes + kXTx);
                    tma_load_2d(smem_u32(region + (it % SLOTS) * sbytes), tw, (kb_first + kb_step * (it % nblk)) *
                                kBlkWords, __ldg(ra.ids + item) * N + wrow0, bar);
                }
        }
    }
    if constexpr (!MOE) pdl_wait();  // x may come from the previous kernel
    if constexpr (DC) {
        if (ra.ids_early) pdl_wait();  // h comes from the previous kernel
    }
    pdl_trigger();
    __syncthreads();
    if constexpr (PUSH && !MOE) cluster_arrive();  // waited on before the partials are pushed

    // issue the copies of iteration `it` (chunk it / nblk, block it % nblk) into
    // its slot; `weights` false: the weight copy (and the transaction count) went out already
    auto issue = [&](int it, bool weights) {
        const int ch = it / nblk, kb = kb_first + kb_step * (it % nblk);
        const int slot = it % SLOTS;
        const int nvalid = DC ? 1 : min(kPerChunk, cnt - ch * kPerChunk);
        int xrow;
        long long unused;
        int row_w = tma_row;
        if constexpr (DC) {
            const int item = (int)blockIdx.z * ra.topk + dc_slot(ch);
            xrow = ra.x_per_slot ? item : item / ra.topk;
            row_w = __ldg(ra.ids + item) * N + wrow0;
        } else {
            slot_rows<MOE>(ra, off0, cnt, ch * kPerChunk + lane, xrow, unused);
        }
        const uint32_t dst = smem_u32(region + slot * sbytes);
        if (lane == 0 && weights) {
            mbar_arrive_expect_tx(bar0 + 8 * slot, kBlkWBytes + nvalid * kXTx);
            tma_load_2d(dst, tw, kb * kBlkWords, row_w, bar0 + 8 * slot);
        }
        __syncwarp();
        if (lane < nvalid) {
            if constexpr (X8) {
                // 256 int8 values (32 x 8-byte elements), then the 8 scales (4 x 8 bytes)
                tma_load_2d(dst + kBlkWBytes + lane * kXBlkBytes, &tmX, kb * (kQK / 8), xrow, bar0 + 8 * slot);
                tma_load_2d(dst + kBlkWBytes + lane * kXBlkBytes + 256, &tmAux, kb * 4, xrow, bar0 + 8 * slot);
            } else {
                tma_load_2d(dst + kBlkWBytes + lane * kXBlkBytes, &tmX, kb * (kQK / 4), xrow, bar0 + 8 * slot);
            }
        }
    };

    const bool early = (!MOE && ra.early_w) || (DC && ra.ids_early);
    for (int it = 0; it < SLOTS && it < total; ++it) issue(it, !early);

    float acc[kRowTiles][NT][4];
    bool aborted = false;
    int it = 0;
    for (int ch = 0; ch < chunks; ++ch) {
#pragma unroll
        for (int rt = 0; rt < kRowTiles; ++rt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[rt][nt][q] = 0.0f;
        const int nvalid = DC ? 1 : min(kPerChunk, cnt - ch * kPerChunk);
        bool live[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) live[nt] = nt * 8 + r < nvalid;

        for (int j = 0; j < nblk && !aborted; ++j, ++it) {
            const int slot = it % SLOTS;
            // every lane observes the copy's completion; the decision to go on is warp-uniform
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar0 + 8 * slot, (it / SLOTS) & 1, status))) {
                aborted = true;
                if (lane == 0) atomicExch(&abort_flag, 1);
                break;
            }
            const uint8_t *wst = region + slot * sbytes;
            const uint8_t *xs = wst + kBlkWBytes;
            if constexpr (!FP4) {
                decode_scales<X8>(wst + lane * kBlockBytes, table + lane * (kTableRowBytes / 4));
                if constexpr (kRows > 32) {
                    if (lane < kRows - 32)
                        decode_scales<X8>(wst + (lane + 32) * kBlockBytes,
                                          table + (lane + 32) * (kTableRowBytes / 4));
                }
            }
            __syncwarp();
            if constexpr (FP4)
                block_mma_fp4<NT, ONE, kRowTiles>(wst, xs, live, acc, r, c);
            else if constexpr (X8)
                block_mma_x8<NT, ONE, kRowTiles>(wst, xs, table, live, nvalid, acc, r, c);
            else
                block_mma<NT, ONE, kRowTiles>(wst, xs, table, live, acc, r, c);
            // the slot is consumed: order the reads before the copy that refills it
            __syncwarp();
            fence_proxy_async_smem();
            if (it + SLOTS < total) issue(it + SLOTS, true);
        }
        if constexpr (DC) {
            // this slot's complete output rows (token 0 of the fragment: lanes with
            // c == 0, accumulators 0 and 2) into row dc_slot(ch) of the [16][kRows] stage
            float *o = reinterpret_cast<float *>(smem + G::red_off(nx, SLOTS)) + dc_slot(ch) * kRows;
            if (c == 0)
#pragma unroll
                for (int rt = 0; rt < kRowTiles; ++rt) {
                    o[rt * 16 + r] = acc[rt][0][0];
                    o[rt * 16 + r + 8] = acc[rt][0][2];
                }
        } else if constexpr (MOE && RS) {
            // row split: this warp stores its own rows of the chunk, staged as
            // [16][kRows] in its scale table (free until the next chunk's first
            // block) so that the stores coalesce
            static_assert(16 * 32 * 4 <= kTableRowBytes * 32, "the stage fits in the table");
            float *mine = table;
#pragma unroll
            for (int rt = 0; rt < kRowTiles; ++rt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int rA = rt * 16 + r, tk = nt * 8 + 2 * c;
                    mine[tk * kRows + rA] = acc[rt][nt][0];
                    mine[(tk + 1) * kRows + rA] = acc[rt][nt][1];
                    mine[tk * kRows + rA + 8] = acc[rt][nt][2];
                    mine[(tk + 1) * kRows + rA + 8] = acc[rt][nt][3];
                }
            __syncwarp();
            if constexpr (GLU) {
                // the gate warp of each pair forms h from its own rows and those of the
                // up warp two places on (same rows), once both are staged
                __syncthreads();
                if (mat == 0 && !*(volatile int *)&abort_flag) {  // warp-uniform
                    const float *mine_u =
                        reinterpret_cast<const float *>(smem + (warp + 2) * G::warp_bytes(nx, SLOTS) + SLOTS * sbytes);
                    const int my_item = lane < nvalid ? item_at(ra, off0 + ch * kPerChunk + lane) : 0;
                    const bool in = wrow0 + lane < N;
                    for (int tk = 0; tk < nvalid; ++tk) {
                        const long long o =
                            (long long)__shfl_sync(0xFFFFFFFFu, my_item, tk) * ra.ldy + wrow0 + lane;
                        if (in) ra.glu.h[o] = swiglu_bf16(mine[tk * kRows + lane], mine_u[tk * kRows + lane]);
                    }
                }
                __syncthreads();  // the up warps' tables are rewritten by the next chunk
            } else {
                if (!aborted && wrow0 + lane < N)
                    for (int tk = 0; tk < nvalid; ++tk)
                        ra.y[(long long)item_at(ra, off0 + ch * kPerChunk + tk) * ra.ldy + wrow0 + lane] =
                            mine[tk * kRows + lane];
            }
            __syncwarp();  // the slice is reused by the next chunk
        } else if constexpr (MOE) {
            // reduce this chunk across the warps (warp order) and store it
            float *red_w = reinterpret_cast<float *>(smem + G::red_off(nx, SLOTS));  // [4][16][kRows]
            float *mine = red_w + warp * 16 * kRows;
#pragma unroll
            for (int rt = 0; rt < kRowTiles; ++rt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int rA = rt * 16 + r, tk = nt * 8 + 2 * c;
                    mine[tk * kRows + rA] = acc[rt][nt][0];
                    mine[(tk + 1) * kRows + rA] = acc[rt][nt][1];
                    mine[tk * kRows + rA + 8] = acc[rt][nt][2];
                    mine[(tk + 1) * kRows + rA + 8] = acc[rt][nt][3];
                }
            if (threadIdx.x < kPerChunk) {
                int xr;
                long long yo;
                slot_rows<MOE>(ra, off0, cnt, ch * kPerChunk + threadIdx.x, xr, yo);
                yoff_s[threadIdx.x] = yo;
            }
            __syncthreads();
            if (!*(volatile int *)&abort_flag) {
                if constexpr (GLU) {
                    // g: the gate pair's partials (warps 0, 1), u: the up pair's (2, 3)
                    for (int e2 = threadIdx.x; e2 < nvalid * kRows; e2 += kThreads) {
                        const float g = red_w[e2] + red_w[16 * kRows + e2];
                        const float u = red_w[2 * 16 * kRows + e2] + red_w[3 * 16 * kRows + e2];
                        const int tk = e2 / kRows, rr = e2 % kRows;
                        if (row0 + rr < N) ra.glu.h[yoff_s[tk] + row0 + rr] = swiglu_bf16(g, u);
                    }
                } else {
                    for (int e2 = threadIdx.x; e2 < nvalid * kRows; e2 += kThreads) {
                        float v = red_w[e2];
#pragma unroll
                        for (int w = 1; w < kWarps; ++w) v += red_w[w * 16 * kRows + e2];
                        const int tk = e2 / kRows, rr = e2 % kRows;
                        if (row0 + rr < N) ra.y[yoff_s[tk] + row0 + rr] = v;
                    }
                }
            }
            __syncthreads();  // red_w and the token table are reused by the next chunk
        }
    }
    if (aborted) drain_ring<SLOTS>(bar0, it, min(total, it + SLOTS), status);
    if constexpr (DC) {
        // the weighted combine of token t over its slots, in slot order; slot j's
        // rows were staged at index j by the cluster rank that owns it ((j / 4) % S),
        // and rank 0 reads the other ranks' over distributed shared memory
        if (S > 1) cluster_sync();
        else __syncthreads();
        const int t = blockIdx.z;
        if (split == 0 && !*(volatile int *)&abort_flag && threadIdx.x < kRows && row0 + (int)threadIdx.x < N) {
            const uint32_t o = smem_u32(smem + G::red_off(nx, SLOTS)) + 4u * threadIdx.x;
            float v = 0.0f;
            for (int j = 0; j < ra.topk; ++j) {
                const int e = __ldg(ra.ids + t * ra.topk + j);
                if (e < 0 || e >= ra.E) continue;
                const uint32_t a = o + 4u * (uint32_t)(j * kRows);
                const int owner = (j / kWarps) % S;
                const float oj = owner == 0 ? *reinterpret_cast<const float *>(smem + G::red_off(nx, SLOTS) +
                                                                                4 * (j * kRows + threadIdx.x))
                                            : ld_shared_cluster_f32(map_shared_rank(a, owner));
                v = fmaf(__ldg(ra.gates + t * ra.topk + j), oj, v);
            }
            ra.y[(long long)t * ra.ldy + row0 + threadIdx.x] = v;
        }
        if (S > 1) cluster_sync();  // keep every rank's stage alive until rank 0 has read it
        return;
    }
    if constexpr (MOE) return;

    __syncthreads();  // all slots consumed: the rings become reduction space
    // per-warp partials, laid out [token][row] so that the final stores coalesce
    float *red_w = reinterpret_cast<float *>(smem);  // [4][16][kRows]
    float *red = red_w + kWarps * 16 * kRows;         // [16][kRows]
    {
        float *mine = red_w + warp * 16 * kRows;
#pragma unroll
        for (int rt = 0; rt < kRowTiles; ++rt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int rA = rt * 16 + r, tk = nt * 8 + 2 * c;
                mine[tk * kRows + rA] = acc[rt][nt][0];
                mine[(tk + 1) * kRows + rA] = acc[rt][nt][1];
                mine[tk * kRows + rA + 8] = acc[rt][nt][2];
                mine[(tk + 1) * kRows + rA + 8] = acc[rt][nt][3];
            }
    }
    if (threadIdx.x < 16) yoff_s[threadIdx.x] = (long long)threadIdx.x * ra.ldy;
    __syncthreads();
    const int elems = cnt * kRows;
    for (int e = threadIdx.x; e < elems; e += kThreads) {
        float v = red_w[e];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) v += red_w[w * 16 * kRows + e];
        red[e] = v;
    }
    if constexpr (PUSH) {
        // ranks 1.. push their partial into rank 0's landing buffer [S-1][elems] (apart
        // from the rings, which rank 0 may still be reading) and arrive on its landing
        // barrier, then leave; rank 0 adds them in rank order, as the pull below does
        __syncthreads();  // red is complete
        cluster_wait();   // the prologue's arrive: rank 0's landing barrier is initialised
        float *land = reinterpret_cast<float *>(smem + G::red_off(nx, SLOTS));
        if (split != 0) {
            const uint32_t dst = map_shared_rank(smem_u32(land + (split - 1) * elems), 0);
            for (int e = threadIdx.x; e < elems; e += kThreads) st_shared_cluster_f32(dst + 4u * e, red[e]);
            mbar_arrive_cluster(map_shared_rank(lbar, 0));
            // second cluster-barrier phase: this rank's stores into rank 0 are done (the
            // arrive above released them); it arrives and leaves without waiting
            cluster_arrive_relaxed();
        } else {
            // (the limit outlasts every bounded wait a pushing rank can make first)
            if (mbar_wait_cluster(lbar, 0, status, (SLOTS + 2) * 4 * kWaitLimitNs)) {
                for (int e = threadIdx.x; e < elems; e += kThreads) {
                    float v = red[e];
                    for (int q = 1; q < S; ++q) v += land[(q - 1) * elems + e];
                    const int tk = e / kRows, rr = e % kRows;
                    if (row0 + rr < N) ra.y[yoff_s[tk] + row0 + rr] = FP4 ? ra.gscale * v : v;
                }
            }
            // rank 0 leaves only after every other rank has arrived on the second phase,
            // that is after its last store into this CTA's shared memory - also when the
            // landing wait above gave up (the other ranks' own waits are bounded)
            cluster_arrive_relaxed();
            cluster_wait();
        }
    } else if (S > 1) {
        cluster_sync();  // every split's partial is in its shared memory
        if (split == 0) {
            const uint32_t base = smem_u32(red);
            for (int e = threadIdx.x; e < elems; e += kThreads) {
                float v = red[e];
                for (int q = 1; q < S; ++q) v += ld_shared_cluster_f32(map_shared_rank(base + 4 * e, q));
                const int tk = e / kRows, rr = e % kRows;
                if (row0 + rr < N) ra.y[yoff_s[tk] + row0 + rr] = FP4 ? ra.gscale * v : v;
            }
        }
        cluster_sync();  // keep every CTA's shared memory alive until rank 0 has read it
    } else {
        __syncthreads();
        for (int e = threadIdx.x; e < elems; e += kThreads) {
            const int tk = e / kRows, rr = e % kRows;
            if (row0 + rr < N) ra.y[yoff_s[tk] + row0 + rr] = FP4 ? ra.gscale * red[e] : red[e];
        }
    }
}

template <int NT, bool MOE, bool ONE, int SLOTS, int ROWS, bool RS = false, int CH = 8 * NT, bool GLU = false,
          bool DC = false, bool X8 = false, bool FP4 = false, bool PUSH = false>
cudaError_t launch_cfg(int S, int tiles, int E, int nx, cudaStream_t s, const CUtensorMap &tmW,
                       const CUtensorMap &tmX, const RowArgs &ra, int N, int KB, unsigned int *status,
                       const CUtensorMap *tmAux = nullptr) {
    // PUSH: rank 0's landing buffer for the other ranks' partials
    const int smem = Geo<ROWS>::smem_total(nx, SLOTS, MOE && !RS) + (PUSH ? (S - 1) * nx * ROWS * 4 : 0);
    auto kern = smallm_kernel<NT, MOE, ONE, SLOTS, ROWS, RS, CH, GLU, DC, X8, FP4, PUSH>;
    cudaError_t e = ensure_smem((const void *)kern, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(S, tiles, E), dim3(kThreads), (size_t)smem, s, dim3(S), tmW, tmAux ? *tmAux : tmW, tmX,
                      ra, N, KB, nx,
                      status);
}

// CTAs of the one-token kernel with ROWS rows that fit on one SM (per device).
template <int ROWS>
int resident_ctas(const DeviceInfo &di) {
    static int cache[64];
    int &slot = cache[di.device < 64 ? di.device : 63];
    if (slot == 0) {
        const int smem = Geo<ROWS>::smem_total(1, 2, false);
        auto kern = smallm_kernel<1, false, true, 2, ROWS>;
        int n = 0;
        cudaError_t e = ensure_smem((const void *)kern, smem);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, smem);
        slot = e == cudaSuccess && n > 0 ? n : 1;
    }
    return slot;
}

// How a dense call splits its work: CTAs of `rows` weight rows (32 or 48), and a
// cluster of S CTAs splitting K when the row tiles alone cannot fill the GPU in
// one wave.  Of the candidates, the one whose busiest SM streams the fewest
// weights wins (ties go to 32 rows).  Depends on (N, K, device) only, never on
// M, so the summation order of a row does not depend on how many tokens share
// the call.
struct Split {
    int rows, S;
};

Split split_for(const DeviceInfo &di, int64_t N, int KB) {
    Split best = {32, 1};
    int64_t best_load = -1;
    const int cand[2] = {32, 48};
    for (int rows : cand) {
        const int64_t tiles = (N + rows - 1) / rows;
        const int64_t fit = (int64_t)(rows == 32 ? resident_ctas<32>(di) : resident_ctas<48>(di)) * di.sm_count;
        int64_t S = fit / tiles;
        if (S > 8) S = 8;
        if (S > KB / kWarps) S = KB / kWarps;  // keep at least one block per warp
        if (S < 1) S = 1;
        const int64_t per_sm = (tiles * S + di.sm_count - 1) / di.sm_count;
        const int64_t load = per_sm * rows * ((KB + S - 1) / S);  // rows x blocks on the busiest SM
        if (best_load < 0 || load < best_load) {
            best = {rows, (int)S};
            best_load = load;
        }
    }
    return best;
}

}  // namespace

cudaError_t launch_smallm(const DeviceInfo &di, const void *w, int64_t N, int64_t K, const uint16_t *x, int64_t M,
                          int64_t ldx, float *y, int64_t ldy, bool early_weights, cudaStream_t s) {
    const int KB = (int)(K / kQK);
    const Split sp = split_for(di, N, KB);
    const int S = sp.S, tiles = (int)((N + sp.rows - 1) / sp.rows);
    CUtensorMap tmW, tmX;
    cudaError_t e = make_weight_tmap(&tmW, w, N, K, sp.rows, kBlkWords);
    if (e != cudaSuccess) return e;
    e = make_act_tmap(&tmX, x, M, K, ldx, kQK / 4);
    if (e != cudaSuccess) return e;
    RowArgs ra = {};
    ra.y = y; ra.ldy = ldy; ra.M = (int)M;
    ra.early_w = early_weights ? 1 : 0;
    const int nx = (int)M, n = (int)N;
    // a K split reduces by pushing the partials to rank 0 (PUSH); without one the
    // kernel has no cluster work at all
    auto go = [&](auto push) -> cudaError_t {
        constexpr bool P = decltype(push)::value;
        if (sp.rows == 48) {
            if (M == 1)
                return launch_cfg<1, false, true, 2, 48, false, 8, false, false, false, false, P>(
                    S, tiles, 1, nx, s, tmW, tmX, ra, n, KB, di.status);
            if (M <= 8)
                return launch_cfg<1, false, false, 2, 48, false, 8, false, false, false, false, P>(
                    S, tiles, 1, nx, s, tmW, tmX, ra, n, KB, di.status);
            return launch_cfg<2, false, false, 2, 48, false, 16, false, false, false, false, P>(
                S, tiles, 1, nx, s, tmW, tmX, ra, n, KB, di.status);
        }
        if (M == 1)
            return launch_cfg<1, false, true, 2, 32, false, 8, false, false, false, false, P>(
                S, tiles, 1, nx, s, tmW, tmX, ra, n, KB, di.status);
        if (M <= 8)
            return launch_cfg<1, false, false, 2, 32, false, 8, false, false, false, false, P>(
                S, tiles, 1, nx, s, tmW, tmX, ra, n, KB, di.status);
        return launch_cfg<2, false, false, 2, 32, false, 16, false, false, false, false, P>(
            S, tiles, 1, nx, s, tmW, tmX, ra, n, KB, di.status);
    };
    return S > 1 ? go(std::true_type{}) : go(std::false_type{});
}

cudaError_t launch_smallm_fp4(const DeviceInfo &di, const void *w, float g, int64_t N, int64_t K, const uint16_t *x,
                              int64_t M, int64_t ldx, float *y, int64_t ldy, bool early_weights, cudaStream_t s) {
    const int KB = (int)(K / kQK);
    const Split sp = split_for(di, N, KB);
    const int S = sp.S, tiles = (int)((N + sp.rows - 1) / sp.rows);
    CUtensorMap tmW, tmX;
    cudaError_t e = make_weight_tmap(&tmW, w, N, K, sp.rows, kBlkWords);
    if (e != cudaSuccess) return e;
    e = make_act_tmap(&tmX, x, M, K, ldx, kQK / 4);
    if (e != cudaSuccess) return e;
    RowArgs ra = {};
    ra.y = y; ra.ldy = ldy; ra.M = (int)M;
    ra.early_w = early_weights ? 1 : 0;
    ra.gscale = g;
    const int nx = (int)M, n = (int)N;
    // a K split reduces by pushing the partials to rank 0 (PUSH), as in launch_smallm
    auto go = [&](auto push) -> cudaError_t {
        constexpr bool P = decltype(push)::value;
        if (sp.rows == 48) {
            if (M == 1)
                return launch_cfg<1, false, true, 2, 48, false, 8, false, false, false, true, P>(
                    S, tiles, 1, nx, s, tmW, tmX, ra, n, KB, di.status);
            if (M <= 8)
                return launch_cfg<1, false, false, 2, 48, false, 8, false, false, false, true, P>(
                    S, tiles, 1, nx, s, tmW, tmX, ra, n, KB, di.status);
            return launch_cfg<2, false, false, 2, 48, false, 16, false, false, false, true, P>(
                S, tiles, 1, nx, s, tmW, tmX, ra, n, KB, di.status);
        }
        if (M == 1)
            return launch_cfg<1, false, true, 2, 32, false, 8, false, false, false, true, P>(
                S, tiles, 1, nx, s, tmW, tmX, ra, n, KB, di.status);
        if (M <= 8)
            return launch_cfg<1, false, false, 2, 32, false, 8, false, false, false, true, P>(
                S, tiles, 1, nx, s, tmW, tmX, ra, n, KB, di.status);
        return launch_cfg<2, false, false, 2, 32, false, 16, false, false, false, true, P>(
            S, tiles, 1, nx, s, tmW, tmX, ra, n, KB, di.status);
    };
    return S > 1 ? go(std::true_type{}) : go(std::false_type{});
}

cudaError_t launch_smallm_x8(const DeviceInfo &di, const void *w, int64_t N, int64_t K, const int8_t *q,
                             const float *sx, int64_t M, float *y, int64_t ldy, bool early_weights, cudaStream_t s) {
    const int KB = (int)(K / kQK);
    const Split sp = split_for(di, N, KB);
    const int S = sp.S, tiles = (int)((N + sp.rows - 1) / sp.rows);
    CUtensorMap tmW, tmX, tmS;
    cudaError_t e = make_weight_tmap(&tmW, w, N, K, sp.rows, kBlkWords);
    if (e != cudaSuccess) return e;
    e = make_bytes_tmap(&tmX, q, M, K, K, kQK);  // per block: 256 int8 values
    if (e != cudaSuccess) return e;
    e = make_bytes_tmap(&tmS, sx, M, K / 8, K / 8, 32);  // per block: 8 fp32 scales
    if (e != cudaSuccess) return e;
    RowArgs ra = {};
    ra.y = y; ra.ldy = ldy; ra.M = (int)M;
    ra.early_w = early_weights ? 1 : 0;
    const int nx = (int)M, n = (int)N;
    // the K split keeps the pull reduction: with the push form the int8 decode step was
    // measured no faster (its steps varied 40-50 us, against 39-40 us with the pull)
    if (sp.rows == 48) {
        if (M == 1)
            return launch_cfg<1, false, true, 2, 48, false, 8, false, false, true>(S, tiles, 1, nx, s, tmW, tmX, ra, n,
                                                                                   KB, di.status, &tmS);
        if (M <= 8)
            return launch_cfg<1, false, false, 2, 48, false, 8, false, false, true>(S, tiles, 1, nx, s, tmW, tmX, ra,
                                                                                    n, KB, di.status, &tmS);
        return launch_cfg<2, false, false, 2, 48, false, 16, false, false, true>(S, tiles, 1, nx, s, tmW, tmX, ra, n,
                                                                                 KB, di.status, &tmS);
    }
    if (M == 1)
        return launch_cfg<1, false, true, 2, 32, false, 8, false, false, true>(S, tiles, 1, nx, s, tmW, tmX, ra, n, KB,
                                                                               di.status, &tmS);
    if (M <= 8)
        return launch_cfg<1, false, false, 2, 32, false, 8, false, false, true>(S, tiles, 1, nx, s, tmW, tmX, ra, n,
                                                                                KB, di.status, &tmS);
    return launch_cfg<2, false, false, 2, 32, false, 16, false, false, true>(S, tiles, 1, nx, s, tmW, tmX, ra, n, KB,
                                                                             di.status, &tmS);
}

namespace {

struct MoeShape {
    bool rs, deep;
    int64_t per_expert;
    bool direct, few;
    int tiles, layers, nx1;
};

// The MoE kernel variant for a call: row split or not, chunk size, ring depth.
template <bool GLU>
cudaError_t moe_variant(const MoeShape &m, cudaStream_t s, const CUtensorMap &tmW, const CUtensorMap *tmAux,
                        const CUtensorMap &tmX, const RowArgs &ra, int n, int KB, unsigned int *status) {
    if (m.rs) {
        // chunks of 4, 8 or 16 token slots for up to 4, 8 or more items per expert
        // on average (every chunk streams the weights once); a third ring slot while
        // the CTAs of the experts with items fit on the SMs at once
        if (m.per_expert <= 4 || m.direct) {
            const int nx = m.nx1 ? 1 : 4;
            return m.deep ? launch_cfg<1, true, false, 3, 32, true, 4, GLU>(1, m.tiles, m.layers, nx, s, tmW, tmX, ra,
                                                                             n, KB, status, tmAux)
                          : launch_cfg<1, true, false, 2, 32, true, 4, GLU>(1, m.tiles, m.layers, nx, s, tmW, tmX, ra,
                                                                             n, KB, status, tmAux);
        }
        if (m.per_expert <= 8)
            return m.deep ? launch_cfg<1, true, false, 3, 32, true, 8, GLU>(1, m.tiles, m.layers, 8, s, tmW, tmX, ra, n,
                                                                             KB, status, tmAux)
                          : launch_cfg<1, true, false, 2, 32, true, 8, GLU>(1, m.tiles, m.layers, 8, s, tmW, tmX, ra, n,
                                                                             KB, status, tmAux);
        return launch_cfg<2, true, false, 2, 32, true, 16, GLU>(1, m.tiles, m.layers, 16, s, tmW, tmX, ra, n, KB,
                                                                 status, tmAux);
    }
    if (m.few)
        return launch_cfg<1, true, false, 3, 32, false, 8, GLU>(1, m.tiles, m.layers, m.nx1 ? 1 : 8, s, tmW, tmX, ra,
                                                                 n, KB, status, tmAux);
    return launch_cfg<2, true, false, 2, 32, false, 16, GLU>(1, m.tiles, m.layers, 16, s, tmW, tmX, ra, n, KB, status, tmAux);
}

}  // namespace

cudaError_t launch_moe_smallm(const DeviceInfo &di, const void *w_experts, int E, int64_t N, int64_t K,
                              const uint16_t *x, int x_per_slot, const int32_t *perm, const int32_t *offsets,
                              const int4 *tok_tiles, const int *n_tiles, const int32_t *ids, int64_t T, int topk,
                              float *out, bool zero_invalid, cudaStream_t s, const GluOut &glu,
                              const void *w_up, const float *gates, bool ids_early) {
    CUtensorMap tmW, tmAux, tmX;
    // all experts stacked: E*N rows of the same pitch
    constexpr int kRows = 32;
    cudaError_t e = make_weight_tmap(&tmW, w_experts, (int64_t)E * N, K, kRows, kBlkWords);
    if (e != cudaSuccess) return e;
    const bool fused = glu.h != nullptr;  // gate (w_experts) and up (w_up) in one pass
    if (fused) {
        if (!w_up) return cudaErrorInvalidValue;
        e = make_weight_tmap(&tmAux, w_up, (int64_t)E * N, K, kRows, kBlkWords);
        if (e != cudaSuccess) return e;
    }
    e = make_act_tmap(&tmX, x, x_per_slot ? T * topk : T, K, K, kQK / 4);
    if (e != cudaSuccess) return e;
    const int KB = (int)(K / kQK);
    // The warps split rows instead of K when K gives them fewer than two blocks
    // each, and with fewer than four when the 128-row CTAs of the experts that can
    // have items still give every SM two CTAs (items spread over many experts).
    const int64_t items_all = T * topk;
    const int64_t rs_ctas = (N + kRows * kWarps - 1) / (kRows * kWarps) * (items_all < E ? items_all : E);
    const bool rs = KB < 2 * kWarps || (KB < 4 * kWarps && rs_ctas >= 2 * (int64_t)di.sm_count);
    // rows per CTA: 32 (K split), 128 (row split), 64 (row split, gate and up fused)
    const int cta_rows = kRows * (rs ? (fused ? 2 : kWarps) : 1);
    const int tiles = (int)((N + cta_rows - 1) / cta_rows);
    RowArgs ra = {};
    ra.y = out; ra.ldy = N; ra.M = 0;
    ra.x_per_slot = x_per_slot; ra.topk = topk; ra.perm = perm; ra.tiles = tok_tiles; ra.n_tiles = n_tiles;
    const int64_t items = T * topk;
    ra.n_valid = offsets + E; ra.n_items = (int)items; ra.zero_invalid = zero_invalid ? 1 : 0;
    ra.direct = moe_direct(items) ? 1 : 0; ra.ids = ids; ra.E = E;
    ra.glu = glu;
    // one grid layer per item (direct), or per possible token tile (+1 to zero the
    // invalid items' rows); layers past the routing's tile count leave at once
    const int layers = ra.direct ? (int)items : (int)moe_max_tiles(E, items) + (zero_invalid ? 1 : 0);
    const int nx1 = ra.direct ? 1 : 0;  // a direct layer has one token: one activation row per slot
    if (ra.direct && gates && !fused) {
        // the weighted combine in the CTA: one grid layer per token, 32-row CTAs in
        // clusters of two that split the token's slots
        ra.gates = gates;
        ra.zero_invalid = 0;
        ra.ids_early = ids_early ? 1 : 0;
        const int t32 = (int)((N + kRows - 1) / kRows);
        return launch_cfg<1, true, true, 3, 32, false, 8, false, true>(2, t32, (int)T, 1, s, tmW, tmX, ra, (int)N,
                                                                        KB, di.status);
    }
    const bool deep = rs_ctas <= di.sm_count;
    const int64_t per_expert = (items + (items < E ? items : E) - 1) / (items < E ? items : E);
    const MoeShape ms = {rs, deep, per_expert, ra.direct != 0, items <= 64 * (int64_t)E, tiles, layers, nx1};
    return fused ? moe_variant<true>(ms, s, tmW, &tmAux, tmX, ra, (int)N, KB, di.status)
                 : moe_variant<false>(ms, s, tmW, nullptr, tmX, ra, (int)N, KB, di.status);
}

}  // namespace q4k
