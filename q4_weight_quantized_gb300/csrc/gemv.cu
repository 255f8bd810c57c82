// Decode GEMV, one token: y[n] = sum_k w[n][k] x[k] over a Q4_K matrix.
//
// Every decode token streams the whole weight matrix once (sparkinfer-server
// README, "Determinism": the decode path carries no floating-point atomics;
// ninfer serving docs, "Determinism": decode kernels are picked by the step's
// token count).  At one token the product is bound by HBM only if the SMs turn
// 0.5625-byte-per-weight blocks into dot products with very few instructions.
// This kernel is built for that:
//
//   * Work split: a CTA owns 64 weight rows; one warp per (row group, K group),
//     where the four K groups take K blocks g, g+4, ..., and narrow N splits K
//     over a thread-block cluster.  Each warp streams its blocks through a
//     private TMA ring (one rows x 144-byte tensor copy per block).  Two launch
//     shapes, chosen from (N, SM count) only:
//       - wide (at least one 64-row tile per SM): 8 warps of 32 rows with 3-slot
//         rings, 2 CTAs per SM;
//       - K split (fewer tiles): 4 warps of 64 rows with 2-slot rings, 3 CTAs
//         per SM.
//     Either way the launch is sized so that all of its CTAs are resident at
//     once, so each warp requests its first blocks the moment its CTA starts (at
//     50 MB per matrix, 40-60 % of the weights are in flight before the first
//     block is consumed): HBM runs from a full queue, where a second wave would
//     start cold.
//   * Columns are sub-blocks, not tokens.  mma.m16n8k16 has 8 columns; with one
//     token, 7 of them would be empty.  Here column s of the B operand holds the
//     token's activations of sub-block s (zero elsewhere), and the 16 k-positions
//     of each MMA carry two weights of each of the 8 sub-blocks of a block.  After
//     the block's 16 MMAs the accumulator holds, per weight row, the 8
//     sub-block sums C_s = sum_l q_l x_l, spread over the 4 lanes of a quad (lane
//     c: sub-blocks 2c and 2c+1), and y += sum_s (d sc_s) C_s - sum_s (dmin m_s) S_s
//     needs two scale multiply-adds per row and lane per block.
//   * The codes enter the MMA as bf16 bit patterns without a magic exponent:
//     a nibble in bits 0-3 of a 16-bit lane is the subnormal q * 2^-133, in bits
//     4-7 it is q * 2^-129 (subnormal and the lowest normal binade share one
//     spacing, so the value stays linear in q).  The tensor cores multiply these
//     exactly.  Lane c of a quad takes group c of a row (bytes 32c..32c+31: low
//     nibbles = sub-block 2c, high = 2c+1); one 32-bit word of codes gives four
//     operand registers with one shift and four ANDs: (w, w >> 8) & 0x000F000F
//     and & 0x00F000F0.  Those pair the weights of bytes (0, 2) and (1, 3), so the
//     activations are staged in that order.
//   * Each warp stages one block of activations at a time (the next block's are
//     loaded while the current one computes): multiplied by 2^64 (exact, so that
//     the products are normal fp32 numbers), permuted into MMA order per
//     sub-block, with the sub-block sums S_s beside them.  The four lanes whose
//     column is their own sub-block read them; the others read zeros.
//   * The bias term sum_s dmin m_s S_s is accumulated by the lane that decodes a
//     row's block header (lane = row), so the quad lanes only scale C_s.  The
//     decoding lane writes the row's 8 scales over the row's first code bytes in
//     the ring slot (consumed by then), so the scales need no shared memory of
//     their own; that, and one activation stage per warp, are what let the
//     rings above fit.
//
// Results are run-to-run deterministic: fixed summation orders within the
// tensor core's accumulator, across the quad (butterfly), across the warps
// (warp order) and across the K-split cluster (rank order).  They differ in
// rounding (not in what is computed) from the small-M kernel's, which puts
// tokens in the MMA columns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>
#include <type_traits>

#include "q4k_internal.h"
#include "q4k_ptx.cuh"

namespace q4k {
namespace {

constexpr int kKGroups = 4;                  // warps per row group: K blocks g, g+4, ...
constexpr int kBlkWordsG = kBlockBytes / 4;  // 36 (TMA box inner dim, uint32)
constexpr int kXsBytes = 512;                // one block's staged activations: 8 sub-blocks x 16 pairs
constexpr int kSumBytes = 32;                // one block's 8 scaled sub-block sums
constexpr float kXScale = 18446744073709551616.0f;   // 2^64
constexpr float kSumScale = 1.6940658945086007e-21f;  // 2^-69 = 2^64 * 2^-133
constexpr float kYScale = 590295810358705651712.0f;   // 2^69

// Launch shape: a CTA is HALVES row groups of ROWS_W weight rows, one warp per
// (row group, K group); each warp streams its blocks through a SLOTS-deep ring;
// CTAS CTAs fit on an SM.
template <int ROWS_W, int HALVES, int SLOTS, int CTAS>
struct GemvCfg {
    static constexpr int kHalves = HALVES;
    static constexpr int kWarpsG = kKGroups * kHalves;
    static constexpr int kThreadsG = kWarpsG * 32;
    static constexpr int kRowsW = ROWS_W;                // weight rows per warp
    static constexpr int kRowsG = kRowsW * kHalves;      // weight rows per CTA
    static constexpr int kSlotsG = SLOTS;
    static constexpr int kDecRows = kRowsW / 32;         // rows each lane decodes
    static constexpr int kCtasPerSm = CTAS;
    static constexpr int kRT = kRowsW / 16;                  // 16-row MMA tiles per warp
    static constexpr int kSlotBytes = kRowsW * kBlockBytes;  // one block column of the warp's rows
    static constexpr int kRingBytes = kSlotsG * kSlotBytes;
    // CTA: [warp rings][warp activation stages (one block each)][64 zero bytes]
    //      [ring barriers][landing barrier]
    static constexpr int kXsOff = kWarpsG * kRingBytes;
    static constexpr int kZeroOff = kXsOff + kWarpsG * (kXsBytes + kSumBytes);
    static constexpr int kBarsOff = kZeroOff + 64;
    static constexpr int kSmem = kBarsOff + kWarpsG * kSlotsG * 8 + 16;
    static_assert(kSlotBytes % 128 == 0, "TMA destinations stay 128-byte aligned");
    static_assert(kXsOff % 16 == 0 && kZeroOff % 16 == 0 && kBarsOff % 8 == 0, "aligned regions");
    // after the loop: the reduction buffers [4][rows] + [rows] floats reuse warp 0's
    // ring, the K split's landing buffer [7][rows] warp 1's
    static_assert((kKGroups + 1) * kRowsG * 4 <= kRingBytes, "reduction buffers fit a ring");
    static_assert(7 * kRowsG * 4 <= kRingBytes, "landing buffer fits a ring");
    static_assert(kRowsW % 32 == 0 && kWarpsG >= 2, "whole decode rows per lane; a second ring for the landing");
    static_assert(CTAS * (kSmem + 128 + 1024) <= 233472, "CTAS CTAs fit an SM's shared memory");
};
// Many row tiles (no K split needed to fill the GPU): 8 warps of 32 rows, 3-slot
// rings, 2 CTAs per SM.
using CfgWide = GemvCfg<32, 2, 3, 2>;
// Few row tiles (the K split fills the GPU): 4 warps of 64 rows, 2-slot rings, 3
// CTAs per SM.
using CfgSplit = GemvCfg<64, 1, 2, 3>;

__device__ __forceinline__ float byte_as_float(uint32_t w, int i) {  // 2^23 + byte i of w
    return __uint_as_float(prmt(w, 0x4B000000u, 0x7440u | (uint32_t)i));
}

// One row's block header -> the 8 scales of its MMA columns (d sc_s, with the
// -1/16 of the high-nibble columns folded in for odd s) into trow[0..8), and
// bias += sum_s (dmin m_s) S_s over the block's scaled sub-block sums sv.  Every
// product is exact: d, dmin are fp16 values and sc_s, m_s < 64.
__device__ __forceinline__ void decode_row(const uint8_t *blk, float *trow, const float (&sv)[8], float &bias) {
    const uint4 h = *reinterpret_cast<const uint4 *>(blk);
    const float d = __half2float(__ushort_as_half((unsigned short)(h.x & 0xFFFFu)));
    const float dmin = __half2float(__ushort_as_half((unsigned short)(h.x >> 16)));
    const float d16 = d * -0.0625f;  // odd columns hold -16 C_s
    const uint32_t sc_lo = h.y & 0x3F3F3F3Fu;
    const uint32_t m_lo = h.z & 0x3F3F3F3Fu;
    const uint32_t sc_hi = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
    const uint32_t m_hi = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float dj = (j & 1) ? d16 : d;
        v[j] = fmaf(byte_as_float(j < 4 ? sc_lo : sc_hi, j & 3), dj, -8388608.0f * dj);
        const float dm = fmaf(byte_as_float(j < 4 ? m_lo : m_hi, j & 3), dmin, -8388608.0f * dmin);
        bias = fmaf(dm, sv[j], bias);
    }
    float4 *dst = reinterpret_cast<float4 *>(trow);
    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
}

__device__ __forceinline__ uint32_t bf16x2_scale(uint32_t u, __nv_bfloat162 k) {
    const __nv_bfloat162 t = __hmul2(*reinterpret_cast<const __nv_bfloat162 *>(&u), k);
    return *reinterpret_cast<const uint32_t *>(&t);
}

// Stages one block's activations for the MMA: lane l holds elements 8l..8l+7 of
// the block (v), i.e. elements 8i..8i+7 (i = l & 3) of sub-block s = l >> 2,
// which are the pairs of MMAs 4i..4i+3 of that sub-block; they are multiplied by
// 2^64 and stored in MMA pair order, and S_s (the eight values in order, then the
// quad, butterfly) is stored scaled by 2^-69.  Warp-collective.
__device__ __forceinline__ void stage_x(const uint4 v, uint8_t *xs, float *sums, int lane) {
    const __nv_bfloat162 k64 = __floats2bfloat162_rn(kXScale, kXScale);
    const int s = lane >> 2, i = lane & 3;
    float t = __uint_as_float(v.x << 16);
    t += __uint_as_float(v.x & 0xFFFF0000u);
    t += __uint_as_float(v.y << 16);
    t += __uint_as_float(v.y & 0xFFFF0000u);
    t += __uint_as_float(v.z << 16);
    t += __uint_as_float(v.z & 0xFFFF0000u);
    t += __uint_as_float(v.w << 16);
    t += __uint_as_float(v.w & 0xFFFF0000u);
    t += __shfl_xor_sync(0xFFFFFFFFu, t, 1);
    t += __shfl_xor_sync(0xFFFFFFFFu, t, 2);
    const uint32_t a = bf16x2_scale(v.x, k64), bb = bf16x2_scale(v.y, k64);
    const uint32_t cc = bf16x2_scale(v.z, k64), dd = bf16x2_scale(v.w, k64);
    *reinterpret_cast<uint4 *>(xs + s * 64 + 16 * i) =
        make_uint4(prmt(a, bb, 0x5410u), prmt(a, bb, 0x7632u), prmt(cc, dd, 0x5410u), prmt(cc, dd, 0x7632u));
    if (i == 0) sums[s] = t * kSumScale;
}

template <class C, bool PUSH>
__global__ void __launch_bounds__(C::kThreadsG, C::kCtasPerSm) gemv_kernel(const __grid_constant__ CUtensorMap tmW,
                                                         const uint16_t *__restrict__ x, float *__restrict__ y,
                                                         int N, int KB, int early_w, unsigned int *status,
                                                         unsigned long long wait_ns) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int abort_flag;
    using G = C;
    constexpr int kRT = C::kRT, kHalves = C::kHalves, kWarpsG = C::kWarpsG, kThreadsG = C::kThreadsG;
    constexpr int kRowsW = C::kRowsW, kRowsG = C::kRowsG, kSlotsG = C::kSlotsG, kDecRows = C::kDecRows;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kg = warp % kKGroups, half = warp / kKGroups;
    const int r = lane >> 2, c = lane & 3;
    const int S = gridDim.x, split = blockIdx.x;  // K split = cluster rank
    const int row0 = blockIdx.y * kRowsG, wrow0 = row0 + half * kRowsW;
    const int kb0 = (int)((int64_t)KB * split / S), kb1 = (int)((int64_t)KB * (split + 1) / S);
    // (a row half wholly past N has no blocks: its partial sums stay zero and are never stored)
    const int nblk = wrow0 < N && kb1 - kb0 > kg ? (kb1 - kb0 - kg + kKGroups - 1) / kKGroups : 0;

    uint8_t *ring = smem + warp * G::kRingBytes;
    uint8_t *xs = smem + G::kXsOff + warp * (kXsBytes + kSumBytes);
    float *sums = reinterpret_cast<float *>(xs + kXsBytes);
    const uint8_t *zeros = smem + G::kZeroOff;
    const uint32_t bar0 = smem_u32(smem + G::kBarsOff) + warp * kSlotsG * 8;
    const uint32_t lbar = smem_u32(smem + G::kBarsOff) + kWarpsG * kSlotsG * 8;

    if (threadIdx.x == 0) abort_flag = 0;
    if (threadIdx.x < 16) reinterpret_cast<float *>(smem + G::kZeroOff)[threadIdx.x] = 0.0f;
    if constexpr (PUSH) {
        if (threadIdx.x == 0) mbar_init(lbar, (S - 1) * kThreadsG);
    }
    auto issue = [&](int it, int slot) {  // lane 0: the weight copy of this warp's block it into `slot`
        const uint32_t bar = bar0 + 8 * slot;
        mbar_arrive_expect_tx(bar, G::kSlotBytes);
        tma_load_2d(smem_u32(ring + slot * G::kSlotBytes), &tmW, (kb0 + kg + kKGroups * it) * kBlkWordsG, wrow0, bar);
    };
    if (lane == 0) {
        for (int i = 0; i < kSlotsG; ++i) mbar_init(bar0 + 8 * i, 1);
        fence_mbar_init();
        prefetch_tmap(&tmW);
        // static weights: the first blocks go out before waiting on the previous kernel
        if (early_w)
            for (int it = 0; it < kSlotsG && it < nblk; ++it) issue(it, it);
    }
    pdl_wait();  // x may come from the previous kernel
    // this lane's 8 activations of the warp's block i are xw[i * kKGroups * 32]
    const uint4 *xw = reinterpret_cast<const uint4 *>(x) + (size_t)(kb0 + kg) * 32 + lane;
    uint4 xn = make_uint4(0u, 0u, 0u, 0u), xn2 = make_uint4(0u, 0u, 0u, 0u);
    if (nblk > 0) xn = __ldg(xw);
    if (nblk > 1) xn2 = __ldg(xw + kKGroups * 32);
    pdl_trigger();
    __syncthreads();
    if (lane == 0 && !early_w)
        for (int it = 0; it < kSlotsG && it < nblk; ++it) issue(it, it);
    if (nblk > 0) stage_x(xn, xs, sums, lane);
    __syncwarp();

    // B operand: column s holds sub-block s's activations where the MMA's k
    // positions carry that sub-block's codes.  Lane (r, c) feeds column r at k 2c,
    // 2c+1 (the full code bytes: sub-block 2c's low nibble plus 16 x its neighbour's
    // high nibble) and at k 2c+8, 2c+9 (-16 x the high nibbles): column 2c takes
    // both, so the high nibbles cancel and it sums sub-block 2c's codes; column
    // 2c+1 takes the second only and sums -16 x sub-block 2c+1's codes.
    const uint8_t *xa = r == 2 * c ? xs + r * 64 : zeros;
    const uint8_t *xb = (r >> 1) == c ? xs + r * 64 : zeros;
    // this lane's row r, code group c, within a slot
    const int lrow = r * kBlockBytes + 16 + 32 * c;

    float acc[kRT][2];
#pragma unroll
    for (int rt = 0; rt < kRT; ++rt) acc[rt][0] = acc[rt][1] = 0.0f;
    float bias[kDecRows];  // the rows this lane decodes: lane + 32 i
#pragma unroll
    for (int i = 0; i < kDecRows; ++i) bias[i] = 0.0f;
    // each lane writes its rows' 8 scales over the rows' first 32 code bytes
    auto decode = [&](uint8_t *wst, const float (&sv)[8]) {
#pragma unroll
        for (int i = 0; i < kDecRows; ++i) {
            uint8_t *row = wst + (lane + 32 * i) * kBlockBytes;
            decode_row(row, reinterpret_cast<float *>(row + 16), sv, bias[i]);
        }
    };
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};

    // Half h of a block's MMAs (code bytes 16h..16h+15 of each group): C_s of every
    // row of the warp, accumulated into d (started at zero by h = 0).
    auto mma_half = [&](const uint8_t *wl, int h, float (&d)[kRT][4]) {
        // B registers of MMAs 8h..8h+7: column r's pairs (zero unless r is this quad's sub-block)
        const uint4 a0 = *reinterpret_cast<const uint4 *>(xa + 32 * h);
        const uint4 a1 = *reinterpret_cast<const uint4 *>(xa + 32 * h + 16);
        const uint4 b0 = *reinterpret_cast<const uint4 *>(xb + 32 * h);
        const uint4 b1 = *reinterpret_cast<const uint4 *>(xb + 32 * h + 16);
        const uint32_t BA[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint32_t BB[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int rt = 0; rt < kRT; ++rt) {
            // words 4h..4h+3 of group c of rows rt*16 + r and rt*16 + r + 8
            const uint4 wa = *reinterpret_cast<const uint4 *>(wl + rt * 16 * kBlockBytes + 16 * h);
            const uint4 wb = *reinterpret_cast<const uint4 *>(wl + (rt * 16 + 8) * kBlockBytes + 16 * h);
            const uint32_t WA[4] = {wa.x, wa.y, wa.z, wa.w}, WB[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                // bytes (0, 2) as whole bytes b = q_lo + 16 q_hi (k 2c, 2c+1) and as -16 q_hi
                // (k 2c+8, 2c+9): a byte in bits 0-7 of a bf16 is the exact value b * 2^-133
                const uint32_t A0[4] = {WA[j] & 0x00FF00FFu, WB[j] & 0x00FF00FFu, (WA[j] & 0x00F000F0u) | 0x80008000u,
                                        (WB[j] & 0x00F000F0u) | 0x80008000u};
                // bytes (1, 3), moved down into bytes (0, 2)
                const uint32_t pa = prmt(WA[j], 0u, 0x4341u), pb = prmt(WB[j], 0u, 0x4341u);
                const uint32_t A1[4] = {pa, pb, (pa & 0x00F000F0u) | 0x80008000u, (pb & 0x00F000F0u) | 0x80008000u};
                if (h == 0 && j == 0)
                    mma_bf16_16816(d[rt], A0, BA[0], BB[0], zero4);
                else
                    mma_bf16_16816(d[rt], A0, BA[2 * j], BB[2 * j], d[rt]);
                mma_bf16_16816(d[rt], A1, BA[2 * j + 1], BB[2 * j + 1], d[rt]);
            }
        }
    };
    // y += (d sc_s) C_s for this quad's sub-blocks 2c, 2c+1 of rows rt*16 + r and + 8,
    // with the scales the decoding lanes wrote into the slot at wst
    auto scale = [&](const uint8_t *wst, const float (&d)[kRT][4]) {
        const uint8_t *tl = wst + lrow - 24 * c;
#pragma unroll
        for (int rt = 0; rt < kRT; ++rt) {
            const float2 sa = *reinterpret_cast<const float2 *>(tl + rt * 16 * kBlockBytes);
            const float2 sb = *reinterpret_cast<const float2 *>(tl + (rt * 16 + 8) * kBlockBytes);
            acc[rt][0] = fmaf(sa.x, d[rt][0], acc[rt][0]);
            acc[rt][0] = fmaf(sa.y, d[rt][1], acc[rt][0]);
            acc[rt][1] = fmaf(sb.x, d[rt][2], acc[rt][1]);
            acc[rt][1] = fmaf(sb.y, d[rt][3], acc[rt][1]);
        }
    };
    auto load_sums = [&](float (&sv)[8]) {
        const float4 s0 = *reinterpret_cast<const float4 *>(sums);
        const float4 s1 = *reinterpret_cast<const float4 *>(sums + 4);
        sv[0] = s0.x, sv[1] = s0.y, sv[2] = s0.z, sv[3] = s0.w, sv[4] = s1.x, sv[5] = s1.y, sv[6] = s1.z, sv[7] = s1.w;
    };
    // every lane observes the copy's completion; the decision to go on is warp-uniform
    // (main-loop waits take wait_ns; the drain after a give-up keeps the full limit)
    auto wait_slot = [&](int sl, uint32_t ph) {
        return __all_sync(0xFFFFFFFFu, mbar_wait_limit(bar0 + 8 * sl, ph, status, wait_ns));
    };

    bool aborted = false;
    int it = 0, slot = 0;
    uint32_t phase = 0;
    for (; it < nblk; ++it) {
        // the activations of the block after next (xn2 holds the next block's)
        uint4 xn3 = make_uint4(0u, 0u, 0u, 0u);
        if (it + 2 < nblk) xn3 = __ldg(xw + (size_t)(it + 2) * kKGroups * 32);
        if (!wait_slot(slot, phase)) {
            aborted = true;
            break;
        }
        uint8_t *wst = ring + slot * G::kSlotBytes;
        float sv[8], d[kRT][4];
        load_sums(sv);
        mma_half(wst + lrow, 0, d);
        mma_half(wst + lrow, 1, d);
        // the block's codes and activations are consumed: the activation stage takes
        // the next block, the decoding lanes write the block's scales into the slot
        __syncwarp();
        if (it + 1 < nblk) stage_x(xn2, xs, sums, lane);
        xn2 = xn3;
        decode(wst, sv);
        __syncwarp();
        scale(wst, d);
        // the slot is consumed: order its reads and writes before the refill
        __syncwarp();
        fence_proxy_async_smem();
        if (lane == 0 && it + kSlotsG < nblk) issue(it + kSlotsG, slot);
        if (++slot == kSlotsG) {
            slot = 0;
            phase ^= 1u;
        }
    }
    if (aborted) {
        if (lane == 0) atomicExch(&abort_flag, 1);
        // wait (bounded) for this warp's copies still in flight: blocks it .. it + slots - 1
        for (int k = it; k < min(nblk, it + kSlotsG); ++k) (void)mbar_wait(bar0 + 8 * (k % kSlotsG), (k / kSlotsG) & 1, status);
    }

    // each row's sum over the quad's four column pairs (butterfly: the same bits in every lane)
#pragma unroll
    for (int rt = 0; rt < kRT; ++rt)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float v = acc[rt][q];
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
            acc[rt][q] = v;
        }
    __syncthreads();  // every ring consumed: warp 0's ring becomes the reduction buffer
    // K split: this rank's ring is free (the landing buffer of rank 0 lies in it)
    if constexpr (PUSH) cluster_arrive();
    float *red_w = reinterpret_cast<float *>(smem);  // [4 K groups][64 rows]
    float *red = red_w + kKGroups * kRowsG;           // [64 rows]
    float *myred = red_w + kg * kRowsG + half * kRowsW;
    if (c == 0)
#pragma unroll
        for (int rt = 0; rt < kRT; ++rt) {
            myred[rt * 16 + r] = acc[rt][0];
            myred[rt * 16 + r + 8] = acc[rt][1];
        }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < kDecRows; ++i) myred[lane + 32 * i] -= bias[i];
    __syncthreads();
    if (threadIdx.x < kRowsG) {
        float v = red_w[threadIdx.x];
#pragma unroll
        for (int g = 1; g < kKGroups; ++g) v += red_w[g * kRowsG + threadIdx.x];
        red[threadIdx.x] = v;
    }
    if constexpr (PUSH) {
        // ranks 1.. push their partial into rank 0's landing buffer (warp 1's ring,
        // free once rank 0 has arrived above) and leave; rank 0 adds them in rank order
        __syncthreads();  // red is complete
        cluster_wait();   // every rank has left its loop
        float *land = reinterpret_cast<float *>(smem + G::kRingBytes);
        if (split != 0) {
            const uint32_t dst = map_shared_rank(smem_u32(land + (split - 1) * kRowsG), 0);
            if (threadIdx.x < kRowsG) st_shared_cluster_f32(dst + 4u * threadIdx.x, red[threadIdx.x]);
            mbar_arrive_cluster(map_shared_rank(lbar, 0));
            cluster_arrive_relaxed();  // second phase: this rank's stores into rank 0 are done
        } else {
            // (the limit outlasts every bounded wait a pushing rank can make first)
            if (mbar_wait_cluster(lbar, 0, status, (kSlotsG + 2) * 4 * kWaitLimitNs) && !*(volatile int *)&abort_flag &&
                threadIdx.x < kRowsG) {
                float v = red[threadIdx.x];
                for (int q = 1; q < S; ++q) v += land[(q - 1) * kRowsG + threadIdx.x];
                if (row0 + (int)threadIdx.x < N) y[row0 + threadIdx.x] = v * kYScale;
            }
            // rank 0 leaves only after every other rank has passed its stores into this CTA
            cluster_arrive_relaxed();
            cluster_wait();
        }
    } else {
        __syncthreads();
        if (threadIdx.x < kRowsG && row0 + (int)threadIdx.x < N && !*(volatile int *)&abort_flag)
            y[row0 + threadIdx.x] = red[threadIdx.x] * kYScale;
    }
}

template <class C, bool PUSH>
const void *gemv_fn() {
    return (const void *)gemv_kernel<C, PUSH>;
}

// The K split S of an N x KB matrix: every CTA of the launch is resident at once
// (one wave: each warp's ring then requests its first blocks the moment the CTA
// starts), and within that the largest split up to 8 that leaves every warp at
// least one block, so that the most weight bytes are in flight.  Cached per
// (device, N, KB); depends on nothing else (not on the token count).
template <class C>
cudaError_t gemv_split(const DeviceInfo &di, int64_t N, int KB, int *out) {
    struct Entry {
        int device;
        int64_t N;
        int KB;
        int S;
    };
    static std::mutex mu;
    static Entry cache[64];
    static int used = 0, next = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < used; ++i)
            if (cache[i].device == di.device && cache[i].N == N && cache[i].KB == KB) {
                *out = cache[i].S;
                return cudaSuccess;
            }
    }
    const int64_t tiles = (N + C::kRowsG - 1) / C::kRowsG;
    int best = 1;
    for (int S = 2; S <= 8 && KB / S >= kKGroups; ++S) {
        const int smem = C::kSmem;
        if ((size_t)smem > di.smem_optin) break;
        const void *fn = gemv_fn<C, true>();
        cudaError_t e = ensure_smem(fn, smem);
        if (e != cudaSuccess) return e;
        int occ = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, C::kThreadsG, smem);
        if (e != cudaSuccess) return e;
        if (tiles * S > (int64_t)occ * di.sm_count) break;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(S, (unsigned)tiles, 1);
        cfg.blockDim = dim3(C::kThreadsG);
        cfg.dynamicSmemBytes = (size_t)smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = S;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();  // a split the device cannot place is simply not taken
            break;
        }
        if (tiles > clusters) break;
        best = S;
    }
    std::lock_guard<std::mutex> lock(mu);
    Entry &en = cache[used < 64 ? used++ : (next++ % 64)];
    en = {di.device, N, KB, best};
    *out = best;
    return cudaSuccess;
}

template <class C, bool PUSH>
cudaError_t gemv_launch(const DeviceInfo &di, const CUtensorMap &tmW, const uint16_t *x, float *y, int N, int KB,
                        int S, bool early_weights, unsigned long long wait_ns, cudaStream_t s) {
    const int smem = C::kSmem;
    auto kern = gemv_kernel<C, PUSH>;
    cudaError_t e = ensure_smem((const void *)kern, smem);
    if (e != cudaSuccess) return e;
    const int tiles = (N + C::kRowsG - 1) / C::kRowsG;
    return launch_pdl(kern, dim3(S, tiles, 1), dim3(C::kThreadsG), (size_t)smem, s, dim3(S), tmW, x, y, N, KB,
                      early_weights ? 1 : 0, di.status, wait_ns);
}

template <class C>
cudaError_t launch_cfg(const DeviceInfo &di, const void *w, int64_t N, int64_t K, const uint16_t *x, float *y,
                       bool early_weights, unsigned long long wait_ns, cudaStream_t s) {
    const int KB = (int)(K / kQK);
    int S = 1;
    cudaError_t e = gemv_split<C>(di, N, KB, &S);
    if (e != cudaSuccess) return e;
    CUtensorMap tmW;
    e = make_weight_tmap(&tmW, w, N, K, C::kRowsW, kBlkWordsG);
    if (e != cudaSuccess) return e;
    const int n = (int)N;
    return S > 1 ? gemv_launch<C, true>(di, tmW, x, y, n, KB, S, early_weights, wait_ns, s)
                 : gemv_launch<C, false>(di, tmW, x, y, n, KB, 1, early_weights, wait_ns, s);
}

}  // namespace

// The wide shape when the 64-row tiles alone give every SM a CTA, else the
// K-split shape.  Depends on (N, SM count) only.
cudaError_t launch_gemv(const DeviceInfo &di, const void *w, int64_t N, int64_t K, const uint16_t *x, float *y,
                        bool early_weights, unsigned long long wait_ns, cudaStream_t s) {
    const int64_t tiles = (N + CfgWide::kRowsG - 1) / CfgWide::kRowsG;
    return tiles >= di.sm_count ? launch_cfg<CfgWide>(di, w, N, K, x, y, early_weights, wait_ns, s)
                                : launch_cfg<CfgSplit>(di, w, N, K, x, y, early_weights, wait_ns, s);
}

}  // namespace q4k
