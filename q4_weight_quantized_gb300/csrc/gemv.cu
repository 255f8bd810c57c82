// Decode GEMV, one token: y[n] = sum_k w[n][k] x[k] over a Q4_K matrix.
//
// Every decode token streams the whole weight matrix once (sparkinfer-server
// README, "Determinism": the decode path carries no floating-point atomics;
// ninfer serving docs, "Determinism": decode kernels are picked by the step's
// token count).  At one token the product is bound by HBM only if the SMs turn
// 0.5625-byte-per-weight blocks into dot products with very few instructions.
// This kernel is built for that:
//
//   * Work split as in the small-M kernel: a CTA owns ROWS (32 or 48) weight
//     rows, its four warps take K blocks w, w+4, ..., and narrow N splits K over
//     a thread-block cluster.  Each warp streams its blocks through a private
//     2-slot TMA ring (one ROWS x 144-byte tensor copy per block).
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
//   * The activations are staged once per warp (its blocks only): multiplied by
//     2^64 (exact, so that the products are normal fp32 numbers), permuted into
//     MMA order per sub-block, with the sub-block sums S_s beside them.  The four
//     lanes whose column is their own sub-block read them; the others read zeros.
//   * The bias term sum_s dmin m_s S_s is accumulated by the lane that decodes a
//     row's block header (lane = row), so the quad lanes only scale C_s.
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

constexpr int kWarpsG = 4;  // split the CTA's K blocks
constexpr int kThreadsG = kWarpsG * 32;
constexpr int kSlotsG = 2;
constexpr int kBlkWordsG = kBlockBytes / 4;  // 36 (TMA box inner dim, uint32)
constexpr int kXsBytes = 512;                // one block's staged activations: 8 sub-blocks x 16 pairs
constexpr int kSumBytes = 32;                // one block's 8 scaled sub-block sums
constexpr float kXScale = 18446744073709551616.0f;   // 2^64
constexpr float kSumScale = 1.6940658945086007e-21f;  // 2^-69 = 2^64 * 2^-133
constexpr float kYScale = 590295810358705651712.0f;   // 2^69

template <int ROWS>
struct GemvGeo {
    static constexpr int kRT = ROWS / 16;               // 16-row MMA tiles per warp
    static constexpr int kSlotBytes = ROWS * kBlockBytes;  // one block column of the CTA's rows
    static constexpr int kTableBytes = ROWS * 32;          // 8 scales per row
    // per warp: [ring][scale table][staged activations nbw x 512][sub-block sums nbw x 32], 128-byte multiple
    __host__ __device__ static constexpr int warp_bytes(int nbw) {
        return (kSlotsG * kSlotBytes + kTableBytes + nbw * (kXsBytes + kSumBytes) + 127) / 128 * 128;
    }
    // CTA: [warp regions][64 zero bytes][ring barriers][landing barrier][landing buffer (K split)]
    __host__ __device__ static constexpr int zero_off(int nbw) { return kWarpsG * warp_bytes(nbw); }
    __host__ __device__ static constexpr int bars_off(int nbw) { return zero_off(nbw) + 64; }
    __host__ __device__ static constexpr int land_off(int nbw) { return bars_off(nbw) + kWarpsG * kSlotsG * 8 + 16; }
    __host__ __device__ static constexpr int smem_total(int nbw, int S) {
        return land_off(nbw) + (S > 1 ? (S - 1) * ROWS * 4 : 0);
    }
    static_assert(kSlotBytes % 128 == 0 && kTableBytes % 128 == 0, "TMA destinations stay 128-byte aligned");
    static_assert(ROWS % 16 == 0 && ROWS <= 64, "rows per CTA");
    // the reduction buffers [4][ROWS] + [ROWS] floats reuse warp 0's ring
    static_assert((kWarpsG + 1) * ROWS * 4 <= kSlotsG * kSlotBytes, "reduction buffers fit the ring");
};

__device__ __forceinline__ float byte_as_float(uint32_t w, int i) {  // 2^23 + byte i of w
    return __uint_as_float(prmt(w, 0x4B000000u, 0x7440u | (uint32_t)i));
}

// One row's block header -> the 8 scales of its MMA columns (d sc_s, with the
// 1/16 of the high-nibble columns folded in for odd s) into trow[0..8), and
// bias += sum_s (dmin m_s) S_s over the block's scaled sub-block sums.  Every
// product is exact: d, dmin are fp16 values and sc_s, m_s < 64.
__device__ __forceinline__ void decode_row(const uint8_t *blk, float *trow, const float *sums, float &bias) {
    const uint4 h = *reinterpret_cast<const uint4 *>(blk);
    const float d = __half2float(__ushort_as_half((unsigned short)(h.x & 0xFFFFu)));
    const float dmin = __half2float(__ushort_as_half((unsigned short)(h.x >> 16)));
    const float d16 = d * 0.0625f;
    const uint32_t sc_lo = h.y & 0x3F3F3F3Fu;
    const uint32_t m_lo = h.z & 0x3F3F3F3Fu;
    const uint32_t sc_hi = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
    const uint32_t m_hi = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
    const float4 s0 = *reinterpret_cast<const float4 *>(sums);
    const float4 s1 = *reinterpret_cast<const float4 *>(sums + 4);
    const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
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

template <int ROWS, bool PUSH>
__global__ void __launch_bounds__(kThreadsG, 3) gemv_kernel(const __grid_constant__ CUtensorMap tmW,
                                                         const uint16_t *__restrict__ x, float *__restrict__ y,
                                                         int N, int KB, int nbw, int early_w,
                                                         unsigned int *status) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int abort_flag;
    using G = GemvGeo<ROWS>;
    constexpr int kRT = G::kRT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, c = lane & 3;
    const int S = gridDim.x, split = blockIdx.x;  // K split = cluster rank
    const int row0 = blockIdx.y * ROWS;
    const int kb0 = (int)((int64_t)KB * split / S), kb1 = (int)((int64_t)KB * (split + 1) / S);
    const int nblk = kb1 - kb0 > warp ? (kb1 - kb0 - warp + kWarpsG - 1) / kWarpsG : 0;  // <= nbw

    uint8_t *ring = smem + warp * G::warp_bytes(nbw);
    float *table = reinterpret_cast<float *>(ring + kSlotsG * G::kSlotBytes);
    uint8_t *xs = ring + kSlotsG * G::kSlotBytes + G::kTableBytes;
    float *sums = reinterpret_cast<float *>(xs + nbw * kXsBytes);
    const uint8_t *zeros = smem + G::zero_off(nbw);
    const uint32_t bar0 = smem_u32(smem + G::bars_off(nbw)) + warp * kSlotsG * 8;
    const uint32_t lbar = smem_u32(smem + G::bars_off(nbw)) + kWarpsG * kSlotsG * 8;

    if (threadIdx.x == 0) abort_flag = 0;
    if (threadIdx.x < 16) reinterpret_cast<float *>(smem + G::zero_off(nbw))[threadIdx.x] = 0.0f;
    if constexpr (PUSH) {
        if (threadIdx.x == 0) mbar_init(lbar, (S - 1) * kThreadsG);
    }
    auto issue = [&](int it) {  // lane 0: the weight copy of this warp's block it
        const uint32_t bar = bar0 + 8 * (it % kSlotsG);
        mbar_arrive_expect_tx(bar, G::kSlotBytes);
        tma_load_2d(smem_u32(ring + (it % kSlotsG) * G::kSlotBytes), &tmW, (kb0 + warp + kWarpsG * it) * kBlkWordsG,
                    row0, bar);
    };
    if (lane == 0) {
        for (int i = 0; i < kSlotsG; ++i) mbar_init(bar0 + 8 * i, 1);
        fence_mbar_init();
        prefetch_tmap(&tmW);
        // static weights: the first blocks go out before waiting on the previous kernel
        if (early_w)
            for (int it = 0; it < kSlotsG && it < nblk; ++it) issue(it);
    }
    pdl_wait();  // x may come from the previous kernel
    pdl_trigger();
    __syncthreads();
    if constexpr (PUSH) cluster_arrive();  // waited on before the partials are pushed
    if (lane == 0 && !early_w)
        for (int it = 0; it < kSlotsG && it < nblk; ++it) issue(it);

    // Stage this warp's activations: lane l holds elements 8l..8l+7 of a block,
    // i.e. elements 8i..8i+7 (i = l & 3) of sub-block s = l >> 2, which are the
    // pairs of MMAs 4i..4i+3 of that sub-block.
    {
        const __nv_bfloat162 k64 = __floats2bfloat162_rn(kXScale, kXScale);
        const int s = lane >> 2, i = lane & 3;
        for (int b = 0; b < nblk; ++b) {
            const int kb = kb0 + warp + kWarpsG * b;
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)kb * kQK) + lane);
            // S_s: the eight values in order, then the quad (butterfly: every lane the same sum)
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
            *reinterpret_cast<uint4 *>(xs + b * kXsBytes + s * 64 + 16 * i) =
                make_uint4(prmt(a, bb, 0x5410u), prmt(a, bb, 0x7632u), prmt(cc, dd, 0x5410u), prmt(cc, dd, 0x7632u));
            if (i == 0) sums[b * 8 + s] = t * kSumScale;
        }
        __syncwarp();
    }

    // the quad lanes whose column is their own low (A) or high (B) sub-block
    const uint8_t *xa_base = r == 2 * c ? xs + r * 64 : zeros;
    const uint8_t *xb_base = r == 2 * c + 1 ? xs + r * 64 : zeros;
    const int xa_step = r == 2 * c ? kXsBytes : 0, xb_step = r == 2 * c + 1 ? kXsBytes : 0;

    float acc[kRT][2];
#pragma unroll
    for (int rt = 0; rt < kRT; ++rt) acc[rt][0] = acc[rt][1] = 0.0f;
    float bias0 = 0.0f, bias1 = 0.0f;  // decode rows lane and 32 + lane
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    bool aborted = false;
    int it = 0;
    for (; it < nblk; ++it) {
        const int slot = it % kSlotsG;
        // every lane observes the copy's completion; the decision to go on is warp-uniform
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar0 + 8 * slot, (it / kSlotsG) & 1, status))) {
            aborted = true;
            if (lane == 0) atomicExch(&abort_flag, 1);
            break;
        }
        const uint8_t *wst = ring + slot * G::kSlotBytes;
        decode_row(wst + lane * kBlockBytes, table + lane * 8, sums + it * 8, bias0);
        if constexpr (ROWS > 32) {
            if (lane < ROWS - 32)
                decode_row(wst + (lane + 32) * kBlockBytes, table + (lane + 32) * 8, sums + it * 8, bias1);
        }
        __syncwarp();
        const uint8_t *xa = xa_base + it * xa_step, *xb = xb_base + it * xb_step;
        float d[kRT][4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
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
                const uint4 wa = *reinterpret_cast<const uint4 *>(wst + (rt * 16 + r) * kBlockBytes + 16 + 32 * c + 16 * h);
                const uint4 wb =
                    *reinterpret_cast<const uint4 *>(wst + (rt * 16 + r + 8) * kBlockBytes + 16 + 32 * c + 16 * h);
                const uint32_t WA[4] = {wa.x, wa.y, wa.z, wa.w}, WB[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t ta = WA[j] >> 8, tb = WB[j] >> 8;
                    // bytes (0, 2): low nibbles -> sub-block 2c (k 2c, 2c+1), high -> 2c+1 (k 2c+8, 2c+9)
                    const uint32_t A0[4] = {WA[j] & 0x000F000Fu, WB[j] & 0x000F000Fu, WA[j] & 0x00F000F0u,
                                            WB[j] & 0x00F000F0u};
                    // bytes (1, 3)
                    const uint32_t A1[4] = {ta & 0x000F000Fu, tb & 0x000F000Fu, ta & 0x00F000F0u, tb & 0x00F000F0u};
                    if (h == 0 && j == 0)
                        mma_bf16_16816(d[rt], A0, BA[0], BB[0], zero4);
                    else
                        mma_bf16_16816(d[rt], A0, BA[2 * j], BB[2 * j], d[rt]);
                    mma_bf16_16816(d[rt], A1, BA[2 * j + 1], BB[2 * j + 1], d[rt]);
                }
            }
        }
        // y += (d sc_s) C_s for this quad's sub-blocks 2c, 2c+1 of rows rt*16 + r and + 8
#pragma unroll
        for (int rt = 0; rt < kRT; ++rt) {
            const float2 sa = *reinterpret_cast<const float2 *>(table + (rt * 16 + r) * 8 + 2 * c);
            const float2 sb = *reinterpret_cast<const float2 *>(table + (rt * 16 + r + 8) * 8 + 2 * c);
            acc[rt][0] = fmaf(sa.x, d[rt][0], acc[rt][0]);
            acc[rt][0] = fmaf(sa.y, d[rt][1], acc[rt][0]);
            acc[rt][1] = fmaf(sb.x, d[rt][2], acc[rt][1]);
            acc[rt][1] = fmaf(sb.y, d[rt][3], acc[rt][1]);
        }
        // the slot and the table are consumed: order the reads before the refill and the next decode
        __syncwarp();
        fence_proxy_async_smem();
        if (lane == 0 && it + kSlotsG < nblk) issue(it + kSlotsG);
    }
    // after a wait gave up: wait (bounded) for this warp's copies still in flight
    if (aborted)
        for (int k = it; k < min(nblk, it + kSlotsG); ++k) (void)mbar_wait(bar0 + 8 * (k % kSlotsG), (k / kSlotsG) & 1, status);

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
    float *red_w = reinterpret_cast<float *>(smem);  // [4][ROWS]
    float *red = red_w + kWarpsG * ROWS;             // [ROWS]
    if (c == 0)
#pragma unroll
        for (int rt = 0; rt < kRT; ++rt) {
            red_w[warp * ROWS + rt * 16 + r] = acc[rt][0];
            red_w[warp * ROWS + rt * 16 + r + 8] = acc[rt][1];
        }
    __syncwarp();
    red_w[warp * ROWS + lane] -= bias0;
    if constexpr (ROWS > 32) {
        if (lane < ROWS - 32) red_w[warp * ROWS + 32 + lane] -= bias1;
    }
    __syncthreads();
    if (threadIdx.x < ROWS) {
        float v = red_w[threadIdx.x];
#pragma unroll
        for (int w = 1; w < kWarpsG; ++w) v += red_w[w * ROWS + threadIdx.x];
        red[threadIdx.x] = v;
    }
    if constexpr (PUSH) {
        // ranks 1.. push their partial into rank 0's landing buffer and leave; rank 0
        // adds them in rank order
        __syncthreads();  // red is complete
        cluster_wait();   // the prologue's arrive: rank 0's landing barrier is initialised
        float *land = reinterpret_cast<float *>(smem + G::land_off(nbw));
        if (split != 0) {
            const uint32_t dst = map_shared_rank(smem_u32(land + (split - 1) * ROWS), 0);
            if (threadIdx.x < ROWS) st_shared_cluster_f32(dst + 4u * threadIdx.x, red[threadIdx.x]);
            mbar_arrive_cluster(map_shared_rank(lbar, 0));
            cluster_arrive_relaxed();  // second phase: this rank's stores into rank 0 are done
        } else {
            // (the limit outlasts every bounded wait a pushing rank can make first)
            if (mbar_wait_cluster(lbar, 0, status, (kSlotsG + 2) * 4 * kWaitLimitNs) && !*(volatile int *)&abort_flag &&
                threadIdx.x < ROWS) {
                float v = red[threadIdx.x];
                for (int q = 1; q < S; ++q) v += land[(q - 1) * ROWS + threadIdx.x];
                if (row0 + (int)threadIdx.x < N) y[row0 + threadIdx.x] = v * kYScale;
            }
            // rank 0 leaves only after every other rank has passed its stores into this CTA
            cluster_arrive_relaxed();
            cluster_wait();
        }
    } else {
        __syncthreads();
        if (threadIdx.x < ROWS && row0 + (int)threadIdx.x < N && !*(volatile int *)&abort_flag)
            y[row0 + threadIdx.x] = red[threadIdx.x] * kYScale;
    }
}

template <int ROWS, bool PUSH>
const void *gemv_fn() {
    return (const void *)gemv_kernel<ROWS, PUSH>;
}

// Blocks per warp: at most ceil(ceil(KB / S) / 4).
int blocks_per_warp(int KB, int S) { return ((KB + S - 1) / S + kWarpsG - 1) / kWarpsG; }

int smem_for(int rows, int KB, int S) {
    const int nbw = blocks_per_warp(KB, S);
    return rows == 32 ? GemvGeo<32>::smem_total(nbw, S) : GemvGeo<48>::smem_total(nbw, S);
}

struct GemvSplit {
    int rows, S;
};

// (rows, S) for an N x KB matrix: among CTAs of 32 or 48 rows and K splits of
// 1..8 (at least one block per warp), the pair whose busiest SM streams the
// fewest weights in one wave (occupancy from the CUDA occupancy calculator at
// that pair's shared memory); ties go to the smaller split, then to 32 rows.
// Cached per (device, N, KB); depends on nothing else.
cudaError_t gemv_split(const DeviceInfo &di, int64_t N, int KB, GemvSplit *out) {
    struct Entry {
        int device;
        int64_t N;
        int KB;
        GemvSplit sp;
    };
    static std::mutex mu;
    static Entry cache[64];
    static int used = 0, next = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < used; ++i)
            if (cache[i].device == di.device && cache[i].N == N && cache[i].KB == KB) {
                *out = cache[i].sp;
                return cudaSuccess;
            }
    }
    GemvSplit best = {32, 1};
    int64_t best_load = -1;
    for (int rows : {32, 48}) {
        const int64_t tiles = (N + rows - 1) / rows;
        for (int S = 1; S <= 8; ++S) {
            if (S > 1 && KB / S < kWarpsG) break;  // keep at least one block per warp
            const int smem = smem_for(rows, KB, S);
            if ((size_t)smem > di.smem_optin) continue;
            const void *fn = rows == 32 ? (S > 1 ? gemv_fn<32, true>() : gemv_fn<32, false>())
                                        : (S > 1 ? gemv_fn<48, true>() : gemv_fn<48, false>());
            cudaError_t e = ensure_smem(fn, smem);
            if (e != cudaSuccess) return e;
            int occ = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, kThreadsG, smem);
            if (e != cudaSuccess) return e;
            if (occ < 1) continue;
            const int64_t fit = (int64_t)occ * di.sm_count;
            if (S > 1 && tiles * S > fit) break;  // a split must fit one wave
            const int64_t per_sm = (tiles * S + di.sm_count - 1) / di.sm_count;
            const int64_t load = per_sm * rows * ((KB + S - 1) / S);
            if (best_load < 0 || load < best_load) {
                best = {rows, S};
                best_load = load;
            }
        }
    }
    std::lock_guard<std::mutex> lock(mu);
    Entry &en = cache[used < 64 ? used++ : (next++ % 64)];
    en = {di.device, N, KB, best};
    *out = best;
    return cudaSuccess;
}

template <int ROWS, bool PUSH>
cudaError_t gemv_launch(const DeviceInfo &di, const CUtensorMap &tmW, const uint16_t *x, float *y, int N, int KB,
                        int S, bool early_weights, cudaStream_t s) {
    const int nbw = blocks_per_warp(KB, S);
    const int smem = GemvGeo<ROWS>::smem_total(nbw, S);
    auto kern = gemv_kernel<ROWS, PUSH>;
    cudaError_t e = ensure_smem((const void *)kern, smem);
    if (e != cudaSuccess) return e;
    const int tiles = (N + ROWS - 1) / ROWS;
    return launch_pdl(kern, dim3(S, tiles, 1), dim3(kThreadsG), (size_t)smem, s, dim3(S), tmW, x, y, N, KB, nbw,
                      early_weights ? 1 : 0, di.status);
}

}  // namespace

cudaError_t launch_gemv(const DeviceInfo &di, const void *w, int64_t N, int64_t K, const uint16_t *x, float *y,
                        bool early_weights, cudaStream_t s) {
    const int KB = (int)(K / kQK);
    GemvSplit sp;
    cudaError_t e = gemv_split(di, N, KB, &sp);
    if (e != cudaSuccess) return e;
    CUtensorMap tmW;
    e = make_weight_tmap(&tmW, w, N, K, sp.rows, kBlkWordsG);
    if (e != cudaSuccess) return e;
    const int n = (int)N;
    if (sp.rows == 48)
        return sp.S > 1 ? gemv_launch<48, true>(di, tmW, x, y, n, KB, sp.S, early_weights, s)
                        : gemv_launch<48, false>(di, tmW, x, y, n, KB, 1, early_weights, s);
    return sp.S > 1 ? gemv_launch<32, true>(di, tmW, x, y, n, KB, sp.S, early_weights, s)
                    : gemv_launch<32, false>(di, tmW, x, y, n, KB, 1, early_weights, s);
}

}  // namespace q4k
