// Small-M Q4_K matmul: decode GEMV (M = 1) and speculative-verify GEMM (M <= 16).
//
// The decode projections of the pages run one token per lane, or 1 + accepted
// drafts per lane when a drafter proposes --draft-tokens N (ninfer serving docs,
// "Start the server" and "Determinism"), and carry no floating-point atomics
// (sparkinfer-server README, "Determinism").  At these M the product is bound by
// streaming the 0.5625-byte-per-weight Q4_K matrix from HBM once, so the kernel
// is built around keeping HBM busy and the per-weight instruction count low:
//
//   * TMA streams the raw blocks: a CTA owns R = 32 consecutive weight rows; each
//     pipeline stage is one 2-D bulk-tensor copy of 32 rows x 4 blocks (18 KiB)
//     into shared memory, issued by a producer warp and completed on an mbarrier.
//     Rows past N and blocks past K/256 are zero-filled by the copy and decode to
//     zero weights.
//   * Four consumer warps each take one block of the stage.  A lane turns one
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
#include <cuda.h>
#include <cuda_fp16.h>

#include "q4k_internal.h"
#include "q4k_ptx.cuh"

namespace q4k {
namespace {

constexpr int kRows = 32;                          // weight rows per CTA
constexpr int kRowTiles = kRows / 16;              // 16-row MMA tiles per CTA
constexpr int kBlocksPerStage = 4;                 // one block per consumer warp
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + producer warp
constexpr int kStageRowBytes = kBlocksPerStage * kBlockBytes;  // 576
constexpr int kStageBytes = kRows * kStageRowBytes;            // 18432
constexpr int kStageWords = kStageRowBytes / 4;                // 144 (TMA box inner dim, uint32)
constexpr int kTableRowBytes = 80;  // 8 x (dsc, bias) + 16 pad: conflict-free 16-byte reads
constexpr int kTableBytes = kConsumerWarps * kRows * kTableRowBytes;
constexpr int kStages = 2;

constexpr size_t smem_bytes() {
    return (size_t)kStages * kStageBytes + kTableBytes + 2 * kStages * 8 + 16;
}

static_assert(kConsumerWarps * kRows * 16 * 4 + kRows * 16 * 4 <= kStages * kStageBytes,
              "reduction buffers alias the stage buffers");

__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t &lo01, uint32_t &lo23, uint32_t &hi01,
                                            uint32_t &hi23) {
    const uint32_t t01 = prmt(w, 0u, 0x4140u);  // bytes 0,1 -> 16-bit lanes
    const uint32_t t23 = prmt(w, 0u, 0x4342u);  // bytes 2,3
    lo01 = lop3_and_or(t01, 0x000F000Fu, 0x43004300u);
    lo23 = lop3_and_or(t23, 0x000F000Fu, 0x43004300u);
    hi01 = lop3_and_or(t01 >> 4, 0x000F000Fu, 0x43004300u);
    hi23 = lop3_and_or(t23 >> 4, 0x000F000Fu, 0x43004300u);
}

// Decode one row's block header (d, dmin, 12 scale bytes) into 8 (d*sc, bias) pairs.
__device__ __forceinline__ void decode_scales(const uint8_t *blk, float *table_row) {
    const uint4 h = *reinterpret_cast<const uint4 *>(blk);
    const float d = __half2float(__ushort_as_half((unsigned short)(h.x & 0xFFFFu)));
    const float dmin = __half2float(__ushort_as_half((unsigned short)(h.x >> 16)));
    const uint32_t sc_lo = h.y & 0x3F3F3F3Fu;
    const uint32_t m_lo = h.z & 0x3F3F3F3Fu;
    const uint32_t sc_hi = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
    const uint32_t m_hi = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
    float v[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t sc = ((j < 4 ? sc_lo : sc_hi) >> (8 * (j & 3))) & 0xFFu;
        const uint32_t m = ((j < 4 ? m_lo : m_hi) >> (8 * (j & 3))) & 0xFFu;
        const float dsc = d * (float)sc;
        v[2 * j] = dsc;
        v[2 * j + 1] = fmaf(dmin, (float)m, 128.0f * dsc);
    }
    float4 *dst = reinterpret_cast<float4 *>(table_row);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

// Where each token slot of a chunk reads its activation row and writes its
// output row.  Dense: slot n is token n.  MoE: slot n of expert e's list is the
// (token, k-slot) item perm[offsets[e] + n].
struct RowArgs {
    const uint16_t *x;
    int64_t ldx;          // dense: activation row stride; MoE: K
    float *y;
    int64_t ldy;          // dense: output row stride; MoE: N
    int M;                // dense: number of tokens (<= 16)
    int x_per_slot;       // MoE: activation row is the item (1) or its token (0)
    int topk;             // MoE
    const int32_t *perm;  // MoE routing permutation
    const int32_t *offsets;
};

__device__ __forceinline__ void consumer_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

template <int NT, bool MOE>
__global__ void __launch_bounds__(kThreads, 4) smallm_kernel(const __grid_constant__ CUtensorMap tmW, RowArgs ra, int N,
                                                          int KB, unsigned int *status) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *stages = smem;
    float *tables = reinterpret_cast<float *>(smem + kStages * kStageBytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes + kTableBytes);
    // MoE keeps its reduction buffers apart from the stages (the pipeline runs on
    // into the next token chunk while a chunk is reduced)
    float *moe_red = reinterpret_cast<float *>(smem + kStages * kStageBytes + kTableBytes + 2 * kStages * 8 + 16);
    __shared__ int abort_flag;
    __shared__ long long xoff_s[16], yoff_s[16];

    constexpr int kPerChunk = 8 * NT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = gridDim.x;       // K split = cluster size (always 1 for MoE)
    const int split = blockIdx.x;  // == cluster rank
    const int row0 = blockIdx.y * kRows;
    const int n_stage_total = (KB + kBlocksPerStage - 1) / kBlocksPerStage;
    const int st0 = (int)((int64_t)n_stage_total * split / S);
    const int st1 = (int)((int64_t)n_stage_total * (split + 1) / S);
    const int nst = st1 - st0;

    int off0 = 0, cnt = ra.M, tma_row = row0;
    if constexpr (MOE) {
        const int e = blockIdx.z;
        off0 = __ldg(ra.offsets + e);
        cnt = __ldg(ra.offsets + e + 1) - off0;
        if (cnt <= 0) return;  // expert without tokens: the whole CTA leaves before any barrier
        tma_row = e * N + row0;
    }
    const int chunks = (cnt + kPerChunk - 1) / kPerChunk;
    const int total_it = chunks * nst;

    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kStages);
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < kStages; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, kConsumerWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    float acc[kRowTiles][NT][4];

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------- producer warp
        if (lane == 0) {
            prefetch_tmap(&tmW);
            for (int it = 0; it < total_it; ++it) {
                const int slot = it % kStages;
                if (it >= kStages && !mbar_wait(empty0 + 8 * slot, ((it / kStages) - 1) & 1, status)) {
                    atomicExch(&abort_flag, 1);
                    break;
                }
                if (*(volatile int *)&abort_flag) break;
                mbar_arrive_expect_tx(full0 + 8 * slot, kStageBytes);
                tma_load_2d(smem_u32(stages + slot * kStageBytes), &tmW, (st0 + it % nst) * kStageWords, tma_row,
                            full0 + 8 * slot);
            }
        }
    } else {
        // ------------------------------------------------------ consumer warps
        const int c = lane & 3, r = lane >> 2;
        const uint32_t ones[4] = {0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u};
        const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
        float *table = tables + warp * (kRows * kTableRowBytes / 4);
        for (int ch = 0; ch < chunks; ++ch) {
            if (threadIdx.x < kPerChunk) {
                const int n = ch * kPerChunk + threadIdx.x;
                long long xo = -1, yo = -1;
                if (n < cnt) {
                    if constexpr (MOE) {
                        const int item = __ldg(ra.perm + off0 + n);
                        xo = (long long)(ra.x_per_slot ? item : item / ra.topk) * ra.ldx;
                        yo = (long long)item * ra.ldy;
                    } else {
                        xo = (long long)n * ra.ldx;
                        yo = (long long)n * ra.ldy;
                    }
                }
                xoff_s[threadIdx.x] = xo;
                yoff_s[threadIdx.x] = yo;
            }
            consumer_bar();
            long long xrow[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) xrow[nt] = xoff_s[nt * 8 + r];
#pragma unroll
            for (int rt = 0; rt < kRowTiles; ++rt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[rt][nt][i] = 0.0f;

            for (int i = 0; i < nst; ++i) {
                const int it = ch * nst + i;
                const int slot = it % kStages;
                // every lane observes the stage's completion; the decision to go on is warp-uniform
                const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(full0 + 8 * slot, (it / kStages) & 1, status));
                if (!ok && lane == 0) atomicExch(&abort_flag, 1);
                if (__any_sync(0xFFFFFFFFu, *(volatile int *)&abort_flag != 0)) break;
                const int kb = (st0 + i) * kBlocksPerStage + warp;
                if (kb < KB) {
                    const uint8_t *stage = stages + slot * kStageBytes + warp * kBlockBytes;
                    decode_scales(stage + lane * kStageRowBytes, table + lane * (kTableRowBytes / 4));
                    __syncwarp();
#pragma unroll 1
                    for (int g = 0; g < 4; ++g) {
                        // activations for sub-blocks 2g (xl) and 2g+1 (xh), per 8-token tile
                        uint32_t xl[NT][4], xh[NT][4];
                        float sl[NT][4], sh[NT][4];
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
                            if (xrow[nt] >= 0) {
                                const uint16_t *xp = ra.x + xrow[nt] + (int64_t)kb * kQK + 64 * g + 8 * c;
                                a = __ldg(reinterpret_cast<const uint4 *>(xp));
                                b = __ldg(reinterpret_cast<const uint4 *>(xp + 32));
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
                            const uint2 wa =
                                *reinterpret_cast<const uint2 *>(stage + rA * kStageRowBytes + 16 + 32 * g + 8 * c);
                            const uint2 wb =
                                *reinterpret_cast<const uint2 *>(stage + rB * kStageRowBytes + 16 + 32 * g + 8 * c);
                            uint32_t alo0[4], alo1[4], ahi0[4], ahi1[4];
                            // word 0 (elements 8c..8c+3) feeds MMA 0, word 1 (8c+4..8c+7) MMA 1
                            unpack_word(wa.x, alo0[0], alo0[2], ahi0[0], ahi0[2]);
                            unpack_word(wb.x, alo0[1], alo0[3], ahi0[1], ahi0[3]);
                            unpack_word(wa.y, alo1[0], alo1[2], ahi1[0], ahi1[2]);
                            unpack_word(wb.y, alo1[1], alo1[3], ahi1[1], ahi1[3]);
                            const float4 sa =
                                *reinterpret_cast<const float4 *>(table + rA * (kTableRowBytes / 4) + 4 * g);
                            const float4 sb =
                                *reinterpret_cast<const float4 *>(table + rB * (kTableRowBytes / 4) + 4 * g);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                float cl[4], chh[4];
                                mma_bf16_16816(cl, alo0, xl[nt][0], xl[nt][1], zero4);
                                mma_bf16_16816(cl, alo1, xl[nt][2], xl[nt][3], cl);
                                mma_bf16_16816(chh, ahi0, xh[nt][0], xh[nt][1], zero4);
                                mma_bf16_16816(chh, ahi1, xh[nt][2], xh[nt][3], chh);
                                float *a4 = acc[rt][nt];
                                // sub-block 2g
                                a4[0] = fmaf(sa.x, cl[0], a4[0]); a4[0] = fmaf(-sa.y, sl[nt][0], a4[0]);
                                a4[1] = fmaf(sa.x, cl[1], a4[1]); a4[1] = fmaf(-sa.y, sl[nt][1], a4[1]);
                                a4[2] = fmaf(sb.x, cl[2], a4[2]); a4[2] = fmaf(-sb.y, sl[nt][2], a4[2]);
                                a4[3] = fmaf(sb.x, cl[3], a4[3]); a4[3] = fmaf(-sb.y, sl[nt][3], a4[3]);
                                // sub-block 2g+1
                                a4[0] = fmaf(sa.z, chh[0], a4[0]); a4[0] = fmaf(-sa.w, sh[nt][0], a4[0]);
                                a4[1] = fmaf(sa.z, chh[1], a4[1]); a4[1] = fmaf(-sa.w, sh[nt][1], a4[1]);
                                a4[2] = fmaf(sb.z, chh[2], a4[2]); a4[2] = fmaf(-sb.w, sh[nt][2], a4[2]);
                                a4[3] = fmaf(sb.z, chh[3], a4[3]); a4[3] = fmaf(-sb.w, sh[nt][3], a4[3]);
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty0 + 8 * slot);
            }
            if constexpr (MOE) {
                // reduce this chunk across the consumer warps (warp order) and store it
                float *red_w = moe_red;  // [4][16][kRows]
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
                consumer_bar();
                const int valid = min(kPerChunk, cnt - ch * kPerChunk);
                for (int e2 = threadIdx.x; e2 < valid * kRows; e2 += 128) {
                    float v = red_w[e2];
#pragma unroll
                    for (int w = 1; w < kConsumerWarps; ++w) v += red_w[w * 16 * kRows + e2];
                    const int tk = e2 / kRows, rr = e2 % kRows;
                    if (row0 + rr < N) ra.y[yoff_s[tk] + row0 + rr] = v;
                }
                consumer_bar();  // red_w and the token table are reused by the next chunk
            }
        }
    }
    if constexpr (MOE) return;

    __syncthreads();  // all stages consumed: the stage buffers become reduction space
    // per-warp partials, laid out [token][row] so that the final stores coalesce
    float *red_w = reinterpret_cast<float *>(stages);  // [4][16][kRows]
    float *red = red_w + kConsumerWarps * 16 * kRows;   // [16][kRows]
    if (warp < kConsumerWarps) {
        const int c = lane & 3, r = lane >> 2;
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
    __syncthreads();
    const int elems = cnt * kRows;
    for (int e = threadIdx.x; e < elems; e += kThreads) {
        float v = red_w[e];
#pragma unroll
        for (int w = 1; w < kConsumerWarps; ++w) v += red_w[w * 16 * kRows + e];
        red[e] = v;
    }
    if (S > 1) {
        cluster_sync();  // every split's partial is in its shared memory
        if (split == 0) {
            const uint32_t base = smem_u32(red);
            for (int e = threadIdx.x; e < elems; e += kThreads) {
                float v = red[e];
                for (int q = 1; q < S; ++q) v += ld_shared_cluster_f32(map_shared_rank(base + 4 * e, q));
                const int tk = e / kRows, rr = e % kRows;
                if (row0 + rr < N) ra.y[yoff_s[tk] + row0 + rr] = v;
            }
        }
        cluster_sync();  // keep every CTA's shared memory alive until rank 0 has read it
    } else {
        __syncthreads();
        for (int e = threadIdx.x; e < elems; e += kThreads) {
            const int tk = e / kRows, rr = e % kRows;
            if (row0 + rr < N) ra.y[yoff_s[tk] + row0 + rr] = red[e];
        }
    }
}

}  // namespace

namespace {

template <int NT, bool MOE>
cudaError_t launch_cfg(int S, int tiles, int E, size_t smem, cudaStream_t s, const CUtensorMap &tm,
                       const RowArgs &ra, int N, int KB, unsigned int *status) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S, tiles, E);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = S > 1 ? 1 : 0;
    cudaError_t e = cudaFuncSetAttribute(smallm_kernel<NT, MOE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, smallm_kernel<NT, MOE>, tm, ra, N, KB, status);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

int split_for(const DeviceInfo &di, int64_t units, int KB) {
    // Split K across a cluster only when the row tiles cannot fill the GPU at the
    // design occupancy of 4 CTAs per SM.  Depends on (N, K, device), never on M.
    const int n_stage_total = (KB + kBlocksPerStage - 1) / kBlocksPerStage;
    int64_t S = (4 * (int64_t)di.sm_count) / (units > 0 ? units : 1);
    if (S > 8) S = 8;
    if (S > n_stage_total) S = n_stage_total;
    if (S < 1) S = 1;
    return (int)S;
}

}  // namespace

cudaError_t launch_smallm(const DeviceInfo &di, const void *w, int64_t N, int64_t K, const uint16_t *x, int64_t M,
                          int64_t ldx, float *y, int64_t ldy, cudaStream_t s) {
    CUtensorMap tm;
    cudaError_t e = make_weight_tmap(&tm, w, N, K, kRows, kStageWords);
    if (e != cudaSuccess) return e;
    const int KB = (int)(K / kQK);
    const int tiles = (int)((N + kRows - 1) / kRows);
    const int S = split_for(di, tiles, KB);
    RowArgs ra = {};
    ra.x = x; ra.ldx = ldx; ra.y = y; ra.ldy = ldy; ra.M = (int)M;
    const size_t smem = smem_bytes();
    if (M <= 8) return launch_cfg<1, false>(S, tiles, 1, smem, s, tm, ra, (int)N, KB, di.status);
    return launch_cfg<2, false>(S, tiles, 1, smem, s, tm, ra, (int)N, KB, di.status);
}

cudaError_t launch_moe_smallm(const DeviceInfo &di, const void *w_experts, int E, int64_t N, int64_t K,
                              const uint16_t *x, int x_per_slot, const int32_t *perm, const int32_t *offsets,
                              int64_t T, int topk, float *out, cudaStream_t s) {
    CUtensorMap tm;
    // all experts stacked: E*N rows of the same pitch
    cudaError_t e = make_weight_tmap(&tm, w_experts, (int64_t)E * N, K, kRows, kStageWords);
    if (e != cudaSuccess) return e;
    const int KB = (int)(K / kQK);
    const int tiles = (int)((N + kRows - 1) / kRows);
    RowArgs ra = {};
    ra.x = x; ra.ldx = K; ra.y = out; ra.ldy = N; ra.M = 0;
    ra.x_per_slot = x_per_slot; ra.topk = topk; ra.perm = perm; ra.offsets = offsets;
    const size_t smem = smem_bytes() + kConsumerWarps * 16 * kRows * 4;
    const int64_t items = T * topk;
    if (items <= 64 * (int64_t)E) return launch_cfg<1, true>(1, tiles, E, smem, s, tm, ra, (int)N, KB, di.status);
    return launch_cfg<2, true>(1, tiles, E, smem, s, tm, ra, (int)N, KB, di.status);
}

}  // namespace q4k
