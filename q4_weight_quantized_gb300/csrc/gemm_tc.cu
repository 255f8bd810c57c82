// Prefill Q4_K (and NVFP4) GEMM on the tcgen05 tensor cores.
//
// A GGUF target dequantizes Q4_K "into the matrix-multiply operand on every
// prefill pass"; that fixed cost dominates at 128 tokens and is amortized by 4k
// (sparkinfer-server README, "Serve a GGUF instead of NVFP4").  This kernel does
// exactly that, tile by tile, without ever writing a dequantized matrix to HBM:
//
//   * A CTA owns 128 weight rows x BN tokens (BN = 256, or 128 for short
//     prompts).  The weight rows are the MMA's M dimension, the tokens its N.
//   * Warp 0 (TMA): per 256-wide K block, one bulk-tensor copy of the raw Q4_K
//     tile (128 rows x 144 bytes) into a ring of raw slots, refilled as soon as
//     a slot's codes are in the dequant warps' registers.  Warp 2 (TMA): per
//     64-wide K stage, one copy of the activation tile (BN tokens x 64 bf16)
//     with the 128-byte swizzle that the tensor core's K-major layout expects.
//   * Warps 4-11 (dequant): two threads per weight row.  Once per K block each
//     loads the 64 code bytes it will convert (16 of each group) and turns them
//     into 128 bf16 weights for the block's four 64-wide stages (one Q4_K group
//     each: sub-blocks 2g and 2g+1), each the round-to-nearest-even bf16 of the
//     fp32 weight fl32(q * d sc - dmin m) (packed fp32 FMAs, q * d sc exact
//     inside them), i.e. the very value the standalone bf16 dequantization
//     writes; then it hands the stages over one by one as the MMA frees them.
//     They go to tensor memory, not shared memory: the row's lane, two weights
//     per column (tcgen05.st), where the MMA reads its A operand.  The
//     tensor core's operand reads, the activation and raw copies and the
//     dequant stores would otherwise all share the SM's shared-memory bandwidth,
//     which then set the pace of every stage.
//   * Warp 1 (MMA): one elected thread issues four 128 x BN x 16 tcgen05.mma per
//     stage (A from tensor memory, B from shared memory) into an fp32
//     accumulator in tensor memory.  It waits on one barrier per stage (the
//     dequant warps and the activation copy both arrive on it) and commits the
//     stage's completion to one barrier that frees both halves of the stage.
//   * Warps 4-11 then read the accumulator (tcgen05.ld, one 32-lane quarter and
//     half the columns per warp) and store fp32 rows of y with coalesced
//     128-byte writes.
//   * When the output has too few tiles to occupy the GPU (short prompts on the
//     narrow down projection), a thread-block cluster splits K: each CTA parks
//     its partial tile in its idle stage buffers and every rank sums one slice of
//     columns over the cluster's distributed shared memory, in rank order - no
//     workspace, no atomics.
// Every wait is bounded.  After one gives up, the producer waits (bounded) for
// the copies it still has in flight and tensor memory is freed only after the
// MMAs issued so far have completed.  The accumulator is a plain sum per output
// element in a fixed order, so the result is run-to-run deterministic.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "q4k_internal.h"
#include "q4k_ptx.cuh"

namespace q4k {
namespace {

constexpr int kTileRows = 128;                    // weight rows per CTA (MMA M)
constexpr int kStageK = 64;                       // K per pipeline stage (one swizzle row of bf16)
constexpr int kRawBytes = kTileRows * kBlockBytes;  // 18 KiB raw Q4_K tile per block
constexpr int kDqWarp0 = 4;                       // first dequant warp: warp w may use tensor-memory lanes 32 (w % 4) ..
constexpr int kDqWarps = 8;                       // two threads per weight row
constexpr int kTPR = kDqWarps / 4;                // dequant threads per weight row
constexpr int kEPT = 32 / kTPR;                   // code bytes of a group per dequant thread and stage
constexpr int kWPT = kEPT / 4;                    // the same in 32-bit words
constexpr int kThreads = (kDqWarp0 + kDqWarps) * 32;
constexpr int kStageCols = kStageK / 2;           // tensor-memory columns of one stage's operand (bf16 pairs)
constexpr uint32_t kTmemCols = 512;               // accumulator + operand stages, whole allocation

// Rings: NS stages, each an activation tile in shared memory plus the
// dequantized weight operand in tensor memory, and RS raw Q4_K slots in shared
// memory.  A stage's activation copy can only start once the MMAs of the stage
// NS before are done, and it crosses L2: NS stages of MMA time must cover an L2
// round trip under load.  A stage is full once the dequant warps have written
// its operand and its activation copy has landed (one barrier), and one commit
// frees both halves, so that the MMA thread waits once and commits once per
// stage.  A raw slot is free again as soon as the dequant warps have read its
// codes into registers, and its own producer refills it at once, RS - 1 blocks
// ahead.
template <int BN>
struct Cfg {
    static constexpr int NS = BN == 128 ? 8 : 4;        // stages
    static constexpr int RS = 3;                        // raw Q4_K slots
    static constexpr int XB = BN * kStageK * 2;         // activation bytes per stage
    static constexpr int x_off = 0;
    static constexpr int raw_off = x_off + NS * XB;
    static constexpr int bar_off = raw_off + RS * kRawBytes;
    static constexpr int n_bars = 2 * NS + 2 * RS + 1;
    static constexpr int misc_off = bar_off + n_bars * 8;
    static constexpr int bytes = misc_off + 16 + 1024;  // + slack to align the base to 1024
    static_assert(bytes <= 227 * 1024, "dynamic shared memory per CTA");
};

__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t u) { return *reinterpret_cast<__nv_bfloat162 *>(&u); }
__device__ __forceinline__ uint32_t as_u32(__nv_bfloat162 v) { return *reinterpret_cast<uint32_t *>(&v); }


// FP4: the weights are NVFP4 blocks (16 e4m3 scales, then 128 bytes of e2m1
// pairs) instead of Q4_K; each operand element is the exact e2m1 * e4m3 product
// in bf16, and the epilogue multiplies by the tensor scale gscale.
template <int BN, bool FP4>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW,
                                                              const __grid_constant__ CUtensorMap tmX, float *y,
                                                              int64_t ldy, int M, int N, int KB, float gscale,
                                                              int late_wait, unsigned int *status) {
    // late_wait: this launch is the remainder of a split problem, queued right after
    // the main launch, which waited for the producers of x and w before letting it
    // start; it waits for the main launch only before it ends, so that a later
    // kernel that waits on this one also sees the main launch's outputs
    if (!late_wait) pdl_wait();  // the activations may come from the previous kernel
    pdl_trigger();
    using C = Cfg<BN>;
    constexpr int NS = C::NS, RS = C::RS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *xs = base + C::x_off;
    uint8_t *raw = base + C::raw_off;
    const uint32_t bar = smem_u32(base + C::bar_off);
    // full: the dequant warps wrote the stage's operand and its activation copy
    // landed (tx bytes); empty: the MMAs reading the stage are done; rfull / rempty:
    // the raw tile ring; accfull: all MMAs of the tile are done
    const uint32_t full0 = bar, empty0 = bar + 8 * NS, rfull0 = empty0 + 8 * NS, rempty0 = rfull0 + 8 * RS,
                   accfull = rempty0 + 8 * RS;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(base + C::misc_off);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + C::misc_off + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * kTileRows;
    const int m0 = blockIdx.y * BN;
    // split K over a cluster of gridDim.z CTAs: this CTA takes blocks [kbeg, kbeg + KBs)
    const int S = gridDim.z, split = blockIdx.z;
    const int kbeg = (int)((int64_t)KB * split / S);
    const int KBs = (int)((int64_t)KB * (split + 1) / S) - kbeg;
    const int total = KBs * 4;  // 64-wide stages

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full0 + 8 * s, kDqWarps + 1);  // the dequant warps and the activation producer
            mbar_init(empty0 + 8 * s, 1);            // tcgen05.commit
        }
        for (int r = 0; r < RS; ++r) {
            mbar_init(rfull0 + 8 * r, 1);
            mbar_init(rempty0 + 8 * r, kDqWarps);
        }
        mbar_init(accfull, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    // columns [0, BN): the accumulator; then NS operand stages of kStageCols
    const uint32_t a_col0 = (uint32_t)BN;

    if (warp == 0) {
        // ------------------------------------------------------- TMA: raw Q4_K
        if (lane == 0) {
            prefetch_tmap(&tmW);
            int issued = 0;
            for (int kb = 0; kb < KBs && !*abort_flag; ++kb) {
                const int r = kb % RS;
                if (kb >= RS && !mbar_wait(rempty0 + 8 * r, ((kb / RS) - 1) & 1, status)) {
                    *abort_flag = 1;
                    break;
                }
                mbar_arrive_expect_tx(rfull0 + 8 * r, kRawBytes);
                tma_load_2d(smem_u32(raw + r * kRawBytes), &tmW, (kbeg + kb) * (kBlockBytes / 4), n0, rfull0 + 8 * r);
                ++issued;
            }
            // no copy may still be landing when the CTA leaves (bounded waits; on the
            // normal path the dequant warps have consumed every block already)
            for (int j = issued > RS ? issued - RS : 0; j < issued; ++j)
                (void)mbar_wait(rfull0 + 8 * (j % RS), (j / RS) & 1, status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA
        if (lane == 0) {
            const uint32_t idesc = umma_idesc_bf16_f32(kTileRows, BN);
            for (int i = 0; i < total; ++i) {
                const int s = i % NS;
                if (!mbar_wait(full0 + 8 * s, (i / NS) & 1, status)) {
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
                const uint64_t bd = umma_desc_sw128(smem_u32(xs + s * C::XB));
                const uint32_t at = tmem + a_col0 + (uint32_t)(kStageCols * s);
#pragma unroll
                for (int kk = 0; kk < kStageK / 16; ++kk)  // A: +8 columns, B: +32 bytes per 16-wide step
                    umma_bf16_ts(tmem, at + 8 * kk, bd + 2 * kk, idesc, (i | kk) != 0);
                umma_commit(empty0 + 8 * s);
            }
            // completes once every MMA issued above has (also after an abort, so
            // that tensor memory is freed only after the MMAs that write it)
            umma_commit(accfull);
        }
    } else if (warp >= kDqWarp0) {
        // ---------------------------------------------------- dequant warps
        const int t = threadIdx.x - 32 * kDqWarp0;
        const int row = t & (kTileRows - 1);  // weight row within the tile = tensor-memory lane
        const int h = t >> 7;                 // which kEPT code bytes of each group: elements kEPT h ..
        const uint32_t arow0 = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + a_col0;
        bool ok = true;
        for (int kb = 0; kb < KBs && ok; ++kb) {
            const int r = kb % RS;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(rfull0 + 8 * r, (kb / RS) & 1, status))) {
                ok = false;
                break;
            }
            // the block's header and this thread's code bytes, read once; the raw slot
            // is free for the next copy as soon as every dequant warp has them
            const uint8_t *rowp = raw + r * kRawBytes + row * kBlockBytes;
            const uint4 hd = *reinterpret_cast<const uint4 *>(rowp);
            uint32_t qv[4][kWPT];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const uint8_t *src = rowp + 16 + 32 * g + kEPT * h;
                if constexpr (kWPT == 4) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(src);
                    qv[g][0] = v.x, qv[g][1] = v.y, qv[g][2] = v.z, qv[g][3] = v.w;
                } else {
                    const uint2 v = *reinterpret_cast<const uint2 *>(src);
                    qv[g][0] = v.x, qv[g][1] = v.y;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(rempty0 + 8 * r);
            if constexpr (FP4) {
                // all four stages of the block first (registers), then the hand-offs.
                // Stage g4: weights 64*g4 .. +63 of the block, scales 4*g4 .. +3 (16
                // weights each); this thread takes weights 2 kEPT h .. +2 kEPT - 1 of the
                // stage (code word j: scale kEPT h / 8 + j / 2)
                uint32_t p[4][2 * kEPT / 2];  // stage columns kEPT h .. : two weights each
#pragma unroll
                for (int g4 = 0; g4 < 4; ++g4) {
                    const uint32_t scw = g4 == 0 ? hd.x : g4 == 1 ? hd.y : g4 == 2 ? hd.z : hd.w;
                    __nv_bfloat162 sv[kEPT / 8];
#pragma unroll
                    for (int q = 0; q < kEPT / 8; ++q) {
                        const float f = e4m3_to_f32(scw >> (8 * (kEPT * h / 8 + q)));
                        sv[q] = __floats2bfloat162_rn(f, f);  // exact: e4m3 values are bf16 values
                    }
#pragma unroll
                    for (int j = 0; j < kWPT; ++j) {
                        e2m1x8_to_bf16(qv[g4][j], p[g4][4 * j], p[g4][4 * j + 1], p[g4][4 * j + 2], p[g4][4 * j + 3]);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            p[g4][4 * j + q] = as_u32(__hmul2(as_bf2(p[g4][4 * j + q]), sv[j >> 1]));  // exact
                    }
                }
#pragma unroll
                for (int g4 = 0; g4 < 4; ++g4) {
                    const int i = kb * 4 + g4, s = i % NS;
                    if (i >= NS &&
                        !__all_sync(0xFFFFFFFFu, mbar_wait(empty0 + 8 * s, ((i / NS) - 1) & 1, status))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();  // after the wait for the MMAs that read this stage
                    tmem_st(arow0 + (uint32_t)(kStageCols * s + kEPT * h), p[g4]);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(full0 + 8 * s);
                }
                continue;
            }
            const float d = __half2float(__ushort_as_half((unsigned short)(hd.x & 0xFFFFu)));
            const float dmin = __half2float(__ushort_as_half((unsigned short)(hd.x >> 16)));
            const uint32_t sc_lo = hd.y & 0x3F3F3F3Fu, m_lo = hd.z & 0x3F3F3F3Fu;
            const uint32_t sc_hi = (hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u);
            const uint32_t m_hi = ((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u);
            // all four stages of the block are converted first, in registers (they need
            // only the codes), and handed to the MMA one by one as its stages free up:
            // the conversions of the block overlap each other and those waits.
            // Stage g: elements kEPT h .. of sub-block 2g (stage columns kEPT h / 2 ..)
            // and of 2g+1 (16 + kEPT h / 2 ..)
            uint32_t lo[4][2 * kWPT], hi[4][2 * kWPT];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                // scales of sub-blocks 2g (low nibbles) and 2g+1 (high nibbles)
                const uint32_t scw = g < 2 ? sc_lo : sc_hi, mw = g < 2 ? m_lo : m_hi;
                const int b0 = (2 * g) & 3, b1 = (2 * g + 1) & 3;
                const float dsc0 = d * (float)((scw >> (8 * b0)) & 0xFFu), dm0 = dmin * (float)((mw >> (8 * b0)) & 0xFFu);
                const float dsc1 = d * (float)((scw >> (8 * b1)) & 0xFFu), dm1 = dmin * (float)((mw >> (8 * b1)) & 0xFFu);
                const GroupScales gs = group_scales(dsc0, dm0, dsc1, dm1);
#pragma unroll
                for (int j = 0; j < kWPT; ++j)
                    q4k_word_to_bf16(qv[g][j], gs, lo[g][2 * j], lo[g][2 * j + 1], hi[g][2 * j], hi[g][2 * j + 1]);
            }
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const int i = kb * 4 + g, s = i % NS;
                if (i >= NS && !__all_sync(0xFFFFFFFFu, mbar_wait(empty0 + 8 * s, ((i / NS) - 1) & 1, status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();  // after the wait for the MMAs that read this stage
                const uint32_t at = arow0 + (uint32_t)(kStageCols * s + kEPT / 2 * h);
                tmem_st(at, lo[g]);
                tmem_st(at + 16, hi[g]);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(full0 + 8 * s);
            }
        }
        if (!ok && lane == 0) *abort_flag = 1;
        // ------------------------------------------------------- epilogue
        if (ok && __all_sync(0xFFFFFFFFu, mbar_wait(accfull, 0, status)) && !*abort_flag) {
            tc_fence_after();
            const int q = warp & 3;  // tensor-memory lane quarter this warp may read
            const int rl = 32 * q + lane, n = n0 + rl;
            constexpr int kCC = BN / 32 / kTPR;           // 32-column chunks per warp
            const int share = (warp - kDqWarp0) >> 2;     // which share of the columns this warp takes
            // with a K split, the partial tile goes to this CTA's (now idle) stage
            // buffers, column-major [BN][128], for the cluster reduction below
            float *part = reinterpret_cast<float *>(base);
#pragma unroll 1
            for (int cc = share * kCC; cc < (share + 1) * kCC; ++cc) {
                uint32_t v[32];
                tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + 32 * cc, v);
                tmem_ld_wait();
                if (S > 1) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) part[(32 * cc + j) * kTileRows + rl] = __uint_as_float(v[j]);
                } else if (n < N) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int m = m0 + 32 * cc + j;
                        if (m < M) y[(int64_t)m * ldy + n] = FP4 ? gscale * __uint_as_float(v[j]) : __uint_as_float(v[j]);
                    }
                }
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------ TMA: activations
        if (lane == 0) {
            prefetch_tmap(&tmX);
            int issued = 0;
            for (int i = 0; i < total && !*abort_flag; ++i) {
                const int kb = i >> 2, g = i & 3, s = i % NS;
                if (i >= NS && !mbar_wait(empty0 + 8 * s, ((i / NS) - 1) & 1, status)) {
                    *abort_flag = 1;
                    break;
                }
                mbar_arrive_expect_tx(full0 + 8 * s, C::XB);
                tma_load_2d(smem_u32(xs + s * C::XB), &tmX, (kbeg + kb) * kQK + kStageK * g, m0, full0 + 8 * s);
                ++issued;
            }
            // (on the normal path the MMAs have consumed every stage already; after an
            // abort these bounded waits may run out, the copies having landed or not)
            for (int j = issued > NS ? issued - NS : 0; j < issued; ++j)
                (void)mbar_wait(full0 + 8 * (j % NS), (j / NS) & 1, status);
        }
    }
    if (S > 1) {
        // every rank's partial is in its shared memory; rank r sums the columns
        // [r*BN/S, (r+1)*BN/S) over the ranks in rank order and stores them
        cluster_sync();
        if (!*abort_flag) {
            const int r = (int)cluster_ctarank();
            const int c0 = BN * r / S, c1 = BN * (r + 1) / S;
            const uint32_t pbase = smem_u32(base);
            for (int e = threadIdx.x; e < (c1 - c0) * kTileRows; e += kThreads) {
                const int c = c0 + e / kTileRows, rr = e % kTileRows;
                const uint32_t off = pbase + 4u * (uint32_t)(c * kTileRows + rr);
                float v = 0.0f;
                for (int qr = 0; qr < S; ++qr) v += ld_shared_cluster_f32(map_shared_rank(off, qr));
                const int m = m0 + c, n = n0 + rr;
                if (m < M && n < N) y[(int64_t)m * ldy + n] = FP4 ? gscale * v : v;
            }
        }
        cluster_sync();  // keep every partial alive until all ranks have read it
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        // every MMA has completed (immediate on the normal path; after an abort,
        // a bounded wait for the MMAs still running) before the columns are freed
        (void)mbar_wait(accfull, 0, status);
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (late_wait) pdl_wait();
}

// The cluster K split of an N x K problem with `tiles` output tiles: when the
// tiles leave more than half of the SMs idle (one CTA per SM), split K over up to
// 8 CTAs, at least four K blocks each.
int k_split(const DeviceInfo &di, int64_t tiles, int KB) {
    int S = 1;
    if (2 * tiles <= di.sm_count) {
        int64_t want = di.sm_count / tiles;
        if (want > 8) want = 8;
        if (want > KB / 4) want = KB / 4;
        if (want > 1) S = (int)want;
    }
    return S;
}

// S: the cluster K split (1: none).
template <int BN, bool FP4>
cudaError_t launch_bn(const DeviceInfo &di, const void *w, int64_t N, int64_t K, const uint16_t *x, int64_t M,
                      int64_t ldx, float *y, int64_t ldy, float g, cudaStream_t s, int S, int late_wait = 0) {
    CUtensorMap tmW, tmX;
    cudaError_t e = make_weight_tmap(&tmW, w, N, K, kTileRows, kBlockBytes / 4);
    if (e != cudaSuccess) return e;
    e = make_act_tmap_sw128(&tmX, x, M, K, ldx, BN);
    if (e != cudaSuccess) return e;
    using C = Cfg<BN>;
    const int smem = C::bytes;
    static_assert(C::raw_off >= BN * kTileRows * 4, "the partial tile fits in the activation stages");
    static_assert(BN + C::NS * kStageCols <= (int)kTmemCols, "the accumulator and the operand stages fit");
    e = ensure_smem((const void *)gemm_tc_kernel<BN, FP4>, smem);
    if (e != cudaSuccess) return e;
    const int KB = (int)(K / kQK);
    const dim3 grid((unsigned)((N + kTileRows - 1) / kTileRows), (unsigned)((M + BN - 1) / BN), (unsigned)S);
    return launch_pdl(gemm_tc_kernel<BN, FP4>, grid, dim3(kThreads), (size_t)smem, s, dim3(1, 1, (unsigned)S), tmW,
                      tmX, y, ldy, (int)M, (int)N, KB, g, late_wait, di.status);
}

// One CTA per SM: when the tiles' last wave would run mostly empty and a row of
// token tiles is narrow enough for the cluster K split, the last token tiles
// become a second launch that splits K and fills the idle SMs.  Returns the
// number of tokens of the main launch (M when nothing is split off).
int64_t main_part(const DeviceInfo &di, int64_t N, int64_t M) {
    const int64_t tn = (N + kTileRows - 1) / kTileRows, tm = (M + 255) / 256;
    const int64_t total = tn * tm, full = total / di.sm_count * di.sm_count, rem = total - full;
    if (M <= 256 || full == 0 || rem == 0 || 2 * rem > di.sm_count) return M;
    const int64_t r = (rem + tn - 1) / tn;  // token tiles to peel off
    if (r >= tm || 2 * r * tn > di.sm_count) return M;  // the remainder must leave room for a K split
    return (tm - r) * 256;
}

// Default: the K split follows the tile count (so it depends on M), and a mostly
// empty last wave becomes a second, K-split launch.  Batch-invariant: the K split
// is the one the weight rows alone would get (one token tile), for every M, and
// nothing is split off; each output element is then summed over the same K
// ranges in the same order whatever M is.
template <bool FP4>
cudaError_t launch_split(const DeviceInfo &di, const void *w, int64_t N, int64_t K, const uint16_t *x, int64_t M,
                         int64_t ldx, float *y, int64_t ldy, float g, bool invariant, cudaStream_t s) {
    const int KB = (int)(K / kQK);
    const int64_t tn = (N + kTileRows - 1) / kTileRows;
    if (invariant) {
        // at most 2 ways over a cluster pair, at every M (3 ways measured slower
        // at large M)
        const int S = k_split(di, tn, KB) > 1 ? 2 : 1;
        if (M <= 128) return launch_bn<128, FP4>(di, w, N, K, x, M, ldx, y, ldy, g, s, S);
        return launch_bn<256, FP4>(di, w, N, K, x, M, ldx, y, ldy, g, s, S);
    }
    if (M <= 128) return launch_bn<128, FP4>(di, w, N, K, x, M, ldx, y, ldy, g, s, k_split(di, tn, KB));
    const int64_t m1 = main_part(di, N, M);
    cudaError_t e = launch_bn<256, FP4>(di, w, N, K, x, m1, ldx, y, ldy, g, s, k_split(di, tn * ((m1 + 255) / 256), KB));
    if (e != cudaSuccess || m1 == M) return e;
    const int64_t m2 = M - m1;
    const uint16_t *x2 = x + m1 * ldx;
    float *y2 = y + m1 * ldy;
    return m2 <= 128 ? launch_bn<128, FP4>(di, w, N, K, x2, m2, ldx, y2, ldy, g, s, k_split(di, tn, KB), 1)
                     : launch_bn<256, FP4>(di, w, N, K, x2, m2, ldx, y2, ldy, g, s,
                                           k_split(di, tn * ((m2 + 255) / 256), KB), 1);
}

}  // namespace

cudaError_t launch_gemm_tc(const DeviceInfo &di, const void *w, int64_t N, int64_t K, const uint16_t *x, int64_t M,
                           int64_t ldx, float *y, int64_t ldy, bool invariant, cudaStream_t s) {
    return launch_split<false>(di, w, N, K, x, M, ldx, y, ldy, 1.0f, invariant, s);
}

cudaError_t launch_gemm_tc_nvfp4(const DeviceInfo &di, const void *w, float g, int64_t N, int64_t K,
                                 const uint16_t *x, int64_t M, int64_t ldx, float *y, int64_t ldy, bool invariant,
                                 cudaStream_t s) {
    return launch_split<true>(di, w, N, K, x, M, ldx, y, ldy, g, invariant, s);
}

}  // namespace q4k
