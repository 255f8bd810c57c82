// Persistent MoE expert Q4_K GEMM on the tcgen05 tensor cores.
//
// Same arithmetic as gemm_tc.cu (per-tile dequantization of Q4_K into a bf16
// operand in shared memory, tcgen05.mma into an fp32 tensor-memory accumulator;
// sparkinfer-server README, "Serve a GGUF instead of NVFP4"), organized so that
// one CTA per SM streams tile after tile without draining its pipeline:
//
//   * warp 0    TMA: per 256-wide K block the raw Q4_K tile of 128 weight rows
//               (two slots, issued one block ahead, across tile boundaries), per
//               64-wide stage the token tile's activation rows (128-byte swizzle;
//               one or two 96-row boxes, as the tile's count needs);
//   * warp 1    MMA: one thread issues 4 x tcgen05.mma (128 x N x 16) per stage,
//               A from tensor memory, B from shared memory, into one of two
//               192-column accumulators in tensor memory;
//   * warps 2-9 dequant: two threads per weight row.  Each reads the 64 code
//               bytes it converts once per block (16 of each group: elements
//               16h .. 16h+15 of both sub-blocks 2g and 2g+1) and writes the bf16
//               operand of each stage into tensor memory (tcgen05.st: the row's
//               lane, two weights per column, four stages after the
//               accumulators), off the shared-memory bandwidth that the
//               activation copies and the tensor core's B reads use;
//   * warps 10-13 epilogue: tcgen05.ld of the finished accumulator and fp32
//               stores, while the MMA warp already fills the other accumulator.
// Tiles are (128-row weight tile, token tile of the routing's list) pairs taken
// round-robin (tile = CTA + k * grid).  A token tile is (expert, first item,
// count <= 192) of the expert-sorted activation rows; the MMA width is the count
// rounded up to 16, and output column j goes to the row of item perm[first + j].
// Every wait is bounded; the sum per output element runs in a fixed order, so
// results are run-to-run deterministic.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "q4k_internal.h"
#include "q4k_ptx.cuh"

namespace q4k {
namespace {

constexpr int kTileRows = 128;                      // weight rows per tile (MMA M)
constexpr int kBN = kMoeTileItems;                  // tokens per tile (MMA N at most): 192
constexpr int kStageK = 64;                         // K per stage: one 128-byte swizzle row of bf16
constexpr int kNS = 4;                              // stages
constexpr int kXB = kBN * kStageK * 2;              // 24 KiB activations per stage
constexpr int kXBox = kBN / 2;                      // activation rows per TMA box
constexpr int kXBoxBytes = kXBox * kStageK * 2;     // 12 KiB: rows kXBox.. land right after, as one 192-row box would
constexpr int kStageCols = kStageK / 2;             // tensor-memory columns of one stage's operand (bf16 pairs)
constexpr int kRawBytes = kTileRows * kBlockBytes;  // 18 KiB raw Q4_K per block
constexpr int kDqWarps = 8, kEpWarps = 4;
constexpr int kThreads = (2 + kDqWarps + kEpWarps) * 32;
constexpr int kX = 0, kRaw = kNS * kXB, kBar = kRaw + 2 * kRawBytes;
constexpr int kNBars = 2 * kNS + 2 + 2 + 2 + 2 + 1;
constexpr int kMisc = kBar + kNBars * 8;
constexpr int kOrow = kMisc + 16;                   // [2][kBN] output rows (MoE)
constexpr int kSmem = kOrow + 2 * kBN * 4 + 1024;   // + slack to align the base to 1024
constexpr uint32_t kAcol0 = 2 * kBN;                // the operand stages follow the two accumulators
constexpr uint32_t kTmemCols = 512;
static_assert(kAcol0 + kNS * kStageCols <= kTmemCols, "accumulators and operand stages fit in tensor memory");
static_assert(kBN % 16 == 0 && kXBoxBytes % 1024 == 0, "MMA width and 1024-byte swizzle atoms");

struct Tile {
    int n0, m0, cnt, wrow0;
};

struct Params {
    float *y;
    int64_t ldy;
    int N, KB;
    int tiles_n;           // 128-row weight tiles per expert
    const int32_t *perm;   // routing permutation
    const int4 *tiles;     // MoE: (expert, first item, count, -)
    const int *n_tiles;    // number of token tiles; then the routing's (E, items, stamp)
    int E, n_items;        // this call's shape, checked against the routing's
    unsigned int *status;
    GluOut glu;            // SwiGLU epilogue (up projection of an expert FFN)
};

__device__ __forceinline__ Tile tile_of(const Params &p, int k) {
    const int tile = blockIdx.x + k * gridDim.x;
    const int nt = tile % p.tiles_n, mt = tile / p.tiles_n;
    const int4 tl = __ldg(p.tiles + mt);
    Tile t;
    t.n0 = nt * kTileRows;
    t.m0 = tl.y;
    t.cnt = tl.z;
    t.wrow0 = tl.x * p.N + t.n0;
    return t;
}

__global__ void __launch_bounds__(kThreads, 1) gemm_tcp_kernel(const __grid_constant__ CUtensorMap tmW,
                                                               const __grid_constant__ CUtensorMap tmX, Params p) {
    pdl_wait();  // the tile list and the sorted activations come from the routing and gather kernels
    pdl_trigger();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *xs = base + kX;
    uint8_t *raw = base + kRaw;
    const uint32_t bar = smem_u32(base + kBar);
    // full: the dequant warps wrote the stage's operand and its activation copy
    // landed (one barrier, so that the MMA thread waits once per stage); empty: its
    // MMAs are done; rfull / rempty: raw Q4_K ring; accfull / accempty: the two
    // tensor-memory accumulators; mmadone: every MMA issued
    const uint32_t full0 = bar, empty0 = bar + 8 * kNS, rfull0 = bar + 16 * kNS,
                   rempty0 = rfull0 + 16, accfull0 = rempty0 + 16, accempty0 = accfull0 + 16,
                   mmadone = accempty0 + 16;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(base + kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + kMisc + 4);
    int *orow = reinterpret_cast<int *>(base + kOrow);
    unsigned int *status = p.status;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // a routing made for another shape: leave before any barrier or allocation
    if (!routing_matches(p.n_tiles, p.E, p.n_items, status)) return;
    const int tiles_m = __ldg(p.n_tiles);
    const int total_tiles = p.tiles_n * tiles_m;
    const int my_tiles =
        (int)blockIdx.x < total_tiles ? (total_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
    if (my_tiles == 0) return;  // no work: leave before any barrier or allocation
    const int KB = p.KB;
    const int nblocks = my_tiles * KB;  // raw blocks this CTA streams, in order

    if (threadIdx.x == 0) {
        for (int s = 0; s < kNS; ++s) {
            mbar_init(full0 + 8 * s, kDqWarps + 1);  // the dequant warps and the activation producer (+ tx bytes)
            mbar_init(empty0 + 8 * s, 1);        // tcgen05.commit
        }
        for (int r = 0; r < 2; ++r) {
            mbar_init(rfull0 + 8 * r, 1);
            mbar_init(rempty0 + 8 * r, kDqWarps);
            mbar_init(accfull0 + 8 * r, 1);          // tcgen05.commit
            mbar_init(accempty0 + 8 * r, kEpWarps);  // epilogue warps
        }
        mbar_init(mmadone, 1);  // tcgen05.commit after the last MMA
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

    if (warp == 0) {
        // ------------------------------------------------------------- TMA
        if (lane == 0) {
            prefetch_tmap(&tmW);
            prefetch_tmap(&tmX);
            // raw block b = k * KB + kb (tile k of this CTA, block kb)
            int raw_issued = 0, x_issued = 0;
            auto issue_raw = [&](int b) -> bool {
                const Tile t = tile_of(p, b / KB);
                const int r = b & 1;
                if (b >= 2 && !mbar_wait(rempty0 + 8 * r, ((b >> 1) - 1) & 1, status)) return false;
                mbar_arrive_expect_tx(rfull0 + 8 * r, kRawBytes);
                tma_load_2d(smem_u32(raw + r * kRawBytes), &tmW, (b % KB) * (kBlockBytes / 4), t.wrow0,
                            rfull0 + 8 * r);
                ++raw_issued;
                return true;
            };
            bool ok = issue_raw(0);
            Tile t = tile_of(p, 0);
            for (int b = 0; b < nblocks && ok; ++b) {
                const int kb = b % KB;
                if (kb == 0 && b > 0) t = tile_of(p, b / KB);
                if (b + 1 < nblocks && !issue_raw(b + 1)) {
                    ok = false;
                    break;
                }
                for (int g = 0; g < 4; ++g) {
                    const int i = b * 4 + g, s = i % kNS;
                    if (i >= kNS && !mbar_wait(empty0 + 8 * s, ((i / kNS) - 1) & 1, status)) {
                        ok = false;
                        break;
                    }
                    if (*abort_flag) {
                        ok = false;
                        break;
                    }
                    // one kXBox-row box for a tile of at most kXBox tokens, two otherwise:
                    // the MMA reads only the tile's rows
                    const int nbox = t.cnt > kXBox ? 2 : 1;
                    mbar_arrive_expect_tx(full0 + 8 * s, nbox * kXBoxBytes);
                    for (int q = 0; q < nbox; ++q)
                        tma_load_2d(smem_u32(xs + s * kXB + q * kXBoxBytes), &tmX, kb * kQK + kStageK * g,
                                    t.m0 + q * kXBox, full0 + 8 * s);
                    ++x_issued;
                }
            }
            if (!ok) *abort_flag = 1;
            if (*abort_flag) {
                // a wait gave up somewhere: wait (bounded) for this CTA's copies still in flight
                for (int j = raw_issued > 2 ? raw_issued - 2 : 0; j < raw_issued; ++j)
                    (void)mbar_wait(rfull0 + 8 * (j & 1), (j >> 1) & 1, status);
                for (int j = x_issued > kNS ? x_issued - kNS : 0; j < x_issued; ++j)
                    (void)mbar_wait(full0 + 8 * (j % kNS), (j / kNS) & 1, status);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA
        if (lane == 0) {
            bool ok = true;
            Tile tn = tile_of(p, 0);  // the next tile's record, loaded a tile ahead
            for (int k = 0; k < my_tiles && ok; ++k) {
                const Tile t = tn;
                if (k + 1 < my_tiles) tn = tile_of(p, k + 1);
                const int mma_n = (t.cnt + 15) & ~15;
                const uint32_t idesc = umma_idesc_bf16_f32(kTileRows, mma_n);
                const int buf = k & 1;
                // another role that gave up is seen here, once per tile (a stage whose
                // producers gave up never completes, and its wait is bounded)
                if ((k >= 2 && !mbar_wait(accempty0 + 8 * buf, ((k >> 1) - 1) & 1, status)) || *abort_flag) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(buf * kBN);
                for (int j = 0; j < KB * 4; ++j) {
                    const int i = k * KB * 4 + j, s = i % kNS;
                    if (!mbar_wait(full0 + 8 * s, (i / kNS) & 1, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t at = tmem + kAcol0 + (uint32_t)(kStageCols * s);
                    const uint64_t bd = umma_desc_sw128(smem_u32(xs + s * kXB));
#pragma unroll
                    for (int kk = 0; kk < kStageK / 16; ++kk)  // A: +8 columns, B: +32 bytes per 16-wide step
                        umma_bf16_ts(d, at + 8 * kk, bd + 2 * kk, idesc, (j | kk) != 0);
                    umma_commit(empty0 + 8 * s);
                }
                if (ok) umma_commit(accfull0 + 8 * buf);
            }
            if (!ok) *abort_flag = 1;
            umma_commit(mmadone);  // completes once every MMA issued above has
        }
    } else if (warp < 2 + kDqWarps) {
        // ---------------------------------------------------- dequant warps
        // warp w may reach tensor-memory lanes 32 (w % 4) .. +31: its rows are those lanes
        const int row = ((warp & 3) << 5) | lane;  // weight row within the tile
        const int h = (warp - 2) >> 2;              // which 16 code bytes of each group: elements 16h..16h+15
        const uint32_t arow0 = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + kAcol0;
        bool ok = true;
        for (int b = 0; b < nblocks && ok; ++b) {
            const int r = b & 1;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(rfull0 + 8 * r, (b >> 1) & 1, status))) {
                ok = false;
                break;
            }
            // the block's header and this thread's 64 code bytes, read once; the raw
            // slot is free for the next copy as soon as every dequant warp has them
            const uint8_t *rowp = raw + r * kRawBytes + row * kBlockBytes;
            const uint4 hd = *reinterpret_cast<const uint4 *>(rowp);
            uint4 qv[4];
#pragma unroll
            for (int g = 0; g < 4; ++g) qv[g] = *reinterpret_cast<const uint4 *>(rowp + 16 + 32 * g + 16 * h);
            __syncwarp();
            if (lane == 0) mbar_arrive(rempty0 + 8 * r);
            const float d = __half2float(__ushort_as_half((unsigned short)(hd.x & 0xFFFFu)));
            const float dmin = __half2float(__ushort_as_half((unsigned short)(hd.x >> 16)));
            const uint32_t sc_lo = hd.y & 0x3F3F3F3Fu, m_lo = hd.z & 0x3F3F3F3Fu;
            const uint32_t sc_hi = (hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u);
            const uint32_t m_hi = ((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u);
            for (int g = 0; g < 4; ++g) {
                const int i = b * 4 + g, s = i % kNS;
                if (i >= kNS &&
                    !__all_sync(0xFFFFFFFFu, mbar_wait(empty0 + 8 * s, ((i / kNS) - 1) & 1, status))) {
                    ok = false;
                    break;
                }
                // scales of sub-blocks 2g (low nibbles) and 2g+1 (high nibbles)
                const uint32_t scw = g < 2 ? sc_lo : sc_hi, mw = g < 2 ? m_lo : m_hi;
                const int b0 = (2 * g) & 3, b1 = (2 * g + 1) & 3;
                const float dsc0 = d * (float)((scw >> (8 * b0)) & 0xFFu), dm0 = dmin * (float)((mw >> (8 * b0)) & 0xFFu);
                const float dsc1 = d * (float)((scw >> (8 * b1)) & 0xFFu), dm1 = dmin * (float)((mw >> (8 * b1)) & 0xFFu);
                const GroupScales gs = group_scales(dsc0, dm0, dsc1, dm1);
                // elements 16h .. 16h+15 of sub-block 2g (stage columns 8h ..) and of 2g+1 (16 + 8h ..)
                uint32_t lo[8], hi[8];
                q4k_word_to_bf16(qv[g].x, gs, lo[0], lo[1], hi[0], hi[1]);
                q4k_word_to_bf16(qv[g].y, gs, lo[2], lo[3], hi[2], hi[3]);
                q4k_word_to_bf16(qv[g].z, gs, lo[4], lo[5], hi[4], hi[5]);
                q4k_word_to_bf16(qv[g].w, gs, lo[6], lo[7], hi[6], hi[7]);
                tc_fence_after();  // after the wait for the MMAs that read this stage
                const uint32_t at = arow0 + (uint32_t)(kStageCols * s + 8 * h);
                tmem_st8(at, lo);
                tmem_st8(at + 16, hi);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(full0 + 8 * s);
            }
            if (*abort_flag) ok = false;
        }
        if (!ok && lane == 0) *abort_flag = 1;
    } else {
        // ------------------------------------------------------- epilogue
        const int q = warp & 3;  // tensor-memory lane quarter this warp may read
        const int et = threadIdx.x - (2 + kDqWarps) * 32;
        for (int k = 0; k < my_tiles; ++k) {
            const Tile t = tile_of(p, k);
            const int buf = k & 1;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(accfull0 + 8 * buf, (k >> 1) & 1, status))) {
                if (lane == 0) *abort_flag = 1;
                break;
            }
            tc_fence_after();
            int *orw = orow + buf * kBN;
            for (int j = et; j < t.cnt; j += kEpWarps * 32) orw[j] = __ldg(p.perm + t.m0 + j);
            asm volatile("bar.sync 2, %0;" ::"n"(kEpWarps * 32) : "memory");
            const int n = t.n0 + 32 * q + lane;
            if (!p.glu.h) {
#pragma unroll 1
                for (int cc = 0; cc < (t.cnt + 31) / 32; ++cc) {
                    uint32_t v[32];
                    tmem_ld32(tmem + (uint32_t)(buf * kBN) + ((uint32_t)(32 * q) << 16) + 32 * cc, v);
                    tmem_ld_wait();
                    if (n < p.N) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int col = 32 * cc + j;
                            if (col < t.cnt) p.y[(int64_t)orw[col] * p.ldy + n] = __uint_as_float(v[j]);
                        }
                    }
                }
            } else {
                // SwiGLU epilogue: the 32 gate values of column group cc + 1 are
                // loaded while group cc is converted and stored
                const int nch = (t.cnt + 31) / 32;
                float gv[32];
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    gv[j] = n < p.N && j < t.cnt ? __ldg(p.glu.g + (int64_t)orw[j] * p.ldy + n) : 0.0f;
#pragma unroll 1
                for (int cc = 0; cc < nch; ++cc) {
                    float gn[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int col = 32 * (cc + 1) + j;
                        gn[j] = n < p.N && col < t.cnt ? __ldg(p.glu.g + (int64_t)orw[col] * p.ldy + n) : 0.0f;
                    }
                    uint32_t v[32];
                    tmem_ld32(tmem + (uint32_t)(buf * kBN) + ((uint32_t)(32 * q) << 16) + 32 * cc, v);
                    tmem_ld_wait();
                    if (n < p.N) {
                        if (p.glu.h_sorted) {
                            // rows t.m0 + col: consecutive, one pitch apart
                            uint16_t *hp = p.glu.h + (int64_t)(t.m0 + 32 * cc) * p.ldy + n;
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                if (32 * cc + j < t.cnt) *hp = swiglu_bf16(gv[j], __uint_as_float(v[j]));
                                hp += p.ldy;
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                const int col = 32 * cc + j;
                                if (col < t.cnt)
                                    p.glu.h[(int64_t)orw[col] * p.ldy + n] = swiglu_bf16(gv[j], __uint_as_float(v[j]));
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) gv[j] = gn[j];
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(accempty0 + 8 * buf);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        (void)mbar_wait(mmadone, 0, status);  // no MMA still writes the columns
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

cudaError_t launch(const CUtensorMap &tmW, const CUtensorMap &tmX, const Params &p, int grid, cudaStream_t s) {
    cudaError_t e = ensure_smem((const void *)gemm_tcp_kernel, kSmem);
    if (e != cudaSuccess) return e;
    return launch_pdl(gemm_tcp_kernel, dim3(grid), dim3(kThreads), kSmem, s, dim3(1), tmW, tmX, p);
}

}  // namespace

cudaError_t launch_moe_tcp(const DeviceInfo &di, const void *w_experts, int E, int64_t N, int64_t K,
                           const uint16_t *x_sorted, int64_t n_items, const int32_t *perm, const int4 *tiles,
                           const int *n_tiles, float *out, cudaStream_t s, const GluOut &glu) {
    CUtensorMap tmW, tmX;
    cudaError_t e = make_weight_tmap(&tmW, w_experts, (int64_t)E * N, K, kTileRows, kBlockBytes / 4);
    if (e != cudaSuccess) return e;
    e = make_act_tmap_sw128(&tmX, x_sorted, n_items, K, K, kXBox);
    if (e != cudaSuccess) return e;
    Params p = {};
    p.y = out;
    p.ldy = N;
    p.N = (int)N;
    p.KB = (int)(K / kQK);
    p.tiles_n = (int)((N + kTileRows - 1) / kTileRows);
    p.perm = perm;
    p.tiles = tiles;
    p.n_tiles = n_tiles;
    p.E = E;
    p.n_items = (int)n_items;
    p.status = di.status;
    p.glu = glu;
    return launch(tmW, tmX, p, di.sm_count, s);
}

}  // namespace q4k
