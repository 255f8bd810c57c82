// MoE routing permutation and the weighted combine.
//
// The pages' MoE models route each token to its top-k experts, and the routed
// down projection ends in a combine whose fp32 atomicAdd order is one of the two
// sources of run-to-run nondeterminism they report (sparkinfer-server README,
// "Determinism").  Here the (token, slot) items are grouped by expert with a
// stable counting sort, every item's output row is written by exactly one CTA,
// and the combine sums each token's slots in slot order: the result does not
// depend on scheduling.
#include <cuda_runtime.h>

#include "q4k_internal.h"
#include "q4k_ptx.cuh"

namespace q4k {
namespace {

constexpr int kRouteThreads = 1024;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kHistStride = kRouteWarps + 1;  // [E][33]: the warps' columns of one expert, padded
constexpr int kRouteUnroll = 8;               // id loads in flight per lane

// Expert of item i; E (a pseudo-expert after the last) for an id outside
// [0, E); -1 for i past `hi`.
__device__ __forceinline__ int route_expert(const int32_t *ids, int i, int hi, int E) {
    if (i >= hi) return -1;
    const int e = __ldg(ids + i);
    return e >= 0 && e < E ? e : E;
}

// One CTA.  Warp w owns the contiguous item range [n*w/32, n*(w+1)/32), so a
// stable order is: expert, then warp, then item within the warp.
//   1. each warp counts its items per expert (lanes with equal ids are grouped
//      with a match, and the group's first lane adds the group size to the
//      warp's private column: no atomics);
//   2. per expert, an exclusive scan over the 32 warp columns, then an
//      exclusive scan of the expert totals gives offsets[];
//   3. each warp walks its range again in item order: an item's position is
//      its expert's offset + its warp's base + the running count of that
//      expert in the warp + its rank among equal lanes of the same round.
// Items with an invalid id form a pseudo-expert E placed after the valid ones:
// with invalid_tail they fill perm[offsets[E] ..) in item order (the expert
// kernels zero their per-slot rows); otherwise that tail is -1.
// Two reads of the ids and four block barriers, independent of the item count.
__global__ void __launch_bounds__(kRouteThreads) route_kernel(const int32_t *__restrict__ ids, int n_items, int E,
                                                              int32_t *__restrict__ offsets,
                                                              int32_t *__restrict__ perm, int invalid_tail,
                                                              int4 *__restrict__ tiles, int *__restrict__ n_tiles) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ int route_smem[];
    int *base = route_smem;                    // [E + 1]: expert offsets (base[E]: the invalid items)
    int *hist = route_smem + E + 1;            // [E + 1][kHistStride]: per-warp counts, then running positions
    __shared__ int warp_tot[kRouteWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int lo = (int)((int64_t)n_items * warp / kRouteWarps);
    const int hi = (int)((int64_t)n_items * (warp + 1) / kRouteWarps);
    const unsigned lt_mask = (1u << lane) - 1u;

    for (int k = tid; k < (E + 1) * kHistStride; k += kRouteThreads) hist[k] = 0;
    __syncthreads();
    // 1. per-warp counts
    for (int i0 = lo; i0 < hi; i0 += 32 * kRouteUnroll) {
        int ev[kRouteUnroll];
#pragma unroll
        for (int u = 0; u < kRouteUnroll; ++u) ev[u] = route_expert(ids, i0 + 32 * u + lane, hi, E);
#pragma unroll
        for (int u = 0; u < kRouteUnroll; ++u) {
            const unsigned same = __match_any_sync(0xFFFFFFFFu, ev[u]);
            if (ev[u] >= 0 && (same & lt_mask) == 0) hist[ev[u] * kHistStride + warp] += __popc(same);
            __syncwarp();
        }
    }
    __syncthreads();
    // 2a. per expert: exclusive scan over the warp columns (one warp per expert, lane = column)
    for (int ex = warp; ex <= E; ex += kRouteWarps) {
        const int c = hist[ex * kHistStride + lane];
        int inc = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xFFFFFFFFu, inc, o);
            if (lane >= o) inc += t;
        }
        hist[ex * kHistStride + lane] = inc - c;
        if (lane == 31 && ex < E) base[ex] = inc;  // the expert's total, for now
    }
    __syncthreads();
    // 2b. exclusive scan of the expert totals (E <= 1024: one per thread)
    const int v = tid < E ? base[tid] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = warp_tot[lane];
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xFFFFFFFFu, wi, o);
            if (lane >= o) wi += t;
        }
        warp_tot[lane] = wi - w;  // exclusive over warps
    }
    __syncthreads();
    const int excl = incl - v + warp_tot[warp];
    if (tid < E) {
        base[tid] = excl;
        offsets[tid] = excl;
    }
    if (tid == E - 1) {
        base[E] = excl + v;
        offsets[E] = excl + v;
    }
    __syncthreads();
    const int n_valid = base[E];
    // 3. stable scatter: each warp walks its own range in item order
    for (int i0 = lo; i0 < hi; i0 += 32 * kRouteUnroll) {
        int ev[kRouteUnroll];
#pragma unroll
        for (int u = 0; u < kRouteUnroll; ++u) ev[u] = route_expert(ids, i0 + 32 * u + lane, hi, E);
#pragma unroll
        for (int u = 0; u < kRouteUnroll; ++u) {
            const int e = ev[u];
            const unsigned same = __match_any_sync(0xFFFFFFFFu, e);
            const bool place = e >= 0 && (e < E || invalid_tail);
            int *run = hist + (e >= 0 ? e : 0) * kHistStride + warp;
            if (place) perm[base[e] + *run + __popc(same & lt_mask)] = i0 + 32 * u + lane;
            __syncwarp();
            if (place && (same & lt_mask) == 0) *run += __popc(same);
            __syncwarp();
        }
    }
    if (tiles) {
        // token tiles of up to kMoeTileItems items per expert, listed in expert order
        const int cnt = tid < E ? base[tid + 1] - base[tid] : 0;
        const int nt = (cnt + kMoeTileItems - 1) / kMoeTileItems;
        int ti = nt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xFFFFFFFFu, ti, o);
            if (lane >= o) ti += t;
        }
        __shared__ int tile_tot[kRouteWarps];
        if (lane == 31) tile_tot[warp] = ti;
        __syncthreads();
        if (warp == 0) {
            const int w = tile_tot[lane];
            int wi = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xFFFFFFFFu, wi, o);
                if (lane >= o) wi += t;
            }
            tile_tot[lane] = wi - w;
            if (lane == 31) *n_tiles = wi;
        }
        __syncthreads();
        const int first = ti - nt + tile_tot[warp];
        for (int k = 0; k < nt; ++k)
            tiles[first + k] = make_int4(tid, base[tid] + k * kMoeTileItems, min(kMoeTileItems, cnt - k * kMoeTileItems), 0);
    }
    if (!invalid_tail)
        for (int k = n_valid + tid; k < n_items; k += kRouteThreads) perm[k] = -1;
}

// y[t][n] = sum_{j < topk} g[t][j] * out[(t*topk + j)][n], j in increasing order;
// items whose expert id is invalid contribute nothing.
__global__ void combine_kernel(const float *__restrict__ out, const float *__restrict__ gates,
                               const int32_t *__restrict__ ids, int E, int64_t T, int topk, int64_t N,
                               float *__restrict__ y) {
    pdl_wait();
    pdl_trigger();
    const int64_t n4 = N / 4;
    const int64_t total = T * n4;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < total; q += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = q / n4, c = (q % n4) * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < topk; ++j) {
            const int e = __ldg(ids + t * topk + j);
            if (e < 0 || e >= E) continue;
            const float g = __ldg(gates + t * topk + j);
            const float4 o = __ldg(reinterpret_cast<const float4 *>(out + (t * topk + j) * N + c));
            acc.x = fmaf(g, o.x, acc.x);
            acc.y = fmaf(g, o.y, acc.y);
            acc.z = fmaf(g, o.z, acc.z);
            acc.w = fmaf(g, o.w, acc.w);
        }
        *reinterpret_cast<float4 *>(y + t * N + c) = acc;
    }
}

// x_sorted[p] = activation row of item perm[p], one warp per row, 16-byte
// accesses.  Rows past the valid item count (offsets[E]) are left alone.  With
// zero_y, the per-slot output rows (N floats) of the items with an invalid id,
// listed in perm[offsets[E] .. n_items), are zeroed.
__global__ void gather_kernel(const uint16_t *__restrict__ x, int x_per_slot, int topk,
                              const int32_t *__restrict__ perm, const int32_t *__restrict__ offsets, int E,
                              int64_t K, uint16_t *__restrict__ x_sorted, float *__restrict__ zero_y, int64_t N,
                              int n_items) {
    pdl_wait();
    pdl_trigger();
    const int n_valid = __ldg(offsets + E);
    const int lane = threadIdx.x & 31;
    const int64_t chunks = K / 8;  // 16-byte chunks per row
    const int64_t w0 = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5), nw = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t p = w0; p < n_valid; p += nw) {
        const int item = __ldg(perm + p);
        const int64_t src = x_per_slot ? item : item / topk;
        const uint4 *s = reinterpret_cast<const uint4 *>(x + src * K);
        uint4 *d = reinterpret_cast<uint4 *>(x_sorted + p * K);
        for (int64_t c = lane; c < chunks; c += 32) d[c] = __ldg(s + c);
    }
    if (zero_y)
        for (int64_t p = n_valid + w0; p < n_items; p += nw) {
            float *row = zero_y + (int64_t)__ldg(perm + p) * N;
            for (int64_t c = lane; c < N; c += 32) row[c] = 0.0f;
        }
}

}  // namespace

cudaError_t launch_moe_gather(const DeviceInfo &di, const uint16_t *x, int x_per_slot, int topk, const int32_t *perm,
                              const int32_t *offsets, int E, int64_t n_items, int64_t K, uint16_t *x_sorted,
                              float *zero_y, int64_t N, cudaStream_t s) {
    int64_t blocks = (n_items + 7) / 8;
    const int64_t cap = (int64_t)di.sm_count * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(gather_kernel, dim3((unsigned)blocks), dim3(256), 0, s, dim3(1), x, x_per_slot, topk, perm, offsets,
                      E, K, x_sorted, zero_y, N, (int)n_items);
}

size_t route_smem_bytes(int E) { return (size_t)(E + 1) * 4 + (size_t)kHistStride * (E + 1) * 4; }

cudaError_t launch_moe_route(const int32_t *ids, int64_t n_items, int E, int32_t *offsets, int32_t *perm,
                             bool invalid_tail, int4 *tiles, int *n_tiles, cudaStream_t s) {
    const size_t smem = route_smem_bytes(E);
    cudaError_t e = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(route_kernel, dim3(1), dim3(kRouteThreads), smem, s, dim3(1), ids, (int)n_items, E, offsets, perm,
                      invalid_tail ? 1 : 0, tiles, n_tiles);
}

cudaError_t launch_moe_combine(const DeviceInfo &di, const float *out, const float *gates, const int32_t *ids, int E,
                               int64_t T, int topk, int64_t N, float *y, cudaStream_t s) {
    const int64_t total = T * (N / 4);
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)di.sm_count * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(combine_kernel, dim3((unsigned)blocks), dim3(256), 0, s, dim3(1), out, gates, ids, E, T, topk, N, y);
}

}  // namespace q4k
