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

constexpr int kRouteThreads = 512;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kWhStride = kRouteWarps + 1;  // [E+1][17]: the warps' columns of one expert, padded
constexpr int kRouteMaxCtas = 128;

// Expert of item i; E (a pseudo-expert after the last) for an id outside
// [0, E); -1 for i past `hi`.
__device__ __forceinline__ int route_expert(const int32_t *ids, int i, int hi, int E) {
    if (i >= hi) return -1;
    const int e = __ldg(ids + i);
    return e >= 0 && e < E ? e : E;
}

// Exclusive prefix sums of a0, a1 (two consecutive values per thread, in thread
// order) over the CTA; *total receives the sum of all.  Every thread calls it.
__device__ __forceinline__ void block_scan2(int a0, int a1, int &x0, int &x1, int &total, int *scratch) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int v = a0 + a1;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += t;
    }
    if (lane == 31) scratch[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < kRouteWarps ? scratch[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xFFFFFFFFu, wi, o);
            if (lane >= o) wi += t;
        }
        if (lane < kRouteWarps) scratch[lane] = wi - w;
        if (lane == kRouteWarps - 1) scratch[kRouteWarps] = wi;
    }
    __syncthreads();
    x0 = inc - v + scratch[warp];
    x1 = x0 + a0;
    total = scratch[kRouteWarps];
    __syncthreads();  // scratch is reused by the next call
}

// Stable counting sort of the items by expert over many CTAs, with no
// cross-CTA communication.  CTA c owns the contiguous item range [c*R, (c+1)*R):
//   1. it counts every item per expert, and separately those before its range
//      (integer shared-memory atomics: the counts do not depend on order), which
//      gives the expert offsets and where its own items of each expert start;
//   2. its warps split the range into contiguous runs; each warp counts its run
//      per expert (lanes with equal ids grouped by a match, the group's first
//      lane adds the group size to the warp's private column: no atomics), an
//      exclusive scan over the warp columns gives each warp's start;
//   3. each warp walks its run again in item order: an item's position is its
//      expert's start in this CTA + its warp's start + the warp's running count
//      of that expert + its rank among equal lanes of the round.
// Items with an invalid id form a pseudo-expert E placed after the valid ones:
// with invalid_tail they fill perm[offsets[E] ..) in item order (the expert
// kernels zero their per-slot rows); otherwise that tail is -1.  CTA 0 writes
// offsets[] and the token-tile list.
__global__ void __launch_bounds__(kRouteThreads) route_kernel(const int32_t *__restrict__ ids, int n_items, int E,
                                                              int range, int32_t *__restrict__ offsets,
                                                              int32_t *__restrict__ perm, int invalid_tail,
                                                              int4 *__restrict__ tiles, int *__restrict__ n_tiles) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ int route_smem[];
    const int E1 = E + 1;
    int *total = route_smem;                     // [E+1] items per expert (E: invalid ids)
    int *start_e = route_smem + E1;              // [E+1] items before this range, then this range's first position
    int *wh = route_smem + 2 * E1;               // [E+1][kWhStride] per-warp counts, then running positions
    __shared__ int scratch[kRouteWarps + 1];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c0 = blockIdx.x * range, c1 = min(c0 + range, n_items);
    const int lo = c0 + (int)((int64_t)(c1 - c0) * warp / kRouteWarps);
    const int hi = c0 + (int)((int64_t)(c1 - c0) * (warp + 1) / kRouteWarps);
    const unsigned lt_mask = (1u << lane) - 1u;

    for (int k = tid; k < E1; k += kRouteThreads) total[k] = 0, start_e[k] = 0;
    for (int k = tid; k < E1 * kWhStride; k += kRouteThreads) wh[k] = 0;
    __syncthreads();
    // 1. counts of all items, and of the items before this range
    for (int i = tid; i < n_items; i += kRouteThreads) {
        const int e = route_expert(ids, i, n_items, E);
        atomicAdd(&total[e], 1);
        if (i < c0) atomicAdd(&start_e[e], 1);
    }
    // 2. per-warp counts of this range
    for (int i0 = lo; i0 < hi; i0 += 32) {
        const int e = route_expert(ids, i0 + lane, hi, E);
        const unsigned same = __match_any_sync(0xFFFFFFFFu, e);
        if (e >= 0 && (same & lt_mask) == 0) wh[e * kWhStride + warp] += __popc(same);
        __syncwarp();
    }
    __syncthreads();
    // expert offsets: exclusive scan of total[0..E) (two experts per thread)
    const int e0 = 2 * tid, e1 = 2 * tid + 1;
    int x0, x1, n_valid;
    block_scan2(e0 < E ? total[e0] : 0, e1 < E ? total[e1] : 0, x0, x1, n_valid, scratch);
    // this range's first position per expert (the pseudo-expert E follows the valid items)
    if (e0 < E) start_e[e0] += x0;
    if (e1 < E) start_e[e1] += x1;
    if (tid == 0) start_e[E] += n_valid;
    if (blockIdx.x == 0) {
        if (e0 < E) offsets[e0] = x0;
        if (e1 < E) offsets[e1] = x1;
        if (tid == 0) offsets[E] = n_valid;
    }
    // per expert: exclusive scan over the warp columns
    for (int ex = tid; ex < E1; ex += kRouteThreads) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < kRouteWarps; ++w) {
            const int t = wh[ex * kWhStride + w];
            wh[ex * kWhStride + w] = run;
            run += t;
        }
    }
    if (blockIdx.x == 0 && tiles) {
        // token tiles of up to kMoeTileItems items per expert, listed in expert order
        const int nt0 = e0 < E ? (total[e0] + kMoeTileItems - 1) / kMoeTileItems : 0;
        const int nt1 = e1 < E ? (total[e1] + kMoeTileItems - 1) / kMoeTileItems : 0;
        int f0, f1, nt;
        block_scan2(nt0, nt1, f0, f1, nt, scratch);
        for (int k = 0; k < nt0; ++k)
            tiles[f0 + k] = make_int4(e0, x0 + k * kMoeTileItems, min(kMoeTileItems, total[e0] - k * kMoeTileItems), 0);
        for (int k = 0; k < nt1; ++k)
            tiles[f1 + k] = make_int4(e1, x1 + k * kMoeTileItems, min(kMoeTileItems, total[e1] - k * kMoeTileItems), 0);
        if (tid == 0) {
            n_tiles[0] = nt;
            n_tiles[1] = E;  // the shape this routing was made for (checked on reuse)
            n_tiles[2] = n_items;
            n_tiles[3] = kRoutingStamp;
        }
    }
    __syncthreads();
    // 3. stable scatter: each warp walks its run in item order
    for (int i0 = lo; i0 < hi; i0 += 32) {
        const int e = route_expert(ids, i0 + lane, hi, E);
        const unsigned same = __match_any_sync(0xFFFFFFFFu, e);
        const bool place = e >= 0 && (e < E || invalid_tail);
        int *run = wh + (e >= 0 ? e : 0) * kWhStride + warp;
        if (place) perm[start_e[e] + *run + __popc(same & lt_mask)] = i0 + lane;
        __syncwarp();
        if (place && (same & lt_mask) == 0) *run += __popc(same);
        __syncwarp();
    }
    if (!invalid_tail && blockIdx.x == 0)
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
        // up to 8 slots' loads in flight at once, then their FMAs in increasing j
        for (int j0 = 0; j0 < topk; j0 += 8) {
            float4 o[8];
            float g[8];
            bool v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int j = j0 + u;
                const int e = j < topk ? __ldg(ids + t * topk + j) : -1;
                v[u] = e >= 0 && e < E;
                if (v[u]) {
                    g[u] = __ldg(gates + t * topk + j);
                    o[u] = __ldg(reinterpret_cast<const float4 *>(out + (t * topk + j) * N + c));
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (!v[u]) continue;
                acc.x = fmaf(g[u], o[u].x, acc.x);
                acc.y = fmaf(g[u], o[u].y, acc.y);
                acc.z = fmaf(g[u], o[u].z, acc.z);
                acc.w = fmaf(g[u], o[u].w, acc.w);
            }
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
                              int n_items, const int *__restrict__ hdr, unsigned int *status) {
    pdl_wait();
    pdl_trigger();
    if (!routing_matches(hdr, E, n_items, status)) return;  // not this call's routing: read none of it
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
                              float *zero_y, int64_t N, const int *hdr, cudaStream_t s) {
    int64_t blocks = (n_items + 7) / 8;
    const int64_t cap = (int64_t)di.sm_count * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(gather_kernel, dim3((unsigned)blocks), dim3(256), 0, s, dim3(1), x, x_per_slot, topk, perm, offsets,
                      E, K, x_sorted, zero_y, N, (int)n_items, hdr, di.status);
}

size_t route_smem_bytes(int E) { return (size_t)(E + 1) * (2 + kWhStride) * 4; }

cudaError_t launch_moe_route(const int32_t *ids, int64_t n_items, int E, int32_t *offsets, int32_t *perm,
                             bool invalid_tail, int4 *tiles, int *n_tiles, cudaStream_t s) {
    const size_t smem = route_smem_bytes(E);
    cudaError_t e = ensure_smem((const void *)route_kernel, (int)smem);
    if (e != cudaSuccess) return e;
    // ranges of a multiple of 512 items, at most kRouteMaxCtas of them
    int64_t range = (n_items + kRouteMaxCtas - 1) / kRouteMaxCtas;
    range = (range + kRouteThreads - 1) / kRouteThreads * kRouteThreads;
    if (range < kRouteThreads) range = kRouteThreads;
    const int ctas = (int)((n_items + range - 1) / range);
    return launch_pdl(route_kernel, dim3(ctas > 0 ? ctas : 1), dim3(kRouteThreads), smem, s, dim3(1), ids, (int)n_items,
                      E, (int)range, offsets, perm, invalid_tail ? 1 : 0, tiles, n_tiles);
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
