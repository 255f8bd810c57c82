// Host-side launchers shared between the library's translation units.  Each
// returns a cudaError_t from the launch; arguments were validated by the C-ABI
// layer (api.cu) before any of these is called.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace q4k {

constexpr int kQK = 256;          // weights per Q4_K block
constexpr int kBlockBytes = 144;  // bytes per Q4_K block

struct DeviceInfo {
    int device;
    int sm_count;
    int cc_major, cc_minor;
    size_t smem_optin;
    unsigned int *status;  // device address of the status word
};

// Current device's cached properties (first call per device, and per context
// of that device, queries them).
cudaError_t device_info(DeviceInfo *out);

// Unique id of the calling thread's current CUDA context (cuCtxGetId), 0 if no
// context is current.  Caches of device addresses are keyed on it, so that a
// context re-created after cudaDeviceReset never sees a stale address.
unsigned long long context_id();

cudaError_t launch_dequant_f32(const void *w, int64_t N, int64_t K, float *out, cudaStream_t s);
cudaError_t launch_dequant_bf16(const void *w, int64_t N, int64_t K, uint16_t *out, cudaStream_t s);
// NVFP4 blocks (16 e4m3 scales, then 128 bytes of e2m1 pairs, per 256 weights)
// with tensor scale g: w = g * e4m3 * e2m1 in fp32 (dequant.cu)
cudaError_t launch_nvfp4_dequant(const void *w, float g, int64_t N, int64_t K, float *out, cudaStream_t s);

// M in [1, 16].  early_weights: the first weight blocks may be copied before
// the kernel has waited on the previous kernel in the stream (static weights).
cudaError_t launch_smallm(const DeviceInfo &di, const void *w, int64_t N, int64_t K, const uint16_t *x, int64_t M,
                          int64_t ldx, float *y, int64_t ldy, bool early_weights, cudaStream_t s);

// M = 1: the decode GEMV kernel (gemv.cu): sub-blocks in the MMA columns, codes as
// bare bf16 bit patterns, activations staged once per warp.  Deterministic; its
// rounding differs from launch_smallm's at M = 1.
// wait_ns: the limit of the main-loop waits (kWaitLimitNs unless a test shortens it)
cudaError_t launch_gemv(const DeviceInfo &di, const void *w, int64_t N, int64_t K, const uint16_t *x, float *y,
                        bool early_weights, unsigned long long wait_ns, cudaStream_t s);

// M in [1, 16] with int8 activations: q [M][K] int8 and sx [M][K/32] fp32 scales,
// both dense and 16-byte aligned (smallm.cu, int8 mode).
cudaError_t launch_smallm_x8(const DeviceInfo &di, const void *w, int64_t N, int64_t K, const int8_t *q,
                             const float *sx, int64_t M, float *y, int64_t ldy, bool early_weights, cudaStream_t s);

// M in [1, 16] with NVFP4 weights (same 144-byte block size), y = g * (x . W^T)
// (smallm.cu, FP4 mode).
cudaError_t launch_smallm_fp4(const DeviceInfo &di, const void *w, float g, int64_t N, int64_t K, const uint16_t *x,
                              int64_t M, int64_t ldx, float *y, int64_t ldy, bool early_weights, cudaStream_t s);

// Per-32 int8 quantization of bf16 rows (x8.cu).
cudaError_t launch_quantize_x8(const DeviceInfo &di, const uint16_t *x, int64_t M, int64_t K, int64_t ldx, int8_t *q,
                               float *sx, cudaStream_t s);
// xh[M][K] bf16 = bf16(s * q), the tensor-core operand of int8 activations (x8.cu)
cudaError_t launch_expand_x8(const DeviceInfo &di, const int8_t *q, const float *sx, int64_t M, int64_t K,
                             uint16_t *xh, cudaStream_t s);

// M > 16: per-tile dequantization into shared memory + tcgen05 MMA (gemm_tc.cu).
// invariant: the K split depends on (N, K, SM count) only, never on M.
cudaError_t launch_gemm_tc(const DeviceInfo &di, const void *w, int64_t N, int64_t K, const uint16_t *x, int64_t M,
                           int64_t ldx, float *y, int64_t ldy, bool invariant, cudaStream_t s);

// SwiGLU epilogue of a routed expert's up projection: instead of its fp32
// output u, the kernel stores h = swiglu_bf16(g, u), g being the gate
// projection's fp32 output at the same row and column (rows of N, addressed
// like the output).  h_sorted (tensor-core path only): h's row is the item's
// position in the expert-sorted order rather than the item, so the down
// projection reads h as its expert-sorted activations without a gather.
struct GluOut {
    const float *g = nullptr;
    uint16_t *h = nullptr;  // null: plain fp32 output
    int h_sorted = 0;
};

// NVFP4 weights through the same tensor-core kernel: the operand is the exact
// bf16 e2m1 * e4m3 product, y = g * (x . operand^T) (gemm_tc.cu)
cudaError_t launch_gemm_tc_nvfp4(const DeviceInfo &di, const void *w, float g, int64_t N, int64_t K,
                                 const uint16_t *x, int64_t M, int64_t ldx, float *y, int64_t ldy, bool invariant,
                                 cudaStream_t s);

// MoE expert GEMM on the tensor cores: a persistent kernel (one CTA per SM,
// double-buffered tensor-memory accumulators) walking the routing's token tiles
// over the expert-sorted activation rows x_sorted (gemm_tcp.cu).
cudaError_t launch_moe_tcp(const DeviceInfo &di, const void *w_experts, int E, int64_t N, int64_t K,
                           const uint16_t *x_sorted, int64_t n_items, const int32_t *perm, const int4 *tiles,
                           const int *n_tiles, float *out, cudaStream_t s, const GluOut &glu = GluOut());

// MoE: all experts stacked as E*N rows; rows of x and of out are chosen through
// the routing permutation (perm/offsets from launch_moe_route).  With glu.h set,
// w_experts and w_up are an expert FFN's gate and up matrices (same shape),
// computed in one pass, and h = bf16(silu(g) * u) is stored instead of out
// (glu.g is not used).  With gates set and very few items (moe_direct), out is
// the combined y [T][N]: y[t] = sum_j gates[t][j] * (slot j's row), j in
// increasing order and invalid ids skipped, the same bits as launch_moe_combine
// over the per-slot rows.
// With zero_invalid, the per-slot rows of the items with an invalid id
// (perm[offsets[E] .. T*topk)) are zeroed.  With very few items (moe_direct),
// no routing is read: each item is its own grid layer, its expert ids[item].
// ids_early (with gates, very few items): the ids and the first expert weight
// blocks are read before waiting on the previous kernel - only for a call whose
// previous kernel itself waited for the ids' writer, and with static weights.
inline bool moe_direct(int64_t n_items) { return n_items <= 16; }
cudaError_t launch_moe_smallm(const DeviceInfo &di, const void *w_experts, int E, int64_t N, int64_t K,
                              const uint16_t *x, int x_per_slot, const int32_t *perm, const int32_t *offsets,
                              const int4 *tok_tiles, const int *n_tiles, const int32_t *ids, int64_t T, int topk,
                              float *out, bool zero_invalid, cudaStream_t s, const GluOut &glu = GluOut(),
                              const void *w_up = nullptr, const float *gates = nullptr, bool ids_early = false);

// Stable counting sort of items by expert (E <= 1024).  Items with an id
// outside [0, E) are left out of offsets; with invalid_tail they follow the
// valid items in perm (item order), otherwise that tail of perm is -1.  When
// tiles is given, it also lists every (expert, first item, item count) token
// tile of at most kMoeTileItems items, and n_tiles[0..3] receives their number,
// E, n_items and kRoutingStamp.
constexpr int kMoeTileItems = 192;
size_t route_smem_bytes(int E);
cudaError_t launch_moe_route(const int32_t *ids, int64_t n_items, int E, int32_t *offsets, int32_t *perm,
                             bool invalid_tail, int4 *tiles, int *n_tiles, cudaStream_t s);

// Upper bound on the number of token tiles the routing can produce: an expert
// with c > 0 items gives ceil(c / T) <= 1 + (c - 1) / T tiles (T = kMoeTileItems), and at most
// min(E, n_items) experts have items.
inline int64_t moe_max_tiles(int E, int64_t n_items) {
    return (n_items < E ? n_items : (int64_t)E) + (n_items + kMoeTileItems - 1) / kMoeTileItems;
}

// x_sorted[p] = activation row of item perm[p] (p < offsets[E]): per-token rows
// (x[item / topk]) or per-slot rows (x[item]), K bf16 each.  With zero_y, the N
// floats of zero_y's row of every invalid item (perm[offsets[E] .. n_items)) are
// zeroed.
// hdr: the routing header (tile count, E, items, stamp) written by the routing
// kernel; a header made for another (E, n_items) makes the kernel record
// kDevRouting and leave (so do the expert kernels).
cudaError_t launch_moe_gather(const DeviceInfo &di, const uint16_t *x, int x_per_slot, int topk, const int32_t *perm,
                              const int32_t *offsets, int E, int64_t n_items, int64_t K, uint16_t *x_sorted,
                              float *zero_y, int64_t N, const int *hdr, cudaStream_t s);

// y[t] = sum_j gates[t][j] * out[t*topk+j] in slot order (N % 4 == 0)
cudaError_t launch_moe_combine(const DeviceInfo &di, const float *out, const float *gates, const int32_t *ids, int E,
                               int64_t T, int topk, int64_t N, float *y, cudaStream_t s);

// Launches kern<<<grid, block, smem, s>>>(args...) with programmatic stream
// serialization (the kernel may begin while the previous kernel in the stream
// drains; it waits for it with griddepcontrol.wait before touching global
// memory) and, when `cluster` holds more than one CTA, thread-block clusters of
// that shape.
template <typename... Exp, typename... Act>
cudaError_t launch_pdl(void (*kern)(Exp...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, dim3 cluster,
                       Act &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster.x * cluster.y * cluster.z > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster.x;
        attr[n].val.clusterDim.y = cluster.y;
        attr[n].val.clusterDim.z = cluster.z;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = (unsigned)n;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<Act &&>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Raises `kern`'s dynamic shared-memory limit on the current device to at least
// `bytes`; calls cudaFuncSetAttribute only the first time a larger limit is
// needed (process-wide cache, thread-safe).
cudaError_t ensure_smem(const void *kern, int bytes);

// TMA descriptor of a Q4_K matrix viewed as uint32 words: dims {K/256*36, N},
// row pitch K/256*144 bytes, box {box_words, box_rows}, zero fill outside.
cudaError_t make_weight_tmap(CUtensorMap *m, const void *w, int64_t N, int64_t K, int box_rows, int box_words);

// TMA descriptor of bf16 activations [rows][ld] viewed as uint64 (4 activations
// each): dims {K/4, rows}, box {box_elems, 1} = one row segment of 4*box_elems.
cudaError_t make_act_tmap(CUtensorMap *m, const void *x, int64_t rows, int64_t K, int64_t ld, int box_elems);
// Rows of raw bytes [rows][pitch] (row_bytes used) as a 2-D uint64 tensor: box
// {box_bytes / 8, 1 row}.  row_bytes, pitch and box_bytes multiples of 16.
cudaError_t make_bytes_tmap(CUtensorMap *m, const void *p, int64_t rows, int64_t row_bytes, int64_t pitch,
                            int box_bytes);

// bf16 activations [rows][ld], box {64, box_rows}, 128-byte swizzle (tcgen05 operand)
cudaError_t make_act_tmap_sw128(CUtensorMap *m, const void *x, int64_t rows, int64_t K, int64_t ld, int box_rows);

}  // namespace q4k
