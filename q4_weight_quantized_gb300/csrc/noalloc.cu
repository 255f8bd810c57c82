// Allocation-free variant of the MoE grouped GEMM.
//
// Some callers cannot hand the library a workspace:
//   * code that must not call cudaMalloc / cudaFree at all, because those calls
//     synchronize the whole device and stall every stream mid-step;
//   * engines that reserve device memory once at start-up and hand all of it to
//     their own pools (a serving process typically sizes its KV-cache pool to
//     fill what is left after the weights), so there is no allocator to ask;
//   * thin foreign-language callers that only pass tensors they already own.
// For them, q4k_moe_grouped_gemm_noalloc keeps its scratch - the routing
// offsets and permutation and, for the weighted combine, the per-slot fp32
// rows - in one fixed array that lives in the library itself.
//
// The array is a file-scope __device__ object, so every GPU that loads this
// library holds Q4K_MOE_NOALLOC_SCRATCH_BYTES of device memory for it until the
// process exits.  In host code its name is only a stand-in: the device address
// is looked up with cudaGetSymbolAddress, with the device current, the first
// time the entry point runs on a device - and again the first time it runs in a
// context of that device made since (cudaDeviceReset destroys the context the
// address belonged to; the array may land elsewhere in the next one).
#include <cuda_runtime.h>

#include <mutex>

#include "q4k.h"
#include "q4k_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_moe_scratch[Q4K_MOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices];              // device address of g_moe_scratch, per device
unsigned long long g_scratch_ctx[kMaxDevices];  // the context that address belongs to

// Device address of the scratch array in the current device's current context
// (looked up on first use there).
q4k_status scratch_for_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return Q4K_ERR_DEVICE;
    const unsigned long long ctx = q4k::context_id();  // 0: no context current yet
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_moe_scratch);
        if (e != cudaSuccess || !p) return e == cudaErrorNoDevice ? Q4K_ERR_DEVICE : Q4K_ERR_CUDA;
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = q4k::context_id();  // the lookup made the context current
    }
    *out = g_scratch_ptr[dev];
    return Q4K_OK;
}

}  // namespace

extern "C" q4k_status q4k_moe_grouped_gemm_noalloc(const void *w_experts, int32_t n_experts, int64_t N, int64_t K,
                                                   const uint16_t *x, int x_mode, const int32_t *topk_ids,
                                                   const float *gates, int64_t T, int32_t topk, float *y, int y_mode,
                                                   void *stream) {
    void *scratch = nullptr;
    const q4k_status st = scratch_for_current_device(&scratch);
    if (st != Q4K_OK) return st;
    // Every scratch byte a call reads was written earlier in the same call (the
    // routing kernel rebuilds the offsets and permutation, the grouped GEMM writes
    // every per-slot row the combine reads), so nothing has to be cleared first.
    // Requests larger than the array fail with Q4K_ERR_WORKSPACE before any launch.
    return q4k_moe_grouped_gemm(w_experts, n_experts, N, K, x, x_mode, topk_ids, gates, T, topk, y, y_mode, scratch,
                                (size_t)Q4K_MOE_NOALLOC_SCRATCH_BYTES, stream);
}
