// C-ABI of the q4k library: argument validation, device checks, TMA descriptor
// construction and dispatch to the kernels.  Declarations and the contract of
// every entry point are in include/q4k.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "q4k.h"
#include "q4k_internal.h"
#include "q4k_ptx.cuh"

namespace q4k {

__device__ unsigned int g_status_word;  // kernels OR Q4K_DEV_* bits here

// q4k_set_static_weights (process-wide, default off)
static std::atomic<int> g_static_weights{0};
// q4k_set_batch_invariant (process-wide, default off)
static std::atomic<int> g_batch_invariant{0};
// q4k_set_gemv_wait_limit_ns (process-wide, 0 = the standard limit)
static std::atomic<unsigned long long> g_gemv_wait_ns{0};

namespace {

thread_local int t_last_cuda_error = 0;

q4k_status cuda_fail(cudaError_t e) {
    t_last_cuda_error = (int)e;
    return Q4K_ERR_CUDA;
}

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
bool g_dev_ready[kMaxDevices];
unsigned long long g_dev_ctx[kMaxDevices];  // context the cached entry was made in
DeviceInfo g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool k_ok(int64_t K) { return K > 0 && K % kQK == 0 && K <= (int64_t)1 << 30; }

}  // namespace

unsigned long long context_id() {
    std::call_once(g_ctx_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    });
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (!g_ctx_current || !g_ctx_id || g_ctx_current(&c) != CUDA_SUCCESS || !c || g_ctx_id(c, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

cudaError_t device_info(DeviceInfo *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    // the status word's address belongs to the device's current context: a context
    // made since the entry was cached (after cudaDeviceReset, say) is looked up anew
    unsigned long long ctx = context_id();
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_dev_ready[dev] || ctx == 0 || ctx != g_dev_ctx[dev]) {
        DeviceInfo di = {};
        di.device = dev;
        if ((e = cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&di.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&di.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) return e;
        int optin = 0;
        if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
        di.smem_optin = (size_t)optin;
        if (di.cc_major == 10 && di.cc_minor == 3) {
            void *p = nullptr;
            if ((e = cudaGetSymbolAddress(&p, g_status_word)) != cudaSuccess) return e;
            di.status = static_cast<unsigned int *>(p);
        }
        g_dev[dev] = di;
        g_dev_ready[dev] = true;
        g_dev_ctx[dev] = context_id();  // the symbol lookup above made the context current
    }
    *out = g_dev[dev];
    return cudaSuccess;
}

cudaError_t ensure_smem(const void *kern, int bytes) {
    // keyed by context as well: a re-created context starts from the default limit
    struct Entry {
        const void *kern;
        unsigned long long ctx;
        int device, bytes;
    };
    static std::mutex mu;
    static Entry table[256];
    static int used = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long ctx = context_id();
    std::lock_guard<std::mutex> lock(mu);
    int i = 0;
    while (i < used && !(table[i].kern == kern && table[i].device == dev)) ++i;
    if (i < used && ctx != 0 && table[i].ctx == ctx && table[i].bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    if (i < used) {
        if (table[i].ctx != ctx || table[i].bytes < bytes) table[i].bytes = bytes;
        table[i].ctx = ctx;
    } else if (used < 256) {
        table[used++] = {kern, ctx, dev, bytes};
    }
    return cudaSuccess;
}

// Encoding a descriptor costs host time on every call; the last few per thread
// are kept, keyed by everything that goes into them.
struct TmapKey {
    const void *ptr;
    int64_t d0, d1, stride;
    int box0, box1, kind;
    bool operator==(const TmapKey &o) const {
        return ptr == o.ptr && d0 == o.d0 && d1 == o.d1 && stride == o.stride && box0 == o.box0 && box1 == o.box1 &&
               kind == o.kind;
    }
};

static cudaError_t encode_cached(CUtensorMap *m, const TmapKey &k, CUtensorMapDataType dtype, CUtensorMapSwizzle sw) {
    constexpr int kSlots = 16;
    thread_local TmapKey keys[kSlots];
    thread_local CUtensorMap maps[kSlots];
    thread_local bool valid[kSlots] = {};
    thread_local int next = 0;
    for (int i = 0; i < kSlots; ++i)
        if (valid[i] && keys[i] == k) {
            *m = maps[i];
            return cudaSuccess;
        }
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)k.d0, (cuuint64_t)k.d1};
    cuuint64_t strides[1] = {(cuuint64_t)k.stride};
    cuuint32_t box[2] = {(cuuint32_t)k.box0, (cuuint32_t)k.box1};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, dtype, 2, const_cast<void *>(k.ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    keys[next] = k;
    maps[next] = *m;
    valid[next] = true;
    next = (next + 1) % kSlots;
    return cudaSuccess;
}

// Weight matrix as a 2-D uint32 tensor: dims {K/256*36, N}, row pitch K/256*144
// bytes; tiles of box_rows rows x box_words words, no swizzle, zero fill outside.
cudaError_t make_weight_tmap(CUtensorMap *m, const void *w, int64_t N, int64_t K, int box_rows, int box_words) {
    const int64_t KB = K / kQK;
    const TmapKey k = {w, KB * (kBlockBytes / 4), N, KB * kBlockBytes, box_words, box_rows, 0};
    return encode_cached(m, k, CU_TENSOR_MAP_DATA_TYPE_UINT32, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Activations [rows][ld] bf16 as a 2-D uint64 tensor (4 bf16 per element): dims
// {K/4, rows}, row pitch ld*2 bytes, box {box_elems, 1 row}.
cudaError_t make_act_tmap(CUtensorMap *m, const void *x, int64_t rows, int64_t K, int64_t ld, int box_elems) {
    const TmapKey k = {x, K / 4, rows, ld * 2, box_elems, 1, 1};
    return encode_cached(m, k, CU_TENSOR_MAP_DATA_TYPE_UINT64, CU_TENSOR_MAP_SWIZZLE_NONE);
}

cudaError_t make_bytes_tmap(CUtensorMap *m, const void *p, int64_t rows, int64_t row_bytes, int64_t pitch,
                            int box_bytes) {
    const TmapKey k = {p, row_bytes / 8, rows, pitch, box_bytes / 8, 1, 3};
    return encode_cached(m, k, CU_TENSOR_MAP_DATA_TYPE_UINT64, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Activations [rows][ld] bf16 for the tensor-core path: dims {K, rows}, box {64,
// box_rows}, 128-byte swizzle (the K-major operand layout tcgen05.mma reads).
cudaError_t make_act_tmap_sw128(CUtensorMap *m, const void *x, int64_t rows, int64_t K, int64_t ld, int box_rows) {
    const TmapKey k = {x, K, rows, ld * 2, 64, box_rows, 2};
    return encode_cached(m, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace q4k

using namespace q4k;

namespace {

// Common device gate: a cc 10.3 device must be current.
q4k_status check_device(DeviceInfo *di) {
    cudaError_t e = device_info(di);
    if (e != cudaSuccess) {
        if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver || e == cudaErrorInvalidDevice) {
            t_last_cuda_error = (int)e;
            return Q4K_ERR_DEVICE;
        }
        return cuda_fail(e);
    }
    if (di->cc_major != 10 || di->cc_minor != 3 || di->status == nullptr) return Q4K_ERR_DEVICE;
    return Q4K_OK;
}

}  // namespace

extern "C" {

const char *q4k_status_string(int status) {
    switch (status) {
        case Q4K_OK: return "ok";
        case Q4K_ERR_NULL: return "a required pointer is NULL";
        case Q4K_ERR_SHAPE: return "a size argument is out of range";
        case Q4K_ERR_ALIGN: return "a pointer or leading dimension is misaligned";
        case Q4K_ERR_WORKSPACE: return "the workspace is too small";
        case Q4K_ERR_DEVICE: return "the current device is not a compute capability 10.3 GPU";
        case Q4K_ERR_CUDA: return "a CUDA runtime call failed";
        case Q4K_ERR_TIMEOUT: return "a kernel gave up waiting on a barrier";
        case Q4K_ERR_ROUTING: return "a call reusing a routing found one made for another shape";
        default: return "unknown status";
    }
}

int q4k_last_cuda_error(void) { return t_last_cuda_error; }

size_t q4k_row_bytes(int64_t K) { return k_ok(K) ? (size_t)(K / kQK) * kBlockBytes : 0; }

int q4k_version(void) { return 100; }

int q4k_set_static_weights(int enable) { return g_static_weights.exchange(enable ? 1 : 0); }

int q4k_set_batch_invariant(int enable) { return g_batch_invariant.exchange(enable ? 1 : 0); }

unsigned long long q4k_set_gemv_wait_limit_ns(unsigned long long ns) { return g_gemv_wait_ns.exchange(ns); }

q4k_status q4k_check_device(void *stream) {
    DeviceInfo di;
    q4k_status st = check_device(&di);
    if (st != Q4K_OK) return st;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned int v = 0;
    if ((e = cudaMemcpyFromSymbol(&v, g_status_word, sizeof(v))) != cudaSuccess) return cuda_fail(e);
    if (v != 0) {
        const unsigned int zero = 0;
        if ((e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero))) != cudaSuccess) return cuda_fail(e);
        return (v & kDevTimeout) ? Q4K_ERR_TIMEOUT : Q4K_ERR_ROUTING;
    }
    return Q4K_OK;
}

static q4k_status dequant_common(const void *w, int64_t N, int64_t K, void *out, int out_align, bool bf16,
                                 void *stream) {
    if (!w || !out) return Q4K_ERR_NULL;
    if (N < 1 || !k_ok(K) || N > ((int64_t)1 << 31) - 1) return Q4K_ERR_SHAPE;
    if (!aligned(w, 16) || !aligned(out, (uintptr_t)out_align)) return Q4K_ERR_ALIGN;
    DeviceInfo di;
    q4k_status st = check_device(&di);
    if (st != Q4K_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = bf16 ? launch_dequant_bf16(w, N, K, static_cast<uint16_t *>(out), s)
                         : launch_dequant_f32(w, N, K, static_cast<float *>(out), s);
    return e == cudaSuccess ? Q4K_OK : cuda_fail(e);
}

q4k_status q4k_dequant(const void *w, int64_t N, int64_t K, float *out, void *stream) {
    return dequant_common(w, N, K, out, 16, false, stream);
}

q4k_status q4k_dequant_bf16(const void *w, int64_t N, int64_t K, uint16_t *out, void *stream) {
    return dequant_common(w, N, K, out, 16, true, stream);
}

size_t q4k_gemm_workspace_size(int64_t M, int64_t N, int64_t K) {
    (void)M; (void)N; (void)K;
    return 0;
}

q4k_status q4k_gemm(const void *w, int64_t N, int64_t K, const uint16_t *x, int64_t M, int64_t ldx, float *y,
                    int64_t ldy, void *ws, size_t ws_bytes, void *stream) {
    if (!w || !x || !y) return Q4K_ERR_NULL;
    if (M < 1 || N < 1 || !k_ok(K) || ldx < K || ldy < N) return Q4K_ERR_SHAPE;
    if (N > ((int64_t)1 << 31) - 1 || M > ((int64_t)1 << 31) - 1) return Q4K_ERR_SHAPE;
    if (!aligned(w, 16) || !aligned(x, 16) || (ldx % 8) != 0 || !aligned(y, 4)) return Q4K_ERR_ALIGN;
    if (M > 16 && (!aligned(y, 16) || (ldy % 4) != 0)) return Q4K_ERR_ALIGN;
    const size_t need = q4k_gemm_workspace_size(M, N, K);
    if (need > 0 && (!ws || ws_bytes < need)) return Q4K_ERR_WORKSPACE;
    if (ws && !aligned(ws, 256)) return Q4K_ERR_ALIGN;
    DeviceInfo di;
    q4k_status st = check_device(&di);
    if (st != Q4K_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // M = 1: the decode GEMV kernel, unless batch invariance is asked for (then the
    // small-M kernel, whose rows do not depend on M); M <= 16: small-M kernel;
    // otherwise the tensor-core kernel, one CTA per output tile (with a cluster K
    // split when the tiles leave the GPU half idle)
    const bool early = g_static_weights.load(std::memory_order_relaxed) != 0;
    const bool invariant = g_batch_invariant.load(std::memory_order_relaxed) != 0;
    cudaError_t e;
    if (M == 1 && !invariant) {
        const unsigned long long lim = g_gemv_wait_ns.load(std::memory_order_relaxed);
        e = launch_gemv(di, w, N, K, x, y, early, lim ? lim : kWaitLimitNs, s);
    }
    else if (M <= 16) e = launch_smallm(di, w, N, K, x, M, ldx, y, ldy, early, s);
    else e = launch_gemm_tc(di, w, N, K, x, M, ldx, y, ldy, invariant, s);
    return e == cudaSuccess ? Q4K_OK : cuda_fail(e);
}

q4k_status q4k_quantize_x8(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, int8_t *q, float *s, void *stream) {
    if (!x || !q || !s) return Q4K_ERR_NULL;
    if (M < 1 || !k_ok(K) || ldx < K || M > ((int64_t)1 << 31) - 1) return Q4K_ERR_SHAPE;
    if (!aligned(x, 4) || !aligned(q, 16) || !aligned(s, 16)) return Q4K_ERR_ALIGN;
    DeviceInfo di;
    q4k_status st = check_device(&di);
    if (st != Q4K_OK) return st;
    cudaError_t e = launch_quantize_x8(di, x, M, K, ldx, q, s, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? Q4K_OK : cuda_fail(e);
}

size_t q4k_gemm_x8_workspace_size(int64_t M, int64_t K) {
    if (M <= 16 || M < 1 || !k_ok(K)) return 0;
    return (size_t)M * (size_t)K * 2;  // the bf16 operand xh [M][K]
}

q4k_status q4k_gemm_x8(const void *w, int64_t N, int64_t K, const int8_t *q, const float *s, int64_t M, float *y,
                       int64_t ldy, void *ws, size_t ws_bytes, void *stream) {
    if (!w || !q || !s || !y) return Q4K_ERR_NULL;
    if (M < 1 || N < 1 || !k_ok(K) || ldy < N || N > ((int64_t)1 << 31) - 1 || M > ((int64_t)1 << 31) - 1)
        return Q4K_ERR_SHAPE;
    if (!aligned(w, 16) || !aligned(q, 16) || !aligned(s, 16) || !aligned(y, 4)) return Q4K_ERR_ALIGN;
    if (M > 16 && (!aligned(y, 16) || (ldy % 4) != 0)) return Q4K_ERR_ALIGN;
    const size_t need = q4k_gemm_x8_workspace_size(M, K);
    if (need > 0 && (!ws || ws_bytes < need)) return Q4K_ERR_WORKSPACE;
    if (need > 0 && !aligned(ws, 256)) return Q4K_ERR_ALIGN;
    DeviceInfo di;
    q4k_status st = check_device(&di);
    if (st != Q4K_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (M <= 16) {
        e = launch_smallm_x8(di, w, N, K, q, s, M, y, ldy, g_static_weights.load(std::memory_order_relaxed) != 0, cs);
    } else {
        // prefill: s * q rounded to bf16 in the workspace, then the tensor-core GEMM
        uint16_t *xh = static_cast<uint16_t *>(ws);
        e = launch_expand_x8(di, q, s, M, K, xh, cs);
        if (e == cudaSuccess)
            e = launch_gemm_tc(di, w, N, K, xh, M, K, y, ldy,
                               g_batch_invariant.load(std::memory_order_relaxed) != 0, cs);
    }
    return e == cudaSuccess ? Q4K_OK : cuda_fail(e);
}

q4k_status q4k_nvfp4_dequant(const void *w, float g, int64_t N, int64_t K, float *out, void *stream) {
    if (!w || !out) return Q4K_ERR_NULL;
    if (N < 1 || !k_ok(K)) return Q4K_ERR_SHAPE;
    if (!aligned(w, 16) || !aligned(out, 16)) return Q4K_ERR_ALIGN;
    DeviceInfo di;
    q4k_status st = check_device(&di);
    if (st != Q4K_OK) return st;
    cudaError_t e = launch_nvfp4_dequant(w, g, N, K, out, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? Q4K_OK : cuda_fail(e);
}

q4k_status q4k_nvfp4_gemm(const void *w, float g, int64_t N, int64_t K, const uint16_t *x, int64_t M, int64_t ldx,
                          float *y, int64_t ldy, void *stream) {
    if (!w || !x || !y) return Q4K_ERR_NULL;
    if (M < 1 || N < 1 || !k_ok(K) || ldx < K || ldy < N) return Q4K_ERR_SHAPE;
    if (N > ((int64_t)1 << 31) - 1 || M > ((int64_t)1 << 31) - 1) return Q4K_ERR_SHAPE;
    if (!aligned(w, 16) || !aligned(x, 16) || (ldx % 8) != 0 || !aligned(y, 4)) return Q4K_ERR_ALIGN;
    DeviceInfo di;
    q4k_status st = check_device(&di);
    if (st != Q4K_OK) return st;
    // M <= 16: the small-M kernel in its NVFP4 mode; otherwise the tensor-core kernel
    cudaError_t e = M <= 16 ? launch_smallm_fp4(di, w, g, N, K, x, M, ldx, y, ldy,
                                                g_static_weights.load(std::memory_order_relaxed) != 0,
                                                static_cast<cudaStream_t>(stream))
                            : launch_gemm_tc_nvfp4(di, w, g, N, K, x, M, ldx, y, ldy,
                                                   g_batch_invariant.load(std::memory_order_relaxed) != 0,
                                                   static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? Q4K_OK : cuda_fail(e);
}

q4k_status q4k_gemv(const void *w, int64_t N, int64_t K, const uint16_t *x, float *y, void *stream) {
    return q4k_gemm(w, N, K, x, 1, K, y, N, nullptr, 0, stream);
}

static size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

static bool moe_shape_ok(int32_t E, int64_t N, int64_t K, int64_t T, int32_t topk) {
    if (E < 1 || E > 1024 || N < 1 || !k_ok(K) || T < 1 || topk < 1 || topk > E) return false;
    if (T * (int64_t)topk >= ((int64_t)1 << 31) || (int64_t)E * N >= ((int64_t)1 << 31)) return false;
    return true;
}

q4k_status q4k_moe_route(const int32_t *topk_ids, int64_t T, int32_t topk, int32_t n_experts, int32_t *offsets,
                         int32_t *perm, void *stream) {
    if (!topk_ids || !offsets || !perm) return Q4K_ERR_NULL;
    if (T < 1 || topk < 1 || n_experts < 1 || n_experts > 1024 || topk > n_experts ||
        T * (int64_t)topk >= ((int64_t)1 << 31))
        return Q4K_ERR_SHAPE;
    if (!aligned(topk_ids, 4) || !aligned(offsets, 4) || !aligned(perm, 4)) return Q4K_ERR_ALIGN;
    DeviceInfo di;
    q4k_status st = check_device(&di);
    if (st != Q4K_OK) return st;
    cudaError_t e = launch_moe_route(topk_ids, T * topk, n_experts, offsets, perm, false, nullptr, nullptr,
                                     static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? Q4K_OK : cuda_fail(e);
}

// Many items per expert (32 or more on average): tensor-core tiles of up to 192
// expert-sorted tokens; otherwise the small-M kernel over each expert's few tokens.
static bool moe_uses_tc(int32_t E, int64_t T, int32_t topk) { return T * (int64_t)topk >= 32 * (int64_t)E; }

// workspace: [offsets E+1][perm T*topk][tile list][tile count][expert-sorted
// activations (tensor-core path only)][per-slot rows (combine only)]
size_t q4k_moe_workspace_size(int32_t n_experts, int64_t N, int64_t K, int64_t T, int32_t topk, int y_mode) {
    if (!moe_shape_ok(n_experts, N, K, T, topk)) return 0;
    size_t b = align256((size_t)(n_experts + 1) * 4) + align256((size_t)(T * topk) * 4) +
               align256((size_t)moe_max_tiles(n_experts, T * topk) * sizeof(int4)) + 256;
    if (moe_uses_tc(n_experts, T, topk)) b += align256((size_t)(T * topk) * (size_t)K * 2);
    if (y_mode == Q4K_MOE_Y_COMBINE) b += align256((size_t)(T * topk) * (size_t)N * 4);
    return b;
}

// route: compute the routing into ws; otherwise use the one a previous call left there
static q4k_status moe_common(const void *w_experts, int32_t n_experts, int64_t N, int64_t K, const uint16_t *x,
                             int x_mode, const int32_t *topk_ids, const float *gates, int64_t T, int32_t topk, float *y,
                             int y_mode, void *ws, size_t ws_bytes, void *stream, bool route) {
    if (!w_experts || !x || !topk_ids || !y || !ws) return Q4K_ERR_NULL;
    if (y_mode == Q4K_MOE_Y_COMBINE && !gates) return Q4K_ERR_NULL;
    if (!moe_shape_ok(n_experts, N, K, T, topk)) return Q4K_ERR_SHAPE;
    if ((x_mode != Q4K_MOE_X_PER_TOKEN && x_mode != Q4K_MOE_X_PER_SLOT) ||
        (y_mode != Q4K_MOE_Y_PER_SLOT && y_mode != Q4K_MOE_Y_COMBINE))
        return Q4K_ERR_SHAPE;
    if (y_mode == Q4K_MOE_Y_COMBINE && N % 4 != 0) return Q4K_ERR_SHAPE;
    if (!aligned(w_experts, 16) || !aligned(x, 16) || !aligned(y, 16) || !aligned(topk_ids, 4) || !aligned(ws, 256) ||
        (gates && !aligned(gates, 4)))
        return Q4K_ERR_ALIGN;
    if (ws_bytes < q4k_moe_workspace_size(n_experts, N, K, T, topk, y_mode)) return Q4K_ERR_WORKSPACE;
    DeviceInfo di;
    q4k_status st = check_device(&di);
    if (st != Q4K_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *p = static_cast<uint8_t *>(ws);
    int32_t *offsets = reinterpret_cast<int32_t *>(p);
    p += align256((size_t)(n_experts + 1) * 4);
    int32_t *perm = reinterpret_cast<int32_t *>(p);
    p += align256((size_t)(T * topk) * 4);
    int4 *tiles = reinterpret_cast<int4 *>(p);
    p += align256((size_t)moe_max_tiles(n_experts, T * topk) * sizeof(int4));
    int *n_tiles = reinterpret_cast<int *>(p);
    p += 256;
    const bool tc = moe_uses_tc(n_experts, T, topk);
    uint16_t *x_sorted = nullptr;
    if (tc) {
        x_sorted = reinterpret_cast<uint16_t *>(p);
        p += align256((size_t)(T * topk) * (size_t)K * 2);
    }
    const bool per_slot = y_mode == Q4K_MOE_Y_PER_SLOT;
    float *slot_out = per_slot ? y : reinterpret_cast<float *>(p);
    cudaError_t e = cudaSuccess;
    // with very few items the expert kernel reads the ids directly: nothing to sort
    if (route && (tc || !moe_direct(T * topk)))
        e = launch_moe_route(topk_ids, T * topk, n_experts, offsets, perm, true, tiles, n_tiles, s);
    if (e == cudaSuccess && tc)
        e = launch_moe_gather(di, x, x_mode, topk, perm, offsets, n_experts, T * topk, K, x_sorted,
                              per_slot ? y : nullptr, N, n_tiles, s);
    // with very few items the small-M kernel combines in the CTA, straight into y
    const bool dcomb = !tc && !per_slot && moe_direct(T * topk);
    if (e == cudaSuccess)
        e = tc ? launch_moe_tcp(di, w_experts, n_experts, N, K, x_sorted, T * topk, perm, tiles, n_tiles, slot_out, s)
               : launch_moe_smallm(di, w_experts, n_experts, N, K, x, x_mode, perm, offsets, tiles, n_tiles, topk_ids,
                                   T, topk, dcomb ? y : slot_out, per_slot, s, GluOut(), nullptr,
                                   dcomb ? gates : nullptr);
    if (e == cudaSuccess && !per_slot && !dcomb)
        e = launch_moe_combine(di, slot_out, gates, topk_ids, n_experts, T, topk, N, y, s);
    return e == cudaSuccess ? Q4K_OK : cuda_fail(e);
}

q4k_status q4k_moe_grouped_gemm(const void *w_experts, int32_t n_experts, int64_t N, int64_t K, const uint16_t *x,
                                int x_mode, const int32_t *topk_ids, const float *gates, int64_t T, int32_t topk,
                                float *y, int y_mode, void *ws, size_t ws_bytes, void *stream) {
    return moe_common(w_experts, n_experts, N, K, x, x_mode, topk_ids, gates, T, topk, y, y_mode, ws, ws_bytes, stream,
                      true);
}

q4k_status q4k_moe_grouped_gemm_reuse_routing(const void *w_experts, int32_t n_experts, int64_t N, int64_t K,
                                              const uint16_t *x, int x_mode, const int32_t *topk_ids,
                                              const float *gates, int64_t T, int32_t topk, float *y, int y_mode,
                                              void *ws, size_t ws_bytes, void *stream) {
    return moe_common(w_experts, n_experts, N, K, x, x_mode, topk_ids, gates, T, topk, y, y_mode, ws, ws_bytes, stream,
                      false);
}

// routing part of the workspace: [offsets E+1][perm T*topk][tile list][tile count]
static size_t moe_routing_bytes(int32_t E, int64_t n_items) {
    return align256((size_t)(E + 1) * 4) + align256((size_t)n_items * 4) +
           align256((size_t)moe_max_tiles(E, n_items) * sizeof(int4)) + 256;
}

// FFN workspace: [routing][g fp32 T*topk*H][h bf16 T*topk*H][o fp32 T*topk*D]
// [expert-sorted x bf16 T*topk*D (tensor-core path only)]
size_t q4k_moe_ffn_workspace_size(int32_t n_experts, int64_t H, int64_t D, int64_t T, int32_t topk) {
    if (!moe_shape_ok(n_experts, H, D, T, topk) || !moe_shape_ok(n_experts, D, H, T, topk)) return 0;
    const size_t n = (size_t)(T * topk);
    size_t b = moe_routing_bytes(n_experts, T * topk) + align256(n * (size_t)H * 4) + align256(n * (size_t)H * 2) +
               align256(n * (size_t)D * 4);
    if (moe_uses_tc(n_experts, T, topk)) b += align256(n * (size_t)D * 2);
    return b;
}

q4k_status q4k_moe_ffn(const void *w_gate, const void *w_up, const void *w_down, int32_t n_experts, int64_t H,
                       int64_t D, const uint16_t *x, const int32_t *topk_ids, const float *gates, int64_t T,
                       int32_t topk, float *y, void *ws, size_t ws_bytes, void *stream) {
    if (!w_gate || !w_up || !w_down || !x || !topk_ids || !gates || !y || !ws) return Q4K_ERR_NULL;
    if (!moe_shape_ok(n_experts, H, D, T, topk) || !moe_shape_ok(n_experts, D, H, T, topk)) return Q4K_ERR_SHAPE;
    if (!aligned(w_gate, 16) || !aligned(w_up, 16) || !aligned(w_down, 16) || !aligned(x, 16) || !aligned(y, 16) ||
        !aligned(topk_ids, 4) || !aligned(gates, 4) || !aligned(ws, 256))
        return Q4K_ERR_ALIGN;
    if (ws_bytes < q4k_moe_ffn_workspace_size(n_experts, H, D, T, topk)) return Q4K_ERR_WORKSPACE;
    DeviceInfo di;
    q4k_status st = check_device(&di);
    if (st != Q4K_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t n = T * topk;
    const int E = n_experts;
    uint8_t *p = static_cast<uint8_t *>(ws);
    int32_t *offsets = reinterpret_cast<int32_t *>(p);
    p += align256((size_t)(E + 1) * 4);
    int32_t *perm = reinterpret_cast<int32_t *>(p);
    p += align256((size_t)n * 4);
    int4 *tiles = reinterpret_cast<int4 *>(p);
    p += align256((size_t)moe_max_tiles(E, n) * sizeof(int4));
    int *n_tiles = reinterpret_cast<int *>(p);
    p += 256;
    float *g = reinterpret_cast<float *>(p);
    p += align256((size_t)n * (size_t)H * 4);
    uint16_t *h = reinterpret_cast<uint16_t *>(p);
    p += align256((size_t)n * (size_t)H * 2);
    float *o = reinterpret_cast<float *>(p);
    p += align256((size_t)n * (size_t)D * 4);
    const bool tc = moe_uses_tc(E, T, topk);
    cudaError_t e = cudaSuccess;
    if (tc || !moe_direct(n)) e = launch_moe_route(topk_ids, n, E, offsets, perm, true, tiles, n_tiles, s);
    if (tc) {
        // gate and up read one expert-sorted copy of x; up stores h in that order too,
        // which is the down projection's expert-sorted activation matrix
        uint16_t *x_sorted = reinterpret_cast<uint16_t *>(p);
        GluOut glu;
        glu.g = g;
        glu.h = h;
        glu.h_sorted = 1;
        if (e == cudaSuccess)
            e = launch_moe_gather(di, x, 0, topk, perm, offsets, E, n, D, x_sorted, nullptr, H, n_tiles, s);
        if (e == cudaSuccess) e = launch_moe_tcp(di, w_gate, E, H, D, x_sorted, n, perm, tiles, n_tiles, g, s);
        if (e == cudaSuccess)
            e = launch_moe_tcp(di, w_up, E, H, D, x_sorted, n, perm, tiles, n_tiles, nullptr, s, glu);
        if (e == cudaSuccess) e = launch_moe_tcp(di, w_down, E, D, H, h, n, perm, tiles, n_tiles, o, s);
    } else {
        // gate and up in one pass: h straight from the two accumulators
        GluOut glu;
        glu.h = h;
        if (e == cudaSuccess)
            e = launch_moe_smallm(di, w_gate, E, H, D, x, 0, perm, offsets, tiles, n_tiles, topk_ids, T, topk, nullptr,
                                  false, s, glu, w_up);
        // very few items: the down projection combines in the CTA, straight into y
        const bool dcomb = moe_direct(n);
        // (its ids were waited for by the gate and up kernel just before: with static
        // weights its first expert weight blocks go out before its own wait)
        if (e == cudaSuccess)
            e = launch_moe_smallm(di, w_down, E, D, H, h, 1, perm, offsets, tiles, n_tiles, topk_ids, T, topk,
                                  dcomb ? y : o, false, s, GluOut(), nullptr, dcomb ? gates : nullptr,
                                  dcomb && g_static_weights.load(std::memory_order_relaxed) != 0);
        if (e == cudaSuccess && !dcomb) e = launch_moe_combine(di, o, gates, topk_ids, E, T, topk, D, y, s);
        return e == cudaSuccess ? Q4K_OK : cuda_fail(e);
    }
    if (e == cudaSuccess) e = launch_moe_combine(di, o, gates, topk_ids, E, T, topk, D, y, s);
    return e == cudaSuccess ? Q4K_OK : cuda_fail(e);
}

}  // extern "C"
