// Per-32 int8 quantization of bf16 activation rows.
//
// The pages' pipeline requantizes activations to int8 at each layer
// (sparkinfer-server README, "Determinism"); the format is not given there.  Per
// block of 32 consecutive elements of a row, in fp32: a = max |x|, s = a / 127,
// q = rint(x / s) (ties to even), and q = 0, s = 0 for an all-zero block.  The
// divisions are IEEE round-to-nearest, so every q and s is bit-determined.
#include <cuda_runtime.h>

#include "q4k_internal.h"
#include "q4k_ptx.cuh"

namespace q4k {
namespace {

// One warp per 32-element block, one element per lane.
__global__ void quantize_x8_kernel(const uint16_t *__restrict__ x, int64_t M, int64_t K, int64_t ldx,
                                   int8_t *__restrict__ q, float *__restrict__ sx) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t nb = K / 32, total = M * nb;
    const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t b = w0; b < total; b += nw) {
        const int64_t m = b / nb, j = b % nb;
        const float v = __uint_as_float((uint32_t)__ldg(x + m * ldx + 32 * j + lane) << 16);
        // |v| orders like its bit pattern: the warp maximum as an integer reduction
        const float a = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(v))));
        const float s = a / 127.0f;
        float r = a > 0.0f ? rintf(v / s) : 0.0f;
        r = fminf(fmaxf(r, -127.0f), 127.0f);
        q[m * K + 32 * j + lane] = (int8_t)r;
        if (lane == 0) sx[m * nb + j] = s;
    }
}

}  // namespace

cudaError_t launch_quantize_x8(const DeviceInfo &di, const uint16_t *x, int64_t M, int64_t K, int64_t ldx, int8_t *q,
                               float *sx, cudaStream_t s) {
    const int64_t blocks32 = M * (K / 32);
    int64_t ctas = (blocks32 + 7) / 8;  // 8 warps per CTA
    const int64_t cap = (int64_t)di.sm_count * 8;
    if (ctas > cap) ctas = cap;
    if (ctas < 1) ctas = 1;
    return launch_pdl(quantize_x8_kernel, dim3((unsigned)ctas), dim3(256), 0, s, dim3(1), x, M, K, ldx, q, sx);
}

}  // namespace q4k
