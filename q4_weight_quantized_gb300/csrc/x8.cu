// Per-32 int8 quantization of bf16 activation rows.
//
// The pages' pipeline requantizes activations to int8 at each layer
// (sparkinfer-server README, "Determinism"); the format is not given there.  Per
// block of 32 consecutive elements of a row, in fp32: a = max |x|, s = a / 127,
// q = rint(x / s) (ties to even), and q = 0, s = 0 for an all-zero block.  The
// divisions are IEEE round-to-nearest, so every q and s is bit-determined.
#include <cuda_bf16.h>
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

// Prefill with int8 activations: xh[m][k] = bf16(s[m][k/32] * q[m][k]) (the fp32
// product, rounded once more to nearest-even bf16), the tensor-core operand.  One
// thread per 8 consecutive elements.
__global__ void expand_x8_kernel(const int8_t *__restrict__ q, const float *__restrict__ sx, int64_t M, int64_t K,
                                 uint16_t *__restrict__ xh) {
    pdl_wait();
    pdl_trigger();
    const int64_t n8 = M * K / 8;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t e = 8 * i, m = e / K, k = e % K;
        const float s = __ldg(sx + m * (K / 32) + k / 32);
        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(q + e));
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t wv = j < 2 ? v.x : v.y;
            const int sh = 16 * (j & 1);
            const float a = __fmul_rn(s, (float)(int8_t)(wv >> sh));
            const float b = __fmul_rn(s, (float)(int8_t)(wv >> (sh + 8)));
            const __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
            o[j] = *reinterpret_cast<const uint32_t *>(&p);
        }
        *reinterpret_cast<uint4 *>(xh + e) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace

cudaError_t launch_expand_x8(const DeviceInfo &di, const int8_t *q, const float *sx, int64_t M, int64_t K,
                             uint16_t *xh, cudaStream_t s) {
    const int64_t n8 = M * K / 8;
    int64_t ctas = (n8 + 255) / 256;
    const int64_t cap = (int64_t)di.sm_count * 8;
    if (ctas > cap) ctas = cap;
    if (ctas < 1) ctas = 1;
    return launch_pdl(expand_x8_kernel, dim3((unsigned)ctas), dim3(256), 0, s, dim3(1), q, sx, M, K, xh);
}

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
