// Standalone Q4_K dequantization (fp32 and bf16 outputs), and NVFP4 (fp32).
//
// This is the step a GGUF target repeats on every prefill pass ("dequantizing it
// into the matrix-multiply operand", sparkinfer-server README, "Serve a GGUF
// instead of NVFP4"), exposed on its own.  It is HBM-bound: 0.5625 bytes read and
// 4 (fp32) or 2 (bf16) bytes written per weight, so the kernel only has to keep
// the loads and stores wide and coalesced.
//
// Mapping: one warp per 144-byte block.  Lane L covers qs bytes [4L, 4L+4) of
// the block, i.e. group g = L/8 and elements l = 4(L%8) .. +3 of sub-blocks 2g
// (low nibbles) and 2g+1 (high nibbles).  Each lane stores two 16-byte vectors
// (fp32) or two 8-byte vectors (bf16); a warp's stores cover the block's output
// row segment with full 128-byte lines.
//
// Numerics: w = d*sc*q - dmin*m with d*sc, (d*sc)*q and dmin*m exact in fp32, so
// the final subtraction is the only rounding; the kernel spells the operations
// out with round-to-nearest intrinsics so that no contraction changes them.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "q4k_internal.h"
#include "q4k_ptx.cuh"

namespace q4k {
namespace {

struct SubScale {
    float step;  // d * sc
    float mn;    // dmin * m
};

__device__ __forceinline__ void decode_pair(const uint8_t *sc12, int j, int &sc, int &m) {
    if (j < 4) {
        sc = sc12[j] & 63;
        m = sc12[j + 4] & 63;
    } else {
        sc = (sc12[j + 4] & 15) | ((sc12[j - 4] >> 6) << 4);
        m = (sc12[j + 4] >> 4) | ((sc12[j] >> 6) << 4);
    }
}

template <typename Store>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t *__restrict__ w, int64_t n_blocks,
                                                      Store store) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int g = lane >> 3;
    const int l0 = 4 * (lane & 7);
    for (int64_t b = warp; b < n_blocks; b += nwarps) {
        const uint8_t *blk = w + b * kBlockBytes;
        // header: d, dmin and the 12 scale bytes (every lane reads the same 16 bytes)
        const uint4 hdr = __ldg(reinterpret_cast<const uint4 *>(blk));
        const uint32_t qw = __ldg(reinterpret_cast<const uint32_t *>(blk + 16 + 32 * g + l0));
        const float d = __half2float(__ushort_as_half((unsigned short)(hdr.x & 0xFFFF)));
        const float dmin = __half2float(__ushort_as_half((unsigned short)(hdr.x >> 16)));
        uint8_t sc12[12];
        const uint32_t words[3] = {hdr.y, hdr.z, hdr.w};
#pragma unroll
        for (int i = 0; i < 12; ++i) sc12[i] = (uint8_t)(words[i >> 2] >> (8 * (i & 3)));
        int sc_lo, m_lo, sc_hi, m_hi;
        decode_pair(sc12, 2 * g, sc_lo, m_lo);
        decode_pair(sc12, 2 * g + 1, sc_hi, m_hi);
        const SubScale lo{__fmul_rn(d, (float)sc_lo), __fmul_rn(dmin, (float)m_lo)};
        const SubScale hi{__fmul_rn(d, (float)sc_hi), __fmul_rn(dmin, (float)m_hi)};
        float vlo[4], vhi[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t byte = (qw >> (8 * i)) & 0xFF;
            vlo[i] = __fsub_rn(__fmul_rn(lo.step, (float)(byte & 15)), lo.mn);
            vhi[i] = __fsub_rn(__fmul_rn(hi.step, (float)(byte >> 4)), hi.mn);
        }
        const int64_t base = b * kQK + 64 * g + l0;
        store(base, vlo);
        store(base + 32, vhi);
    }
}

struct StoreF32 {
    float *out;
    __device__ __forceinline__ void operator()(int64_t i, const float (&v)[4]) const {
        *reinterpret_cast<float4 *>(out + i) = make_float4(v[0], v[1], v[2], v[3]);
    }
};

struct StoreBF16 {
    uint16_t *out;
    __device__ __forceinline__ void operator()(int64_t i, const float (&v)[4]) const {
        __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
        __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t *>(&a);
        u.y = *reinterpret_cast<uint32_t *>(&b);
        *reinterpret_cast<uint2 *>(out + i) = u;
    }
};

template <typename Store>
cudaError_t launch(const void *w, int64_t N, int64_t K, Store st, cudaStream_t s) {
    const int64_t n_blocks = N * (K / kQK);
    const int threads = 256;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t want = (n_blocks + 7) / 8;
    int64_t cap = (int64_t)sms * 16;
    int grid = (int)(want < cap ? want : cap);
    if (grid < 1) grid = 1;
    return launch_pdl(dequant_kernel<Store>, dim3(grid), dim3(threads), 0, s, dim3(1), static_cast<const uint8_t *>(w),
                      n_blocks, st);
}

// NVFP4: one warp per 144-byte block; lane L takes value bytes 4L..4L+3
// (weights 8L..8L+7, scale L/2).  w = g * (e4m3 * e2m1): the product is exact
// in fp32, the multiplication by g rounds once.
__global__ void __launch_bounds__(256) nvfp4_dequant_kernel(const uint8_t *__restrict__ w, float g, int64_t n_blocks,
                                                            float *__restrict__ out) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t b = warp; b < n_blocks; b += nwarps) {
        const uint8_t *blk = w + b * kBlockBytes;
        const float sc = e4m3_to_f32(__ldg(blk + (lane >> 1)));
        const uint32_t vw = __ldg(reinterpret_cast<const uint32_t *>(blk + 16 + 4 * lane));
        uint32_t p[4];
        e2m1x8_to_bf16(vw, p[0], p[1], p[2], p[3]);
        float v[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __fmul_rn(g, __fmul_rn(__uint_as_float(p[i] << 16), sc));
            v[2 * i + 1] = __fmul_rn(g, __fmul_rn(__uint_as_float(p[i] & 0xFFFF0000u), sc));
        }
        float *o = out + b * kQK + 8 * lane;
        *reinterpret_cast<float4 *>(o) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4 *>(o + 4) = make_float4(v[4], v[5], v[6], v[7]);
    }
}

}  // namespace

cudaError_t launch_nvfp4_dequant(const void *w, float g, int64_t N, int64_t K, float *out, cudaStream_t s) {
    const int64_t n_blocks = N * (K / kQK);
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t want = (n_blocks + 7) / 8;
    const int64_t cap = (int64_t)sms * 16;
    const int grid = (int)(want < cap ? (want > 0 ? want : 1) : cap);
    return launch_pdl(nvfp4_dequant_kernel, dim3(grid), dim3(256), 0, s, dim3(1), static_cast<const uint8_t *>(w), g,
                      n_blocks, out);
}

cudaError_t launch_dequant_f32(const void *w, int64_t N, int64_t K, float *out, cudaStream_t s) {
    return launch(w, N, K, StoreF32{out}, s);
}

cudaError_t launch_dequant_bf16(const void *w, int64_t N, int64_t K, uint16_t *out, cudaStream_t s) {
    return launch(w, N, K, StoreBF16{out}, s);
}

}  // namespace q4k
