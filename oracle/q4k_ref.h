/*
 * Q4_K matmul oracle: plain, slow, obviously correct CPU code.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * loads this code; only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code with the CUDA path.
 *
 * What it computes (the method): the pages are serving READMEs that only name
 * the operation - a GGUF target "dequantizes Q4_K into the matrix-multiply
 * operand" on every prefill pass (sparkinfer-server README, "Serve a GGUF instead
 * of NVFP4"); decode projections run over the same weights (ninfer serving docs,
 * "Determinism"); the routed MoE down projection ends in a weighted combine
 * (sparkinfer-server README, "Determinism").  The bit layout of a Q4_K block is
 * not on the pages; it is the public GGUF Q4_K definition:
 *
 *   bytes [0,2)    d     IEEE binary16, little-endian
 *   bytes [2,4)    dmin  IEEE binary16
 *   bytes [4,16)   scales[12]: eight 6-bit (sc_j, m_j) pairs
 *                    j < 4 : sc_j = scales[j] & 63,   m_j = scales[j+4] & 63
 *                    j >= 4: sc_j = (scales[j+4] & 15) | (scales[j-4] >> 6) << 4
 *                            m_j  = (scales[j+4] >> 4) | (scales[j]   >> 6) << 4
 *   bytes [16,144) qs[128]: for g = 0..3, l = 0..31, byte qs[32g+l] holds the
 *                  code of weight 64g+l in its low nibble and of weight
 *                  64g+32+l in its high nibble.
 *
 *   weight 32s+l of the block:  w = d*sc_s*q - dmin*m_s
 *
 * Dequantization is done in fp32: d*sc_s, (d*sc_s)*q and dmin*m_s are exact in
 * fp32 (at most 21 significant bits), so the only rounding is the final
 * subtraction.  Matrix products accumulate in fp64 in increasing k; each product
 * of an fp32 weight and a bf16 activation is exact in fp64.
 *
 * A weight matrix W is N x K (K % 256 == 0) stored as N rows of K/256 blocks,
 * rows contiguous; y[m][n] = sum_k x[m][k] * W[n][k].
 */
#ifndef Q4K_REF_H
#define Q4K_REF_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

float q4k_ref_f16_to_f32(uint16_t h);
float q4k_ref_bf16_to_f32(uint16_t b);
uint16_t q4k_ref_f32_to_bf16(float f);

/* (sc_j, m_j) for j = 0..7 from the 12-byte field */
void q4k_ref_scale_min(const uint8_t *scales, int j, int *sc, int *m);

/* one 144-byte block -> 256 fp32 weights */
void q4k_ref_dequant_block(const uint8_t *blk, float *out);

/* whole matrix -> N x K fp32 / bf16; returns 0, or -1 on a bad shape */
int q4k_ref_dequant(const uint8_t *w, int64_t N, int64_t K, float *out);
int q4k_ref_dequant_bf16(const uint8_t *w, int64_t N, int64_t K, uint16_t *out);

/* y[M][N] (fp64) = x[M][K] (bf16) * W^T, fp64 accumulation in increasing k */
int q4k_ref_gemm(const uint8_t *w, int64_t N, int64_t K, const uint16_t *x, int64_t M, double *y);
/* same result, rows of W split across `threads` pthreads (for timing) */
int q4k_ref_gemm_mt(const uint8_t *w, int64_t N, int64_t K, const uint16_t *x, int64_t M, double *y,
                    int threads);

/* MoE routing: stable counting sort of the T*topk (token, slot) items by expert.
 * offsets[E+1] (offsets[e]..offsets[e+1] are expert e's items), perm[T*topk]
 * holds item indices t*topk+j in sorted order.  Returns the number of items
 * whose expert id is outside [0,E) (those are left out of perm). */
int64_t q4k_ref_moe_route(const int32_t *ids, int64_t T, int32_t topk, int32_t E, int32_t *offsets,
                          int32_t *perm);

/* MoE per-slot outputs out[T][topk][N] (fp64).  w_experts is [E][N][K/256]
 * blocks.  x_per_slot = 0: x is [T][K] and every slot of token t reads x[t];
 * x_per_slot = 1: x is [T][topk][K].  A slot whose expert id is outside [0,E)
 * gets zeros. */
int q4k_ref_moe_slots(const uint8_t *w_experts, int32_t E, int64_t N, int64_t K, const uint16_t *x,
                      int x_per_slot, const int32_t *ids, int64_t T, int32_t topk, double *out,
                      int threads);

/* y[T][N] = sum_{j=0..topk-1} gates[t][j] * out[t][j][:], in j order, fp64 */
void q4k_ref_moe_combine(const double *out, const float *gates, int64_t T, int32_t topk, int64_t N, double *y);

/* int8 activations (sparkinfer-server README, "Determinism": the pipeline
 * requantizes activations to int8 at each layer).  The pages do not give the
 * format; the reading taken: blocks of 32 consecutive elements of a row (the
 * span of one Q4_K sub-block), in fp32 arithmetic:
 *     a = max |x_i|,  s = a / 127,  q_i = rint(x_i / s)  (ties to even),
 * and q_i = 0, s = 0 for an all-zero block.  |q_i| <= 127.  x is [M][K] bf16,
 * q [M][K], s [M][K/32].  K must be a multiple of 32. */
void q4k_ref_quantize_x8(const uint16_t *x, int64_t M, int64_t K, int8_t *q, float *s);

/* y[m][n] = sum_k w[n][k] * xh[m][k] with xh[m][k] = s[m][k/32] * q[m][k], the
 * dequantized int8 activations, in fp64 over the fp32 dequantized weights.
 * Returns 0, or -1 on a bad shape. */
int q4k_ref_gemm_x8(const uint8_t *w, int64_t N, int64_t K, const int8_t *q, const float *s, int64_t M, double *y);

/* NVFP4 weights (the pages serve NVFP4 checkpoints next to GGUF Q4_K:
 * sparkinfer-server README, "Serve a GGUF instead of NVFP4"; the format is not
 * spelled out there).  Reading taken: NVIDIA's NVFP4 - 4-bit e2m1 values (sign,
 * 2-bit exponent with bias 1, 1-bit mantissa: magnitudes 0, 0.5, 1, 1.5, 2, 3,
 * 4, 6), one e4m3 scale (sign, 4-bit exponent with bias 7, 3-bit mantissa;
 * exponent 0 subnormal; 0x7F/0xFF NaN) per 16 consecutive weights, and one fp32
 * scale g per tensor: w = g * e4m3 * e2m1.  Byte layout (this library's, like
 * GGUF's for Q4_K): a row is K/256 blocks of 144 bytes, each 16 scale bytes
 * (scale j for weights 16j..16j+15) then 128 value bytes (weight 2i in the low
 * nibble of byte i, 2i+1 in the high nibble). */
float q4k_ref_e2m1_to_f32(uint8_t code);
float q4k_ref_e4m3_to_f32(uint8_t bits);
/* 256 weights of one block, each g * (e4m3 * e2m1) rounded once to fp32 (the
 * product e4m3 * e2m1 is exact in fp32) */
void q4k_ref_nvfp4_dequant_block(const uint8_t *blk, float g, float *out);
int q4k_ref_nvfp4_dequant(const uint8_t *w, float g, int64_t N, int64_t K, float *out);
/* y[m][n] = sum_k w[n][k] * x[m][k], with w = g * e4m3 * e2m1 exact in fp64 */
int q4k_ref_nvfp4_gemm(const uint8_t *w, float g, int64_t N, int64_t K, const uint16_t *x, int64_t M, double *y,
                       int threads);

/* Round a double to the nearest bf16 (ties to even), once; returns its bits.
 * Finite normal range only (|v| from 2^-126 to the bf16 maximum, or 0). */
uint16_t q4k_ref_f64_to_bf16(double v);

/* Routed SwiGLU expert layer: the projections on either side of the routed
 * grouped GEMM and its combine (sparkinfer-server README, "Determinism": the
 * routed MoE down projection and its combine).  The activation between the
 * projections is not on the pages; the reading taken is SwiGLU.  For every item
 * (t, j) whose expert e = ids[t][j] is in [0, E):
 *     g = x[t] . W_gate[e]^T,  u = x[t] . W_up[e]^T        (H values each, fp64)
 *     h = bf16( g / (1 + exp(-g)) * u )                   (rounded once, ties to even)
 *     out[t][j] = h . W_down[e]^T                          (D values, fp64)
 * and y[T][D] = sum_j gates[t][j] * out[t][j] in j order (items with an invalid
 * id have out = 0).  w_gate, w_up are [E][H][D/256] blocks, w_down [E][D][H/256];
 * x is [T][D] bf16.  Returns 0, or -1 on a bad shape. */
int q4k_ref_moe_ffn(const uint8_t *w_gate, const uint8_t *w_up, const uint8_t *w_down, int32_t E, int64_t H,
                    int64_t D, const uint16_t *x, const int32_t *ids, const float *gates, int64_t T, int32_t topk,
                    double *y, int threads);

#ifdef __cplusplus
}
#endif
#endif
