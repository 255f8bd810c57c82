/*
 * q4k — matrix products against GGUF Q4_K block-quantized weights on GB300 (sm_103a).
 *
 * The operation.  A GGUF serving target "dequantizes Q4_K into the matrix-multiply
 * operand" on every prefill pass, a fixed cost that dominates at 128 tokens and is
 * amortized by 4k (sparkinfer-server README, "Serve a GGUF instead of NVFP4").
 * Decode runs the same projections with one token per lane, and speculative
 * verification with 1 + draft tokens per lane (ninfer serving docs, "Start the
 * server": --draft-tokens N, MTP 1..5, DFlash 1..15; "Determinism": decode kernels
 * are chosen by the step's token count).  A routed MoE layer ends in a weighted
 * combine of its experts' down projections (sparkinfer-server README,
 * "Determinism").  This library computes exactly those products:
 *
 *     y[m][n] = sum_k x[m][k] * w[n][k]
 *
 * with w an N x K matrix stored as GGUF Q4_K blocks, x bf16 activations and y fp32.
 *
 * Q4_K block (144 bytes, 256 consecutive weights of one row; public GGUF format):
 *     [0,2) d (fp16)  [2,4) dmin (fp16)  [4,16) scales[12]  [16,144) qs[128]
 *     eight 6-bit (sc_j, m_j) pairs:  j < 4: sc = scales[j] & 63, m = scales[j+4] & 63
 *                 j >= 4: sc = (scales[j+4] & 15) | (scales[j-4] >> 6) << 4
 *                          m = (scales[j+4] >> 4) | (scales[j]   >> 6) << 4
 *     qs[32g+l]: low nibble = code of weight 64g+l, high nibble = weight 64g+32+l
 *     weight 32s+l = d*sc_s*q - dmin*m_s
 *
 * Matrix layout.  Row n of w (output feature n) is K/256 consecutive blocks;
 * rows are consecutive, so row n starts at byte n*q4k_row_bytes(K).  K must be a
 * positive multiple of 256.  x is row-major [M][ldx] bf16 (uint16 bit patterns),
 * y is row-major [M][ldy] fp32.
 *
 * Conventions for every call.
 *   - All data pointers are DEVICE pointers owned by the caller.  The library keeps
 *     no pointer after it returns.  Scratch memory, where a call needs it, is the
 *     caller's `ws` buffer; no call allocates device memory.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL is
 *     the legacy default stream) and enqueue their kernels in order on it.
 *   - Outputs are overwritten (never accumulated into).
 *   - Arguments are validated on the host before anything is launched; a call that
 *     returns an error has enqueued nothing.  Q4K_ERR_NULL: a required pointer is
 *     NULL.  Q4K_ERR_SHAPE: a size is out of range (K % 256 != 0, N or M < 1,
 *     ldx < K, ldy < N, ...).  Q4K_ERR_ALIGN: a pointer or leading dimension breaks
 *     the alignment stated for it.  Q4K_ERR_WORKSPACE: ws is smaller than the size
 *     query returns.  Q4K_ERR_DEVICE: the current device is not compute capability
 *     10.3.  Q4K_ERR_CUDA: a CUDA runtime call failed (q4k_last_cuda_error() gives
 *     the cudaError_t, per thread).
 *   - Faults inside a kernel surface at the caller's next synchronization, as with
 *     any CUDA library.  No kernel spins without a bound: a wait that runs past
 *     its limit records Q4K_ERR_TIMEOUT in a device status word and the kernel
 *     returns; q4k_check_device() reports and clears it.
 *   - Every result is run-to-run deterministic: no floating-point atomics, fixed
 *     reduction orders.
 */
#ifndef Q4K_H
#define Q4K_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    Q4K_OK = 0,
    Q4K_ERR_NULL = 1,
    Q4K_ERR_SHAPE = 2,
    Q4K_ERR_ALIGN = 3,
    Q4K_ERR_WORKSPACE = 4,
    Q4K_ERR_DEVICE = 5,
    Q4K_ERR_CUDA = 6,
    Q4K_ERR_TIMEOUT = 7,
    Q4K_ERR_ROUTING = 8
} q4k_status;

/* Static English text for a status code; never NULL. */
const char *q4k_status_string(int status);

/* The cudaError_t behind this thread's most recent Q4K_ERR_CUDA (0 if none). */
int q4k_last_cuda_error(void);

/* Bytes of one Q4_K row of K weights: K/256*144; 0 if K is not a positive
 * multiple of 256. */
size_t q4k_row_bytes(int64_t K);

/* Library version as major*10000 + minor*100 + patch. */
int q4k_version(void);

/* Synchronizes `stream`, then reads and clears the device status word that the
 * kernels set when a bounded wait gives up (Q4K_ERR_TIMEOUT) or when a call of
 * q4k_moe_grouped_gemm_reuse_routing found no routing for its shape in its
 * workspace (Q4K_ERR_ROUTING; a timeout is reported first).  Returns Q4K_OK,
 * one of those two, or Q4K_ERR_CUDA if the synchronization itself failed. */
q4k_status q4k_check_device(void *stream);

/* Declares whether the weight matrices read by the small-M calls (q4k_gemv,
 * q4k_gemm with M <= 16, q4k_gemm_x8, q4k_nvfp4_gemm with M <= 16, and the down
 * projection of q4k_moe_ffn with at most 16 items) are static: never written by
 * the kernel enqueued on the same stream immediately before the call.  Every kernel of the library is
 * launched so that it may start while the previous kernel on its stream drains,
 * and it waits for that kernel to finish before it touches memory.  With static
 * weights on, the small-M kernels already copy their first weight blocks into
 * shared memory during that wait, which hides part of each call's start-up
 * (about 1.5 us on a 50 MB GEMV).  In q4k_moe_ffn the down projection then also
 * reads topk_ids early; its gate/up kernel has already waited for the ids' writer
 * by then.  That is the usual inference setting: weights
 * are uploaded once, by copies, and only read afterwards.  Keep it off (the
 * default) when a kernel may write a weight buffer right before a q4k call reads
 * it, for example a fill or an on-device quantization kernel: the early copies
 * could then see the old contents.  Activations and outputs are never touched
 * early.  Process-wide; applies to calls enqueued after it returns.  Returns the
 * previous setting (0 or 1). */
int q4k_set_static_weights(int enable);

/* Batch-invariant mode.  The pages' serving engines pick their decode kernels by
 * the step's token count, so a token's logits can change with how many tokens
 * share the step; their deterministic mode removes that for a small cost
 * (sparkinfer-server README, "Determinism").  Here every call is run-to-run
 * deterministic in either mode; this switch is about batch invariance:
 *   off (default): M = 1 runs the decode GEMV kernel (sub-blocks in the MMA
 *       columns: the fastest one-token form), whose rounding differs from the
 *       2..16-token kernel's (both within the small-M bar).  Rows of calls with
 *       2 <= M <= 16 tokens equal each other bit for bit.
 *   on: M = 1 runs the 2..16-token kernel as well, so row m of any call with
 *       M <= 16 equals the one-token call on row m bit for bit.  Calls with
 *       M > 16 (the tensor-core path of q4k_gemm and q4k_nvfp4_gemm) split K
 *       in two or not at all, as the weight shape alone dictates (never by M),
 *       and split off no last-wave launch, so a token's row has the same bits
 *       in every call of 17 tokens or more, wherever it sits in the batch.  The
 *       two K halves are summed over a thread-block cluster pair, half 0 plus
 *       half 1.
 *       Cost: none where the weight rows fill the GPU without a K split (the
 *       K 5120 -> N 17408 prefill shape); on the narrow K 17408 -> N 5120 shape
 *       about +34 % time at 128 tokens, +25 % at 1024, +22 % at 4096 on one
 *       GB300.
 * The boundary between the two paths stays: rows of calls with M <= 16 and
 * M > 16 differ in rounding (different kernels, each within its bar).
 * Process-wide; applies to calls enqueued after it returns.  Returns the previous
 * setting (0 or 1). */
int q4k_set_batch_invariant(int enable);

/* Failure-detection test hook (no counterpart on the pages).  Every wait inside
 * the kernels is bounded (2 s); a wait that runs out makes its kernel abandon
 * its work, wait for its own copies in flight, reach all of its barriers and
 * set a device status word that q4k_check_device reports as Q4K_ERR_TIMEOUT.
 * This sets the limit of the decode GEMV's main-loop waits (q4k_gemv, and
 * q4k_gemm with M = 1 outside batch-invariant mode) to `ns`, so that a test can
 * make that path run out without faulting or hanging anything; 0 restores the
 * standard limit.  Under 1000 ns a wait tests its copy once, without blocking,
 * and gives up at once if it has not landed.  A GEMV whose wait ran out leaves
 * its output undefined.
 * Process-wide; applies to calls enqueued after it returns.  Returns the
 * previous setting (0 = standard). */
unsigned long long q4k_set_gemv_wait_limit_ns(unsigned long long ns);

/* ----------------------------------------------------------------- dequant --
 * Standalone dequantization of an N x K Q4_K matrix:
 *     out[n][k] = d*sc_s*q - dmin*m_s   (fp32, computed as fp32 multiplies and one
 *                                        final fp32 subtraction: bit-exact)
 * q4k_dequant_bf16 stores the round-to-nearest-even bf16 of that fp32 value.
 * This is the "dequantize Q4_K into the matrix-multiply operand" step of the
 * sparkinfer-server README ("Serve a GGUF instead of NVFP4") on its own.
 *   w    device, N*q4k_row_bytes(K) bytes, 16-byte aligned
 *   out  device, N*K elements, row-major, 16-byte aligned
 * Errors: NULL, SHAPE (N < 1, bad K), ALIGN, DEVICE, CUDA. */
q4k_status q4k_dequant(const void *w, int64_t N, int64_t K, float *out, void *stream);
q4k_status q4k_dequant_bf16(const void *w, int64_t N, int64_t K, uint16_t *out, void *stream);

/* -------------------------------------------------------------------- GEMV --
 * Decode projection, one token:  y[n] = sum_k x[k] * w[n][k]   (n < N, k < K)
 * Same as q4k_gemm with M = 1 and the same bits.  The decode path of the pages
 * carries no floating-point atomics (sparkinfer-server README, "Determinism");
 * neither does this one.  Activations must be finite and below 2^63 in
 * magnitude (the kernel scales them by 2^64 inside its tensor-core operands);
 * magnitudes below 2^-56 lose relative precision there.
 *   w  device Q4_K blocks, 16-byte aligned;  x  device bf16[K], 16-byte aligned;
 *   y  device fp32[N], 4-byte aligned.
 * Errors: NULL, SHAPE, ALIGN, DEVICE, CUDA. */
q4k_status q4k_gemv(const void *w, int64_t N, int64_t K, const uint16_t *x, float *y, void *stream);

/* -------------------------------------------------------------------- GEMM --
 * y[m][n] = sum_k x[m*ldx + k] * w[n][k]  for m < M, n < N; y[m*ldy + n].
 *   M <= 16 : the small-M path (decode and speculative verification, 1 + drafts
 *             tokens per lane; ninfer serving docs "Determinism"): exact integer
 *             tensor-core products per 32-weight sub-block, fp32 scaling and
 *             accumulation.  M = 1 is the decode GEMV (q4k_gemv).  For 2 <= M <=
 *             16, row m of the result does not depend on M; with
 *             q4k_set_batch_invariant(1) that holds for M = 1 too.
 *   M >  16 : the prefill path (sparkinfer-server README, "Serve a GGUF instead of
 *             NVFP4"): each weight tile is dequantized to bf16 in shared memory and
 *             multiplied on the tcgen05 tensor cores with fp32 accumulation in
 *             tensor memory.
 *   w   device Q4_K blocks, 16-byte aligned
 *   x   device bf16, 16-byte aligned, ldx >= K and ldx % 8 == 0
 *   y   device fp32, ldy >= N; 4-byte aligned for M <= 16, 16-byte aligned with
 *       ldy % 4 == 0 for M > 16
 *   ws  device scratch of at least q4k_gemm_workspace_size(M, N, K) bytes,
 *       256-byte aligned (may be NULL when that size is 0).  Its contents need not
 *       be initialized and are garbage afterwards.
 * Errors: NULL, SHAPE (M < 1, N < 1, bad K, ldx < K, ldy < N), ALIGN, WORKSPACE,
 * DEVICE, CUDA. */
size_t q4k_gemm_workspace_size(int64_t M, int64_t N, int64_t K);
q4k_status q4k_gemm(const void *w, int64_t N, int64_t K, const uint16_t *x, int64_t M, int64_t ldx, float *y,
                    int64_t ldy, void *ws, size_t ws_bytes, void *stream);

/* -------------------------------------------------------- int8 activations --
 * The pages' serving pipeline requantizes activations to int8 at each layer
 * (sparkinfer-server README, "Determinism"); their format is not given.  The
 * reading taken: blocks of 32 consecutive elements of a row (one Q4_K
 * sub-block's span), in fp32: a = max |x|, s = a / 127, q = rint(x / s) with
 * ties to even, and q = 0, s = 0 for an all-zero block.
 *
 * q4k_quantize_x8: x -> (q, s).
 *   x  device bf16 [M][ldx], ldx >= K, 4-byte aligned
 *   q  device int8 [M][K], dense, 16-byte aligned
 *   s  device fp32 [M][K/32], dense, 16-byte aligned
 * Bit-exact: every q and s follows from the IEEE round-to-nearest divisions
 * above.  Errors: NULL, SHAPE (M < 1, K not a positive multiple of 256,
 * ldx < K), ALIGN, DEVICE, CUDA. */
q4k_status q4k_quantize_x8(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, int8_t *q, float *s, void *stream);

/* q4k_gemm_x8: y = xh . W^T, where xh[m][k] = s[m][k/32] * q[m][k] are the
 * int8 activations (layouts as q4k_quantize_x8).
 *   M <= 16: the integer dot products of each 32-weight sub-block are exact; the
 *            scaling and accumulation are fp32.  Row m of the result does not
 *            depend on M.  No workspace.
 *   M >  16 (prefill, where the pages requantize the next layer's input): the
 *            activation scale changes every 32 elements of K, which an MMA
 *            accumulating over K cannot apply, so a pre-pass writes
 *            bf16(s * q) (the fp32 product rounded to nearest-even bf16) into
 *            the workspace and the tcgen05 prefill GEMM multiplies it like bf16
 *            activations (within the tensor-core bar, 1e-2).
 *   y   fp32 [M][ldy], ldy >= N; 4-byte aligned for M <= 16, 16-byte aligned with
 *       ldy % 4 == 0 for M > 16
 *   ws  device scratch of at least q4k_gemm_x8_workspace_size(M, K) bytes (M*K*2
 *       for M > 16, else 0), 256-byte aligned; garbage afterwards
 * Errors: NULL, SHAPE (M < 1, N < 1, bad K, ldy < N), ALIGN, WORKSPACE, DEVICE,
 * CUDA. */
size_t q4k_gemm_x8_workspace_size(int64_t M, int64_t K);
q4k_status q4k_gemm_x8(const void *w, int64_t N, int64_t K, const int8_t *q, const float *s, int64_t M, float *y,
                       int64_t ldy, void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------- NVFP4 weights --
 * The pages serve NVFP4 checkpoints as well as GGUF Q4_K (sparkinfer-server
 * README, "Serve a GGUF instead of NVFP4"); they do not spell the format out.
 * Reading taken: NVIDIA's NVFP4, w = g * e4m3 * e2m1 - 4-bit e2m1 values
 * (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 and a sign bit), one e4m3 scale per 16
 * consecutive weights of a row, one fp32 scale g per tensor.  Byte layout (this
 * library's): a row is K/256 blocks of 144 bytes (q4k_row_bytes(K)), each 16
 * e4m3 scale bytes (scale j covers weights 16j..16j+15) followed by 128 bytes
 * of e2m1 pairs (weight 2i in the low nibble of byte i, 2i+1 in the high one).
 *
 * q4k_nvfp4_dequant: out[N][K] fp32 = g * (e4m3 * e2m1), the product exact and
 * the multiplication by g rounded once: bit-exact.  w and out 16-byte aligned.
 * q4k_nvfp4_gemm: y[M][ldy] = x[M][ldx] . W^T for any M >= 1, on the tcgen05
 * tensor cores: each weight enters the MMA as the exact bf16 value e4m3 * e2m1,
 * the fp32 accumulator is multiplied by g in the epilogue.  x 16-byte aligned,
 * ldx % 8 == 0; y 4-byte aligned.  Deterministic (no atomics).
 * Errors: NULL, SHAPE (M or N < 1, K not a positive multiple of 256, ldx < K,
 * ldy < N), ALIGN, DEVICE, CUDA. */
q4k_status q4k_nvfp4_dequant(const void *w, float g, int64_t N, int64_t K, float *out, void *stream);
q4k_status q4k_nvfp4_gemm(const void *w, float g, int64_t N, int64_t K, const uint16_t *x, int64_t M, int64_t ldx,
                          float *y, int64_t ldy, void *stream);

/* --------------------------------------------------------------------- MoE --
 * Routed-expert layer over E experts, each an N x K Q4_K matrix; the pages' MoE
 * models route each token to its top-k experts and combine the experts' outputs
 * weighted by the gates (sparkinfer-server README, "Determinism": the routed MoE
 * down-projection combine, done there with fp32 atomicAdd; here in slot order,
 * with no atomics).
 *
 * q4k_moe_route: stable counting sort of the T*topk (token t, slot j) items by
 * expert id.  Item i = t*topk + j.
 *   topk_ids  device int32[T*topk]
 *   offsets   device int32[E+1]: items of expert e are perm[offsets[e] .. offsets[e+1])
 *   perm      device int32[T*topk]: item indices, grouped by expert, increasing
 *             within an expert.  Items whose id is outside [0,E) are left out
 *             (offsets[E] counts the valid items; perm beyond it is -1).
 * This is the routing step of q4k_moe_grouped_gemm exposed on its own.
 * Errors: NULL, SHAPE (T < 1, topk < 1, E < 1 or E > 1024, topk > E,
 * T*topk >= 2^31), ALIGN (a pointer not 4-byte aligned), DEVICE, CUDA. */
q4k_status q4k_moe_route(const int32_t *topk_ids, int64_t T, int32_t topk, int32_t n_experts, int32_t *offsets,
                         int32_t *perm, void *stream);

typedef enum {
    Q4K_MOE_X_PER_TOKEN = 0, /* x is [T][K]: every slot of token t multiplies x[t] */
    Q4K_MOE_X_PER_SLOT = 1   /* x is [T][topk][K]: slot (t,j) multiplies x[t][j] */
} q4k_moe_x_mode;

typedef enum {
    Q4K_MOE_Y_PER_SLOT = 0, /* y is [T][topk][N]: y[t][j] = x_row . w_{ids[t][j]}^T */
    Q4K_MOE_Y_COMBINE = 1   /* y is [T][N]: y[t] = sum_{j=0..topk-1} gates[t][j] * out[t][j],
                               summed in increasing j */
} q4k_moe_y_mode;

/* q4k_moe_grouped_gemm: every (token, slot) item multiplies its activation row by
 * its expert's matrix; one call covers all experts.
 *   w_experts  device, E*N*q4k_row_bytes(K) bytes: expert e's matrix starts at byte
 *              e*N*q4k_row_bytes(K); 16-byte aligned
 *   x          device bf16 rows of K (dense, ld = K), 16-byte aligned
 *   topk_ids   device int32[T][topk]; ids outside [0,E) give zero output rows and
 *              are not an error (they cannot be checked without a synchronization)
 *   gates      device fp32[T][topk]; required for Q4K_MOE_Y_COMBINE, else ignored
 *   y          device fp32, dense, 16-byte aligned
 *   ws         device scratch, >= q4k_moe_workspace_size(...) bytes, 256-byte aligned;
 *              holds the routing permutation and, for Q4K_MOE_Y_COMBINE, the
 *              per-slot fp32 rows; contents need not be initialized
 * Errors: NULL, SHAPE (as q4k_moe_route, plus N < 1, bad K, E*N >= 2^31, an
 * unknown mode, N % 4 != 0 with Q4K_MOE_Y_COMBINE), ALIGN, WORKSPACE, DEVICE,
 * CUDA.  q4k_moe_workspace_size returns 0 for arguments that would give SHAPE.
 * It takes the output mode as well as the shape (an addition to the plain
 * shape query): only Q4K_MOE_Y_COMBINE needs room for the per-slot rows. */
size_t q4k_moe_workspace_size(int32_t n_experts, int64_t N, int64_t K, int64_t T, int32_t topk, int y_mode);
q4k_status q4k_moe_grouped_gemm(const void *w_experts, int32_t n_experts, int64_t N, int64_t K, const uint16_t *x,
                                int x_mode, const int32_t *topk_ids, const float *gates, int64_t T, int32_t topk,
                                float *y, int y_mode, void *ws, size_t ws_bytes, void *stream);

/* q4k_moe_grouped_gemm_reuse_routing: q4k_moe_grouped_gemm without the routing
 * step.  The gate, up and down projections of one routed layer share the same
 * top-k ids (sparkinfer-server README, "Determinism": discrete top-k expert
 * routing), so after one q4k_moe_grouped_gemm call has sorted the items into
 * `ws`, the layer's other projections can use that sort instead of repeating it.
 * Same arguments, results and errors as q4k_moe_grouped_gemm (same bits), under
 * these conditions:
 *   - `ws` holds the routing written by the last q4k_moe_grouped_gemm call that
 *     used it (calls to this function leave it unchanged, so any number of them
 *     may follow one routing call), ordered before this call on the GPU;
 *   - that call had the same n_experts and the same number of items T*topk, and
 *     topk_ids has not changed since.
 * The routing records the (n_experts, T*topk) it was made for, and the kernels
 * check it on the GPU before reading any of it: a workspace holding a routing
 * for another shape, or none, makes the call write nothing, and the next
 * q4k_check_device reports Q4K_ERR_ROUTING.  (With at most 16 items no routing
 * is used at all.)  That topk_ids is unchanged is not checked: changed ids give
 * wrong results, not an error.  N, K, x, x_mode, gates, y and y_mode may differ
 * from the routing call; ws_bytes must cover this call
 * (q4k_moe_workspace_size), and the routing part of the workspace depends only
 * on (n_experts, T, topk). */
q4k_status q4k_moe_grouped_gemm_reuse_routing(const void *w_experts, int32_t n_experts, int64_t N, int64_t K,
                                              const uint16_t *x, int x_mode, const int32_t *topk_ids,
                                              const float *gates, int64_t T, int32_t topk, float *y, int y_mode,
                                              void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------- routed expert FFN layer --
 * One routed SwiGLU feed-forward layer of the pages' MoE models (sparkinfer-server
 * README, "Determinism": discrete top-k expert routing and the routed MoE
 * down-projection combine).  For every token t and slot j with a valid expert
 * e = topk_ids[t][j]:
 *   g = x[t] . Wg_e^T,  u = x[t] . Wu_e^T                     (fp32, H values)
 *   h = bf16(silu(g) * u), silu(g) = g / (1 + e^-g)           (rounded to nearest even)
 *   o = h . Wd_e^T                                            (fp32, D values)
 *   y[t] = sum_{j=0..topk-1} gates[t][j] * o[t][j], summed in increasing j.
 * Slots whose id is outside [0,E) contribute nothing (a token whose ids are all
 * invalid gets a zero row).  The routing is computed once for the three
 * projections; the up projection's epilogue applies SwiGLU to the gate
 * projection's output and stores h in bf16, so u is never written out.
 *   w_gate, w_up  device, E*H*q4k_row_bytes(D) bytes each: expert e's H x D matrix
 *                 starts at byte e*H*q4k_row_bytes(D); 16-byte aligned
 *   w_down        device, E*D*q4k_row_bytes(H) bytes: expert e's D x H matrix at
 *                 byte e*D*q4k_row_bytes(H); 16-byte aligned
 *   x             device bf16 [T][D], dense, 16-byte aligned
 *   topk_ids      device int32 [T][topk];  gates  device fp32 [T][topk]
 *   y             device fp32 [T][D], dense, 16-byte aligned
 *   ws            device scratch, >= q4k_moe_ffn_workspace_size(...) bytes,
 *                 256-byte aligned, contents need not be initialized: the
 *                 routing, g (4*T*topk*H bytes), h (2*T*topk*H), the per-slot
 *                 outputs o (4*T*topk*D) and, from 32*E items on, the
 *                 expert-sorted copy of x (2*T*topk*D)
 * Errors: NULL, SHAPE (E < 1 or E > 1024, topk < 1 or topk > E, T < 1,
 * T*topk >= 2^31, H or D not a positive multiple of 256, E*H or E*D >= 2^31),
 * ALIGN, WORKSPACE, DEVICE, CUDA.  q4k_moe_ffn_workspace_size returns 0 for
 * arguments that would give SHAPE. */
size_t q4k_moe_ffn_workspace_size(int32_t n_experts, int64_t H, int64_t D, int64_t T, int32_t topk);
q4k_status q4k_moe_ffn(const void *w_gate, const void *w_up, const void *w_down, int32_t n_experts, int64_t H,
                       int64_t D, const uint16_t *x, const int32_t *topk_ids, const float *gates, int64_t T,
                       int32_t topk, float *y, void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------- allocation-free MoE --
 * No counterpart on the pages: an addition for callers that cannot provide a
 * workspace - code that must not call cudaMalloc/cudaFree (they synchronize the
 * whole device), engines that hand all device memory to their own pools at
 * start-up, and foreign-language callers that only pass buffers they own.
 *
 * q4k_moe_grouped_gemm_noalloc computes exactly what q4k_moe_grouped_gemm
 * computes (same arguments, same kernels, same bits) but takes no workspace:
 * its scratch is a fixed array of Q4K_MOE_NOALLOC_SCRATCH_BYTES inside the
 * library, which every GPU that loads the library keeps allocated until the
 * process exits.  It allocates nothing itself.
 *   - The first call on a device looks up that device's scratch address
 *     (cudaGetSymbolAddress, with the device current), and so does the first
 *     call in a context of that device created since (cudaDeviceReset destroys
 *     the context the address belonged to).  Make that first call before
 *     capturing a stream into a CUDA graph.
 *   - Every call on a device shares the one array.  Calls whose kernels can
 *     overlap on the GPU (different streams without ordering between them) race
 *     on it and give wrong results; order them on one stream.
 *   - The array keeps the last call's contents; nothing in it needs to start at
 *     zero, because each call writes every scratch byte it later reads.
 *   - A request whose scratch need, q4k_moe_workspace_size(n_experts, N, K, T,
 *     topk, y_mode), exceeds Q4K_MOE_NOALLOC_SCRATCH_BYTES fails with
 *     Q4K_ERR_WORKSPACE before anything is launched.  With Q4K_MOE_Y_PER_SLOT and
 *     fewer than 32*E items the need is only the routing (about 4*(E + T*topk)
 *     bytes); Q4K_MOE_Y_COMBINE adds 4*T*topk*N bytes (for example T = 64,
 *     topk = 8, N = 2048 needs 4 MiB), and from 32*E items on, where the experts
 *     run on the tensor cores, the gathered activation rows add 2*T*topk*K bytes.
 * Other errors are those of q4k_moe_grouped_gemm. */
#define Q4K_MOE_NOALLOC_SCRATCH_BYTES (8u << 20)
q4k_status q4k_moe_grouped_gemm_noalloc(const void *w_experts, int32_t n_experts, int64_t N, int64_t K,
                                        const uint16_t *x, int x_mode, const int32_t *topk_ids, const float *gates,
                                        int64_t T, int32_t topk, float *y, int y_mode, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* Q4K_H */
