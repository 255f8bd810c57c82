/*
 * Q4_K matmul oracle - see q4k_ref.h for the format and what is computed.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
 * benchmark's CPU-baseline leg; never by the product library.
 *
 * Build: gcc -std=c99 -O2 -ffp-contract=off (no fast-math), so that every fp32
 * operation below rounds exactly once, in the order written.
 */
#include "q4k_ref.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define QK 256
#define BB 144

/* IEEE 754 binary16 -> binary32, from the definition: sign, 5-bit biased
 * exponent (bias 15), 10-bit fraction; exponent 0 is subnormal (f * 2^-24),
 * exponent 31 is inf/NaN.  Every binary16 value is exact in binary32. */
float q4k_ref_f16_to_f32(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    float v;
    if (e == 0) {
        v = ldexpf((float)f, -24);
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexpf((float)(1024 + f), e - 25);
    }
    return sign ? -v : v;
}

/* bf16 is the top half of a binary32 */
float q4k_ref_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* binary32 -> bf16, round to nearest, ties to even; NaN stays NaN */
uint16_t q4k_ref_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if (isnan(f)) return (uint16_t)(0x7FC0 | ((u >> 16) & 0x8000));
    uint32_t upper = u >> 16, lower = u & 0xFFFF;
    if (lower > 0x8000 || (lower == 0x8000 && (upper & 1))) upper += 1;
    return (uint16_t)upper;
}

void q4k_ref_scale_min(const uint8_t *scales, int j, int *sc, int *m) {
    if (j < 4) {
        *sc = scales[j] & 63;
        *m = scales[j + 4] & 63;
    } else {
        *sc = (scales[j + 4] & 15) | ((scales[j - 4] >> 6) << 4);
        *m = (scales[j + 4] >> 4) | ((scales[j] >> 6) << 4);
    }
}

/* the 4-bit code of weight i (0..255) of a block */
static int code_of(const uint8_t *qs, int i) {
    int g = i / 64;          /* 64-weight group */
    int r = i % 64;
    int l = r % 32;          /* byte within the group's 32 bytes */
    int high = r >= 32;      /* second sub-block of the group uses high nibbles */
    uint8_t b = qs[32 * g + l];
    return high ? (b >> 4) : (b & 15);
}

void q4k_ref_dequant_block(const uint8_t *blk, float *out) {
    float d = q4k_ref_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
    float dmin = q4k_ref_f16_to_f32((uint16_t)(blk[2] | (blk[3] << 8)));
    const uint8_t *scales = blk + 4;
    const uint8_t *qs = blk + 16;
    for (int i = 0; i < QK; ++i) {
        int s = i / 32;
        int sc, m;
        q4k_ref_scale_min(scales, s, &sc, &m);
        float step = d * (float)sc;            /* exact */
        float a = step * (float)code_of(qs, i); /* exact */
        float b = dmin * (float)m;              /* exact */
        out[i] = a - b;                         /* the one rounding */
    }
}

static int shape_ok(int64_t N, int64_t K) { return N >= 0 && K > 0 && K % QK == 0; }

int q4k_ref_dequant(const uint8_t *w, int64_t N, int64_t K, float *out) {
    if (!shape_ok(N, K)) return -1;
    int64_t nb = N * (K / QK);
    for (int64_t b = 0; b < nb; ++b) q4k_ref_dequant_block(w + b * BB, out + b * QK);
    return 0;
}

int q4k_ref_dequant_bf16(const uint8_t *w, int64_t N, int64_t K, uint16_t *out) {
    if (!shape_ok(N, K)) return -1;
    float tmp[QK];
    int64_t nb = N * (K / QK);
    for (int64_t b = 0; b < nb; ++b) {
        q4k_ref_dequant_block(w + b * BB, tmp);
        for (int i = 0; i < QK; ++i) out[b * QK + i] = q4k_ref_f32_to_bf16(tmp[i]);
    }
    return 0;
}

/* rows [n0, n1) of y = x * W^T; wrow is a K-float scratch row */
static void gemm_rows(const uint8_t *w, int64_t N, int64_t K, const double *xd, int64_t M, double *y,
                      int64_t n0, int64_t n1, float *wrow) {
    int64_t row_bytes = (K / QK) * BB;
    for (int64_t n = n0; n < n1; ++n) {
        q4k_ref_dequant(w + n * row_bytes, 1, K, wrow);
        for (int64_t m = 0; m < M; ++m) {
            const double *xm = xd + m * K;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += (double)wrow[k] * xm[k];
            y[m * N + n] = acc;
        }
    }
}

typedef struct {
    const uint8_t *w;
    int64_t N, K, M, n0, n1;
    const double *xd;
    double *y;
    int rc;
} gemm_job;

static void *gemm_worker(void *arg) {
    gemm_job *j = (gemm_job *)arg;
    float *wrow = (float *)malloc(sizeof(float) * (size_t)j->K);
    if (!wrow) { j->rc = -2; return NULL; }
    gemm_rows(j->w, j->N, j->K, j->xd, j->M, j->y, j->n0, j->n1, wrow);
    free(wrow);
    j->rc = 0;
    return NULL;
}

int q4k_ref_gemm_mt(const uint8_t *w, int64_t N, int64_t K, const uint16_t *x, int64_t M, double *y,
                    int threads) {
    if (!shape_ok(N, K) || M < 0) return -1;
    if (threads < 1) threads = 1;
    if (threads > N && N > 0) threads = (int)N;
    double *xd = (double *)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    if (!xd) return -2;
    for (int64_t i = 0; i < M * K; ++i) xd[i] = (double)q4k_ref_bf16_to_f32(x[i]);
    gemm_job *jobs = (gemm_job *)calloc((size_t)threads, sizeof(gemm_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
    int rc = 0;
    for (int t = 0; t < threads; ++t) {
        gemm_job *j = &jobs[t];
        j->w = w; j->N = N; j->K = K; j->M = M; j->xd = xd; j->y = y;
        j->n0 = N * t / threads; j->n1 = N * (t + 1) / threads;
        if (threads == 1) gemm_worker(j);
        else pthread_create(&tid[t], NULL, gemm_worker, j);
    }
    for (int t = 0; t < threads; ++t) {
        if (threads > 1) pthread_join(tid[t], NULL);
        if (jobs[t].rc) rc = jobs[t].rc;
    }
    free(tid); free(jobs); free(xd);
    return rc;
}

int q4k_ref_gemm(const uint8_t *w, int64_t N, int64_t K, const uint16_t *x, int64_t M, double *y) {
    return q4k_ref_gemm_mt(w, N, K, x, M, y, 1);
}

int64_t q4k_ref_moe_route(const int32_t *ids, int64_t T, int32_t topk, int32_t E, int32_t *offsets,
                          int32_t *perm) {
    int64_t n = T * topk, bad = 0;
    for (int32_t e = 0; e <= E; ++e) offsets[e] = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= E) { ++bad; continue; }
        offsets[ids[i] + 1] += 1;             /* histogram */
    }
    for (int32_t e = 0; e < E; ++e) offsets[e + 1] += offsets[e]; /* exclusive scan */
    int32_t *fill = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    for (int32_t e = 0; e < E; ++e) fill[e] = offsets[e];
    for (int64_t i = 0; i < n; ++i) {           /* stable scatter, increasing i */
        if (ids[i] < 0 || ids[i] >= E) continue;
        perm[fill[ids[i]]++] = (int32_t)i;
    }
    free(fill);
    return bad;
}

typedef struct {
    const uint8_t *w;
    int32_t E;
    int64_t N, K, T;
    const double *xd;
    int x_per_slot;
    const int32_t *ids;
    int32_t topk;
    double *out;
    int64_t i0, i1; /* item range */
    int rc;
} moe_job;

static void *moe_worker(void *arg) {
    moe_job *j = (moe_job *)arg;
    int64_t row_bytes = (j->K / QK) * BB;
    int64_t mat_bytes = j->N * row_bytes;
    float *wrow = (float *)malloc(sizeof(float) * (size_t)j->K);
    if (!wrow) { j->rc = -2; return NULL; }
    for (int64_t i = j->i0; i < j->i1; ++i) {
        int64_t t = i / j->topk;
        int32_t e = j->ids[i];
        double *o = j->out + i * j->N;
        if (e < 0 || e >= j->E) {
            for (int64_t n = 0; n < j->N; ++n) o[n] = 0.0;
            continue;
        }
        const double *xr = j->xd + (j->x_per_slot ? i : t) * j->K;
        /* this slot's output row is one GEMV against expert e */
        gemm_rows(j->w + (int64_t)e * mat_bytes, j->N, j->K, xr, 1, o, 0, j->N, wrow);
    }
    free(wrow);
    j->rc = 0;
    return NULL;
}

int q4k_ref_moe_slots(const uint8_t *w_experts, int32_t E, int64_t N, int64_t K, const uint16_t *x,
                      int x_per_slot, const int32_t *ids, int64_t T, int32_t topk, double *out,
                      int threads) {
    if (!shape_ok(N, K) || T < 0 || topk < 1 || E < 1) return -1;
    int64_t items = T * topk;
    int64_t xrows = x_per_slot ? items : T;
    double *xd = (double *)malloc(sizeof(double) * (size_t)(xrows * K > 0 ? xrows * K : 1));
    if (!xd) return -2;
    for (int64_t i = 0; i < xrows * K; ++i) xd[i] = (double)q4k_ref_bf16_to_f32(x[i]);
    if (threads < 1) threads = 1;
    if (items > 0 && threads > items) threads = (int)items;
    moe_job *jobs = (moe_job *)calloc((size_t)threads, sizeof(moe_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
    int rc = 0;
    for (int t = 0; t < threads; ++t) {
        moe_job *j = &jobs[t];
        j->w = w_experts; j->E = E; j->N = N; j->K = K; j->T = T; j->xd = xd;
        j->x_per_slot = x_per_slot; j->ids = ids; j->topk = topk; j->out = out;
        j->i0 = items * t / threads; j->i1 = items * (t + 1) / threads;
        if (threads == 1) moe_worker(j);
        else pthread_create(&tid[t], NULL, moe_worker, j);
    }
    for (int t = 0; t < threads; ++t) {
        if (threads > 1) pthread_join(tid[t], NULL);
        if (jobs[t].rc) rc = jobs[t].rc;
    }
    free(tid); free(jobs); free(xd);
    return rc;
}

void q4k_ref_moe_combine(const double *out, const float *gates, int64_t T, int32_t topk, int64_t N, double *y) {
    for (int64_t t = 0; t < T; ++t)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int32_t j = 0; j < topk; ++j)
                acc += (double)gates[t * topk + j] * out[(t * topk + j) * N + n];
            y[t * N + n] = acc;
        }
}

uint16_t q4k_ref_f64_to_bf16(double v) {
    if (v == 0.0) return signbit(v) ? 0x8000u : 0u;
    int e;
    const double m = frexp(v, &e);             /* v = m * 2^e, 0.5 <= |m| < 1 */
    const double r = nearbyint(ldexp(m, 8));   /* 8 significant bits, ties to even */
    const float f = (float)ldexp(r, e - 8);    /* exact in fp32 (and in bf16) */
    return q4k_ref_f32_to_bf16(f);
}

int q4k_ref_moe_ffn(const uint8_t *w_gate, const uint8_t *w_up, const uint8_t *w_down, int32_t E, int64_t H,
                    int64_t D, const uint16_t *x, const int32_t *ids, const float *gates, int64_t T, int32_t topk,
                    double *y, int threads) {
    if (!shape_ok(H, D) || !shape_ok(D, H) || T < 0 || topk < 1 || E < 1) return -1;
    const int64_t items = T * topk;
    double *g = (double *)malloc(sizeof(double) * (size_t)(items * H > 0 ? items * H : 1));
    double *u = (double *)malloc(sizeof(double) * (size_t)(items * H > 0 ? items * H : 1));
    uint16_t *h = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(items * H > 0 ? items * H : 1));
    double *out = (double *)malloc(sizeof(double) * (size_t)(items * D > 0 ? items * D : 1));
    int rc = (g && u && h && out) ? 0 : -2;
    if (rc == 0) rc = q4k_ref_moe_slots(w_gate, E, H, D, x, 0, ids, T, topk, g, threads);
    if (rc == 0) rc = q4k_ref_moe_slots(w_up, E, H, D, x, 0, ids, T, topk, u, threads);
    if (rc == 0) {
        for (int64_t i = 0; i < items * H; ++i) h[i] = q4k_ref_f64_to_bf16(g[i] / (1.0 + exp(-g[i])) * u[i]);
        rc = q4k_ref_moe_slots(w_down, E, D, H, h, 1, ids, T, topk, out, threads);
    }
    if (rc == 0) q4k_ref_moe_combine(out, gates, T, topk, D, y);
    free(g); free(u); free(h); free(out);
    return rc;
}

void q4k_ref_quantize_x8(const uint16_t *x, int64_t M, int64_t K, int8_t *q, float *s) {
    for (int64_t m = 0; m < M; ++m)
        for (int64_t b = 0; b < K / 32; ++b) {
            const uint16_t *xb = x + m * K + 32 * b;
            float a = 0.0f;
            for (int i = 0; i < 32; ++i) {
                const float v = fabsf(q4k_ref_bf16_to_f32(xb[i]));
                if (v > a) a = v;
            }
            const float sc = a / 127.0f;
            s[m * (K / 32) + b] = sc;
            for (int i = 0; i < 32; ++i) {
                float r = 0.0f;
                if (a > 0.0f) r = rintf(q4k_ref_bf16_to_f32(xb[i]) / sc);
                if (r > 127.0f) r = 127.0f;
                if (r < -127.0f) r = -127.0f;
                q[m * K + 32 * b + i] = (int8_t)r;
            }
        }
}

int q4k_ref_gemm_x8(const uint8_t *w, int64_t N, int64_t K, const int8_t *q, const float *s, int64_t M, double *y) {
    if (!shape_ok(N, K) || M < 0) return -1;
    float *wrow = (float *)malloc(sizeof(float) * (size_t)K);
    if (!wrow) return -2;
    const int64_t row_bytes = (K / QK) * BB;
    for (int64_t n = 0; n < N; ++n) {
        q4k_ref_dequant(w + n * row_bytes, 1, K, wrow);
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += (double)wrow[k] * ((double)s[m * (K / 32) + k / 32] * (double)q[m * K + k]);
            y[m * N + n] = acc;
        }
    }
    free(wrow);
    return 0;
}

/* e2m1: bit 3 sign, bits 2-1 exponent (bias 1), bit 0 mantissa; exponent 0 is
 * subnormal (0 or 0.5) */
float q4k_ref_e2m1_to_f32(uint8_t code) {
    const int sign = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    const float v = e == 0 ? 0.5f * (float)m : ldexpf(1.0f + 0.5f * (float)m, e - 1);
    return sign ? -v : v;
}

/* e4m3 (the finite variant): bit 7 sign, bits 6-3 exponent (bias 7), bits 2-0
 * mantissa; exponent 0 is subnormal (m * 2^-9); exponent 15 with mantissa 7 is NaN */
float q4k_ref_e4m3_to_f32(uint8_t bits) {
    const int sign = (bits >> 7) & 1, e = (bits >> 3) & 15, m = bits & 7;
    float v;
    if (e == 15 && m == 7) v = NAN;
    else if (e == 0) v = ldexpf((float)m, -9);
    else v = ldexpf((float)(8 + m), e - 10);
    return sign ? -v : v;
}

void q4k_ref_nvfp4_dequant_block(const uint8_t *blk, float g, float *out) {
    for (int i = 0; i < 256; ++i) {
        const uint8_t byte = blk[16 + i / 2];
        const uint8_t code = (i & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
        const float sv = q4k_ref_e4m3_to_f32(blk[i / 16]) * q4k_ref_e2m1_to_f32(code); /* exact */
        out[i] = g * sv;
    }
}

int q4k_ref_nvfp4_dequant(const uint8_t *w, float g, int64_t N, int64_t K, float *out) {
    if (!shape_ok(N, K)) return -1;
    const int64_t nb = K / QK;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < nb; ++b) q4k_ref_nvfp4_dequant_block(w + (n * nb + b) * BB, g, out + n * K + b * QK);
    return 0;
}

typedef struct {
    const uint8_t *w;
    double g;
    int64_t N, K, M, n0, n1;
    const uint16_t *x;
    double *y;
} nvfp4_job;

static void *nvfp4_worker(void *arg) {
    nvfp4_job *j = (nvfp4_job *)arg;
    const int64_t nb = j->K / QK;
    double *wrow = (double *)malloc(sizeof(double) * (size_t)j->K);
    for (int64_t n = j->n0; n < j->n1 && wrow; ++n) {
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t *blk = j->w + (n * nb + b) * BB;
            for (int i = 0; i < 256; ++i) {
                const uint8_t byte = blk[16 + i / 2];
                const uint8_t code = (i & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
                wrow[b * QK + i] = j->g * (double)q4k_ref_e4m3_to_f32(blk[i / 16]) * (double)q4k_ref_e2m1_to_f32(code);
            }
        }
        for (int64_t m = 0; m < j->M; ++m) {
            double acc = 0.0;
            for (int64_t k = 0; k < j->K; ++k) acc += wrow[k] * (double)q4k_ref_bf16_to_f32(j->x[m * j->K + k]);
            j->y[m * j->N + n] = acc;
        }
    }
    free(wrow);
    return NULL;
}

int q4k_ref_nvfp4_gemm(const uint8_t *w, float g, int64_t N, int64_t K, const uint16_t *x, int64_t M, double *y,
                       int threads) {
    if (!shape_ok(N, K) || M < 0) return -1;
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    pthread_t tid[256];
    nvfp4_job jobs[256];
    for (int t = 0; t < threads; ++t) {
        jobs[t] = (nvfp4_job){w, (double)g, N, K, M, N * t / threads, N * (t + 1) / threads, x, y};
        if (threads == 1) nvfp4_worker(&jobs[t]);
        else pthread_create(&tid[t], NULL, nvfp4_worker, &jobs[t]);
    }
    if (threads > 1)
        for (int t = 0; t < threads; ++t) pthread_join(tid[t], NULL);
    return 0;
}
