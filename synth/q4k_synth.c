/*
 * Seeded synthetic inputs for the Q4_K matmul workloads.
 *
 * This file is input generation only.  It is shared by the oracle's tests and by
 * the GPU benchmark and tests, and it holds none of the arithmetic under test: it
 * never decodes a Q4_K block and never forms a product.  It provides
 *
 *   - splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
 *     generators", OOPSLA 2014), uniforms from its top 53 bits;
 *   - Box-Muller normals, both outputs used;
 *   - float -> bf16 round-to-nearest-even (activations are drawn in fp32 then
 *     stored as bf16);
 *   - outlier injection (a fixed fraction of 32-weight sub-blocks scaled by 10);
 *   - top-k routing (distinct experts per token by partial Fisher-Yates) with
 *     Dirichlet(1,...,1) gate weights;
 *   - the reference quantizer that encodes fp32 weights into GGUF Q4_K blocks.
 *
 * The quantizer is the encoder of the GGUF Q4_K format (the weight format the
 * sparkinfer-server README serves, "Serve a GGUF instead of NVFP4"): per 256-weight
 * block an fp16 d and dmin, twelve bytes packing eight 6-bit (scale, min) pairs,
 * and 128 bytes of 4-bit codes.  Its output blocks feed both the oracle and the
 * CUDA kernels, so agreement between the two does not depend on how it picks its
 * codes; it only has to produce valid blocks.  The packer here is written apart
 * from every decoder, so a packing test that round-trips through it checks the
 * decoder against an independent encoder.
 *
 * Build: plain C99, gcc -O2 -ffp-contract=off.  No x86-specific code.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QK_K 256
#define BLOCK_BYTES 144

/* ---------------------------------------------------------------- RNG --- */

typedef struct { uint64_t s; } sm64;

static uint64_t sm64_next(sm64 *g) {
    uint64_t z = (g->s += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* uniform in [0,1) from the top 53 bits */
static double sm64_uniform(sm64 *g) {
    return (double)(sm64_next(g) >> 11) * (1.0 / 9007199254740992.0);
}

/* uniform in (0,1] */
static double sm64_uniform_open0(sm64 *g) { return 1.0 - sm64_uniform(g); }

uint64_t q4k_synth_splitmix64(uint64_t *state) {
    sm64 g = {*state};
    uint64_t r = sm64_next(&g);
    *state = g.s;
    return r;
}

/* n normals N(mean, std^2), rounded once to fp32. */
void q4k_synth_normal_f32(uint64_t seed, int64_t n, double mean, double std, float *out) {
    sm64 g = {seed};
    const double two_pi = 6.283185307179586476925286766559;
    int64_t i = 0;
    while (i < n) {
        double u1 = sm64_uniform_open0(&g);
        double u2 = sm64_uniform(&g);
        double r = sqrt(-2.0 * log(u1));
        out[i++] = (float)(mean + std * r * cos(two_pi * u2));
        if (i < n) out[i++] = (float)(mean + std * r * sin(two_pi * u2));
    }
}

/* ---------------------------------------------------------------- bf16 --- */

static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u); /* quiet NaN */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

void q4k_synth_f32_to_bf16(const float *in, int64_t n, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne(in[i]);
}

/* normals drawn in fp32, stored as bf16 */
void q4k_synth_normal_bf16(uint64_t seed, int64_t n, double mean, double std, uint16_t *out) {
    const int64_t chunk = 1 << 16;
    float *tmp = (float *)malloc(sizeof(float) * (size_t)(n < chunk ? (n > 0 ? n : 1) : chunk));
    /* draw in one stream so that the values do not depend on the chunking */
    sm64 g = {seed};
    const double two_pi = 6.283185307179586476925286766559;
    int64_t i = 0;
    while (i < n) {
        int64_t m = n - i < chunk ? n - i : chunk;
        int64_t j = 0;
        while (j < m) {
            double u1 = sm64_uniform_open0(&g);
            double u2 = sm64_uniform(&g);
            double r = sqrt(-2.0 * log(u1));
            tmp[j++] = (float)(mean + std * r * cos(two_pi * u2));
            /* chunk is even, so a pair is only cut at the very end of the stream */
            if (j < m) tmp[j++] = (float)(mean + std * r * sin(two_pi * u2));
        }
        q4k_synth_f32_to_bf16(tmp, m, out + i);
        i += m;
    }
    free(tmp);
}

/* ------------------------------------------------------------ outliers --- */

/* Multiplies by `factor` the 32 weights of exactly round(frac * S) of the
 * S = n_weights/32 sub-blocks, chosen by a partial Fisher-Yates shuffle.
 * Returns the number of sub-blocks scaled, or -1 on allocation failure. */
int64_t q4k_synth_outliers(uint64_t seed, float *w, int64_t n_weights, double frac, float factor) {
    int64_t S = n_weights / 32;
    int64_t count = (int64_t)floor(frac * (double)S + 0.5);
    if (count <= 0 || S <= 0) return 0;
    if (count > S) count = S;
    int64_t *idx = (int64_t *)malloc(sizeof(int64_t) * (size_t)S);
    if (!idx) return -1;
    for (int64_t i = 0; i < S; ++i) idx[i] = i;
    sm64 g = {seed};
    for (int64_t i = 0; i < count; ++i) {
        int64_t j = i + (int64_t)(sm64_uniform(&g) * (double)(S - i));
        if (j >= S) j = S - 1;
        int64_t t = idx[i]; idx[i] = idx[j]; idx[j] = t;
        float *p = w + idx[i] * 32;
        for (int l = 0; l < 32; ++l) p[l] *= factor;
    }
    free(idx);
    return count;
}

/* ------------------------------------------------------------- routing --- */

/* For each of T tokens: topk distinct experts in [0,E) in draw order
 * (partial Fisher-Yates over 0..E-1), and gate weights g_j = e_j / sum(e),
 * e_j = -log(u_j) ~ Exp(1), which is Dirichlet(1,...,1).  Returns 0, or -1 if
 * topk is out of range. */
int q4k_synth_routing(uint64_t seed_ids, uint64_t seed_gates, int64_t T, int32_t E, int32_t topk,
                      int32_t *ids, float *gates) {
    if (topk < 1 || topk > E) return -1;
    int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    if (!perm) return -1;
    sm64 gi = {seed_ids}, gg = {seed_gates};
    double *e = (double *)malloc(sizeof(double) * (size_t)topk);
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t i = 0; i < E; ++i) perm[i] = i;
        for (int32_t j = 0; j < topk; ++j) {
            int32_t r = j + (int32_t)(sm64_uniform(&gi) * (double)(E - j));
            if (r >= E) r = E - 1;
            int32_t tmp = perm[j]; perm[j] = perm[r]; perm[r] = tmp;
            ids[t * topk + j] = perm[j];
        }
        if (gates) {
            double s = 0.0;
            for (int32_t j = 0; j < topk; ++j) { e[j] = -log(sm64_uniform_open0(&gg)); s += e[j]; }
            for (int32_t j = 0; j < topk; ++j) gates[t * topk + j] = (float)(e[j] / s);
        }
    }
    free(e);
    free(perm);
    return 0;
}

/* ----------------------------------------------------------- quantizer --- */

/* double -> IEEE binary16 bits, round to nearest even, computed directly from
 * the double (no intermediate float) so that there is a single rounding.
 * Inputs here are finite and >= 0. */
static uint16_t f64_to_f16_rne(double x) {
    if (!(x > 0.0)) return 0;
    if (x >= 65520.0) return 0x7C00; /* rounds to inf */
    int e;
    double m = frexp(x, &e); /* x = m * 2^e, m in [0.5,1) */
    /* binary16 normal: 1.f * 2^(E-15), E in 1..30  <=>  e-1 in -14..15 */
    int E = e - 1 + 15;
    if (E >= 1) {
        double scaled = ldexp(m, 11); /* in [1024, 2048): 11 significant bits */
        double r = nearbyint(scaled);  /* default rounding mode: to nearest even */
        if (r >= 2048.0) { r = 1024.0; E += 1; }
        if (E >= 31) return 0x7C00;
        return (uint16_t)((E << 10) | ((int)r - 1024));
    }
    /* subnormal: value = f * 2^-24, f in 0..1023 */
    double f = nearbyint(ldexp(x, 24));
    if (f >= 1024.0) return (uint16_t)(1 << 10); /* rounds up to the smallest normal */
    return (uint16_t)f;
}

static double f16_bits_to_f64(uint16_t h) {
    int E = (h >> 10) & 31, f = h & 1023;
    if (E == 0) return ldexp((double)f, -24);
    if (E == 31) return f ? NAN : INFINITY;
    return ldexp((double)(1024 + f), E - 25);
}

/* Pack eight 6-bit scales and eight 6-bit mins into the 12-byte GGUF Q4_K field:
 * pairs 0..3 sit in the low 6 bits of bytes 0..3 (scale) and 4..7 (min); pairs
 * 4..7 put their low nibbles in bytes 8..11 (scale low, min high) and their top
 * two bits in the top two bits of bytes 0..3 (scale) and 4..7 (min). */
void q4k_synth_pack_scales(const uint8_t sc[8], const uint8_t mn[8], uint8_t out[12]) {
    memset(out, 0, 12);
    for (int j = 0; j < 4; ++j) {
        out[j] = (uint8_t)(sc[j] & 63);
        out[j + 4] = (uint8_t)(mn[j] & 63);
    }
    for (int j = 4; j < 8; ++j) {
        out[j + 4] = (uint8_t)((sc[j] & 15) | ((mn[j] & 15) << 4));
        out[j - 4] |= (uint8_t)(((sc[j] >> 4) & 3) << 6);
        out[j] |= (uint8_t)(((mn[j] >> 4) & 3) << 6);
    }
}

/* Write the 128 code bytes: group g (32 bytes) holds sub-block 2g in its low
 * nibbles and sub-block 2g+1 in its high nibbles, element l at byte l. */
static void pack_codes(const uint8_t q[256], uint8_t qs[128]) {
    for (int g = 0; g < 4; ++g)
        for (int l = 0; l < 32; ++l)
            qs[32 * g + l] = (uint8_t)((q[64 * g + l] & 15) | ((q[64 * g + 32 + l] & 15) << 4));
}

/* Assemble one block from its fields. */
void q4k_synth_make_block(uint16_t d_bits, uint16_t dmin_bits, const uint8_t sc[8], const uint8_t mn[8],
                          const uint8_t q[256], uint8_t *blk) {
    blk[0] = (uint8_t)(d_bits & 255); blk[1] = (uint8_t)(d_bits >> 8);
    blk[2] = (uint8_t)(dmin_bits & 255); blk[3] = (uint8_t)(dmin_bits >> 8);
    q4k_synth_pack_scales(sc, mn, blk + 4);
    pack_codes(q, blk + 16);
}

static void quantize_block(const float *w, uint8_t *blk) {
    double lo[8], hi[8];
    double maxneg = 0.0;
    for (int s = 0; s < 8; ++s) {
        double a = 0.0, b = -INFINITY;
        for (int l = 0; l < 32; ++l) {
            double v = (double)w[32 * s + l];
            if (v < a) a = v;
            if (v > b) b = v;
        }
        lo[s] = a; hi[s] = b;
        if (-a > maxneg) maxneg = -a;
    }
    /* dmin: fp16, large enough that every min fits in 6 bits */
    uint16_t dmin_bits = f64_to_f16_rne(maxneg / 63.0);
    if (maxneg > 0.0 && dmin_bits == 0) dmin_bits = 1;
    for (;;) {
        double dm = f16_bits_to_f64(dmin_bits);
        int ok = 1;
        for (int s = 0; s < 8 && dm > 0.0; ++s)
            if (ceil(-lo[s] / dm) > 63.0) { ok = 0; break; }
        if (ok || dmin_bits >= 0x7BFF) break;
        ++dmin_bits;
    }
    double dmin = f16_bits_to_f64(dmin_bits);
    uint8_t mn[8], sc[8], q[256];
    double need[8], maxneed = 0.0;
    for (int s = 0; s < 8; ++s) {
        double m = dmin > 0.0 ? ceil(-lo[s] / dmin) : 0.0;
        if (m > 63.0) m = 63.0;
        mn[s] = (uint8_t)m;
        need[s] = (hi[s] + dmin * m) / 15.0;
        if (need[s] < 0.0) need[s] = 0.0;
        if (need[s] > maxneed) maxneed = need[s];
    }
    uint16_t d_bits = f64_to_f16_rne(maxneed / 63.0);
    if (maxneed > 0.0 && d_bits == 0) d_bits = 1;
    for (;;) {
        double d = f16_bits_to_f64(d_bits);
        int ok = 1;
        for (int s = 0; s < 8 && d > 0.0; ++s)
            if (ceil(need[s] / d) > 63.0) { ok = 0; break; }
        if (ok || d_bits >= 0x7BFF) break;
        ++d_bits;
    }
    double d = f16_bits_to_f64(d_bits);
    for (int s = 0; s < 8; ++s) {
        double c = d > 0.0 ? ceil(need[s] / d) : 0.0;
        if (c > 63.0) c = 63.0;
        sc[s] = (uint8_t)c;
        double step = d * (double)sc[s];
        for (int l = 0; l < 32; ++l) {
            double v = 0.0;
            if (step > 0.0) v = nearbyint(((double)w[32 * s + l] + dmin * (double)mn[s]) / step);
            if (v < 0.0) v = 0.0;
            if (v > 15.0) v = 15.0;
            q[32 * s + l] = (uint8_t)v;
        }
    }
    q4k_synth_make_block(d_bits, dmin_bits, sc, mn, q, blk);
}

/* Quantize an N x K fp32 matrix (row-major, K % 256 == 0) into N*K/256 blocks,
 * row n occupying blocks [n*K/256, (n+1)*K/256).  Returns 0, or -1 on bad K. */
int q4k_synth_quantize(const float *w, int64_t N, int64_t K, uint8_t *out) {
    if (K <= 0 || K % QK_K != 0 || N < 0) return -1;
    int64_t nb = N * (K / QK_K);
    for (int64_t b = 0; b < nb; ++b) quantize_block(w + b * QK_K, out + b * BLOCK_BYTES);
    return 0;
}

/* Weights for one workload matrix: N x K draws from N(0, std^2) with the given
 * seed, optional outliers (frac of sub-blocks x factor, seed_outliers), then
 * quantized.  Avoids holding more than one row band of fp32 at a time. */
int q4k_synth_weights(uint64_t seed, int64_t N, int64_t K, double std, double outlier_frac,
                      double outlier_factor, uint64_t seed_outliers, uint8_t *out) {
    if (K <= 0 || K % QK_K != 0 || N < 0) return -1;
    float *w = (float *)malloc(sizeof(float) * (size_t)(N * K > 0 ? N * K : 1));
    if (!w) return -2;
    q4k_synth_normal_f32(seed, N * K, 0.0, std, w);
    if (outlier_frac > 0.0) q4k_synth_outliers(seed_outliers, w, N * K, outlier_frac, (float)outlier_factor);
    int rc = q4k_synth_quantize(w, N, K, out);
    free(w);
    return rc;
}
