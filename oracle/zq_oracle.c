/*
 * zq_oracle.c -- plain, slow, single-threaded CPU oracle of the quantized
 * projection: RMSNorm fused with Q8_1 activation packing, then Q4_K x Q8_1
 * matrix products.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this file.
 * Only the test-suite, the smoke check and the CPU-baseline leg of the
 * benchmark load it.  It shares no code, header, table or helper with the
 * CUDA library; both read the same seeded input bytes and nothing else.
 *
 * Sources (page title, then section):
 *   - ZINC docs "ROCm backend", section "Build and verify": RMS normalization
 *     and Q8 activation packing run as one per-token kernel; hot Q4_K
 *     projections consume packed Q8 activations; gate and up run as paired
 *     Q4 projections.
 *   - MIInfer README, "Status" (project list): Q4_K x Q8_1 MMVQ-style
 *     projections for FFN down, gate/up and attention gate; Q4_K metadata
 *     staging; packed int8 dot4.
 *   The pages name Q4_K and Q8_1 but print neither a byte layout nor a
 *   formula.  The definitions below are the readings used throughout:
 *
 *   Q8_1 block (32 activations): int8 q[32], scale d, sum s.
 *     amax = max |xh_i|, d = amax / 127, q_i = round-half-away(xh_i / d)
 *     (computed as xh_i * (1/d)), s = d * sum(q_i); d and s are stored as
 *     IEEE binary16.  Planar storage: qs int8 [B][K], d fp16 [B][K/32],
 *     s fp16 [B][K/32].
 *
 *   Q4_K super-block (256 weights, 144 bytes):
 *     bytes 0..1  d     (binary16)
 *     bytes 2..3  dmin  (binary16)
 *     bytes 4..15 twelve bytes holding eight 6-bit scales sc[j] and eight
 *                 6-bit mins m[j]:
 *                   j < 4 : sc[j] = S[j] & 63,     m[j] = S[j+4] & 63
 *                   j >= 4: sc[j] = (S[j+4] & 15) | ((S[j-4] >> 6) << 4)
 *                           m[j]  = (S[j+4] >> 4) | ((S[j]   >> 6) << 4)
 *                 (S = the twelve bytes)
 *     bytes 16..143  128 bytes of 4-bit quants: weight i (0..31) of
 *                 sub-block j lives in byte 32*(j/2)+i, low nibble for even
 *                 j, high nibble for odd j.
 *     weight value  w = d*sc[j]*q - dmin*m[j].
 *   A Q4_K matrix of N rows and K columns (K % 256 == 0) stores row n as
 *   K/256 consecutive super-blocks; rows are consecutive.
 *
 *   Output (integer-domain product, per token t and row n):
 *     y[t][n] = sum over super-blocks b and sub-blocks j of
 *               d_b*sc_j*d8_{t,bj}*I_{t,n,b,j} - dmin_b*m_j*s8_{t,bj}
 *     with I the exact integer sum of q4*q8 over the 32 weights of the
 *     sub-block; the float part is accumulated in fp64 here.
 *
 * Build: cc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC
 * (contraction must stay off: the fp32 RMSNorm steps below are rounded one
 * operation at a time, and only the explicit fmaf calls are fused).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------
 * IEEE 754 binary16 conversion, written from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; subnormals have
 * the fixed quantum 2^-24; round to nearest, ties to even; magnitudes that
 * round past 65504 become infinity.  (Used for the Q4_K d/dmin fields and
 * the Q8_1 d/s fields, which the pages call fp16.)
 * ---------------------------------------------------------------------- */
uint16_t zqo_f32_to_f16(float f)
{
    double a = fabs((double)f);
    uint16_t sign = signbit(f) ? 0x8000u : 0u;
    if (isnan(f)) return (uint16_t)(sign | 0x7E00u);
    if (isinf(f)) return (uint16_t)(sign | 0x7C00u);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: count quanta of 2^-24, ties to even */
        double qn = nearbyint(a * ldexp(1.0, 24)); /* exact scaling */
        return (uint16_t)(sign | (uint16_t)qn);    /* qn == 1024 is 2^-14 */
    }
    int e;
    double m = frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
    e -= 1;                  /* a = (2m) * 2^e, 2m in [1, 2) */
    double frac = nearbyint((2.0 * m) * 1024.0); /* 1024..2048, ties even */
    if (frac >= 2048.0) { frac = 1024.0; e += 1; }
    int field = e + 15;
    if (field >= 31) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)(field << 10) | (uint16_t)((int)frac - 1024));
}

void zqo_f32_to_f16_array(const float *f, uint16_t *h, size_t n)
{
    for (size_t i = 0; i < n; ++i) h[i] = zqo_f32_to_f16(f[i]);
}

float zqo_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1, field = (h >> 10) & 31, frac = h & 1023;
    double v;
    if (field == 31) v = frac ? NAN : INFINITY;
    else if (field == 0) v = ldexp((double)frac, -24);
    else v = ldexp(1024.0 + frac, field - 25);
    return (float)(sign ? -v : v);
}

/* ------------------------------------------------------------------------
 * Fused RMSNorm + Q8_1 packing, one token at a time (ZINC docs "ROCm
 * backend", "Build and verify": one per-token kernel normalizes and packs).
 *
 * RMSNorm: xh_k = (x_k * r) * gamma_k with r = 1 / sqrt(ss/K + eps) and
 * ss = sum_k x_k^2.  Every step is one IEEE fp32 operation.  The pages fix no
 * summation order for ss; the fixed order used (so that quantized codes are
 * reproducible bit for bit) is:
 *   1. for each 32-element block b: p_b = fmaf chain over its 32 squares in
 *      index order, starting from +0;
 *   2. 256 slots: slot t = fp32 sum of p_b over b = t (mod 256), increasing b,
 *      starting from +0 (empty slots stay +0);
 *   3. pairwise tree over the slots: for off = 128, 64, ..., 1 and t < off,
 *      slot[t] = slot[t] + slot[t + off]; ss = slot[0].
 * mean = ss / K, r = 1 / sqrt(mean + eps) (IEEE division and square root).
 *
 * Q8_1 per 32-block, as stated at the top of this file.
 * ---------------------------------------------------------------------- */
float zqo_rms_scale(const float *x, int K, float eps)
{
    float slot[256];
    for (int t = 0; t < 256; ++t) slot[t] = 0.0f;
    for (int b = 0; b < K / 32; ++b) {
        float p = 0.0f;
        for (int i = 0; i < 32; ++i) p = fmaf(x[32 * b + i], x[32 * b + i], p);
        slot[b % 256] = slot[b % 256] + p;
    }
    for (int off = 128; off >= 1; off /= 2)
        for (int t = 0; t < off; ++t) slot[t] = slot[t] + slot[t + off];
    float mean = slot[0] / (float)K;
    float root = sqrtf(mean + eps);
    return 1.0f / root;
}

void zqo_rmsnorm_q8_1(const float *x, const float *gamma, int B, int K, float eps,
                      int8_t *qs, uint16_t *d16, uint16_t *s16)
{
    for (int t = 0; t < B; ++t) {
        const float *xt = x + (size_t)t * K;
        float r = zqo_rms_scale(xt, K, eps);
        for (int b = 0; b < K / 32; ++b) {
            float xh[32];
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                int k = 32 * b + i;
                float v = xt[k] * r;
                v = v * gamma[k];
                xh[i] = v;
                if (fabsf(v) > amax) amax = fabsf(v);
            }
            float d = amax / 127.0f;
            float id = (d != 0.0f) ? 1.0f / d : 0.0f;
            int sum = 0;
            for (int i = 0; i < 32; ++i) {
                float q = roundf(xh[i] * id); /* half away from zero */
                if (q > 127.0f) q = 127.0f;
                if (q < -127.0f) q = -127.0f;
                qs[(size_t)t * K + 32 * b + i] = (int8_t)q;
                sum += (int)q;
            }
            float s = d * (float)sum;
            d16[(size_t)t * (K / 32) + b] = zqo_f32_to_f16(d);
            s16[(size_t)t * (K / 32) + b] = zqo_f32_to_f16(s);
        }
    }
}

/* ------------------------------------------------------------------------
 * SiLU(gate) * up packed to Q8_1: the input of the FFN down projection
 * (MIInfer README, "Current phase": a fused SiLU(gate)*up epilogue ahead of
 * the down projection).  The pages fix no precision.  This library defines
 * every step as one IEEE fp32 operation, so that any implementation that
 * follows the steps produces the same codes:
 *   e = exp32(-g);  silu = g / (1 + e);  h = silu * up;  Q8_1 of h as above.
 * exp32(a): a clamped to [-86, 88];  k = rint(a * LOG2E);
 *   r = fma(-k, LN2_HI, a);  r = fma(-k, LN2_LO, r)   (Cody-Waite split of
 *   ln 2: LN2_HI holds its leading 16 bits, so k * LN2_HI is exact);
 *   p = sum_{n<=7} r^n / n! in Horner form with fma, coefficients rounded to
 *   fp32 (|r| <= 0.347: the truncation is below 2^-27 relative);
 *   result = p * 2^k, an exact scaling for k in [-124, 127].
 * ---------------------------------------------------------------------- */
static float zqo_pow2i(int k) /* 2^k for -126 <= k <= 127, exactly */
{
    uint32_t bits = (uint32_t)(k + 127) << 23;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

float zqo_exp32(float a)
{
    /* fp32 roundings of log2(e), of ln 2 split in two, and of 1/n! */
    const float LOG2E = 0x1.715476p+0f;
    const float LN2_HI = 0x1.62e4p-1f;
    const float LN2_LO = 0x1.7f7d1cp-20f;
    a = fminf(fmaxf(a, -86.0f), 88.0f);
    float kf = rintf(a * LOG2E);
    float r = fmaf(-kf, LN2_HI, a);
    r = fmaf(-kf, LN2_LO, r);
    float p = 0x1.a01a02p-13f;        /* 1/7! */
    p = fmaf(p, r, 0x1.6c16c2p-10f);  /* 1/6! */
    p = fmaf(p, r, 0x1.111112p-7f);   /* 1/5! */
    p = fmaf(p, r, 0x1.555556p-5f);   /* 1/4! */
    p = fmaf(p, r, 0x1.555556p-3f);   /* 1/3! */
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    return p * zqo_pow2i((int)kf);
}

float zqo_silu32(float g)
{
    float e = zqo_exp32(-g);
    return g / (1.0f + e);
}

/* h[t][k] = silu(g[t][k]) * u[t][k], packed to Q8_1 like zqo_rmsnorm_q8_1. */
void zqo_silu_mul_q8_1(const float *g, const float *u, int B, int K, int8_t *qs, uint16_t *d16,
                       uint16_t *s16)
{
    for (int t = 0; t < B; ++t) {
        for (int b = 0; b < K / 32; ++b) {
            float h[32];
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                size_t k = (size_t)t * K + 32 * b + i;
                float v = zqo_silu32(g[k]) * u[k];
                h[i] = v;
                if (fabsf(v) > amax) amax = fabsf(v);
            }
            float d = amax / 127.0f;
            float id = (d != 0.0f) ? 1.0f / d : 0.0f;
            int sum = 0;
            for (int i = 0; i < 32; ++i) {
                float q = roundf(h[i] * id); /* half away from zero */
                if (q > 127.0f) q = 127.0f;
                if (q < -127.0f) q = -127.0f;
                qs[(size_t)t * K + 32 * b + i] = (int8_t)q;
                sum += (int)q;
            }
            float s = d * (float)sum;
            d16[(size_t)t * (K / 32) + b] = zqo_f32_to_f16(d);
            s16[(size_t)t * (K / 32) + b] = zqo_f32_to_f16(s);
        }
    }
}

/* ------------------------------------------------------------------------
 * Q4_K super-block decode (MIInfer README, "Status": Q4_K metadata staging
 * decodes the packed 6-bit scales/mins; the layout is the one stated at the
 * top of this file).
 * ---------------------------------------------------------------------- */
void zqo_q4k_unpack(const uint8_t *blk, float *d, float *dmin,
                    uint8_t sc[8], uint8_t m[8], uint8_t q[256])
{
    *d = zqo_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
    *dmin = zqo_f16_to_f32((uint16_t)(blk[2] | (blk[3] << 8)));
    const uint8_t *S = blk + 4;
    for (int j = 0; j < 8; ++j) {
        if (j < 4) {
            sc[j] = S[j] & 63;
            m[j] = S[j + 4] & 63;
        } else {
            sc[j] = (uint8_t)((S[j + 4] & 15) | ((S[j - 4] >> 6) << 4));
            m[j] = (uint8_t)((S[j + 4] >> 4) | ((S[j] >> 6) << 4));
        }
    }
    const uint8_t *Q = blk + 16;
    for (int j = 0; j < 8; ++j)
        for (int i = 0; i < 32; ++i) {
            uint8_t byte = Q[32 * (j / 2) + i];
            q[32 * j + i] = (j % 2 == 0) ? (byte & 15) : (byte >> 4);
        }
}

/* fp64 dequantised weights w[n][k] = d*sc*q - dmin*m (brute-force helper). */
void zqo_q4k_dequant(const uint8_t *W, int N, int K, double *w)
{
    int nb = K / 256;
    for (int n = 0; n < N; ++n)
        for (int b = 0; b < nb; ++b) {
            float d, dmin;
            uint8_t sc[8], m[8], q[256];
            zqo_q4k_unpack(W + ((size_t)n * nb + b) * 144, &d, &dmin, sc, m, q);
            for (int j = 0; j < 8; ++j)
                for (int i = 0; i < 32; ++i)
                    w[(size_t)n * K + 256 * b + 32 * j + i] =
                        (double)d * sc[j] * q[32 * j + i] - (double)dmin * m[j];
        }
}

/* Binary16 dequantised weights, the input of a dequantise-then-GEMM prefill
 * (MIInfer README, "Current phase": Q4_K dequantised to 16-bit weights ahead
 * of a dense GEMM).  In fp32: a = d*sc and b = dmin*m (both exact), then
 * w = a*q - b (a*q exact, one rounding), then w rounded to binary16. */
void zqo_q4k_dequant_f16(const uint8_t *W, int N, int K, uint16_t *w16)
{
    int nb = K / 256;
    for (int n = 0; n < N; ++n)
        for (int b = 0; b < nb; ++b) {
            float d, dmin;
            uint8_t sc[8], m[8], q[256];
            zqo_q4k_unpack(W + ((size_t)n * nb + b) * 144, &d, &dmin, sc, m, q);
            for (int j = 0; j < 8; ++j) {
                float a = d * (float)sc[j];
                float bm = dmin * (float)m[j];
                for (int i = 0; i < 32; ++i) {
                    float w = a * (float)q[32 * j + i] - bm;
                    w16[(size_t)n * K + 256 * b + 32 * j + i] = zqo_f32_to_f16(w);
                }
            }
        }
}

/* Binary16 dequantised activations, the other input of the dequantise-then-
 * GEMM design: x = q8 * d8 in fp32 (exact: 8 x 11 significant bits), then
 * rounded to binary16. */
void zqo_q8_1_dequant_f16(const int8_t *qs, const uint16_t *d16, int B, int K, uint16_t *x16)
{
    for (int t = 0; t < B; ++t)
        for (int k = 0; k < K; ++k) {
            float d = zqo_f16_to_f32(d16[(size_t)t * (K / 32) + k / 32]);
            x16[(size_t)t * K + k] = zqo_f32_to_f16((float)qs[(size_t)t * K + k] * d);
        }
}

/* The dense GEMM of that design on binary16 inputs, by its definition:
 * y[t][r] = sum_k x[t][k] * w[rows[r]][k] in fp64 (each product of two
 * binary16 values is exact in fp64; the fp64 sum rounds at 2^-53 relative,
 * far below the fp32 accumulation it is compared with). */
void zqo_f16_gemm_rows(const uint16_t *x16, const uint16_t *w16, int B, int K, const int *rows, int nrows,
                       double *y)
{
    for (int t = 0; t < B; ++t)
        for (int r = 0; r < nrows; ++r) {
            const uint16_t *wr = w16 + (size_t)rows[r] * K;
            const uint16_t *xt = x16 + (size_t)t * K;
            double acc = 0.0;
            for (int k = 0; k < K; ++k) acc += (double)zqo_f16_to_f32(xt[k]) * (double)zqo_f16_to_f32(wr[k]);
            y[(size_t)t * nrows + r] = acc;
        }
}

/* ------------------------------------------------------------------------
 * Sub-block integer dot sums I[t][n][b*8+j] = sum_i q4 * q8 over the 32
 * weights of sub-block j of super-block b (MIInfer README, "Status": the
 * packed dot4 int8 projection path).
 * ---------------------------------------------------------------------- */
void zqo_q4k_isums(const uint8_t *W, int N, int K, const int8_t *qs, int B,
                   int32_t *I)
{
    int nb = K / 256;
    for (int t = 0; t < B; ++t)
        for (int n = 0; n < N; ++n)
            for (int b = 0; b < nb; ++b) {
                float d, dmin;
                uint8_t sc[8], m[8], q[256];
                zqo_q4k_unpack(W + ((size_t)n * nb + b) * 144, &d, &dmin, sc, m, q);
                for (int j = 0; j < 8; ++j) {
                    int32_t acc = 0;
                    for (int i = 0; i < 32; ++i)
                        acc += (int32_t)q[32 * j + i] *
                               (int32_t)qs[(size_t)t * K + 256 * b + 32 * j + i];
                    I[((size_t)t * N + n) * (K / 32) + 8 * b + j] = acc;
                }
            }
}

/* ------------------------------------------------------------------------
 * The projection y[t][n] for the rows listed in `rows` (all rows when
 * rows == NULL), written to y[t][r] with r the position in the list:
 *   y = sum_b sum_j ( d*sc_j*d8*I - dmin*m_j*s8 ), float part in fp64.
 * Also returns, when S != NULL, the tolerance scale
 *   S[t][r] = sum_k | w_nk * xq_tk |  (fp64),  xq = d8 * q8,
 * the row's sum of |weight x activation| over the dequantised operands.
 * (MIInfer README, "Status": Q4_K x Q8_1 MMVQ-style projections.)
 * ---------------------------------------------------------------------- */
void zqo_q4k_matmul_rows(const uint8_t *W, int N, int K, const int8_t *qs,
                         const uint16_t *d16, const uint16_t *s16, int B,
                         const int32_t *rows, int R, float *y, double *S)
{
    int nb = K / 256;
    for (int t = 0; t < B; ++t)
        for (int r = 0; r < R; ++r) {
            int n = rows ? rows[r] : r;
            double acc = 0.0, abs_acc = 0.0;
            for (int b = 0; b < nb; ++b) {
                float d, dmin;
                uint8_t sc[8], m[8], q[256];
                zqo_q4k_unpack(W + ((size_t)n * nb + b) * 144, &d, &dmin, sc, m, q);
                for (int j = 0; j < 8; ++j) {
                    const int8_t *a = qs + (size_t)t * K + 256 * b + 32 * j;
                    double d8 = zqo_f16_to_f32(d16[(size_t)t * (K / 32) + 8 * b + j]);
                    double s8 = zqo_f16_to_f32(s16[(size_t)t * (K / 32) + 8 * b + j]);
                    int64_t isum = 0;
                    for (int i = 0; i < 32; ++i) isum += (int64_t)q[32 * j + i] * a[i];
                    acc += (double)d * sc[j] * d8 * (double)isum - (double)dmin * m[j] * s8;
                    if (S) {
                        for (int i = 0; i < 32; ++i) {
                            double w = (double)d * sc[j] * q[32 * j + i] - (double)dmin * m[j];
                            abs_acc += fabs(w * (d8 * a[i]));
                        }
                    }
                }
            }
            y[(size_t)t * R + r] = (float)acc;
            if (S) S[(size_t)t * R + r] = abs_acc;
        }
}

void zqo_q4k_matmul(const uint8_t *W, int N, int K, const int8_t *qs,
                    const uint16_t *d16, const uint16_t *s16, int B, float *y,
                    double *S)
{
    zqo_q4k_matmul_rows(W, N, K, qs, d16, s16, B, NULL, N, y, S);
}

/* ------------------------------------------------------------------------
 * Q5_K and Q6_K: the other k-quant blocks of a Q4_K_M checkpoint (MIInfer
 * README, "Status": Q5_K x Q8_1 MMVQ-style recurrent output projection,
 * Q5_K scale/min hoisting and paired nibbles; MMVQ-style Q6_K x Q8_1 LM
 * head; ZINC docs "ROCm backend": packed Q8 activations feed the hot Q4_K,
 * Q5_K and Q6_K projections).  As for Q4_K, the pages name the formats but
 * print no byte layout; the layouts below are the readings used throughout:
 *
 *   Q5_K super-block (256 weights, 176 bytes):
 *     bytes 0..15   d, dmin and the twelve scale/min bytes, exactly as Q4_K;
 *     bytes 16..47  qh: bit j of byte 16+i is bit 4 of weight i of
 *                   sub-block j;
 *     bytes 48..175 the low four bits of the quants, placed as the Q4_K
 *                   nibbles (byte 48 + 32*(j/2) + i, low nibble for even j).
 *     w = d*sc[j]*q - dmin*m[j], q in 0..31.
 *
 *   Q6_K super-block (256 weights, 210 bytes; sixteen sub-blocks of 16):
 *     weight k: h = k/128, c = (k%128)/32, i = k%32;
 *     bytes 0..127   low four bits of q in byte 64h + 32(c%2) + i, low
 *                    nibble for c < 2, high nibble for c >= 2;
 *     bytes 128..191 top two bits of q in bits 2c, 2c+1 of byte 128 + 32h + i;
 *     bytes 192..207 sixteen int8 scales, sc[s] for weights 16s..16s+15;
 *     bytes 208..209 d (binary16).
 *     w = d*sc[k/16]*(q - 32), q in 0..63.
 *
 *   Output, per token t and row n, with exact integer sub-block sums:
 *     Q5_K: as Q4_K, y = sum_b sum_j d*sc_j*d8*I_j - dmin*m_j*s8,
 *           I_j = sum over the 32 weights of q5*q8;
 *     Q6_K: y = sum_b sum_s d*sc_s*d8_{t,k/32}*I_s,
 *           I_s = sum over the 16 weights of (q6 - 32)*q8;
 *   the float part accumulated in fp64.  S[t][r] = sum_k |w*xq| as for Q4_K.
 * ---------------------------------------------------------------------- */
void zqo_q5k_unpack(const uint8_t *blk, float *d, float *dmin,
                    uint8_t sc[8], uint8_t m[8], uint8_t q[256])
{
    /* bytes 0..15 and the low bits share the Q4_K reading; rebuild a Q4_K
     * block from them and add the fifth bit */
    uint8_t q4[144];
    memcpy(q4, blk, 16);
    memcpy(q4 + 16, blk + 48, 128);
    zqo_q4k_unpack(q4, d, dmin, sc, m, q);
    const uint8_t *QH = blk + 16;
    for (int j = 0; j < 8; ++j)
        for (int i = 0; i < 32; ++i)
            q[32 * j + i] = (uint8_t)(q[32 * j + i] | (((QH[i] >> j) & 1) << 4));
}

void zqo_q6k_unpack(const uint8_t *blk, float *d, int8_t sc[16], uint8_t q[256])
{
    for (int k = 0; k < 256; ++k) {
        int h = k / 128, c = (k % 128) / 32, i = k % 32;
        uint8_t lb = blk[64 * h + 32 * (c % 2) + i];
        uint8_t low = (c < 2) ? (lb & 15) : (lb >> 4);
        uint8_t top = (blk[128 + 32 * h + i] >> (2 * c)) & 3;
        q[k] = (uint8_t)(low | (top << 4));
    }
    for (int s = 0; s < 16; ++s) sc[s] = (int8_t)blk[192 + s];
    *d = zqo_f16_to_f32((uint16_t)(blk[208] | (blk[209] << 8)));
}

void zqo_q5k_dequant(const uint8_t *W, int N, int K, double *w)
{
    int nb = K / 256;
    for (int n = 0; n < N; ++n)
        for (int b = 0; b < nb; ++b) {
            float d, dmin;
            uint8_t sc[8], m[8], q[256];
            zqo_q5k_unpack(W + ((size_t)n * nb + b) * 176, &d, &dmin, sc, m, q);
            for (int k = 0; k < 256; ++k)
                w[(size_t)n * K + 256 * b + k] = (double)d * sc[k / 32] * q[k] - (double)dmin * m[k / 32];
        }
}

void zqo_q6k_dequant(const uint8_t *W, int N, int K, double *w)
{
    int nb = K / 256;
    for (int n = 0; n < N; ++n)
        for (int b = 0; b < nb; ++b) {
            float d;
            int8_t sc[16];
            uint8_t q[256];
            zqo_q6k_unpack(W + ((size_t)n * nb + b) * 210, &d, sc, q);
            for (int k = 0; k < 256; ++k)
                w[(size_t)n * K + 256 * b + k] = (double)d * sc[k / 16] * ((int)q[k] - 32);
        }
}

/* Projection of a Q5_K matrix, rows and outputs as zqo_q4k_matmul_rows. */
void zqo_q5k_matmul_rows(const uint8_t *W, int N, int K, const int8_t *qs,
                         const uint16_t *d16, const uint16_t *s16, int B,
                         const int32_t *rows, int R, float *y, double *S)
{
    int nb = K / 256;
    for (int t = 0; t < B; ++t)
        for (int r = 0; r < R; ++r) {
            int n = rows ? rows[r] : r;
            double acc = 0.0, abs_acc = 0.0;
            for (int b = 0; b < nb; ++b) {
                float d, dmin;
                uint8_t sc[8], m[8], q[256];
                zqo_q5k_unpack(W + ((size_t)n * nb + b) * 176, &d, &dmin, sc, m, q);
                for (int j = 0; j < 8; ++j) {
                    const int8_t *a = qs + (size_t)t * K + 256 * b + 32 * j;
                    double d8 = zqo_f16_to_f32(d16[(size_t)t * (K / 32) + 8 * b + j]);
                    double s8 = zqo_f16_to_f32(s16[(size_t)t * (K / 32) + 8 * b + j]);
                    int64_t isum = 0;
                    for (int i = 0; i < 32; ++i) isum += (int64_t)q[32 * j + i] * a[i];
                    acc += (double)d * sc[j] * d8 * (double)isum - (double)dmin * m[j] * s8;
                    if (S) {
                        for (int i = 0; i < 32; ++i) {
                            double w = (double)d * sc[j] * q[32 * j + i] - (double)dmin * m[j];
                            abs_acc += fabs(w * (d8 * a[i]));
                        }
                    }
                }
            }
            y[(size_t)t * R + r] = (float)acc;
            if (S) S[(size_t)t * R + r] = abs_acc;
        }
}

/* Projection of a Q6_K matrix; s16 is not used (the Q6_K offset is inside
 * the integer sums). */
void zqo_q6k_matmul_rows(const uint8_t *W, int N, int K, const int8_t *qs,
                         const uint16_t *d16, int B,
                         const int32_t *rows, int R, float *y, double *S)
{
    int nb = K / 256;
    for (int t = 0; t < B; ++t)
        for (int r = 0; r < R; ++r) {
            int n = rows ? rows[r] : r;
            double acc = 0.0, abs_acc = 0.0;
            for (int b = 0; b < nb; ++b) {
                float d;
                int8_t sc[16];
                uint8_t q[256];
                zqo_q6k_unpack(W + ((size_t)n * nb + b) * 210, &d, sc, q);
                for (int sb = 0; sb < 16; ++sb) {
                    const int8_t *a = qs + (size_t)t * K + 256 * b + 16 * sb;
                    double d8 = zqo_f16_to_f32(d16[(size_t)t * (K / 32) + 8 * b + sb / 2]);
                    int64_t isum = 0;
                    for (int i = 0; i < 16; ++i) isum += (int64_t)((int)q[16 * sb + i] - 32) * a[i];
                    acc += (double)d * sc[sb] * d8 * (double)isum;
                    if (S) {
                        for (int i = 0; i < 16; ++i) {
                            double w = (double)d * sc[sb] * ((int)q[16 * sb + i] - 32);
                            abs_acc += fabs(w * (d8 * a[i]));
                        }
                    }
                }
            }
            y[(size_t)t * R + r] = (float)acc;
            if (S) S[(size_t)t * R + r] = abs_acc;
        }
}

int zqo_version(void) { return 1; }
