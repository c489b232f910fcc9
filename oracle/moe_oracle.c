/*
 * moe_oracle.c -- plain, slow, obviously-correct CPU oracle for the sparse
 * mixture-of-experts layer over Q4_K block-quantised expert weights.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test-suite, the smoke
 * check and the CPU-baseline leg of the benchmark may load this library.  It
 * shares no source, header, table or helper with the CUDA path; the two meet
 * only through the seeded synthetic inputs.
 *
 * Pages this follows (cited by page title and section):
 *  [DSV4]  "【瞎折腾】Strata 改源码去跑 DeepSeek V4 Flash？要不就试试！"
 *          (lcz.me/post/23082).
 *          - section 二 ("实测 A"), GGUF anatomy table: routed experts are the
 *            fused 3-D tensors ffn_{gate,up,down}_exps, all listed with the one
 *            shape 256x2048x4096, quantised Q4_K; the remaining matrices
 *            (shared expert, small projections) are Q8_0; 256 routed experts
 *            plus 1 shared expert, 6 active; "router bias" on most layers.
 *          - section 三 item 4: the per-expert blob constant 1,382,400 bytes at
 *            hidden width 2560 = 3 matrices x 2560 x 320 x 4.5 bits, i.e. 144
 *            bytes per 256 weights and expert FF = 320.
 *  [TEAR]  "Strata 引擎深度拆解：125B MoE 跑进 2×3090 + EPYC" (lcz.me/topic/2098/5).
 *          - section 二 ("架构拆解"): 48 layers x 512 experts, about 10 experts
 *            active per token; a verify window of 3-5 drafted tokens runs as
 *            one forward.
 *          - section 一, CPU ledger: the multi-token expert kernel computes an
 *            expert once for all tokens of a window.
 *  [GAP]   the "Gap" post on lcz.me/user/lunarmoon26/best, item 6 (正确性与长上下文):
 *          the correctness baseline turns off expert skipping and
 *          cache-aware routing bias -- strict top-k routing.
 *
 * The pages print no byte layout, formula or pseudo-code for Q4_K, Q8_0, the
 * router, top-k, bucketing or the expert FFN.  The readings taken here (the
 * plainest ones the rest of the pages support) are:
 *  R1  Q4_K super-block, 144 bytes for 256 weights = 8 sub-blocks of 32:
 *        bytes 0-1 d (fp16, little endian), 2-3 dmin (fp16), 4-15 scales[12],
 *        16-143 qs[128].
 *      6-bit sub-block scale sc_j and min m_j:
 *        j < 4 : sc_j = scales[j] & 63,  m_j = scales[j+4] & 63
 *        j >= 4: sc_j = (scales[j+4] & 15) | ((scales[j-4] >> 6) << 4)
 *                m_j  = (scales[j+4] >> 4) | ((scales[j]   >> 6) << 4)
 *      4-bit quants: for c in 0..3 and l in 0..31, byte qs[32c+l] holds the
 *      quant of element 64c+l in its low nibble and of element 64c+32+l in its
 *      high nibble.
 *      Value: y = fp32(fp32(d)*sc_j) * q - fp32(fp32(dmin)*m_j), every product
 *      and the difference rounded to fp32 on its own (no fused multiply-add).
 *  R2  Q4_K quantiser (deterministic, fp32 IEEE, round-half-even):
 *        per sub-block mn = min(0, min x), mx = max x,
 *                      scale_j = (mx - mn) / 15, nmin_j = -mn;
 *        d = fp16(max_j scale_j / 63), dmin = fp16(max_j nmin_j / 63);
 *        sc_j = d > 0 ? min(63, rint(scale_j / d)) : 0   (m_j alike with dmin);
 *        s = d*sc_j, z = dmin*m_j, q = s > 0 ? clamp(rint((x + z) / s), 0, 15) : 0.
 *      A non-finite input, or a d / dmin that overflows fp16, is an error.
 *  R3  Q8_0 block, 34 bytes for 32 weights: fp16 d then 32 int8 quants;
 *        d = fp16(max|x| / 127), q = d > 0 ? clamp(rint(x / d), -127, 127) : 0,
 *        y = fp32(d * q).
 *  R4  Expert blob = [gate FF x H][up FF x H][down FF x H], every matrix stored
 *      row-major with its Q4_K super-blocks along H.  Down is stored [FF][H]
 *      (the same shape the anatomy table lists for all three tensors, and the
 *      only orientation that keeps the 1,382,400-byte blob at FF = 320) and is
 *      applied as o[h] = sum_f a[f] * Wd[f][h].
 *  R5  Activation a = SiLU(g) * u with SiLU(g) = g / (1 + exp(-g)).
 *  R6  Router logits l_e = sum_h x_h * Wr[e][h] (x bf16, Wr fp32; exact in fp64).
 *      softmax scoring: p = softmax(l); the k largest p are selected;
 *        weights w_r = p_{e_r} / sum_selected p (renormalised over the k).
 *      sigmoid scoring: s_e = 1 / (1 + exp(-l_e)); the k largest s_e + b_e are
 *        selected; weights w_r = s_{e_r} / sum_selected s (bias is for selection
 *        only).
 *      Selection is in descending score order; equal scores go to the lower id.
 *  R7  Bucketing is a stable counting sort of the T*k assignments (value t*k+r)
 *      by expert id: counts[E], offsets[E+1] (exclusive prefix), and within an
 *      expert the assignments stay in ascending t.
 *  R8  y_t = sum_r w_r * o_{t,r} over r ascending, plus (when present) the
 *      always-on shared expert's FFN of x_t with weight 1 and Q8_0 weights.
 *
 *  R9  Tensor-core operand rounding of the dequantised weights (the GPU path
 *      multiplies fp16 weights; the pages fix no precision, so this is the
 *      rounding the GPU path states for itself, written out here so that its
 *      fused dequantisation can be checked bit for bit):
 *        Q4_K: S_j = fp16(d*sc_j), NZ_j = fp16(-(dmin*m_j)) (each product exact
 *              in fp32, rounded once to fp16), w = fp16(q*S_j + NZ_j) with the
 *              sum taken exactly and rounded once;
 *        Q8_0: w = fp16(d*q) (exact product, rounded once).
 *  R10 Q5_K super-block, 176 bytes for 256 weights (the pages' deployments mix
 *      Q4_K and Q5_K experts): bytes 0-1 d (fp16), 2-3 dmin (fp16), 4-15
 *      scales[12] packed as in R1, 16-47 qh[32], 48-175 qs[128].  Quant of
 *      element 64c + 32h + l (c in 0..3, h in 0..1, l in 0..31): its low four
 *      bits are the low (h = 0) or high (h = 1) nibble of qs[32c + l], its
 *      fifth bit is bit 2c + h of qh[l]; q in 0..31.  Value as R1:
 *      y = fp32(fp32(d)*sc_j) * q - fp32(fp32(dmin)*m_j), j = 2c + h.
 *  R11 Q5_K quantiser: R2 with 31 levels -- scale_j = (mx - mn) / 31,
 *      q = s > 0 ? clamp(rint((x + z) / s), 0, 31) : 0; the rest as R2.
 *      Operand rounding of the tensor-core paths as R9 (q up to 31 is exact).
 *
 * Precision: quantise/dequantise in fp32 exactly as R1-R3 state; router,
 * scores, weights and every FFN product and sum in fp64.
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -fopenmp -ffp-contract=off
 * (no -ffast-math: the fp32 steps must round as IEEE single precision).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_QK_K 256            /* weights per Q4_K super-block            */
#define ORC_Q4K_BYTES 144       /* 2 + 2 + 12 + 128                        */
#define ORC_Q5K_BYTES 176       /* 2 + 2 + 12 + 32 + 128                   */
#define ORC_QK8 32              /* weights per Q8_0 block                  */
#define ORC_Q8_BYTES 34         /* 2 + 32                                  */

/* ------------------------------------------------------------------ */
/* scalar conversions                                                  */
/* ------------------------------------------------------------------ */

static float bits_to_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f32_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* bf16 -> fp32: the bf16 bits are the upper half of the fp32 bits. */
float orc_bf16_to_f32(uint16_t b) { return bits_to_f32((uint32_t)b << 16); }

/* IEEE binary16 -> fp32, from the field definitions (exact). */
float orc_f16_to_f32(uint16_t h)
{
    int sign = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 31) return m ? NAN : (sign ? -INFINITY : INFINITY);
    if (e == 0) v = ldexp((double)m, -24);              /* subnormal: m * 2^-24 */
    else v = ldexp((double)(1024 + m), e - 25);          /* 1.m * 2^(e-15)       */
    return (float)(sign ? -v : v);
}

/* fp32 -> IEEE binary16, round to nearest, ties to even.  The magnitude is
 * divided by the fp16 ulp of its binade (exact: a power of two) and rounded
 * with rint(), which rounds half to even in the default rounding mode. */
uint16_t orc_f32_to_f16(float f)
{
    uint16_t sign = (uint16_t)((f32_to_bits(f) >> 16) & 0x8000u);
    if (isnan(f)) return 0x7e00;
    if (isinf(f)) return sign | 0x7c00;
    double a = fabs((double)f);
    if (a == 0.0) return sign;
    int e2;
    frexp(a, &e2);                 /* a in [2^(e2-1), 2^e2) */
    int ex = e2 - 1;
    if (ex < -14) ex = -14;        /* subnormals share the ulp 2^-24 */
    double ulp = ldexp(1.0, ex - 10);
    double r = rint(a / ulp);      /* in [0, 2048] */
    if (r >= 2048.0) { r = 1024.0; ex += 1; }   /* carried into the next binade */
    if (ex > 15) return sign | 0x7c00;           /* overflow -> infinity */
    if (r < 1024.0) return sign | (uint16_t)r;   /* subnormal (ex == -14) */
    return sign | (uint16_t)(((ex + 15) << 10) | ((int)r - 1024));
}

/* fp64 -> IEEE binary16, round to nearest, ties to even: the same steps as
 * orc_f32_to_f16 applied to a double, for values that need more than fp32 to
 * be held exactly before their one rounding (R9). */
uint16_t orc_f64_to_f16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    if (isnan(v)) return 0x7e00;
    if (isinf(v)) return sign | 0x7c00;
    double a = fabs(v);
    if (a == 0.0) return sign;
    int e2;
    frexp(a, &e2);
    int ex = e2 - 1;
    if (ex < -14) ex = -14;
    double ulp = ldexp(1.0, ex - 10);
    double r = rint(a / ulp);
    if (r >= 2048.0) { r = 1024.0; ex += 1; }
    if (ex > 15) return sign | 0x7c00;
    if (r < 1024.0) return sign | (uint16_t)r;
    return sign | (uint16_t)(((ex + 15) << 10) | ((int)r - 1024));
}

/* ------------------------------------------------------------------ */
/* Q4_K (R1, R2)                                                       */
/* ------------------------------------------------------------------ */

static void q4k_get_scale_min(const uint8_t *scales, int j, int *sc, int *m)
{
    if (j < 4) {
        *sc = scales[j] & 63;
        *m = scales[j + 4] & 63;
    } else {
        *sc = (scales[j + 4] & 15) | ((scales[j - 4] >> 6) << 4);
        *m = (scales[j + 4] >> 4) | ((scales[j] >> 6) << 4);
    }
}

/* Quantise 256 fp32 weights into one 144-byte block.  0 on success, -1 when
 * an input is non-finite or d / dmin overflows fp16. */
int orc_q4k_quantize_block(const float *x, uint8_t *blk)
{
    float scale[8], nmin[8];
    for (int j = 0; j < 8; ++j) {
        const float *s = x + 32 * j;
        float mn = s[0], mx = s[0];
        for (int i = 0; i < 32; ++i) {
            if (!isfinite(s[i])) return -1;
            if (s[i] < mn) mn = s[i];
            if (s[i] > mx) mx = s[i];
        }
        if (mn > 0.0f) mn = 0.0f;
        scale[j] = (mx - mn) / 15.0f;
        nmin[j] = -mn;
    }
    float max_scale = 0.0f, max_nmin = 0.0f;
    for (int j = 0; j < 8; ++j) {
        if (scale[j] > max_scale) max_scale = scale[j];
        if (nmin[j] > max_nmin) max_nmin = nmin[j];
    }
    uint16_t d_h = orc_f32_to_f16(max_scale / 63.0f);
    uint16_t dmin_h = orc_f32_to_f16(max_nmin / 63.0f);
    float d = orc_f16_to_f32(d_h), dmin = orc_f16_to_f32(dmin_h);
    if (!isfinite(d) || !isfinite(dmin)) return -1;

    int sc[8], m[8];
    for (int j = 0; j < 8; ++j) {
        sc[j] = d > 0.0f ? (int)fminf(63.0f, rintf(scale[j] / d)) : 0;
        m[j] = dmin > 0.0f ? (int)fminf(63.0f, rintf(nmin[j] / dmin)) : 0;
    }

    memset(blk, 0, ORC_Q4K_BYTES);
    blk[0] = (uint8_t)(d_h & 0xff);
    blk[1] = (uint8_t)(d_h >> 8);
    blk[2] = (uint8_t)(dmin_h & 0xff);
    blk[3] = (uint8_t)(dmin_h >> 8);
    uint8_t *scales = blk + 4;
    for (int j = 0; j < 4; ++j) {
        scales[j] = (uint8_t)(sc[j] | ((sc[j + 4] >> 4) << 6));
        scales[j + 4] = (uint8_t)(m[j] | ((m[j + 4] >> 4) << 6));
        scales[j + 8] = (uint8_t)((sc[j + 4] & 15) | ((m[j + 4] & 15) << 4));
    }

    uint8_t q[ORC_QK_K];
    for (int j = 0; j < 8; ++j) {
        float s = d * (float)sc[j];
        float z = dmin * (float)m[j];
        for (int i = 0; i < 32; ++i) {
            int qi = 0;
            if (s > 0.0f) {
                float v = rintf((x[32 * j + i] + z) / s);
                qi = v < 0.0f ? 0 : (v > 15.0f ? 15 : (int)v);
            }
            q[32 * j + i] = (uint8_t)qi;
        }
    }
    uint8_t *qs = blk + 16;
    for (int c = 0; c < 4; ++c)
        for (int l = 0; l < 32; ++l)
            qs[32 * c + l] = (uint8_t)(q[64 * c + l] | (q[64 * c + 32 + l] << 4));
    return 0;
}

/* Dequantise one 144-byte block into 256 fp32 weights (R1). */
void orc_q4k_dequantize_block(const uint8_t *blk, float *y)
{
    float d = orc_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
    float dmin = orc_f16_to_f32((uint16_t)(blk[2] | (blk[3] << 8)));
    const uint8_t *scales = blk + 4, *qs = blk + 16;
    for (int c = 0; c < 4; ++c) {
        for (int half = 0; half < 2; ++half) {
            int j = 2 * c + half, sc, m;
            q4k_get_scale_min(scales, j, &sc, &m);
            float s = d * (float)sc;
            float z = dmin * (float)m;
            for (int l = 0; l < 32; ++l) {
                int q = half ? (qs[32 * c + l] >> 4) : (qs[32 * c + l] & 15);
                float t = s * (float)q;
                y[64 * c + 32 * half + l] = t - z;
            }
        }
    }
}

/* Row-major [rows][cols] fp32 -> [rows][cols/256] blocks.  0 / -1 (bad shape
 * or non-finite input). */
int orc_q4k_quantize(const float *w, int64_t rows, int64_t cols, uint8_t *out)
{
    if (rows < 0 || cols <= 0 || cols % ORC_QK_K) return -1;
    int64_t nb = rows * (cols / ORC_QK_K);
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t b = 0; b < nb; ++b)
        bad |= orc_q4k_quantize_block(w + b * ORC_QK_K, out + b * ORC_Q4K_BYTES) != 0;
    return bad ? -1 : 0;
}

void orc_q4k_dequantize(const uint8_t *blob, int64_t rows, int64_t cols, float *out)
{
    int64_t nb = rows * (cols / ORC_QK_K);
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nb; ++b)
        orc_q4k_dequantize_block(blob + b * ORC_Q4K_BYTES, out + b * ORC_QK_K);
}

/* ------------------------------------------------------------------ */
/* Q5_K (R10, R11)                                                     */
/* ------------------------------------------------------------------ */

/* Quantise 256 fp32 weights into one 176-byte block.  0 / -1 as Q4_K. */
int orc_q5k_quantize_block(const float *x, uint8_t *blk)
{
    float scale[8], nmin[8];
    for (int j = 0; j < 8; ++j) {
        const float *s = x + 32 * j;
        float mn = s[0], mx = s[0];
        for (int i = 0; i < 32; ++i) {
            if (!isfinite(s[i])) return -1;
            if (s[i] < mn) mn = s[i];
            if (s[i] > mx) mx = s[i];
        }
        if (mn > 0.0f) mn = 0.0f;
        scale[j] = (mx - mn) / 31.0f;
        nmin[j] = -mn;
    }
    float max_scale = 0.0f, max_nmin = 0.0f;
    for (int j = 0; j < 8; ++j) {
        if (scale[j] > max_scale) max_scale = scale[j];
        if (nmin[j] > max_nmin) max_nmin = nmin[j];
    }
    uint16_t d_h = orc_f32_to_f16(max_scale / 63.0f);
    uint16_t dmin_h = orc_f32_to_f16(max_nmin / 63.0f);
    float d = orc_f16_to_f32(d_h), dmin = orc_f16_to_f32(dmin_h);
    if (!isfinite(d) || !isfinite(dmin)) return -1;

    int sc[8], m[8];
    for (int j = 0; j < 8; ++j) {
        sc[j] = d > 0.0f ? (int)fminf(63.0f, rintf(scale[j] / d)) : 0;
        m[j] = dmin > 0.0f ? (int)fminf(63.0f, rintf(nmin[j] / dmin)) : 0;
    }

    memset(blk, 0, ORC_Q5K_BYTES);
    blk[0] = (uint8_t)(d_h & 0xff);
    blk[1] = (uint8_t)(d_h >> 8);
    blk[2] = (uint8_t)(dmin_h & 0xff);
    blk[3] = (uint8_t)(dmin_h >> 8);
    uint8_t *scales = blk + 4;
    for (int j = 0; j < 4; ++j) {
        scales[j] = (uint8_t)(sc[j] | ((sc[j + 4] >> 4) << 6));
        scales[j + 4] = (uint8_t)(m[j] | ((m[j + 4] >> 4) << 6));
        scales[j + 8] = (uint8_t)((sc[j + 4] & 15) | ((m[j + 4] & 15) << 4));
    }

    uint8_t q[ORC_QK_K];
    for (int j = 0; j < 8; ++j) {
        float s = d * (float)sc[j];
        float z = dmin * (float)m[j];
        for (int i = 0; i < 32; ++i) {
            int qi = 0;
            if (s > 0.0f) {
                float v = rintf((x[32 * j + i] + z) / s);
                qi = v < 0.0f ? 0 : (v > 31.0f ? 31 : (int)v);
            }
            q[32 * j + i] = (uint8_t)qi;
        }
    }
    uint8_t *qh = blk + 16, *qs = blk + 48;
    for (int c = 0; c < 4; ++c)
        for (int h = 0; h < 2; ++h)
            for (int l = 0; l < 32; ++l) {
                const int v = q[64 * c + 32 * h + l];
                qs[32 * c + l] |= (uint8_t)((v & 15) << (4 * h));
                qh[l] |= (uint8_t)(((v >> 4) & 1) << (2 * c + h));
            }
    return 0;
}

/* The quant of element 64c + 32h + l of a Q5_K block (R10). */
static int q5k_quant(const uint8_t *blk, int c, int h, int l)
{
    const uint8_t *qh = blk + 16, *qs = blk + 48;
    const int lo = h ? (qs[32 * c + l] >> 4) : (qs[32 * c + l] & 15);
    return lo | (((qh[l] >> (2 * c + h)) & 1) << 4);
}

/* Dequantise one 176-byte block into 256 fp32 weights (R10). */
void orc_q5k_dequantize_block(const uint8_t *blk, float *y)
{
    float d = orc_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
    float dmin = orc_f16_to_f32((uint16_t)(blk[2] | (blk[3] << 8)));
    for (int c = 0; c < 4; ++c)
        for (int h = 0; h < 2; ++h) {
            int sc, m;
            q4k_get_scale_min(blk + 4, 2 * c + h, &sc, &m);
            float s = d * (float)sc;
            float z = dmin * (float)m;
            for (int l = 0; l < 32; ++l) {
                float t = s * (float)q5k_quant(blk, c, h, l);
                y[64 * c + 32 * h + l] = t - z;
            }
        }
}

int orc_q5k_quantize(const float *w, int64_t rows, int64_t cols, uint8_t *out)
{
    if (rows < 0 || cols <= 0 || cols % ORC_QK_K) return -1;
    int64_t nb = rows * (cols / ORC_QK_K);
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t b = 0; b < nb; ++b)
        bad |= orc_q5k_quantize_block(w + b * ORC_QK_K, out + b * ORC_Q5K_BYTES) != 0;
    return bad ? -1 : 0;
}

void orc_q5k_dequantize(const uint8_t *blob, int64_t rows, int64_t cols, float *out)
{
    int64_t nb = rows * (cols / ORC_QK_K);
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nb; ++b)
        orc_q5k_dequantize_block(blob + b * ORC_Q5K_BYTES, out + b * ORC_QK_K);
}

/* ------------------------------------------------------------------ */
/* Q8_0 (R3)                                                           */
/* ------------------------------------------------------------------ */

int orc_q8_0_quantize_block(const float *x, uint8_t *blk)
{
    float amax = 0.0f;
    for (int i = 0; i < ORC_QK8; ++i) {
        if (!isfinite(x[i])) return -1;
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    uint16_t d_h = orc_f32_to_f16(amax / 127.0f);
    float d = orc_f16_to_f32(d_h);
    if (!isfinite(d)) return -1;
    blk[0] = (uint8_t)(d_h & 0xff);
    blk[1] = (uint8_t)(d_h >> 8);
    for (int i = 0; i < ORC_QK8; ++i) {
        int q = 0;
        if (d > 0.0f) {
            float v = rintf(x[i] / d);
            q = v < -127.0f ? -127 : (v > 127.0f ? 127 : (int)v);
        }
        blk[2 + i] = (uint8_t)(int8_t)q;
    }
    return 0;
}

void orc_q8_0_dequantize_block(const uint8_t *blk, float *y)
{
    float d = orc_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
    for (int i = 0; i < ORC_QK8; ++i) y[i] = d * (float)(int8_t)blk[2 + i];
}

int orc_q8_0_quantize(const float *w, int64_t rows, int64_t cols, uint8_t *out)
{
    if (rows < 0 || cols <= 0 || cols % ORC_QK8) return -1;
    int64_t nb = rows * (cols / ORC_QK8);
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t b = 0; b < nb; ++b)
        bad |= orc_q8_0_quantize_block(w + b * ORC_QK8, out + b * ORC_Q8_BYTES) != 0;
    return bad ? -1 : 0;
}

void orc_q8_0_dequantize(const uint8_t *blob, int64_t rows, int64_t cols, float *out)
{
    int64_t nb = rows * (cols / ORC_QK8);
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nb; ++b)
        orc_q8_0_dequantize_block(blob + b * ORC_Q8_BYTES, out + b * ORC_QK8);
}

/* ------------------------------------------------------------------ */
/* fp16 operand rounding of the dequantised weights (R9)               */
/* ------------------------------------------------------------------ */

/* One Q4_K block -> 256 binary16 bit patterns: per sub-block j the scale
 * and negated min rounded to fp16, then q*S + NZ taken exactly (every term
 * fits a double) and rounded once. */
void orc_q4k_dequantize_f16_block(const uint8_t *blk, uint16_t *y)
{
    float d = orc_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
    float dmin = orc_f16_to_f32((uint16_t)(blk[2] | (blk[3] << 8)));
    const uint8_t *scales = blk + 4, *qs = blk + 16;
    for (int c = 0; c < 4; ++c) {
        for (int half = 0; half < 2; ++half) {
            int j = 2 * c + half, sc, m;
            q4k_get_scale_min(scales, j, &sc, &m);
            double S = orc_f16_to_f32(orc_f32_to_f16(d * (float)sc));       /* d*sc exact in fp32 */
            double NZ = orc_f16_to_f32(orc_f32_to_f16(-(dmin * (float)m)));
            for (int l = 0; l < 32; ++l) {
                int q = half ? (qs[32 * c + l] >> 4) : (qs[32 * c + l] & 15);
                y[64 * c + 32 * half + l] = orc_f64_to_f16((double)q * S + NZ);
            }
        }
    }
}

void orc_q4k_dequantize_f16(const uint8_t *blob, int64_t rows, int64_t cols, uint16_t *out)
{
    int64_t nb = rows * (cols / ORC_QK_K);
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nb; ++b)
        orc_q4k_dequantize_f16_block(blob + b * ORC_Q4K_BYTES, out + b * ORC_QK_K);
}

/* One Q8_0 block -> 32 binary16 patterns fp16(d*q) (d*q exact in fp32). */
/* R9 applied to a Q5_K block (R10): S, NZ as for Q4_K, w = fp16(q*S + NZ). */
void orc_q5k_dequantize_f16_block(const uint8_t *blk, uint16_t *y)
{
    float d = orc_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
    float dmin = orc_f16_to_f32((uint16_t)(blk[2] | (blk[3] << 8)));
    for (int c = 0; c < 4; ++c)
        for (int h = 0; h < 2; ++h) {
            int sc, m;
            q4k_get_scale_min(blk + 4, 2 * c + h, &sc, &m);
            const double S = (double)orc_f16_to_f32(orc_f64_to_f16((double)d * (double)sc));
            const double NZ = (double)orc_f16_to_f32(orc_f64_to_f16(-((double)dmin * (double)m)));
            for (int l = 0; l < 32; ++l)
                y[64 * c + 32 * h + l] = orc_f64_to_f16((double)q5k_quant(blk, c, h, l) * S + NZ);
        }
}

void orc_q5k_dequantize_f16(const uint8_t *blob, int64_t rows, int64_t cols, uint16_t *out)
{
    int64_t nb = rows * (cols / ORC_QK_K);
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nb; ++b)
        orc_q5k_dequantize_f16_block(blob + b * ORC_Q5K_BYTES, out + b * ORC_QK_K);
}

void orc_q8_0_dequantize_f16(const uint8_t *blob, int64_t rows, int64_t cols, uint16_t *out)
{
    int64_t nb = rows * (cols / ORC_QK8);
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nb; ++b) {
        const uint8_t *blk = blob + b * ORC_Q8_BYTES;
        float d = orc_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
        for (int i = 0; i < ORC_QK8; ++i)
            out[b * ORC_QK8 + i] = orc_f32_to_f16(d * (float)(int8_t)blk[2 + i]);
    }
}

/* ------------------------------------------------------------------ */
/* Router, top-k and weights (R6)                                      */
/* ------------------------------------------------------------------ */

enum { ORC_SCORE_SOFTMAX = 0, ORC_SCORE_SIGMOID_BIAS = 1 };

/* Logits, scores and selection keys of one token, all in fp64. */
static void token_scores(const uint16_t *xt, const float *wr, const float *bias, int H, int E,
                         int score_fn, double *score, double *key)
{
    double lmax = -INFINITY;
    for (int e = 0; e < E; ++e) {
        double l = 0.0;
        for (int h = 0; h < H; ++h)
            l += (double)orc_bf16_to_f32(xt[h]) * (double)wr[(int64_t)e * H + h];
        score[e] = l;
        if (l > lmax) lmax = l;
    }
    if (score_fn == ORC_SCORE_SOFTMAX) {
        double z = 0.0;
        for (int e = 0; e < E; ++e) {
            score[e] = exp(score[e] - lmax);
            z += score[e];
        }
        for (int e = 0; e < E; ++e) {
            score[e] /= z;                       /* p_e */
            key[e] = score[e];
        }
    } else {
        for (int e = 0; e < E; ++e) {
            score[e] = 1.0 / (1.0 + exp(-score[e]));   /* s_e */
            key[e] = score[e] + (bias ? (double)bias[e] : 0.0);
        }
    }
}

/* The k largest keys in descending order, equal keys to the lower id: k
 * rounds of a linear scan for the largest key not yet taken (a strict '>'
 * over ascending e keeps the first, i.e. lowest, id among equals).  Also
 * returns the best key left over (the (k+1)-th), -inf when none. */
static double select_topk(const double *key, int E, int k, int32_t *ids, unsigned char *taken)
{
    memset(taken, 0, (size_t)E);
    for (int r = 0; r < k; ++r) {
        int best = -1;
        for (int e = 0; e < E; ++e)
            if (!taken[e] && (best < 0 || key[e] > key[best])) best = e;
        ids[r] = best;
        taken[best] = 1;
    }
    double next = -INFINITY;
    for (int e = 0; e < E; ++e)
        if (!taken[e] && key[e] > next) next = key[e];
    return next;
}

/*
 * Route T tokens: ids[T*k], weights w[T*k] (fp64); kth_key[T] and next_key[T]
 * receive the k-th selected key and the best unselected key (for near-tie
 * reporting).  When forced_ids is given the selection is taken from it and
 * only the weights are computed.  Returns 0, or -1 for bad arguments.
 */
int orc_route(const uint16_t *x, const float *wr, const float *bias, int64_t T, int H, int E,
              int k, int score_fn, const int32_t *forced_ids, int32_t *ids, double *w,
              double *kth_key, double *next_key)
{
    if (T < 0 || H <= 0 || E <= 0 || k <= 0 || k > E) return -1;
    if (score_fn != ORC_SCORE_SOFTMAX && score_fn != ORC_SCORE_SIGMOID_BIAS) return -1;
    int bad = 0;
#pragma omp parallel reduction(| : bad)
    {
        double *score = malloc(sizeof(double) * (size_t)E);
        double *key = malloc(sizeof(double) * (size_t)E);
        unsigned char *taken = malloc((size_t)E);
#pragma omp for schedule(dynamic, 4)
        for (int64_t t = 0; t < T; ++t) {
            token_scores(x + t * H, wr, bias, H, E, score_fn, score, key);
            int32_t *it = ids + t * k;
            double next = -INFINITY;
            if (forced_ids) {
                for (int r = 0; r < k; ++r) {
                    it[r] = forced_ids[t * k + r];
                    if (it[r] < 0 || it[r] >= E) bad = 1;
                }
                if (bad) continue;
            } else {
                next = select_topk(key, E, k, it, taken);
            }
            double sum = 0.0;
            for (int r = 0; r < k; ++r) sum += score[it[r]];
            for (int r = 0; r < k; ++r) w[t * k + r] = score[it[r]] / sum;
            if (kth_key) kth_key[t] = key[it[k - 1]];
            if (next_key) next_key[t] = next;
        }
        free(score);
        free(key);
        free(taken);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------ */
/* Bucketing (R7)                                                      */
/* ------------------------------------------------------------------ */

int orc_bucket(const int32_t *ids, int64_t T, int k, int E, int32_t *counts, int32_t *offsets,
               int32_t *assign)
{
    memset(counts, 0, sizeof(int32_t) * (size_t)E);
    for (int64_t a = 0; a < T * k; ++a) {
        if (ids[a] < 0 || ids[a] >= E) return -1;
        counts[ids[a]]++;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t *cursor = malloc(sizeof(int32_t) * (size_t)E);
    memcpy(cursor, offsets, sizeof(int32_t) * (size_t)E);
    for (int64_t a = 0; a < T * k; ++a) assign[cursor[ids[a]]++] = (int32_t)a;
    free(cursor);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Expert FFN (R4, R5) and the layer (R8)                              */
/* ------------------------------------------------------------------ */

/* out[b][:] = Wd^T-stored * (SiLU(Wg xs[b]) * (Wu xs[b])) for n tokens, fp64.
 * Wg, Wu, Wd are [FF][H] fp32 (already dequantised). */
static void expert_ffn(const float *Wg, const float *Wu, const float *Wd, int FF, int H,
                       const double *xs, int64_t n, double *act, double *out)
{
#pragma omp parallel for schedule(static)
    for (int f = 0; f < FF; ++f) {
        const float *wg = Wg + (int64_t)f * H, *wu = Wu + (int64_t)f * H;
        for (int64_t b = 0; b < n; ++b) {
            const double *xb = xs + b * H;
            double g = 0.0, u = 0.0;
            for (int h = 0; h < H; ++h) {
                g += (double)wg[h] * xb[h];
                u += (double)wu[h] * xb[h];
            }
            act[b * FF + f] = g / (1.0 + exp(-g)) * u;
        }
    }
    const int HC = 64;   /* h-chunk per thread */
#pragma omp parallel for schedule(static)
    for (int h0 = 0; h0 < H; h0 += HC) {
        int h1 = h0 + HC < H ? h0 + HC : H;
        for (int64_t b = 0; b < n; ++b) {
            double *ob = out + b * H;
            for (int h = h0; h < h1; ++h) ob[h] = 0.0;
            for (int f = 0; f < FF; ++f) {
                double a = act[b * FF + f];
                const float *wd = Wd + (int64_t)f * H;
                for (int h = h0; h < h1; ++h) ob[h] += a * (double)wd[h];
            }
        }
    }
}

/*
 * The whole layer for T tokens.
 *   x        [T][H] bf16 bits        wr [E][H] fp32      bias [E] fp32 or NULL
 *   blobs    E pointers to expert blobs (R4), NULL allowed for experts that
 *            no token selects
 *   shared   shared-expert blob (Q8_0, same [gate][up][down] order) or NULL
 *   forced   [T*k] ids to use instead of the selection, or NULL
 *   y        [T][H] fp64 output
 * Returns 0, -1 (bad arguments) or -2 (a selected expert has no blob).
 */
int orc_moe_forward_codec(int H, int E, int FF, int k, int score_fn, int has_shared, int shared_ff,
                          const uint16_t *x, const float *wr, const float *bias,
                          const uint8_t *const *blobs, const uint8_t *shared, int64_t T,
                          const int32_t *forced, int codec, double *y)
{
    if (codec != 0 && codec != 1) return -1;
    if (H <= 0 || H % ORC_QK_K || FF <= 0 || T < 0) return -1;
    if (has_shared && (!shared || shared_ff <= 0)) return -1;
    int64_t TK = T * k;
    int32_t *ids = malloc(sizeof(int32_t) * (size_t)(TK > 0 ? TK : 1));
    double *w = malloc(sizeof(double) * (size_t)(TK > 0 ? TK : 1));
    int32_t *counts = malloc(sizeof(int32_t) * (size_t)E);
    int32_t *offsets = malloc(sizeof(int32_t) * (size_t)(E + 1));
    int32_t *assign = malloc(sizeof(int32_t) * (size_t)(TK > 0 ? TK : 1));
    int rc = orc_route(x, wr, bias, T, H, E, k, score_fn, forced, ids, w, NULL, NULL);
    if (rc == 0) rc = orc_bucket(ids, T, k, E, counts, offsets, assign);
    for (int e = 0; rc == 0 && e < E; ++e)
        if (counts[e] > 0 && !blobs[e]) rc = -2;
    if (rc != 0) {
        free(ids); free(w); free(counts); free(offsets); free(assign);
        return rc;
    }

    double *xd = malloc(sizeof(double) * (size_t)(T * H > 0 ? T * H : 1));
    for (int64_t i = 0; i < T * H; ++i) xd[i] = (double)orc_bf16_to_f32(x[i]);

    int64_t mat = (int64_t)FF * H;
    int64_t mat_bytes = (int64_t)FF * (H / ORC_QK_K) * (codec ? ORC_Q5K_BYTES : ORC_Q4K_BYTES);
    float *W = malloc(sizeof(float) * (size_t)(3 * mat));
    double *slot = calloc((size_t)(TK > 0 ? TK : 1) * (size_t)H, sizeof(double));
    int64_t maxc = 0;
    for (int e = 0; e < E; ++e) if (counts[e] > maxc) maxc = counts[e];
    double *xs = malloc(sizeof(double) * (size_t)((maxc > 0 ? maxc : 1) * H));
    double *act = malloc(sizeof(double) * (size_t)((maxc > 0 ? maxc : 1) * FF));
    double *ob = malloc(sizeof(double) * (size_t)((maxc > 0 ? maxc : 1) * H));

    /* expert-major: one expert dequantised at a time, all its tokens at once */
    for (int e = 0; e < E; ++e) {
        int64_t n = counts[e];
        if (n == 0) continue;
        for (int m = 0; m < 3; ++m) {
            if (codec) orc_q5k_dequantize(blobs[e] + m * mat_bytes, FF, H, W + m * mat);
            else orc_q4k_dequantize(blobs[e] + m * mat_bytes, FF, H, W + m * mat);
        }
        for (int64_t b = 0; b < n; ++b) {
            int64_t t = assign[offsets[e] + b] / k;
            memcpy(xs + b * H, xd + t * H, sizeof(double) * (size_t)H);
        }
        expert_ffn(W, W + mat, W + 2 * mat, FF, H, xs, n, act, ob);
        for (int64_t b = 0; b < n; ++b)
            memcpy(slot + (int64_t)assign[offsets[e] + b] * H, ob + b * H, sizeof(double) * (size_t)H);
    }

    /* combine: r ascending per token */
    for (int64_t t = 0; t < T; ++t)
        for (int h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int r = 0; r < k; ++r) acc += w[t * k + r] * slot[(t * k + r) * H + h];
            y[t * H + h] = acc;
        }

    if (has_shared && T > 0) {
        int64_t smat = (int64_t)shared_ff * H;
        int64_t smat_bytes = (int64_t)shared_ff * (H / ORC_QK8) * ORC_Q8_BYTES;
        float *S = malloc(sizeof(float) * (size_t)(3 * smat));
        for (int m = 0; m < 3; ++m) orc_q8_0_dequantize(shared + m * smat_bytes, shared_ff, H, S + m * smat);
        double *sact = malloc(sizeof(double) * (size_t)(T * shared_ff));
        double *so = malloc(sizeof(double) * (size_t)(T * H));
        expert_ffn(S, S + smat, S + 2 * smat, shared_ff, H, xd, T, sact, so);
        for (int64_t i = 0; i < T * H; ++i) y[i] += so[i];
        free(S); free(sact); free(so);
    }

    free(ids); free(w); free(counts); free(offsets); free(assign);
    free(xd); free(W); free(slot); free(xs); free(act); free(ob);
    return 0;
}

/* The layer with Q4_K experts (the codec-0 case above). */
int orc_moe_forward(int H, int E, int FF, int k, int score_fn, int has_shared, int shared_ff,
                    const uint16_t *x, const float *wr, const float *bias,
                    const uint8_t *const *blobs, const uint8_t *shared, int64_t T,
                    const int32_t *forced, double *y)
{
    return orc_moe_forward_codec(H, E, FF, k, score_fn, has_shared, shared_ff, x, wr, bias, blobs, shared, T,
                                 forced, 0, y);
}

/* Threads the OpenMP regions above use (0 or less: leave the default). */
int orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}
