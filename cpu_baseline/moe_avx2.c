/*
 * moe_avx2.c -- a multi-token CPU expert kernel (AVX2 + FMA + F16C), timed as a
 * CPU baseline beside the oracle.  Not part of the product: only tests/ and
 * bench.py's CPU legs load it, and it shares no code with the CUDA library or
 * the oracle.
 *
 * The teardown page ("Strata 引擎深度拆解", lcz.me/topic/2098/5, section 一,
 * CPU ledger) describes the engine's CPU expert kernel: it applies an expert's
 * bytes to every token of a verify window at once (a multi-token kernel), and
 * quotes a down projection at 4.4 GB/s (ggml: 3.2) and a 3-token window in
 * 282 us (ggml: 414) on an AVX2 EPYC.  This kernel does the same work for Q4_K
 * experts: for each selected expert, the quants of each 32-weight sub-block of
 * a weight row are converted to fp32 once (AVX2 integer-to-float converts) and
 * multiplied into the sums of all the expert's tokens; the sub-block's scale
 * and min enter once per sub-block through the affine form of Q4_K (a weight
 * is q * S - Z, so a sub-block contributes S * sum(q x) - Z * sum(x)), not
 * once per weight.  Arithmetic in fp32 with fp32 accumulation (the oracle's
 * fp64 is the reference; the difference stays far inside the layer's
 * tolerance).
 *
 * Work split over `threads` POSIX threads: gate/up by ff rows of every selected
 * expert, then the down projection by 256-column blocks of H (each thread owns
 * its columns of y for every token: no atomics).
 */
#include <immintrin.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#define QK 256
#define Q4K_BYTES 144

static inline float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static inline float f16_to_f32(const uint8_t *p)
{
    uint16_t h;
    memcpy(&h, p, 2);
    return _cvtsh_ss(h);
}

/* 6-bit scale and min of sub-block j (GGUF Q4_K packing). */
static inline void q4k_scale_min(const uint8_t *s, int j, int *sc, int *m)
{
    if (j < 4) {
        *sc = s[j] & 63;
        *m = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        *m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

/* 32 quants (one per byte of q8, 0..15) -> 4 x 8 fp32 (exact small integers). */
static inline void q32_to_f32(__m256i q8, __m256 out[4])
{
    const __m128i lo = _mm256_castsi256_si128(q8), hi = _mm256_extracti128_si256(q8, 1);
    out[0] = _mm256_cvtepi32_ps(_mm256_cvtepu8_epi32(lo));
    out[1] = _mm256_cvtepi32_ps(_mm256_cvtepu8_epi32(_mm_srli_si128(lo, 8)));
    out[2] = _mm256_cvtepi32_ps(_mm256_cvtepu8_epi32(hi));
    out[3] = _mm256_cvtepi32_ps(_mm256_cvtepu8_epi32(_mm_srli_si128(hi, 8)));
}

/* The quants of sub-block sb = 2c + half of a super-block: byte group c (32
 * bytes) holds sub-block 2c in its low nibbles and 2c + 1 in its high ones. */
static inline __m256i q4k_sub(__m256i group, int half)
{
    const __m256i m4 = _mm256_set1_epi8(0x0f);
    return half ? _mm256_and_si256(_mm256_srli_epi16(group, 4), m4) : _mm256_and_si256(group, m4);
}

/* Scale and min of the 8 sub-blocks of a Q4_K super-block: a weight of
 * sub-block j is q * S[j] - Z[j], S[j] = d * sc_j, Z[j] = dmin * m_j. */
static inline void q4k_sm(const uint8_t *blk, float S[8], float Z[8])
{
    const float d = f16_to_f32(blk), dmin = f16_to_f32(blk + 2);
    for (int j = 0; j < 8; ++j) {
        int sc, m;
        q4k_scale_min(blk + 4, j, &sc, &m);
        S[j] = d * (float)sc;
        Z[j] = dmin * (float)m;
    }
}

/* 32 quants (bytes) -> 4 x 8 fp32 weights q * S - Z (the down projection). */
static inline void q32_to_f32_affine(__m256i q8, __m256 S, __m256 Z, __m256 out[4])
{
    const __m128i lo = _mm256_castsi256_si128(q8), hi = _mm256_extracti128_si256(q8, 1);
    out[0] = _mm256_fmsub_ps(_mm256_cvtepi32_ps(_mm256_cvtepu8_epi32(lo)), S, Z);
    out[1] = _mm256_fmsub_ps(_mm256_cvtepi32_ps(_mm256_cvtepu8_epi32(_mm_srli_si128(lo, 8))), S, Z);
    out[2] = _mm256_fmsub_ps(_mm256_cvtepi32_ps(_mm256_cvtepu8_epi32(hi)), S, Z);
    out[3] = _mm256_fmsub_ps(_mm256_cvtepi32_ps(_mm256_cvtepu8_epi32(_mm_srli_si128(hi, 8))), S, Z);
}

static inline float hsum(__m256 v)
{
    __m128 s = _mm_add_ps(_mm256_castps256_ps128(v), _mm256_extractf128_ps(v, 1));
    s = _mm_add_ps(s, _mm_movehl_ps(s, s));
    s = _mm_add_ss(s, _mm_movehdup_ps(s));
    return _mm_cvtss_f32(s);
}

typedef struct {
    int H, FF, nb;
    int n_sel;                  /* selected experts */
    const int32_t *sel;         /* [n_sel] expert ids */
    const int32_t *tok_off;     /* [n_sel + 1] offsets into tok / tw */
    const int32_t *tok;         /* token of each assignment, grouped by expert */
    const float *tw;            /* its routing weight */
    const uint8_t *const *blobs;
    const float *xs;            /* [T][H] fp32 */
    const float *xsum;          /* [T][H / 32]: x summed over each 32-element sub-block */
    float *act;                 /* [assignments][FF] */
    float *y;                   /* [T][H] */
    int nthr, id;
} Job;

#define MAXTOK 64

/* Sum of q[i] * x[i] over a sub-block's 32 weights (two independent chains). */
static inline __m256 qdot32(const __m256 q[4], const float *x)
{
    __m256 a = _mm256_mul_ps(q[0], _mm256_loadu_ps(x)), b = _mm256_mul_ps(q[1], _mm256_loadu_ps(x + 8));
    a = _mm256_fmadd_ps(q[2], _mm256_loadu_ps(x + 16), a);
    b = _mm256_fmadd_ps(q[3], _mm256_loadu_ps(x + 24), b);
    return _mm256_add_ps(a, b);
}

/* gate/up of an expert that one token selected (the usual case of a small
 * window): the sums stay in registers, one chain per sub-block parity. */
static void gateup_one(const Job *j, const uint8_t *blob, int64_t mat, int a0)
{
    const int H = j->H, nb = j->nb, nsb = H / 32;
    const int tk = j->tok[a0];
    const float *xr = j->xs + (int64_t)tk * H, *xsr = j->xsum + (int64_t)tk * nsb;
    for (int f = j->id; f < j->FF; f += j->nthr) {
        __m256 g0 = _mm256_setzero_ps(), g1 = g0, u0 = g0, u1 = g0;
        float zg = 0.0f, zu = 0.0f;
        const uint8_t *rg = blob + (int64_t)f * nb * Q4K_BYTES, *ru = rg + mat;
        for (int b = 0; b < nb; ++b) {
            const uint8_t *bg = rg + b * Q4K_BYTES, *bu = ru + b * Q4K_BYTES;
            float Sg[8], Zg[8], Su[8], Zu[8];
            q4k_sm(bg, Sg, Zg);
            q4k_sm(bu, Su, Zu);
            for (int c = 0; c < 4; ++c) {
                const __m256i vg = _mm256_loadu_si256((const __m256i *)(bg + 16 + 32 * c));
                const __m256i vu = _mm256_loadu_si256((const __m256i *)(bu + 16 + 32 * c));
                const float *x0 = xr + b * QK + 64 * c;
                __m256 q[4];
                q32_to_f32(q4k_sub(vg, 0), q);
                g0 = _mm256_fmadd_ps(qdot32(q, x0), _mm256_set1_ps(Sg[2 * c]), g0);
                q32_to_f32(q4k_sub(vu, 0), q);
                u0 = _mm256_fmadd_ps(qdot32(q, x0), _mm256_set1_ps(Su[2 * c]), u0);
                q32_to_f32(q4k_sub(vg, 1), q);
                g1 = _mm256_fmadd_ps(qdot32(q, x0 + 32), _mm256_set1_ps(Sg[2 * c + 1]), g1);
                q32_to_f32(q4k_sub(vu, 1), q);
                u1 = _mm256_fmadd_ps(qdot32(q, x0 + 32), _mm256_set1_ps(Su[2 * c + 1]), u1);
            }
            for (int sb = 0; sb < 8; ++sb) {
                zg += Zg[sb] * xsr[8 * b + sb];
                zu += Zu[sb] * xsr[8 * b + sb];
            }
        }
        const float g = hsum(_mm256_add_ps(g0, g1)) - zg, u = hsum(_mm256_add_ps(u0, u1)) - zu;
        j->act[(int64_t)a0 * j->FF + f] = g / (1.0f + expf(-g)) * u * j->tw[a0];
    }
}

/* gate/up of ff rows f = id, id + nthr, ... of every selected expert.  With
 * the Q4_K affine form, a sub-block's contribution to row . x is
 * S * sum(q * x) - Z * sum(x): the quants are converted once per sub-block
 * and multiplied into every token's sums; sum(x) is the window's xsum. */
static void *gateup_worker(void *arg)
{
    const Job *j = arg;
    const int H = j->H, nb = j->nb, nsb = H / 32;
    const int64_t mat = (int64_t)j->FF * nb * Q4K_BYTES;
    for (int s = 0; s < j->n_sel; ++s) {
        const int a0 = j->tok_off[s], n = j->tok_off[s + 1] - a0;
        const uint8_t *blob = j->blobs[j->sel[s]];
        if (n == 1) {
            gateup_one(j, blob, mat, a0);
            continue;
        }
        for (int f = j->id; f < j->FF; f += j->nthr) {
            __m256 ag[MAXTOK], au[MAXTOK];
            float zg[MAXTOK], zu[MAXTOK];
            for (int t = 0; t < n; ++t) {
                ag[t] = au[t] = _mm256_setzero_ps();
                zg[t] = zu[t] = 0.0f;
            }
            const uint8_t *rg = blob + (int64_t)f * nb * Q4K_BYTES, *ru = rg + mat;
            for (int b = 0; b < nb; ++b) {
                const uint8_t *bg = rg + b * Q4K_BYTES, *bu = ru + b * Q4K_BYTES;
                float Sg[8], Zg[8], Su[8], Zu[8];
                q4k_sm(bg, Sg, Zg);
                q4k_sm(bu, Su, Zu);
                for (int c = 0; c < 4; ++c) {
                    const __m256i vg = _mm256_loadu_si256((const __m256i *)(bg + 16 + 32 * c));
                    const __m256i vu = _mm256_loadu_si256((const __m256i *)(bu + 16 + 32 * c));
                    for (int half = 0; half < 2; ++half) {
                        const int sb = 2 * c + half;
                        __m256 qg[4], qu[4];
                        q32_to_f32(q4k_sub(vg, half), qg);
                        q32_to_f32(q4k_sub(vu, half), qu);
                        const __m256 sg = _mm256_set1_ps(Sg[sb]), su = _mm256_set1_ps(Su[sb]);
                        for (int t = 0; t < n; ++t) {
                            const int tk = j->tok[a0 + t];
                            const float *xt = j->xs + (int64_t)tk * H + b * QK + 32 * sb;
                            const __m256 x0 = _mm256_loadu_ps(xt), x1 = _mm256_loadu_ps(xt + 8);
                            const __m256 x2 = _mm256_loadu_ps(xt + 16), x3 = _mm256_loadu_ps(xt + 24);
                            __m256 pg = _mm256_mul_ps(qg[0], x0), pu = _mm256_mul_ps(qu[0], x0);
                            pg = _mm256_fmadd_ps(qg[1], x1, pg);
                            pu = _mm256_fmadd_ps(qu[1], x1, pu);
                            pg = _mm256_fmadd_ps(qg[2], x2, pg);
                            pu = _mm256_fmadd_ps(qu[2], x2, pu);
                            pg = _mm256_fmadd_ps(qg[3], x3, pg);
                            pu = _mm256_fmadd_ps(qu[3], x3, pu);
                            ag[t] = _mm256_fmadd_ps(pg, sg, ag[t]);
                            au[t] = _mm256_fmadd_ps(pu, su, au[t]);
                            const float xs = j->xsum[(int64_t)tk * nsb + 8 * b + sb];
                            zg[t] += Zg[sb] * xs;
                            zu[t] += Zu[sb] * xs;
                        }
                    }
                }
            }
            for (int t = 0; t < n; ++t) {
                const float g = hsum(ag[t]) - zg[t], u = hsum(au[t]) - zu[t];
                j->act[(int64_t)(a0 + t) * j->FF + f] = g / (1.0f + expf(-g)) * u * j->tw[a0 + t];
            }
        }
    }
    return NULL;
}

/* down: 256-column blocks b = id, id + nthr, ... of y, every selected expert and token. */
static void *down_worker(void *arg)
{
    const Job *j = arg;
    const int H = j->H, nb = j->nb, FF = j->FF;
    const int64_t mat = (int64_t)FF * nb * Q4K_BYTES;
    for (int b = j->id; b < nb; b += j->nthr) {
        for (int s = 0; s < j->n_sel; ++s) {
            const int a0 = j->tok_off[s], n = j->tok_off[s + 1] - a0;
            const uint8_t *rd = j->blobs[j->sel[s]] + 2 * mat + (int64_t)b * Q4K_BYTES;
            for (int t0 = 0; t0 < n; t0 += 4) {
                const int nt = n - t0 < 4 ? n - t0 : 4;
                __m256 acc[4][QK / 8];
                for (int t = 0; t < nt; ++t)
                    for (int i = 0; i < QK / 8; ++i) acc[t][i] = _mm256_setzero_ps();
                for (int f = 0; f < FF; ++f) {
                    /* the row block's weights, unpacked 32 at a time straight into the sums */
                    const uint8_t *blk = rd + (int64_t)f * nb * Q4K_BYTES;
                    const float d = f16_to_f32(blk), dmin = f16_to_f32(blk + 2);
                    __m256 av[4];
                    for (int t = 0; t < nt; ++t) av[t] = _mm256_set1_ps(j->act[(int64_t)(a0 + t0 + t) * FF + f]);
                    for (int c = 0; c < 4; ++c) {
                        const __m256i v = _mm256_loadu_si256((const __m256i *)(blk + 16 + 32 * c));
                        for (int half = 0; half < 2; ++half) {
                            const int sb = 2 * c + half;
                            int sc, m;
                            q4k_scale_min(blk + 4, sb, &sc, &m);
                            __m256 w[4];
                            q32_to_f32_affine(q4k_sub(v, half), _mm256_set1_ps(d * (float)sc),
                                              _mm256_set1_ps(dmin * (float)m), w);
                            for (int t = 0; t < nt; ++t)
                                for (int i = 0; i < 4; ++i)
                                    acc[t][4 * sb + i] = _mm256_fmadd_ps(w[i], av[t], acc[t][4 * sb + i]);
                        }
                    }
                }
                for (int t = 0; t < nt; ++t) {
                    float *yt = j->y + (int64_t)j->tok[a0 + t0 + t] * H + b * QK;
                    for (int i = 0; i < QK / 8; ++i)
                        _mm256_storeu_ps(yt + 8 * i, _mm256_add_ps(_mm256_loadu_ps(yt + 8 * i), acc[t][i]));
                }
            }
        }
    }

    return NULL;
}

/*
 * y[T][H] (fp32, overwritten) = sum over the window's assignments (t, r) of
 * w[t][r] * FFN_{ids[t][r]}(x_t) for Q4_K expert blobs laid out
 * [gate FF x H][up FF x H][down FF x H].  x: bf16 [T][H].  Returns 0, or -1 on
 * bad arguments (H % 256, an id out of range or without a blob, a missing
 * AVX2/FMA/F16C unit, more than 64 tokens on one expert).
 */
int cpu_moe_window(int H, int E, int FF, int k, int64_t T, const uint16_t *x, const int32_t *ids, const float *w,
                   const uint8_t *const *blobs, int threads, float *y)
{
    if (H <= 0 || H % QK || FF <= 0 || k <= 0 || T < 0 || E <= 0) return -1;
    __builtin_cpu_init();
    if (!__builtin_cpu_supports("avx2") || !__builtin_cpu_supports("fma")) return -1;
    const int64_t TK = T * k;
    for (int64_t i = 0; i < TK; ++i)
        if (ids[i] < 0 || ids[i] >= E || !blobs[ids[i]]) return -1;
    memset(y, 0, sizeof(float) * (size_t)(T * H));
    if (T == 0) return 0;
    /* bucket the assignments by expert (token-ascending within an expert) */
    int32_t *cnt = calloc((size_t)E, sizeof(int32_t)), *off = malloc(sizeof(int32_t) * (size_t)(E + 1));
    for (int64_t i = 0; i < TK; ++i) cnt[ids[i]]++;
    int n_sel = 0;
    off[0] = 0;
    for (int e = 0; e < E; ++e) {
        off[e + 1] = off[e] + cnt[e];
        if (cnt[e]) ++n_sel;
        if (cnt[e] > MAXTOK) {
            free(cnt);
            free(off);
            return -1;
        }
    }
    int32_t *sel = malloc(sizeof(int32_t) * (size_t)(n_sel > 0 ? n_sel : 1));
    int32_t *toff = malloc(sizeof(int32_t) * (size_t)(n_sel + 1));
    int32_t *tok = malloc(sizeof(int32_t) * (size_t)TK), *fill = calloc((size_t)E, sizeof(int32_t));
    float *tw = malloc(sizeof(float) * (size_t)TK);
    for (int e = 0, s = 0; e < E; ++e)
        if (cnt[e]) {
            sel[s] = e;
            toff[s] = off[e];
            ++s;
        }
    toff[n_sel] = (int32_t)TK;
    for (int64_t i = 0; i < TK; ++i) {
        const int e = ids[i];
        const int p = off[e] + fill[e]++;
        tok[p] = (int32_t)(i / k);
        tw[p] = w[i];
    }
    float *xs = malloc(sizeof(float) * (size_t)(T * H)), *xsum = malloc(sizeof(float) * (size_t)(T * (H / 32)));
    for (int64_t i = 0; i < T * H; ++i) xs[i] = bf16_to_f32(x[i]);
    for (int64_t i = 0; i < T * (H / 32); ++i) {
        float a = 0.0f;
        for (int l = 0; l < 32; ++l) a += xs[32 * i + l];
        xsum[i] = a;
    }
    float *act = malloc(sizeof(float) * (size_t)TK * (size_t)FF);

    int nthr = threads > 0 ? threads : 1;
    pthread_t *th = malloc(sizeof(pthread_t) * (size_t)nthr);
    Job *jobs = malloc(sizeof(Job) * (size_t)nthr);
    for (int i = 0; i < nthr; ++i) {
        Job jb = {H, FF, H / QK, n_sel, sel, toff, tok, tw, blobs, xs, xsum, act, y, nthr, i};
        jobs[i] = jb;
    }
    for (int i = 0; i < nthr; ++i) pthread_create(&th[i], NULL, gateup_worker, &jobs[i]);
    for (int i = 0; i < nthr; ++i) pthread_join(th[i], NULL);
    for (int i = 0; i < nthr; ++i) pthread_create(&th[i], NULL, down_worker, &jobs[i]);
    for (int i = 0; i < nthr; ++i) pthread_join(th[i], NULL);

    free(th); free(jobs); free(act); free(xs); free(xsum); free(tw); free(fill); free(tok); free(toff); free(sel);
    free(cnt); free(off);
    return 0;
}
