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
 * experts: for each selected expert, each Q4_K super-block of a weight row is
 * unpacked once (nibbles -> fp32 through the AVX2 integer-to-float converts,
 * sub-block scale and min as one fused multiply-subtract) and multiplied into
 * the accumulators of all the expert's tokens.  Arithmetic in fp32 with fp32
 * accumulation (the oracle's fp64 is the reference; the difference stays far
 * inside the layer's tolerance).
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

/* 32 quants (bytes) -> 4 x 8 fp32 weights q * S - Z. */
static inline void q32_to_f32(__m256i q8, __m256 S, __m256 Z, __m256 out[4])
{
    const __m128i lo = _mm256_castsi256_si128(q8), hi = _mm256_extracti128_si256(q8, 1);
    out[0] = _mm256_fmsub_ps(_mm256_cvtepi32_ps(_mm256_cvtepu8_epi32(lo)), S, Z);
    out[1] = _mm256_fmsub_ps(_mm256_cvtepi32_ps(_mm256_cvtepu8_epi32(_mm_srli_si128(lo, 8))), S, Z);
    out[2] = _mm256_fmsub_ps(_mm256_cvtepi32_ps(_mm256_cvtepu8_epi32(hi)), S, Z);
    out[3] = _mm256_fmsub_ps(_mm256_cvtepi32_ps(_mm256_cvtepu8_epi32(_mm_srli_si128(hi, 8))), S, Z);
}

/* One Q4_K super-block (256 weights) -> w[256] fp32. */
static inline void q4k_block(const uint8_t *blk, float *w)
{
    const float d = f16_to_f32(blk), dmin = f16_to_f32(blk + 2);
    const uint8_t *s = blk + 4, *qs = blk + 16;
    const __m256i m4 = _mm256_set1_epi8(0x0f);
    for (int c = 0; c < 4; ++c) {
        const __m256i v = _mm256_loadu_si256((const __m256i *)(qs + 32 * c));
        const __m256i lo = _mm256_and_si256(v, m4), hi = _mm256_and_si256(_mm256_srli_epi16(v, 4), m4);
        int sc, m;
        __m256 o[4];
        q4k_scale_min(s, 2 * c, &sc, &m);
        q32_to_f32(lo, _mm256_set1_ps(d * (float)sc), _mm256_set1_ps(dmin * (float)m), o);
        for (int i = 0; i < 4; ++i) _mm256_storeu_ps(w + 64 * c + 8 * i, o[i]);
        q4k_scale_min(s, 2 * c + 1, &sc, &m);
        q32_to_f32(hi, _mm256_set1_ps(d * (float)sc), _mm256_set1_ps(dmin * (float)m), o);
        for (int i = 0; i < 4; ++i) _mm256_storeu_ps(w + 64 * c + 32 + 8 * i, o[i]);
    }
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
    float *act;                 /* [assignments][FF] */
    float *y;                   /* [T][H] */
    int nthr, id;
} Job;

#define MAXTOK 64

/* gate/up of ff rows f = id, id + nthr, ... of every selected expert. */
static void *gateup_worker(void *arg)
{
    const Job *j = arg;
    const int H = j->H, nb = j->nb;
    const int64_t mat = (int64_t)j->FF * nb * Q4K_BYTES;
    float *wg = aligned_alloc(32, sizeof(float) * QK), *wu = aligned_alloc(32, sizeof(float) * QK);
    for (int s = 0; s < j->n_sel; ++s) {
        const int a0 = j->tok_off[s], n = j->tok_off[s + 1] - a0;
        const uint8_t *blob = j->blobs[j->sel[s]];
        for (int f = j->id; f < j->FF; f += j->nthr) {
            __m256 ag[MAXTOK], au[MAXTOK];
            for (int t = 0; t < n; ++t) ag[t] = au[t] = _mm256_setzero_ps();
            const uint8_t *rg = blob + (int64_t)f * nb * Q4K_BYTES, *ru = rg + mat;
            for (int b = 0; b < nb; ++b) {
                q4k_block(rg + b * Q4K_BYTES, wg);
                q4k_block(ru + b * Q4K_BYTES, wu);
                for (int t = 0; t < n; ++t) {
                    const float *xt = j->xs + (int64_t)j->tok[a0 + t] * H + b * QK;
                    __m256 g = ag[t], u = au[t];
                    for (int i = 0; i < QK; i += 8) {
                        const __m256 xv = _mm256_loadu_ps(xt + i);
                        g = _mm256_fmadd_ps(_mm256_load_ps(wg + i), xv, g);
                        u = _mm256_fmadd_ps(_mm256_load_ps(wu + i), xv, u);
                    }
                    ag[t] = g;
                    au[t] = u;
                }
            }
            for (int t = 0; t < n; ++t) {
                const float g = hsum(ag[t]), u = hsum(au[t]);
                j->act[(int64_t)(a0 + t) * j->FF + f] = g / (1.0f + expf(-g)) * u * j->tw[a0 + t];
            }
        }
    }
    free(wg);
    free(wu);
    return NULL;
}

/* down: 256-column blocks b = id, id + nthr, ... of y, every selected expert and token. */
static void *down_worker(void *arg)
{
    const Job *j = arg;
    const int H = j->H, nb = j->nb, FF = j->FF;
    const int64_t mat = (int64_t)FF * nb * Q4K_BYTES;
    float *wd = aligned_alloc(32, sizeof(float) * QK);
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
                    q4k_block(rd + (int64_t)f * nb * Q4K_BYTES, wd);
                    for (int t = 0; t < nt; ++t) {
                        const __m256 av = _mm256_set1_ps(j->act[(int64_t)(a0 + t0 + t) * FF + f]);
                        for (int i = 0; i < QK / 8; ++i)
                            acc[t][i] = _mm256_fmadd_ps(_mm256_load_ps(wd + 8 * i), av, acc[t][i]);
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
    free(wd);
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
    float *xs = malloc(sizeof(float) * (size_t)(T * H));
    for (int64_t i = 0; i < T * H; ++i) xs[i] = bf16_to_f32(x[i]);
    float *act = malloc(sizeof(float) * (size_t)TK * (size_t)FF);

    int nthr = threads > 0 ? threads : 1;
    pthread_t *th = malloc(sizeof(pthread_t) * (size_t)nthr);
    Job *jobs = malloc(sizeof(Job) * (size_t)nthr);
    for (int i = 0; i < nthr; ++i) {
        Job jb = {H, FF, H / QK, n_sel, sel, toff, tok, tw, blobs, xs, act, y, nthr, i};
        jobs[i] = jb;
    }
    for (int i = 0; i < nthr; ++i) pthread_create(&th[i], NULL, gateup_worker, &jobs[i]);
    for (int i = 0; i < nthr; ++i) pthread_join(th[i], NULL);
    for (int i = 0; i < nthr; ++i) pthread_create(&th[i], NULL, down_worker, &jobs[i]);
    for (int i = 0; i < nthr; ++i) pthread_join(th[i], NULL);

    free(th); free(jobs); free(act); free(xs); free(tw); free(fill); free(tok); free(toff); free(sel);
    free(cnt); free(off);
    return 0;
}
