// decode.cu -- the layer for decode / MTP-verify windows (T <= 8 tokens).
//
// The teardown page ("Strata 引擎深度拆解", lcz.me/topic/2098/5, section 一,
// CPU ledger) computes each selected expert once for all tokens of a 3-token
// verify window; the decode critical path there is the expert arithmetic
// (section 二 item 5).  Here a window is four kernels chained with
// programmatic dependent launch, so each one is scheduled while its
// predecessor drains:
//
//   k_dec_route   router logits over every SM (each router row read once per
//                 window; the window's x staged in shared memory); also
//                 zeroes the y accumulator and builds the fp16 B-operand
//                 fragments of the window's hidden states.
//   k_dec_gateup  every CTA first routes the window itself (top-k of each
//                 token on its own warp, stable counting sort of the
//                 assignments by expert; CTA 0 publishes the result), then
//                 computes gate/up of every selected expert: one warp per 8
//                 ff indices (8 gate rows + the 8 up rows of the same indices
//                 = one m16n8k16 M tile), each warp streaming its Q4_K rows
//                 through a private cp.async ring; the bytes are dequantised
//                 straight into MMA A fragments (fp16, fp32 accumulation)
//                 with the window's tokens as the 8 MMA columns; SiLU(g)*u in
//                 registers.  (An L2 prefetch of the selected experts' down
//                 matrices during gate/up exists behind a switch; measured
//                 slower, it is off.)
//   k_dec_down    down projection: units of (expert, 256 hidden columns, ff
//                 segment) staged in shared memory with cp.async (segments
//                 chosen so the slowest warp has the fewest rows; one buffer
//                 per warp and 3 CTAs per SM when every warp has one unit); Q4_K
//                 nibbles become exact fp32 values through the mantissa, the
//                 sub-block scale and min are factored out of the sum over ff;
//                 the weighted result is added into an fp32 accumulator of y
//                 (or stored into the slot of the assignment and segment in
//                 deterministic mode, summed in a fixed order at the end).
//   k_dec_finish  y = bf16 of the accumulated (or slot-summed) y, plus the
//                 shared expert's output.
//
// Every selected expert's Q4_K bytes are read once per window.
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_h2(float a, float b)
{
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ __half2 u2h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }
__device__ __forceinline__ uint32_t h22u(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// Q4_K sub-block j scale and negated min as fp16: fp16(d * sc), fp16(-(dmin * m)).
__device__ __forceinline__ void q4k_scales_h(uint4 hdr, int j, __half &s, __half &nz)
{
    const float d = f16_bits_to_f32(hdr.x & 0xffff), dmin = f16_bits_to_f32(hdr.x >> 16);
    uint8_t sc8[12];
    *reinterpret_cast<uint32_t *>(sc8) = hdr.y;
    *reinterpret_cast<uint32_t *>(sc8 + 4) = hdr.z;
    *reinterpret_cast<uint32_t *>(sc8 + 8) = hdr.w;
    int sc, m;
    q4k_scale_min(sc8, j, sc, m);
    s = __float2half_rn(__fmul_rn(d, (float)sc));
    nz = __float2half_rn(-__fmul_rn(dmin, (float)m));
}

// Q4_K sub-block j scale and min in fp32: d * sc, dmin * m (each one rounding).
__device__ __forceinline__ void q4k_scales_f(uint4 hdr, int j, float &s, float &z)
{
    const float d = f16_bits_to_f32(hdr.x & 0xffff), dmin = f16_bits_to_f32(hdr.x >> 16);
    uint8_t sc8[12];
    *reinterpret_cast<uint32_t *>(sc8) = hdr.y;
    *reinterpret_cast<uint32_t *>(sc8 + 4) = hdr.z;
    *reinterpret_cast<uint32_t *>(sc8 + 8) = hdr.w;
    int sc, m;
    q4k_scale_min(sc8, j, sc, m);
    s = __fmul_rn(d, (float)sc);
    z = __fmul_rn(dmin, (float)m);
}

// fp16 pairs (1024 + q) of the low / high nibbles of bytes (b0, b1) and (b2, b3)
// of a 32-bit word, converted to q (exact).
__device__ __forceinline__ void nib_q(uint32_t w, __half2 &lo01, __half2 &lo23, __half2 &hi01, __half2 &hi23)
{
    const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
    const __half2 k1024 = __float2half2_rn(1024.0f);
    lo01 = __hsub2(u2h2(__byte_perm(lo, 0x64646464u, 0x5140)), k1024);
    lo23 = __hsub2(u2h2(__byte_perm(lo, 0x64646464u, 0x5342)), k1024);
    hi01 = __hsub2(u2h2(__byte_perm(hi, 0x64646464u, 0x5140)), k1024);
    hi23 = __hsub2(u2h2(__byte_perm(hi, 0x64646464u, 0x5342)), k1024);
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *src)
{
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// ---------------------------------------------------------------- routing

// Order-preserving map of an fp32 key to uint32 (larger float -> larger
// integer); NaN maps to 0, below every number, and is never selected.
__device__ __forceinline__ uint32_t key_bits(float f)
{
    if (isnan(f)) return 0u;
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Top-k of one token by one warp.  key[e] (shared memory) holds the
// order-preserving integer of expert e's selection score (0 = not
// selectable).  Lane l keeps the keys of experts l, l + 32, ... (NPER) in
// registers and its best one (a reduction tree, equal keys to the lower id);
// each round takes the warp maximum (redux), the lowest expert id among equal
// keys, and only the winning lane clears that key and recomputes its best.
// Weights: softmax over the k selected logits (= the full softmax
// renormalised over the k) or s / sum of the selected s; vals[e] (shared
// memory) holds expert e's logit (softmax) or s = sigmoid(logit).  Lane r < k
// receives selection r.
template <int NPER>
__device__ void warp_topk(const uint32_t *keys, const float *vals, int E, int k, int score_fn, int lane,
                          int &out_id, float &out_w, bool &fault)
{
    uint32_t key[NPER];
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
        const int e = lane + 32 * i;
        key[i] = e < E ? keys[e] : 0u;
    }
    auto best = [&](uint32_t &bk, int &bi) {
        uint32_t kk[NPER];
        int ii[NPER];
#pragma unroll
        for (int i = 0; i < NPER; ++i) {
            kk[i] = key[i];
            ii[i] = i;
        }
#pragma unroll
        for (int w = 1; w < NPER; w <<= 1)
#pragma unroll
            for (int i = 0; i + w < NPER; i += 2 * w)
                if (kk[i + w] > kk[i]) {        // strict: equal keys keep the lower index
                    kk[i] = kk[i + w];
                    ii[i] = ii[i + w];
                }
        bk = kk[0];
        bi = ii[0];
    };
    uint32_t bk;
    int bi;
    best(bk, bi);
    int my_id = 0;
    fault = false;
    for (int r = 0; r < k; ++r) {
        const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
        const int e = (int)__reduce_min_sync(0xffffffffu, bk == mk ? (uint32_t)(lane + 32 * bi) : 0xffffffffu);
        if (mk == 0u) fault = true;          // nothing selectable (non-finite scores)
        if (lane == r) my_id = mk == 0u ? r : e;
        if (mk != 0u && lane == (e & 31)) {
#pragma unroll
            for (int i = 0; i < NPER; ++i)
                if (i == (e >> 5)) key[i] = 0u;
            best(bk, bi);
        }
    }
    const bool sel = lane < k;
    const float lv = sel ? vals[my_id] : 0.0f;
    float num;
    if (score_fn == MOE_SCORE_SOFTMAX) {
        const float lmax = __shfl_sync(0xffffffffu, lv, 0);   // the first pick is the largest
        num = sel ? expf(lv - lmax) : 0.0f;
    } else {
        num = sel ? lv : 0.0f;
    }
    float den = num;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
    out_id = my_id;
    out_w = num / den;
}

// Router logits.  Grid: ceil(E / (8 / P)) CTAs of 8 warps; warp (row r =
// warp / P, part p = warp % P) computes the T partial dot products of router
// row (8 / P) * blockIdx.x + r over columns [p * H / P, (p + 1) * H / P) from
// the window's x staged in shared memory; parts are added in order.  Also
// zeroes the y accumulator and writes the fp16 MMA B fragments of x.
constexpr int kRouteThreads = 256;

__global__ void __launch_bounds__(kRouteThreads) k_dec_route(DecArgs a)
{
    extern __shared__ __align__(16) uint16_t s_x[];     // [T][H] bf16
    __shared__ float s_part[8][kDecTok];                 // [warp][token]

    const int P = a.route_parts, rpc = 8 / P;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rloc = warp / P, part = warp % P;
    const int row = blockIdx.x * rpc + rloc;
    const int T = a.T, H = a.H, E = a.E;
    const int seg = H / P, nv = seg / 128;     // float4 per lane (<= kRouteMaxVec)

    // Router rows are weights: read them before the previous kernel finishes
    // only when the caller allows it.
    if (!a.overlap_prev) griddep_wait();
    float4 wv[kRouteMaxVec];
    const float4 *wrow = reinterpret_cast<const float4 *>(a.wr + (int64_t)min(row, E - 1) * H + part * seg);
#pragma unroll
    for (int i = 0; i < kRouteMaxVec; ++i)
        if (i < nv) wv[i] = __ldg(wrow + i * 32 + lane);
    if (a.overlap_prev) griddep_wait();

    {
        const int nvec = T * H / 8;
        const uint4 *src = reinterpret_cast<const uint4 *>(a.x);
        uint4 *dst = reinterpret_cast<uint4 *>(s_x);
        for (int i0 = threadIdx.x; i0 < nvec; i0 += 8 * kRouteThreads) {   // 8 loads in flight
            uint4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (i0 + j * kRouteThreads < nvec) v[j] = __ldg(src + i0 + j * kRouteThreads);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (i0 + j * kRouteThreads < nvec) dst[i0 + j * kRouteThreads] = v[j];
        }
    }
    // zero the y accumulator; fp16 MMA B fragments of x (token g = MMA column g):
    // k-step s of block column cb, lane (g, t): elements e = 256 cb + 64 t + 4 s + j
    // as b0 = (x[e+0], x[e+2]), b1 = (x[e+1], x[e+3])
    const int gtid = blockIdx.x * kRouteThreads + threadIdx.x, gthreads = gridDim.x * kRouteThreads;
    for (int i = gtid; i < T * H; i += gthreads) {
        a.yacc[i] = 0.0f;
        if (a.sh_out) a.sh_out[i] = 0.0f;
    }
    bool bad = false;
    const int n_frag = (H / 256) * 16 * 32;
    for (int i = gtid; i < n_frag; i += gthreads) {
        const int ln = i & 31, s = (i >> 5) & 15, cb = i >> 9;
        const int g = ln >> 2, t = ln & 3;
        const int h = 256 * cb + 64 * t + 4 * s;
        uint2 v = make_uint2(0u, 0u);
        if (g < T) {
            const uint2 xb = __ldg(reinterpret_cast<const uint2 *>(a.x + (int64_t)g * H + h));
            const float x0 = bf16_bits_to_f32(xb.x & 0xffff), x1 = bf16_bits_to_f32(xb.x >> 16);
            const float x2 = bf16_bits_to_f32(xb.y & 0xffff), x3 = bf16_bits_to_f32(xb.y >> 16);
            v = make_uint2(pack_h2(x0, x2), pack_h2(x1, x3));
            const float m = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
            bad |= m > 65504.0f && m <= 3.4e38f;     // finite but beyond the fp16 range
        }
        reinterpret_cast<uint2 *>(a.xfrag)[((cb * 8 + (s >> 1)) * 32 + ln) * 2 + (s & 1)] = v;
    }
    if (bad) set_status(a.header + kHdrStatus, MOE_ERR_DEVICE_FAULT);
    __syncthreads();

    float acc[kDecTok];
#pragma unroll
    for (int t = 0; t < kDecTok; ++t) acc[t] = 0.0f;
#pragma unroll
    for (int i = 0; i < kRouteMaxVec; ++i) {
        if (i < nv) {
            const int h = part * seg + (i * 32 + lane) * 4;
#pragma unroll
            for (int t = 0; t < kDecTok; ++t) {
                if (t < T) {
                    const uint2 xb = *reinterpret_cast<const uint2 *>(s_x + t * H + h);
                    acc[t] = fmaf(wv[i].x, bf16_bits_to_f32(xb.x & 0xffff), acc[t]);
                    acc[t] = fmaf(wv[i].y, bf16_bits_to_f32(xb.x >> 16), acc[t]);
                    acc[t] = fmaf(wv[i].z, bf16_bits_to_f32(xb.y & 0xffff), acc[t]);
                    acc[t] = fmaf(wv[i].w, bf16_bits_to_f32(xb.y >> 16), acc[t]);
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < kDecTok; ++t) {
        float v = acc[t];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == t) s_part[warp][t] = v;
    }
    __syncthreads();
    if (threadIdx.x < rpc * kDecTok) {
        const int rl = threadIdx.x / kDecTok, t = threadIdx.x % kDecTok, r = blockIdx.x * rpc + rl;
        if (r < E && t < T) {
            float v = 0.0f;
            for (int p = 0; p < P; ++p) v += s_part[rl * P + p][t];
            a.logits[(int64_t)t * E + r] = v;
        }
    }
    griddep_launch();
}

// Routing of the window inside each gate/up CTA (every CTA computes the same
// result; CTA 0 publishes it).  Shared scratch `scr` holds the logits and the
// sort; the plan (active experts and their tokens) stays in `pe` / `ptok`.
struct RouteScratch {
    uint32_t *key;       // [T][E] selection keys
    float *val;          // [T][E] logit (softmax) or sigmoid(logit): what the weight uses
    int32_t *ids;        // [T*k]
    float *w;            // [T*k]
    int32_t *rank;       // [T*k]
    int32_t *cnt;        // [kDecMaxAssign]  per active expert
    int32_t *off;        // [kDecMaxAssign]
    uint32_t *bits;      // [32]             selected-expert bitmap
    int32_t *pre;        // [32]             active experts before word l
};

__device__ void route_window(const DecArgs &a, const RouteScratch &sc, int16_t *pe, int16_t (*ptok)[kDecTok],
                             int *n_active_out)
{
    const int T = a.T, E = a.E, k = a.k, TK = T * k;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nthr = blockDim.x;
    // selection keys of every (token, expert): 4 loads in flight per thread
    for (int i0 = threadIdx.x; i0 < T * E; i0 += 4 * nthr) {
        float v[4], b[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = i0 + j * nthr;
            v[j] = i < T * E ? __ldcg(a.logits + i) : 0.0f;
            b[j] = (i < T * E && a.bias && a.score_fn != MOE_SCORE_SOFTMAX) ? __ldg(a.bias + i % E) : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = i0 + j * nthr;
            if (i < T * E) {
                const float sv = a.score_fn == MOE_SCORE_SOFTMAX ? v[j] : 1.0f / (1.0f + expf(-v[j]));
                sc.val[i] = sv;
                sc.key[i] = key_bits(a.score_fn == MOE_SCORE_SOFTMAX ? sv : sv + b[j]);
            }
        }
    }
    if (threadIdx.x < 32) sc.bits[threadIdx.x] = 0u;
    __syncthreads();
    if (warp < T) {
        int id;
        float wt;
        bool f;
        const uint32_t *kr = sc.key + warp * E;
        const float *lr = sc.val + warp * E;
        if (E <= 256) warp_topk<8>(kr, lr, E, k, a.score_fn, lane, id, wt, f);
        else if (E <= 512) warp_topk<16>(kr, lr, E, k, a.score_fn, lane, id, wt, f);
        else warp_topk<32>(kr, lr, E, k, a.score_fn, lane, id, wt, f);
        if (lane < k) {
            sc.ids[warp * k + lane] = id;
            sc.w[warp * k + lane] = wt;
            atomicOr(&sc.bits[id >> 5], 1u << (id & 31));
        }
        if (f && lane == 0 && blockIdx.x == 0) set_status(a.header + kHdrStatus, MOE_ERR_DEVICE_FAULT);
    }
    __syncthreads();
    if (warp == 0) {
        // active experts in id order: bitmap word l covers experts 32 l .. 32 l + 31
        const uint32_t word = sc.bits[lane];
        const int c = __popc(word);
        int incl = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        const int pre = incl - c, n_active = __shfl_sync(0xffffffffu, incl, 31);
        sc.pre[lane] = pre;
        {
            uint32_t wd = word;
            int j = pre;
            while (wd) {
                const int b = __ffs(wd) - 1;
                wd &= wd - 1;
                pe[j++] = (int16_t)(32 * lane + b);
            }
        }
        for (int u = lane; u < n_active; u += 32) {
            sc.cnt[u] = 0;
#pragma unroll
            for (int t = 0; t < kDecTok; ++t) ptok[u][t] = -1;
        }
        __syncwarp();
        // stable ranks within each expert, 32 assignments at a time
        for (int c0 = 0; c0 < TK; c0 += 32) {
            const int as = c0 + lane;
            const bool valid = as < TK;
            const int e = valid ? sc.ids[as] : -1 - lane;
            const unsigned peers = __match_any_sync(0xffffffffu, e);
            const int rk = __popc(peers & ((1u << lane) - 1u));
            int u = 0, base = 0;
            if (valid) {
                u = sc.pre[e >> 5] + __popc(sc.bits[e >> 5] & ((1u << (e & 31)) - 1u));
                base = sc.cnt[u];
            }
            __syncwarp();
            if (valid) {
                sc.rank[as] = base + rk;
                ptok[u][as / k] = (int16_t)as;
                if (rk == 0) sc.cnt[u] = base + __popc(peers);
            }
            __syncwarp();
        }
        // exclusive scan of the counts over active experts (id order)
        const int per = (n_active + 31) / 32;
        int tot = 0;
        for (int j = 0; j < per; ++j) {
            const int u = lane * per + j;
            if (u < n_active) tot += sc.cnt[u];
        }
        int inc2 = tot;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc2, off);
            if (lane >= off) inc2 += v;
        }
        int run = inc2 - tot;
        for (int j = 0; j < per; ++j) {
            const int u = lane * per + j;
            if (u < n_active) {
                sc.off[u] = run;
                run += sc.cnt[u];
            }
        }
        if (lane == 0) *n_active_out = n_active;
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        // publish: ids, w, counts, offsets, assign, active list, plan, n_active
        const int n_active = *n_active_out;
        for (int i = threadIdx.x; i < TK; i += nthr) {
            a.ids[i] = sc.ids[i];
            a.w[i] = sc.w[i];
            const int e = sc.ids[i];
            const int u = sc.pre[e >> 5] + __popc(sc.bits[e >> 5] & ((1u << (e & 31)) - 1u));
            a.assign[sc.off[u] + sc.rank[i]] = i;
        }
        for (int e = threadIdx.x; e < E; e += nthr) {
            const uint32_t wd = sc.bits[e >> 5];
            const int u = sc.pre[e >> 5] + __popc(wd & ((1u << (e & 31)) - 1u));   // active experts below e
            const bool sel = (wd >> (e & 31)) & 1u;
            a.counts[e] = sel ? sc.cnt[u] : 0;
            a.offsets[e] = u < n_active ? sc.off[u] : TK;
        }
        for (int u = threadIdx.x; u < n_active; u += nthr) {
            a.active[u] = pe[u];
            a.plan[u].e = pe[u];
            a.plan[u].count = sc.cnt[u];
#pragma unroll
            for (int t = 0; t < kDecTok; ++t) a.plan[u].tok_assign[t] = ptok[u][t];
        }
        if (threadIdx.x == 0) {
            a.offsets[E] = TK;
            a.header[kHdrNActive] = (uint32_t)n_active;
        }
    }
}

// ---------------------------------------------------------------- gate / up

// Work item (u, m): active expert u, ff indices 8m .. 8m+7 (8 gate rows + the
// 8 up rows of the same indices = one m16n8k16 M tile), optionally split in
// KS parts along H.  A CTA of 16 warps takes groups of 16 / KS items x KS
// parts (groups blockIdx.x, + gridDim.x, ...).  Each warp streams its stages
// -- one Q4_K block column of its 16 rows -- through its own ring of NST
// shared-memory slots with cp.async, NST - 1 stages ahead, across items.
//
// MMA operands: thread (g, t) holds rows g (gate) and g + 8 (up) and, in
// k-step s of a block, the elements 64t + 4s + {0, 2} (slots 2t, 2t+1) and
// 64t + 4s + {1, 3} (slots 2t+8, 2t+9); s < 8 are the low nibbles of qs bytes
// 32t + 4s .. +3 (sub-block 2t), s >= 8 the high nibbles of bytes
// 32t + 4(s-8) .. (sub-block 2t+1).  Nibbles become fp16 through the exponent
// field (0x6400 | q = 1024 + q; the high nibble in place gives 1024 + 16q).
constexpr int kGuWarps = 16;
constexpr int kMaxSmemPerBlock = 232448;         // sm_100-family opt-in limit (static + dynamic)
constexpr int kGuRowStride = 160;                 // 144 + 16: conflict-free 16-byte reads
constexpr int kGuStage = 16 * kGuRowStride;

// (S_a, S_b) = fp16(d * sc_j), fp16(-(dmin * m_j)) for the two sub-blocks j
// = 2t, 2t+1 of a Q4_K header; sel = byte selector of those two scales.
__device__ __forceinline__ void q4k_pair_scales(uint4 hdr, bool hi_group, uint32_t sel, __half2 &S, __half2 &NZ)
{
    // sc / m of sub-blocks 0..3 and 4..7, one per byte
    const uint32_t sc_lo = hdr.y & 0x3F3F3F3Fu, m_lo = hdr.z & 0x3F3F3F3Fu;
    const uint32_t sc_hi = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
    const uint32_t m_hi = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
    const uint32_t scw = hi_group ? sc_hi : sc_lo, mw = hi_group ? m_hi : m_lo;
    const __half2 k1024 = __float2half2_rn(1024.0f);
    const __half2 scv = __hsub2(u2h2(__byte_perm(scw, 0x64646464u, sel)), k1024);   // exact small integers
    const __half2 mv = __hsub2(u2h2(__byte_perm(mw, 0x64646464u, sel)), k1024);
    const uint32_t dd = __byte_perm(hdr.x, 0, 0x1010), mm = __byte_perm(hdr.x, 0, 0x3232) ^ 0x80008000u;
    S = __hmul2(u2h2(dd), scv);            // one rounding of the exact product
    NZ = __hmul2(u2h2(mm), mv);            // -(dmin * m)
}

template <int NST, int KS>
__global__ void __launch_bounds__(kGuWarps * 32, 1) k_dec_gateup(DecArgs a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    const int H = a.H, FF = a.FF, nb = H / 256, T = a.T, E = a.E, k = a.k;
    uint4 *s_xf = reinterpret_cast<uint4 *>(smem);                        // [H/256][8][32]
    uint8_t *ring = smem + (size_t)H * 16;                                 // [16 warps][NST][16 rows][160]
    float *s_red = reinterpret_cast<float *>(ring + kGuWarps * NST * kGuStage);   // [16][32][4]
    int16_t *pe = reinterpret_cast<int16_t *>(s_red + kGuWarps * 32 * 4);          // [256]
    int16_t(*ptok)[kDecTok] = reinterpret_cast<int16_t(*)[kDecTok]>(pe + kDecMaxAssign);
    const uint8_t **s_blob = reinterpret_cast<const uint8_t **>(ptok + kDecMaxAssign);   // [256]
    const uint8_t **s_tab = s_blob + kDecMaxAssign;                                         // [E]
    __shared__ int s_nact;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    uint8_t *myring = ring + warp * NST * kGuStage;

    // the expert table: before the dependency wait when the weights are static
    if (a.overlap_prev)
        for (int e = threadIdx.x; e < E; e += blockDim.x) s_tab[e] = a.blobs[e];
    griddep_wait();
    if (!a.overlap_prev)
        for (int e = threadIdx.x; e < E; e += blockDim.x) s_tab[e] = a.blobs[e];
    // x fragments into shared memory, asynchronously while the window is routed
    for (int i = threadIdx.x; i < nb * 256; i += blockDim.x) cp_async16(s_xf + i, a.xfrag + i);
    cp_async_commit();
    // route the window (scratch in the ring, which is not in use yet)
    {
        RouteScratch sc;
        uint8_t *p = ring;
        sc.key = reinterpret_cast<uint32_t *>(p);
        p += (size_t)T * E * 4;
        sc.val = reinterpret_cast<float *>(p);
        p += (size_t)T * E * 4;
        sc.ids = reinterpret_cast<int32_t *>(p);
        p += kDecMaxAssign * 4;
        sc.w = reinterpret_cast<float *>(p);
        p += kDecMaxAssign * 4;
        sc.rank = reinterpret_cast<int32_t *>(p);
        p += kDecMaxAssign * 4;
        sc.cnt = reinterpret_cast<int32_t *>(p);
        p += kDecMaxAssign * 4;
        sc.off = reinterpret_cast<int32_t *>(p);
        p += kDecMaxAssign * 4;
        sc.bits = reinterpret_cast<uint32_t *>(p);
        p += 32 * 4;
        sc.pre = reinterpret_cast<int32_t *>(p);
        route_window(a, sc, pe, ptok, &s_nact);
    }
    const int U = s_nact;
    const int64_t rb = (int64_t)nb * 144;
    const int mt = FF / 8, items = U * mt;
    const int ipg = kGuWarps / KS, n_groups = (items + ipg - 1) / ipg;
    const bool in_group = warp < ipg * KS;          // KS not dividing 16 leaves warps idle
    const int cpi = nb / KS;                                               // stages per item part

    for (int u = threadIdx.x; u < U; u += blockDim.x) s_blob[u] = s_tab[pe[u]];
    __syncthreads();
    // L2 prefetch of the down matrices of the selected experts (up to a budget),
    // one chunk per thread over the whole grid, so their bytes stream while
    // gate/up computes.
    if (a.prefetch_down) {
        const int64_t per_e = (int64_t)FF * rb;
        const int64_t total = std::min<int64_t>((int64_t)U * per_e, a.prefetch_budget);
        const int64_t chunk = 8192;
        const int64_t nchunks = (total + chunk - 1) / chunk;
        for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < nchunks; c += (int64_t)gridDim.x * blockDim.x) {
            const int64_t off = c * chunk;
            const int u = (int)(off / per_e);
            const int64_t in = off % per_e;
            const uint8_t *blob = s_blob[u];
            const int64_t len = std::min<int64_t>(chunk, std::min<int64_t>(per_e - in, total - off));
            if (blob) prefetch_l2_bulk(blob + 2 * (int64_t)FF * rb + in, (uint32_t)len);
        }
    }
    cp_async_wait<0>();
    __syncthreads();   // route scratch no longer needed; x fragments visible
    griddep_launch();

    const int my_groups = blockIdx.x < n_groups ? (n_groups - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int n_stages = my_groups * cpi;
    auto issue = [&](int s) {
        if (s < n_stages) {
            const int item = (blockIdx.x + (s / cpi) * gridDim.x) * ipg + warp / KS;
            if (in_group && item < items) {
                const int u = item / mt, f0 = (item % mt) * 8;
                const uint8_t *blob = s_blob[u];
                if (blob) {
                    const int cb = (warp % KS) * cpi + s % cpi;
                    uint8_t *slot = myring + (s % NST) * kGuStage;
                    for (int p = lane; p < 16 * 9; p += 32) {
                        const int r = p / 9, pc = p % 9;
                        const int64_t mrow = r < 8 ? f0 + r : FF + f0 + r - 8;
                        cp_async16(slot + r * kGuRowStride + pc * 16, blob + mrow * rb + (int64_t)cb * 144 + pc * 16);
                    }
                }
            }
        }
        cp_async_commit();
    };
#pragma unroll
    for (int p = 0; p < NST - 1; ++p) issue(p);

    // per-thread constants of the scale decode: sub-blocks 2t, 2t+1
    const bool hi_group = t >= 2;
    const uint32_t sel = t & 1 ? 0x5342u : 0x5140u;   // bytes (2, 3) or (0, 1) of the group's word
    const __half2 k1024 = __float2half2_rn(1024.0f), k16th = __float2half2_rn(0.0625f);

    int s = 0;
    for (int gi = 0; gi < my_groups; ++gi) {
        const int item = (blockIdx.x + gi * gridDim.x) * ipg + warp / KS;
        int u = 0, f0 = 0;
        bool live = in_group && item < items;
        if (live) {
            u = item / mt;
            f0 = (item % mt) * 8;
            if (!s_blob[u]) {
                if (lane == 0) set_status(a.header + kHdrStatus, MOE_ERR_DEVICE_FAULT);
                live = false;
            }
        }
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
        float c2[4] = {0.f, 0.f, 0.f, 0.f}, c3[4] = {0.f, 0.f, 0.f, 0.f};
        for (int ch = 0; ch < cpi; ++ch, ++s) {
            issue(s + NST - 1);
            cp_async_wait<NST - 1>();
            __syncwarp();
            if (live) {
                const uint8_t *slot = myring + (s % NST) * kGuStage;
                const int cb = (warp % KS) * cpi + ch;
                const uint8_t *gr = slot + g * kGuRowStride;
                const uint8_t *ur = slot + (8 + g) * kGuRowStride;
                const uint4 hg = *reinterpret_cast<const uint4 *>(gr);
                const uint4 hu = *reinterpret_cast<const uint4 *>(ur);
                const uint4 qg0 = *reinterpret_cast<const uint4 *>(gr + 16 + 32 * t);
                const uint4 qg1 = *reinterpret_cast<const uint4 *>(gr + 32 + 32 * t);
                const uint4 qu0 = *reinterpret_cast<const uint4 *>(ur + 16 + 32 * t);
                const uint4 qu1 = *reinterpret_cast<const uint4 *>(ur + 32 + 32 * t);
                uint4 bf[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) bf[i] = s_xf[(cb * 8 + i) * 32 + lane];
                __half2 Sg, NZg, Su, NZu;
                q4k_pair_scales(hg, hi_group, sel, Sg, NZg);
                q4k_pair_scales(hu, hi_group, sel, Su, NZu);
                const __half2 SGL = __low2half2(Sg), SGH = __hmul2(__high2half2(Sg), k16th);
                const __half2 NGL = __low2half2(NZg), NGH = __high2half2(NZg);
                const __half2 SUL = __low2half2(Su), SUH = __hmul2(__high2half2(Su), k16th);
                const __half2 NUL = __low2half2(NZu), NUH = __high2half2(NZu);
                const uint32_t wg[8] = {qg0.x, qg0.y, qg0.z, qg0.w, qg1.x, qg1.y, qg1.z, qg1.w};
                const uint32_t wu[8] = {qu0.x, qu0.y, qu0.z, qu0.w, qu1.x, qu1.y, qu1.z, qu1.w};
#pragma unroll
                for (int st = 0; st < 8; ++st) {
                    const uint32_t g8 = wg[st] >> 8, u8 = wu[st] >> 8;
                    // (1024 + q) of bytes (0, 2) and (1, 3), low nibbles; (1024 + 16q) high nibbles
                    const __half2 gl02 = __hsub2(u2h2((wg[st] & 0x000F000Fu) | 0x64006400u), k1024);
                    const __half2 gl13 = __hsub2(u2h2((g8 & 0x000F000Fu) | 0x64006400u), k1024);
                    const __half2 gh02 = __hsub2(u2h2((wg[st] & 0x00F000F0u) | 0x64006400u), k1024);
                    const __half2 gh13 = __hsub2(u2h2((g8 & 0x00F000F0u) | 0x64006400u), k1024);
                    const __half2 ul02 = __hsub2(u2h2((wu[st] & 0x000F000Fu) | 0x64006400u), k1024);
                    const __half2 ul13 = __hsub2(u2h2((u8 & 0x000F000Fu) | 0x64006400u), k1024);
                    const __half2 uh02 = __hsub2(u2h2((wu[st] & 0x00F000F0u) | 0x64006400u), k1024);
                    const __half2 uh13 = __hsub2(u2h2((u8 & 0x00F000F0u) | 0x64006400u), k1024);
                    const uint4 bl = bf[st >> 1], bh = bf[(st + 8) >> 1];
                    const uint32_t b0l = (st & 1) ? bl.z : bl.x, b1l = (st & 1) ? bl.w : bl.y;
                    const uint32_t b0h = (st & 1) ? bh.z : bh.x, b1h = (st & 1) ? bh.w : bh.y;
                    float(&cl)[4] = (st & 1) ? c1 : c0;
                    float(&ch4)[4] = (st & 1) ? c3 : c2;
                    mma16816(cl, h22u(__hfma2(gl02, SGL, NGL)), h22u(__hfma2(ul02, SUL, NUL)),
                             h22u(__hfma2(gl13, SGL, NGL)), h22u(__hfma2(ul13, SUL, NUL)), b0l, b1l);
                    mma16816(ch4, h22u(__hfma2(gh02, SGH, NGH)), h22u(__hfma2(uh02, SUH, NUH)),
                             h22u(__hfma2(gh13, SGH, NGH)), h22u(__hfma2(uh13, SUH, NUH)), b0h, b1h);
                }
            }
            __syncwarp();
        }
        float c[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) c[i] = (c0[i] + c1[i]) + (c2[i] + c3[i]);
        if (KS > 1 && in_group) {
            // the KS warps of this item meet on their own named barrier (ids 1..16/KS)
            const int bar = 1 + warp / KS;
            if (warp % KS != 0) {
#pragma unroll
                for (int i = 0; i < 4; ++i) s_red[(warp * 32 + lane) * 4 + i] = c[i];
            }
            asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(KS * 32) : "memory");
            if (warp % KS == 0) {
                for (int j = 1; j < KS; ++j)
#pragma unroll
                    for (int i = 0; i < 4; ++i) c[i] += s_red[((warp + j) * 32 + lane) * 4 + i];
            }
            asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(KS * 32) : "memory");
        }
        if (live && warp % KS == 0) {
            // c0, c1: gate of ff f0+g for tokens 2t, 2t+1; c2, c3: up
            const int f = f0 + g;
            const int a0 = ptok[u][2 * t], a1 = ptok[u][2 * t + 1];
            if (a0 >= 0) a.act[(int64_t)a0 * FF + f] = silu_mul(c[0], c[2]);
            if (a1 >= 0) a.act[(int64_t)a1 * FF + f] = silu_mul(c[1], c[3]);
        }
    }
    cp_async_wait<0>();
    (void)T;
    (void)k;
}

// ---------------------------------------------------------------- down

// Unit (active expert u, hidden block cb, ff segment fs): the segment's FR <=
// kDnMaxRows rows of block column cb (144 bytes each).  One warp per unit:
// the warp stages its units in its own two shared-memory buffers with
// cp.async, one unit ahead, and the activations of the unit's tokens next to
// them.  Lane (q = lane & 7, rl = lane >> 3) takes the 16 quant bytes q of
// rows rl, rl + 4, ...: 32 weights, 16 of sub-block 2c and 16 of sub-block
// 2c + 1 (c = q / 2).  With v = 0.5 + q/256 (the nibble placed in the fp32
// mantissa) a weight is s*q - z = 256 s v - (128 s + z), so
// sum_f a_f w_f = sum_f (256 a_f s_f) v_f - sum_f a_f (128 s_f + z_f): one
// FMA per weight and token; the second sum once per row and sub-block.
constexpr int kDnWarps = 4;                 // warps (independent units) per CTA
constexpr int kDnThreads = kDnWarps * 32;
constexpr int kDnMaxRows = 80;
constexpr int kDnRowStride = 160;           // 144 + 16 padding
// one unit buffer: FR rows + the activations of 2 tokens for them
__host__ __device__ constexpr int dn_buf_bytes(int FR) { return (FR * kDnRowStride + 2 * FR * 4 + 15) & ~15; }
constexpr int kDnRegCtas = 3;               // CTAs per SM the kernel's registers allow

// fp32 scale and min of the sub-block pair (2c, 2c + 1) of a Q4_K header:
// d * sc and dmin * m, each one rounding (exact integer conversions).
__device__ __forceinline__ void q4k_pair_scales_f(uint4 hdr, int c, float &s0, float &z0, float &s1, float &z1)
{
    const uint32_t sc_lo = hdr.y & 0x3F3F3F3Fu, m_lo = hdr.z & 0x3F3F3F3Fu;
    const uint32_t sc_hi = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
    const uint32_t m_hi = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
    const uint32_t scw = c >= 2 ? sc_hi : sc_lo, mw = c >= 2 ? m_hi : m_lo;
    const uint32_t sel0 = (c & 1) ? 0x4442u : 0x4440u, sel1 = (c & 1) ? 0x4443u : 0x4441u;   // byte -> low byte
    const float k23 = 8388608.0f;
    const float sc0 = __uint_as_float(__byte_perm(scw, 0x4B000000u, sel0 | 0x7000u)) - k23;
    const float sc1 = __uint_as_float(__byte_perm(scw, 0x4B000000u, sel1 | 0x7000u)) - k23;
    const float m0 = __uint_as_float(__byte_perm(mw, 0x4B000000u, sel0 | 0x7000u)) - k23;
    const float m1 = __uint_as_float(__byte_perm(mw, 0x4B000000u, sel1 | 0x7000u)) - k23;
    const float d = f16_bits_to_f32(hdr.x & 0xffff), dmin = f16_bits_to_f32(hdr.x >> 16);
    s0 = __fmul_rn(d, sc0);
    s1 = __fmul_rn(d, sc1);
    z0 = __fmul_rn(dmin, m0);
    z1 = __fmul_rn(dmin, m1);
}

__global__ void __launch_bounds__(kDnThreads, kDnRegCtas) k_dec_down(DecArgs a)
{
    extern __shared__ __align__(16) uint8_t smem[];     // [warp][nbuf][buffer]
    griddep_wait();
    griddep_launch();   // the finish kernel may launch now (it waits for this grid before reading)
    const int U = (int)a.header[kHdrNActive];
    const int H = a.H, FF = a.FF, nb = H / 256, FS = a.fs_dn;
    const int64_t rb = (int64_t)nb * 144;
    const int units = U * nb * FS;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int q = lane & 7, rl = lane >> 3;
    const int c = q >> 1, l0 = 16 * (q & 1);
    const int FR = FF / FS;
    const int NB = a.dn_nbuf, BB = dn_buf_bytes(FR);
    uint8_t *wbuf = smem + warp * NB * BB;
    const int gw = blockIdx.x * kDnWarps + warp, nw = gridDim.x * kDnWarps;

    auto unit_of = [&](int unit, int &u, int &cb, int &fs) {
        u = unit / (nb * FS);
        const int rem = unit % (nb * FS);
        cb = rem / FS;
        fs = rem % FS;
    };
    auto issue = [&](int unit, int buf) {
        if (unit < units) {
            int u, cb, fs;
            unit_of(unit, u, cb, fs);
            const uint8_t *blob = a.blobs[a.plan[u].e];
            if (blob) {
                const uint8_t *src = blob + (2 * (int64_t)FF + (int64_t)fs * FR) * rb + (int64_t)cb * 144;
                uint8_t *dst = wbuf + buf * BB;
                for (int p = lane; p < FR * 9; p += 32) {
                    const int row = p / 9, pc = p % 9;
                    cp_async16(dst + row * kDnRowStride + pc * 16, src + row * rb + pc * 16);
                }
            }
        }
        cp_async_commit();
    };

    // two buffers: the next unit is staged while this one computes; one buffer
    // (a warp with a single unit, the usual case): the next unit, if any, is
    // staged after this one
    issue(gw, 0);
    int buf = 0;
    for (int unit = gw; unit < units; unit += nw, buf ^= (NB - 1)) {
        if (NB == 2) issue(unit + nw, buf ^ 1);
        int u, cb, fs;
        unit_of(unit, u, cb, fs);
        if (!a.blobs[a.plan[u].e]) {
            if (lane == 0) set_status(a.header + kHdrStatus, MOE_ERR_DEVICE_FAULT);
            if (NB == 1) {
                cp_async_wait<0>();
                __syncwarp();
                issue(unit + nw, 0);
            }
            continue;
        }
        // the window tokens routed to this expert (bit t: token t), taken two per pass
        int tok_as[kDecTok];
        uint32_t pm = 0;
#pragma unroll
        for (int tt = 0; tt < kDecTok; ++tt) {
            tok_as[tt] = a.plan[u].tok_assign[tt];
            if (tok_as[tt] >= 0) pm |= 1u << tt;
        }
        const int n = __popc(pm);
        uint8_t *tile = wbuf + buf * BB;
        float *s_act = reinterpret_cast<float *>(tile + FR * kDnRowStride);   // [2][FR]
        for (int p0 = 0; p0 < n; p0 += 2) {
            const int np = min(2, n - p0);
            int as0 = -1, as1 = -1, seen = 0;
#pragma unroll
            for (int tt = 0; tt < kDecTok; ++tt)
                if ((pm >> tt) & 1u) {
                    if (seen == p0) as0 = tok_as[tt];
                    if (seen == p0 + 1) as1 = tok_as[tt];
                    ++seen;
                }
            // activations of the pass's tokens for the segment's rows (written by the previous kernel)
            __syncwarp();
            for (int i = lane; i < 2 * FR; i += 32) {
                const int tk = i / FR, row = i % FR;
                const int as = tk ? as1 : as0;
                s_act[tk * FR + row] = as >= 0 ? __ldg(a.act + (int64_t)as * FF + fs * FR + row) : 0.0f;
            }
            if (NB == 2) cp_async_wait<1>();
            else cp_async_wait<0>();
            __syncwarp();
            float acc[2][32];
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[0][j] = acc[1][j] = 0.0f;
            float zl0 = 0.0f, zh0 = 0.0f, zl1 = 0.0f, zh1 = 0.0f;
#pragma unroll 2
            for (int row = rl; row < FR; row += 4) {
                const uint4 hv = *reinterpret_cast<const uint4 *>(tile + row * kDnRowStride);
                const uint4 qv = *reinterpret_cast<const uint4 *>(tile + row * kDnRowStride + 16 + 16 * q);
                const float av0 = s_act[row], av1 = s_act[FR + row];
                float sl, zl, sh, zh;
                q4k_pair_scales_f(hv, c, sl, zl, sh, zh);
                const float A0l = 256.0f * av0 * sl, A0h = 256.0f * av0 * sh;
                const float A1l = 256.0f * av1 * sl, A1h = 256.0f * av1 * sh;
                zl0 = fmaf(av0, fmaf(128.0f, sl, zl), zl0);
                zh0 = fmaf(av0, fmaf(128.0f, sh, zh), zh0);
                zl1 = fmaf(av1, fmaf(128.0f, sl, zl), zl1);
                zh1 = fmaf(av1, fmaf(128.0f, sh, zh), zh1);
                const uint32_t wds[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
                for (int wi = 0; wi < 4; ++wi) {
                    const uint32_t lo = wds[wi] & 0x0F0F0F0Fu, hi = (wds[wi] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
                    for (int bb = 0; bb < 4; ++bb) {
                        const float vl = __uint_as_float(__byte_perm(lo, 0x3F000000u, 0x7044 | (bb << 8)));
                        const float vh = __uint_as_float(__byte_perm(hi, 0x3F000000u, 0x7044 | (bb << 8)));
                        acc[0][4 * wi + bb] = fmaf(A0l, vl, acc[0][4 * wi + bb]);
                        acc[0][16 + 4 * wi + bb] = fmaf(A0h, vh, acc[0][16 + 4 * wi + bb]);
                        if (np > 1) {
                            acc[1][4 * wi + bb] = fmaf(A1l, vl, acc[1][4 * wi + bb]);
                            acc[1][16 + 4 * wi + bb] = fmaf(A1h, vh, acc[1][16 + 4 * wi + bb]);
                        }
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                acc[0][j] -= zl0;
                acc[0][16 + j] -= zh0;
                acc[1][j] -= zl1;
                acc[1][16 + j] -= zh1;
            }
            // sum the 4 row lanes (lanes q, q + 8, q + 16, q + 24)
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                acc[0][j] += __shfl_xor_sync(0xffffffffu, acc[0][j], 8);
                acc[0][j] += __shfl_xor_sync(0xffffffffu, acc[0][j], 16);
                if (np > 1) {
                    acc[1][j] += __shfl_xor_sync(0xffffffffu, acc[1][j], 8);
                    acc[1][j] += __shfl_xor_sync(0xffffffffu, acc[1][j], 16);
                }
            }
            // lane (q, rl) writes token (rl & 1) and the low (rl < 2) or high 16 columns of its chunk
            const int pt = rl & 1, part = rl >> 1;
            if (pt < np) {
                const int as = pt ? as1 : as0;
                const float wt = a.w[as];
                const int tok = as / a.k;
                const int h = 256 * cb + 64 * c + 32 * part + l0;
                float o[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float lo0 = acc[0][j], hi0 = acc[0][16 + j], lo1 = acc[1][j], hi1 = acc[1][16 + j];
                    o[j] = (part ? (pt ? hi1 : hi0) : (pt ? lo1 : lo0)) * wt;
                }
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    if (a.det) {
                        float *dst = a.slots + ((int64_t)as * FS + fs) * H + h + 4 * v;
                        *reinterpret_cast<float4 *>(dst) = make_float4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
                    } else {
                        float *dst = a.yacc + (int64_t)tok * H + h + 4 * v;
                        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(o[4 * v]),
                                     "f"(o[4 * v + 1]), "f"(o[4 * v + 2]), "f"(o[4 * v + 3])
                                     : "memory");
                    }
                }
            }
        }
        if (NB == 1) {
            __syncwarp();              // every lane is done with the buffer
            issue(unit + nw, 0);
        }
    }
    cp_async_wait<0>();
}

// y = bf16(accumulated y), or the fixed-order sum of the slots in
// deterministic mode, plus the shared expert's output; float4 per thread.
__global__ void __launch_bounds__(256) k_dec_finish(DecArgs a)
{
    // the next call's router may launch now: before its own dependency wait it
    // reads only the (static) router rows
    griddep_launch();
    griddep_wait();
    const int H = a.H, FS = a.fs_dn, k = a.k;
    const int n4 = a.T * H / 4;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += gridDim.x * blockDim.x) {
        float4 v;
        if (a.det) {
            const int t = (4 * i) / H, h = (4 * i) % H;
            v = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int r = 0; r < k; ++r)
                for (int f = 0; f < FS; ++f) {
                    const float4 sv = __ldg(reinterpret_cast<const float4 *>(a.slots + ((int64_t)(t * k + r) * FS + f) * H + h));
                    v.x += sv.x; v.y += sv.y; v.z += sv.z; v.w += sv.w;
                }
        } else {
            v = __ldg(reinterpret_cast<const float4 *>(a.yacc) + i);
        }
        if (a.sh_out) {
            const float4 sv = __ldg(reinterpret_cast<const float4 *>(a.sh_out) + i);
            v.x += sv.x; v.y += sv.y; v.z += sv.z; v.w += sv.w;
        }
        const uint32_t lo = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.x)) |
                            ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.y)) << 16);
        const uint32_t hi = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.z)) |
                            ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.w)) << 16);
        reinterpret_cast<uint2 *>(a.y)[i] = make_uint2(lo, hi);
        if (a.y_f32) reinterpret_cast<float4 *>(a.y_f32)[i] = v;
    }
}

// ---------------------------------------------------------------- launch

static int dec_sms()
{
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

int dec_route_parts(int H)
{
    for (int P = 1; P <= 8; P *= 2)
        if (H % (128 * P) == 0 && H / (128 * P) <= kRouteMaxVec) return P;
    return 0;   // unsupported
}

// ff segments per down unit: at most kDnMaxRows rows each, and enough units
// for two per SM.
// Down units (expert, block column, ff segment) are spread over the warps of
// the grid.  A unit buffer holds FR = ff / fs rows; with one buffer per warp
// (every warp has at most one unit) more CTAs fit on an SM than with two.
static int64_t dn_warps(int64_t units, int FR, int nbuf)
{
    const int64_t smem = (int64_t)kDnWarps * nbuf * dn_buf_bytes(FR);
    const int64_t by_smem = 233472 / (smem + 1024);
    const int64_t per_sm = std::max<int64_t>(1, std::min<int64_t>(by_smem, kDnRegCtas));
    const int64_t ctas = std::min<int64_t>((units + kDnWarps - 1) / kDnWarps, per_sm * dec_sms());
    return ctas * kDnWarps;
}

int dec_down_nbuf(const moe_config &c, int32_t T, int fs)
{
    const int64_t maxu = std::min<int64_t>(c.n_experts, (int64_t)T * c.top_k);
    const int64_t units = maxu * (c.hidden / 256) * fs;
    return units <= dn_warps(units, c.ff / fs, 1) ? 1 : 2;
}

int dec_down_splits(const moe_config &c, int32_t T)
{
    const int64_t maxu = std::min<int64_t>(c.n_experts, (int64_t)T * c.top_k);
    const int64_t nb = c.hidden / 256;
    int fs = 1;
    while (c.ff % fs || c.ff / fs > kDnMaxRows) ++fs;      // segments of at most kDnMaxRows rows
    if (c.flags & MOE_FLAG_DETERMINISTIC) return fs;
    // The slowest warp takes ceil(units / warps) units: pick the segmentation
    // with the least work on that warp (its rows' bytes plus a per-unit cost:
    // the unit's additions into y and its fixed latency).
    int64_t best_cost = -1;
    int best = fs;
    for (int f2 = fs; f2 <= 64; ++f2) {
        if (c.ff % f2 || (f2 > fs && c.ff / f2 < 32)) continue;     // segments of >= 32 rows

        const int64_t units = maxu * nb * f2;
        const int64_t warps = dn_warps(units, c.ff / f2, dec_down_nbuf(c, T, f2));
        const int64_t rounds = (units + warps - 1) / warps;
        const int64_t cost = rounds * ((int64_t)(c.ff / f2) * 144 + (int64_t)T * 2048 + 2048);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = f2;
        }
    }
    return best;
}

template <typename K>
static cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                              const DecArgs &a)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

// Ring depth of the gate/up stages: the deepest (up to four) that shared memory holds.
int dec_gateup_stages(int H, int E)
{
    const size_t fixed = (size_t)H * 16 + kGuWarps * 32 * 4 * sizeof(float) + kDecMaxAssign * 2 * (1 + kDecTok) +
                         kDecMaxAssign * sizeof(void *) + (size_t)E * sizeof(void *);
    for (int nst = 4; nst > 2; --nst)
        if (fixed + (size_t)kGuWarps * nst * kGuStage + 1024 <= (size_t)kMaxSmemPerBlock) return nst;
    return 2;
}

static size_t gateup_smem(const DecArgs &a, int nst)
{
    const size_t ring = (size_t)kGuWarps * nst * kGuStage;
    // the routing scratch lives in the ring before the first stage
    const size_t route = (size_t)a.T * a.E * 8 + 5 * kDecMaxAssign * 4 + 64 * 4;
    return (size_t)a.H * 16 + std::max(ring, route) + kGuWarps * 32 * 4 * sizeof(float) +
           kDecMaxAssign * 2 * (1 + kDecTok) + kDecMaxAssign * sizeof(void *) + (size_t)a.E * sizeof(void *);
}

template <int NST, int KS>
static cudaError_t launch_gateup(const DecArgs &a, int grid, cudaStream_t s)
{
    static bool attr = false;
    if (!attr) {
        cudaFuncAttributes fa{};
        cudaError_t e = cudaFuncGetAttributes(&fa, k_dec_gateup<NST, KS>);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_dec_gateup<NST, KS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kMaxSmemPerBlock - (int)fa.sharedSizeBytes);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    return launch_pdl(k_dec_gateup<NST, KS>, dim3(grid), dim3(kGuWarps * 32), gateup_smem(a, NST), s, true, a);
}

cudaError_t launch_decode(const DecArgs &a0, cudaStream_t s)
{
    DecArgs a = a0;
    if (a.T <= 0) return cudaSuccess;
    cudaError_t e;
    static bool attr = false;
    if (!attr) {
        e = cudaFuncSetAttribute(k_dec_route, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kDecTok * 8192 * (int)sizeof(uint16_t));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_dec_down, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kDnWarps * 2 * dn_buf_bytes(kDnMaxRows));
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const int rpc = 8 / a.route_parts;
    prof_begin(kPhDecRoute, s);
    e = launch_pdl(k_dec_route, dim3((a.E + rpc - 1) / rpc), dim3(kRouteThreads), (size_t)a.T * a.H * 2, s,
                   a.overlap_prev != 0, a);
    prof_end(kPhDecRoute, s);
    if (e != cudaSuccess) return e;

    const int sms = dec_sms();
    const int64_t maxu = std::min<int64_t>(a.E, (int64_t)a.T * a.k);
    const int nb = a.H / 256;
    const int NST = dec_gateup_stages(a.H, a.E);
    const int64_t items = maxu * (a.FF / 8);
    // K split of an item: a divisor of the block count (1, 2, 4, 5, 8, 10, 16);
    // groups of 16 / ks items go round-robin to the CTAs, so the slowest CTA
    // runs ceil(groups / CTAs) groups of nb / ks block columns per warp (plus
    // the ks-way reduction); pick the split with the least of that
    int ks = 1;
    double best_cost = -1.0;
    for (int cand : {1, 2, 4, 5, 8, 10, 16}) {
        if (nb % cand) continue;
        const int64_t grp = (items + kGuWarps / cand - 1) / (kGuWarps / cand);
        const int64_t rounds = (grp + sms - 1) / sms;
        const double cost = (double)rounds * ((double)(nb / cand) + (cand > 1 ? 0.25 : 0.0));
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            ks = cand;
        }
    }
    const int ipg = kGuWarps / ks;
    const int64_t groups = (items + ipg - 1) / ipg;
    const int grid_gu = (int)std::max<int64_t>(1, std::min<int64_t>(groups, sms));
    prof_begin(kPhDecGateUp, s);
#define MOE_GU_CASES(NS)                                                                                           \
    ks == 1 ? launch_gateup<NS, 1>(a, grid_gu, s) : ks == 2 ? launch_gateup<NS, 2>(a, grid_gu, s)                   \
    : ks == 4 ? launch_gateup<NS, 4>(a, grid_gu, s) : ks == 5 ? launch_gateup<NS, 5>(a, grid_gu, s)                 \
    : ks == 8 ? launch_gateup<NS, 8>(a, grid_gu, s) : ks == 10 ? launch_gateup<NS, 10>(a, grid_gu, s)               \
              : launch_gateup<NS, 16>(a, grid_gu, s)
    e = NST == 4 ? (MOE_GU_CASES(4)) : NST == 3 ? (MOE_GU_CASES(3)) : (MOE_GU_CASES(2));
#undef MOE_GU_CASES
    prof_end(kPhDecGateUp, s);
    if (e != cudaSuccess) return e;

    if (a.shared_blob) {
        e = launch_shared_gemv(a, s);
        if (e != cudaSuccess) return e;
    }

    const int64_t units = maxu * nb * a.fs_dn;
    const int FR = a.FF / a.fs_dn;
    const int grid_dn = (int)std::max<int64_t>(1, dn_warps(units, FR, a.dn_nbuf) / kDnWarps);
    prof_begin(kPhDecDown, s);
    e = launch_pdl(k_dec_down, dim3(grid_dn), dim3(kDnThreads), (size_t)kDnWarps * a.dn_nbuf * dn_buf_bytes(FR), s,
                   true, a);
    prof_end(kPhDecDown, s);
    if (e != cudaSuccess) return e;
    const int n4 = a.T * a.H / 4;
    prof_begin(kPhDecFinish, s);
    e = launch_pdl(k_dec_finish, dim3(std::max(1, std::min((n4 + 255) / 256, sms))), dim3(256), 0, s, true, a);
    prof_end(kPhDecFinish, s);
    return e;
}

}  // namespace moe
