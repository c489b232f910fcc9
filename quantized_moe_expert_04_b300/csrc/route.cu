// route.cu -- router scoring, top-k selection and token-to-expert bucketing.
//
// The router picks ~10 of 512 experts per token in the Qwen-shaped model
// ("Strata 引擎深度拆解", lcz.me/topic/2098/5, section 二) and 6 of 256
// with a per-expert router bias in the DeepSeek-shaped one ("Strata 改源码去跑
// DeepSeek V4 Flash？", lcz.me/post/23082, section 二, anatomy table).  The
// multi-token expert kernel of the teardown page (section 一, CPU ledger)
// computes each expert once for all tokens of a window; the bucketing below
// groups a window's (token, slot) assignments by expert for exactly that.
//
// Kernels:
//   k_router_logits  fp32 logits [T][E]: warps own experts, a CTA owns up to
//                    8 tokens whose bf16 rows sit in shared memory, so each
//                    router row is read once per 8 tokens.
//   k_topk           one warp per token, E/32 logits per lane in registers,
//                    sorted per lane, k rounds of a warp arg-max (equal
//                    keys: lower id).
//   k_bucket_*       stable counting sort of the T*k assignments over the grid.
#include <algorithm>
#include <mutex>
#include "moe_internal.cuh"
#include "topk_warp.cuh"

namespace moe {

constexpr int kRouterTokens = 8;     // tokens per CTA in the logits kernel
constexpr int kRouterWarps = 4;      // warps per CTA (one expert row at a time each)

__global__ void __launch_bounds__(kRouterWarps * 32)
k_router_logits(const uint16_t *__restrict__ x, const float *__restrict__ wr, int T, int H, int E,
                int experts_per_cta, float *__restrict__ logits)
{
    extern __shared__ __align__(16) uint16_t xs[];     // [kRouterTokens][H] bf16
    const int t0 = blockIdx.y * kRouterTokens;
    const int nt = min(kRouterTokens, T - t0);
    // stage the token rows (16-byte vectors)
    {
        const int vec_per_row = H / 8;
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (int64_t)t0 * H);
        uint4 *dst = reinterpret_cast<uint4 *>(xs);
        for (int i = threadIdx.x; i < nt * vec_per_row; i += blockDim.x) dst[i] = src[i];
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int e_begin = blockIdx.x * experts_per_cta;
    const int e_end = min(E, e_begin + experts_per_cta);
    for (int e = e_begin + warp; e < e_end; e += kRouterWarps) {
        const float4 *row = reinterpret_cast<const float4 *>(wr + (int64_t)e * H);
        float acc[kRouterTokens];
#pragma unroll
        for (int t = 0; t < kRouterTokens; ++t) acc[t] = 0.0f;
        for (int h4 = lane; h4 < H / 4; h4 += 32) {
            const float4 wv = row[h4];
#pragma unroll
            for (int t = 0; t < kRouterTokens; ++t) {
                if (t < nt) {
                    const uint2 xv = *reinterpret_cast<const uint2 *>(xs + t * H + 4 * h4);
                    acc[t] = fmaf(wv.x, bf16_bits_to_f32(xv.x & 0xffff), acc[t]);
                    acc[t] = fmaf(wv.y, bf16_bits_to_f32(xv.x >> 16), acc[t]);
                    acc[t] = fmaf(wv.z, bf16_bits_to_f32(xv.y & 0xffff), acc[t]);
                    acc[t] = fmaf(wv.w, bf16_bits_to_f32(xv.y >> 16), acc[t]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < kRouterTokens; ++t) {
            float v = acc[t];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if (lane == t && t < nt) logits[(int64_t)(t0 + t) * E + e] = v;
        }
    }
}

// Router logits for larger T on the tensor cores (k_router_tc, gemm_tc.cu):
// each fp32 router weight is split exactly into three bf16 parts (w = w1 + w2
// + w3: 8 significant bits each), so with bf16 x the three bf16 x bf16
// products are exact and the MMAs accumulate them in fp32 -- the logits of an
// fp32 dot product, in another summation order.  The split is done once per
// call, into the workspace.
constexpr int kRmK = 64;                // the tensor-core kernel's K stage: H % kRmK == 0

// w -> (w1, w2, w3) bf16 with w1 + w2 + w3 == w
__device__ __forceinline__ void split3(float w, uint16_t &a, uint16_t &b, uint16_t &c)
{
    const __nv_bfloat16 h1 = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(h1);
    const __nv_bfloat16 h2 = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(h2);
    const __nv_bfloat16 h3 = __float2bfloat16_rn(r2);
    a = __bfloat16_as_ushort(h1);
    b = __bfloat16_as_ushort(h2);
    c = __bfloat16_as_ushort(h3);
}

// The router matrix split once per call for the tensor-core logits:
// planes[sp][e][h] (sp = 0, 1, 2) with planes[0] + planes[1] + planes[2] == wr
// exactly (split3).
__global__ void __launch_bounds__(256) k_router_split(const float *__restrict__ wr, int64_t n,
                                                      uint16_t *__restrict__ planes)
{
    for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n / 4; i += (int64_t)gridDim.x * 256) {
        const float4 w = __ldg(reinterpret_cast<const float4 *>(wr) + i);
        uint16_t h[3][4];
        split3(w.x, h[0][0], h[1][0], h[2][0]);
        split3(w.y, h[0][1], h[1][1], h[2][1]);
        split3(w.z, h[0][2], h[1][2], h[2][2]);
        split3(w.w, h[0][3], h[1][3], h[2][3]);
#pragma unroll
        for (int sp = 0; sp < 3; ++sp)
            reinterpret_cast<uint2 *>(planes + sp * n)[i] =
                make_uint2((uint32_t)h[sp][0] | ((uint32_t)h[sp][1] << 16), (uint32_t)h[sp][2] | ((uint32_t)h[sp][3] << 16));
    }
}

// One warp per token.  Keys: the logit (softmax: the order of p equals the
// order of the logits) or s_e + b_e (sigmoid), as order-preserving integers
// (NaN -> 0, never selected); lane l holds experts l, l + 32, ... (NPER) and
// warp_select (topk_warp.cuh) takes the k largest, ties to the lower id.
// Weights: softmax over the k selected logits (= the full softmax
// renormalised over the k), or s_e / sum of the selected s.
__device__ __forceinline__ uint32_t topk_key(float f)
{
    if (isnan(f)) return 0u;
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The float a non-zero topk_key came from.
__device__ __forceinline__ float topk_key_value(uint32_t key)
{
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// (Four CTAs an SM up to 512 experts: every token's warp resident in one wave
// at T = 4096.)
template <int NPER>
__global__ void __launch_bounds__(256, NPER <= 16 ? 4 : 2)
k_topk(const float *__restrict__ logits, const float *__restrict__ bias, int T, int E, int k,
       int score_fn, int32_t *__restrict__ ids, float *__restrict__ wout, uint32_t *status)
{
    const int lane = threadIdx.x & 31;
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    const float *lrow = logits + (int64_t)t * E;
    // all of the lane's loads in flight first
    float lg[NPER];
#pragma unroll
    for (int i = 0; i < NPER; ++i) lg[i] = __ldg(lrow + min(lane + 32 * i, E - 1));
    uint32_t key[NPER];
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
        const int e = lane + 32 * i;
        key[i] = 0u;
        if (e < E) {
            if (score_fn == MOE_SCORE_SOFTMAX) {
                key[i] = topk_key(lg[i]);
            } else {
                const float sg = 1.0f / (1.0f + expf(-lg[i]));
                key[i] = topk_key(sg + (bias ? __ldg(bias + e) : 0.0f));
            }
        }
    }
    int my_id;
    uint32_t my_key;
    bool fault;
    warp_select<NPER>(key, k, lane, my_id, my_key, fault);
    // weights over the k selected (lane r holds selection r): the selected
    // logit (softmax; recovered from its key) or s = sigmoid(logit), as above
    float my_val = 0.0f;
    if (lane < k && my_key != 0u)
        my_val = score_fn == MOE_SCORE_SOFTMAX ? topk_key_value(my_key)
                                               : 1.0f / (1.0f + expf(-__ldg(lrow + my_id)));
    float num;
    if (score_fn == MOE_SCORE_SOFTMAX) {
        const float lmax = __shfl_sync(0xffffffffu, my_val, 0);   // the first pick is the largest
        num = lane < k ? expf(my_val - lmax) : 0.0f;
    } else {
        num = lane < k ? my_val : 0.0f;
    }
    float den = num;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
    if (lane < k) {
        ids[(int64_t)t * k + lane] = my_id;
        wout[(int64_t)t * k + lane] = num / den;
    }
    if (fault && lane == 0) set_status(status, MOE_ERR_DEVICE_FAULT);
}

// Stable counting sort of the T*k assignments by expert, over the grid: CTA
// b owns the kBucketItems assignments [b*kBucketItems, (b+1)*kBucketItems).
//   1. k_bucket_hist: each CTA's per-expert counts (shared-memory atomics);
//   2. k_bucket_scan (one CTA): per expert, the CTAs' counts prefix-summed in
//      CTA order (in place: bhist[b][e] = how many assignments to e the CTAs
//      before b hold) and the expert totals scanned -> counts, offsets, the
//      ascending list of experts that received tokens;
//   3. k_bucket_scatter: CTA b's first assignment to e goes to offsets[e] +
//      bhist[b][e]; within a CTA, lanes with the same expert are ranked
//      by lane (__match_any_sync) and warps by a per-expert prefix over the
//      warps, so equal keys keep the input order -- the sort is stable.
__global__ void __launch_bounds__(kBucketItems)
k_bucket_hist(const int32_t *__restrict__ ids, int TK, int E, int32_t *__restrict__ bhist, uint32_t *header)
{
    extern __shared__ int32_t h[];               // [E]
    for (int i = threadIdx.x; i < E; i += blockDim.x) h[i] = 0;
    __syncthreads();
    const int a = blockIdx.x * kBucketItems + threadIdx.x;
    bool bad = false;
    if (a < TK) {
        const int e = __ldg(ids + a);
        if (e >= 0 && e < E) atomicAdd(&h[e], 1);
        else bad = true;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < E; i += blockDim.x) bhist[(int64_t)blockIdx.x * E + i] = h[i];
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) set_status(header + kHdrStatus, MOE_ERR_DEVICE_FAULT);
}

__global__ void __launch_bounds__(1024)
k_bucket_scan(int nblk, int E, int32_t *__restrict__ bhist, int32_t *__restrict__ counts,
              int32_t *__restrict__ offsets, int32_t *__restrict__ active, uint32_t *header)
{
    __shared__ int32_t w_tot[32], w_act[32];
    const int e = threadIdx.x, lane = e & 31, warp = e >> 5;   // one thread per expert (E <= 1024)
    int tot = 0;
    if (e < E) {
        // the expert's column over the CTAs: 16 loads in flight, then their
        // exclusive prefix written back in their place
        for (int b0 = 0; b0 < nblk; b0 += 16) {
            int c[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) c[j] = b0 + j < nblk ? bhist[(int64_t)(b0 + j) * E + e] : 0;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (b0 + j < nblk) {
                    bhist[(int64_t)(b0 + j) * E + e] = tot;
                    tot += c[j];
                }
        }
        counts[e] = tot;
    }
    // inclusive scans over the experts of the totals and of (total > 0):
    // within each warp, then over the 32 warps' sums
    int sum = tot, act = tot > 0 ? 1 : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, sum, off), b = __shfl_up_sync(0xffffffffu, act, off);
        if (lane >= off) {
            sum += a;
            act += b;
        }
    }
    if (lane == 31) {
        w_tot[warp] = sum;
        w_act[warp] = act;
    }
    __syncthreads();
    if (warp == 0) {
        int ws = w_tot[lane], wa = w_act[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, ws, off), b = __shfl_up_sync(0xffffffffu, wa, off);
            if (lane >= off) {
                ws += a;
                wa += b;
            }
        }
        w_tot[lane] = ws;
        w_act[lane] = wa;
    }
    __syncthreads();
    if (warp > 0) {
        sum += w_tot[warp - 1];
        act += w_act[warp - 1];
    }
    if (e < E) {
        offsets[e] = sum - tot;
        if (tot > 0) active[act - 1] = e;
    }
    if (e == 1023) {
        offsets[E] = sum;                        // = number of valid assignments
        header[kHdrNActive] = (uint32_t)act;
    }
}

__global__ void __launch_bounds__(kBucketItems)
k_bucket_scatter(const int32_t *__restrict__ ids, int TK, int E, const int32_t *__restrict__ bhist,
                 const int32_t *__restrict__ offsets, int32_t *__restrict__ assign)
{
    extern __shared__ int32_t wh[];              // [32 warps][E]
    for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wh[i] = 0;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int a = blockIdx.x * kBucketItems + threadIdx.x;
    int e = a < TK ? __ldg(ids + a) : -1;
    const bool valid = e >= 0 && e < E;
    if (!valid) e = -1 - lane;                   // a key no other lane holds
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (valid && rank == 0) wh[warp * E + e] = __popc(peers);
    __syncthreads();
    for (int x = threadIdx.x; x < E; x += blockDim.x) {
        int run = 0;
#pragma unroll 8
        for (int w = 0; w < 32; ++w) {
            const int c = wh[w * E + x];
            wh[w * E + x] = run;
            run += c;
        }
    }
    __syncthreads();
    if (valid) assign[__ldg(offsets + e) + bhist[(int64_t)blockIdx.x * E + e] + wh[warp * E + e] + rank] = a;
}

cudaError_t launch_route(const RouteArgs &a, cudaStream_t s)
{
    if (a.T <= 0) {
        // offsets all zero, no active experts
        cudaMemsetAsync(a.offsets, 0, sizeof(int32_t) * (a.E + 1), s);
        cudaMemsetAsync(a.counts, 0, sizeof(int32_t) * a.E, s);
        cudaMemsetAsync(a.header + kHdrNActive, 0, sizeof(uint32_t), s);
        return cudaGetLastError();
    }
    // opt-in shared memory limits: function attributes are per device, set once for
    // each device this process launches on
    {
        static std::mutex mu;
        static bool done[64] = {};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev]) {
            e = cudaFuncSetAttribute(k_router_logits, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)(kRouterTokens * 8192 * sizeof(uint16_t)));
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(k_bucket_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(32 * 1024 * sizeof(int32_t)));
            if (e != cudaSuccess) return e;
            done[dev] = true;
        }
    }
    const size_t xs_bytes = (size_t)kRouterTokens * a.H * sizeof(uint16_t);
    const int experts_per_cta = a.T > kRouterTokens ? 16 * kRouterWarps : kRouterWarps;
    dim3 grid((a.E + experts_per_cta - 1) / experts_per_cta, (a.T + kRouterTokens - 1) / kRouterTokens);
    prof_begin(kPhRouterLogits, s);
    if (router_split_bytes(a.E, a.H, a.T) > 0) {
        // tensor-core logits: the split planes, then tcgen05 tiles
        const int64_t n = (int64_t)a.E * a.H;
        k_router_split<<<(unsigned)std::min<int64_t>((n / 4 + 255) / 256, 148 * 16), 256, 0, s>>>(a.wr, n, a.wsplit);
        const cudaError_t e2 = launch_router_tc(a.x, a.wsplit, a.T, a.H, a.E, a.logits, a.header + kHdrStatus,
                                                debug_wait_cycles(), s);
        if (e2 != cudaSuccess) {
            prof_end(kPhRouterLogits, s);
            return e2;
        }
    } else {
        k_router_logits<<<grid, kRouterWarps * 32, xs_bytes, s>>>(a.x, a.wr, a.T, a.H, a.E, experts_per_cta,
                                                                  a.logits);
    }
    prof_end(kPhRouterLogits, s);
    const int warps_per_block = 8;
    prof_begin(kPhTopk, s);
    {
        const dim3 g((a.T + warps_per_block - 1) / warps_per_block), b(warps_per_block * 32);
        const float *bias = a.score_fn == MOE_SCORE_SIGMOID_BIAS ? a.bias : nullptr;
        if (a.E <= 256) k_topk<8><<<g, b, 0, s>>>(a.logits, bias, a.T, a.E, a.k, a.score_fn, a.ids, a.w, a.header + kHdrStatus);
        else if (a.E <= 512) k_topk<16><<<g, b, 0, s>>>(a.logits, bias, a.T, a.E, a.k, a.score_fn, a.ids, a.w, a.header + kHdrStatus);
        else k_topk<32><<<g, b, 0, s>>>(a.logits, bias, a.T, a.E, a.k, a.score_fn, a.ids, a.w, a.header + kHdrStatus);
    }
    prof_end(kPhTopk, s);
    const int TK = a.T * a.k, nblk = (TK + kBucketItems - 1) / kBucketItems;
    prof_begin(kPhBucket, s);
    k_bucket_hist<<<nblk, kBucketItems, a.E * sizeof(int32_t), s>>>(a.ids, TK, a.E, a.bhist, a.header);
    k_bucket_scan<<<1, 1024, 0, s>>>(nblk, a.E, a.bhist, a.counts, a.offsets, a.active, a.header);
    k_bucket_scatter<<<nblk, kBucketItems, 32 * a.E * sizeof(int32_t), s>>>(a.ids, TK, a.E, a.bhist, a.offsets,
                                                                            a.assign);
    prof_end(kPhBucket, s);
    return cudaGetLastError();
}

// Bytes of the split router planes the tensor-core logits read (0: the call
// takes the scalar logits kernel).
size_t router_split_bytes(int E, int H, int T)
{
    return T > kRouterTokens && H % kRmK == 0 ? (size_t)3 * E * H * sizeof(uint16_t) : 0;
}

}  // namespace moe
