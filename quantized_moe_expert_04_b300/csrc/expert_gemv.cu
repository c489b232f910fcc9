// expert_gemv.cu -- grouped expert GEMV for decode / MTP-verify windows
// (T <= 8 tokens), fp32 arithmetic on exactly dequantised weights.
//
// The teardown page ("Strata 引擎深度拆解", lcz.me/topic/2098/5, section 一,
// CPU ledger) describes a multi-token expert kernel that applies each
// expert's bytes to every token of a 3-token verify window at once; the
// decode critical path there is the expert arithmetic (section 二 item 5).
// Here every selected expert's Q4_K bytes are streamed once per window and
// applied to all of that expert's tokens:
//   k_gateup  warp per (expert, FF row): a = SiLU(Wg x) * (Wu x) for each of
//             the expert's tokens; act is indexed by bucket position.
//   k_down    warp per (expert, 256 hidden columns): o = sum_f a_f Wd[f][:],
//             scaled by the routing weight into the assignment's slot.
// The shared expert (Q8_0) runs through the same kernels as an expert whose
// bucket is every token with weight 1.
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {

constexpr int kChunk = 8;     // tokens whose accumulators a lane keeps in registers

enum Fmt { kFmtQ4K = 0, kFmtQ80 = 1 };

template <int FMT> struct RowFmt;

// Q4_K row along H: lane-group of 8 consecutive weights e0 .. e0+7 (e0 % 8 == 0).
template <> struct RowFmt<kFmtQ4K> {
    static __host__ __device__ int64_t row_bytes(int H) { return (int64_t)(H / kQK) * kQ4KBytes; }
    static __device__ __forceinline__ void load8(const uint8_t *row, int e0, float v[8])
    {
        const uint8_t *blk = row + (e0 / kQK) * kQ4KBytes;
        const int i = e0 % kQK;                       // 0, 8, ..., 248
        const int c = i >> 6, within = i & 63;
        const int half = within >> 5, l0 = within & 31;
        const uint4 hdr = __ldg(reinterpret_cast<const uint4 *>(blk));
        const float d = f16_bits_to_f32(hdr.x & 0xffff), dmin = f16_bits_to_f32(hdr.x >> 16);
        uint8_t scales[12];
        *reinterpret_cast<uint32_t *>(scales) = hdr.y;
        *reinterpret_cast<uint32_t *>(scales + 4) = hdr.z;
        *reinterpret_cast<uint32_t *>(scales + 8) = hdr.w;
        int sc, m;
        q4k_scale_min(scales, 2 * c + half, sc, m);
        const float s = __fmul_rn(d, (float)sc), z = __fmul_rn(dmin, (float)m);
        const uint2 qv = __ldg(reinterpret_cast<const uint2 *>(blk + 16 + 32 * c + l0));
        const int shift = half ? 4 : 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint32_t word = e < 4 ? qv.x : qv.y;
            const int q = (word >> (8 * (e & 3) + shift)) & 15;
            v[e] = __fsub_rn(__fmul_rn(s, (float)q), z);
        }
    }
};

// Q8_0 row along H.
template <> struct RowFmt<kFmtQ80> {
    static __host__ __device__ int64_t row_bytes(int H) { return (int64_t)(H / kQK8) * kQ8Bytes; }
    static __device__ __forceinline__ void load8(const uint8_t *row, int e0, float v[8])
    {
        const uint8_t *blk = row + (e0 / kQK8) * kQ8Bytes;
        const int i = e0 % kQK8;
        const float d = f16_bits_to_f32((uint32_t)blk[0] | ((uint32_t)blk[1] << 8));
        // 2-byte aligned (34-byte blocks): four 16-bit loads
        const uint16_t *q16 = reinterpret_cast<const uint16_t *>(blk + 2 + i);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t pair = q16[e];
            v[2 * e] = __fmul_rn(d, (float)(int8_t)(pair & 0xff));
            v[2 * e + 1] = __fmul_rn(d, (float)(int8_t)(pair >> 8));
        }
    }
};

__device__ __forceinline__ void load_x8(const uint16_t *x, float v[8])
{
    const uint4 p = __ldg(reinterpret_cast<const uint4 *>(x));
    v[0] = bf16_bits_to_f32(p.x & 0xffff); v[1] = bf16_bits_to_f32(p.x >> 16);
    v[2] = bf16_bits_to_f32(p.y & 0xffff); v[3] = bf16_bits_to_f32(p.y >> 16);
    v[4] = bf16_bits_to_f32(p.z & 0xffff); v[5] = bf16_bits_to_f32(p.z >> 16);
    v[6] = bf16_bits_to_f32(p.w & 0xffff); v[7] = bf16_bits_to_f32(p.w >> 16);
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// Bucket of one work unit: routed expert u (active index) or the shared expert.
struct Bucket {
    const uint8_t *blob;
    int begin, count;    // positions in assign order (routed) or tokens (shared)
};

template <bool SHARED>
__device__ __forceinline__ bool get_bucket(const ExpertArgs &a, int u, Bucket &bk)
{
    if (SHARED) {
        bk.blob = a.shared_blob;
        bk.begin = 0;
        bk.count = a.T;
        return u == 0;
    }
    const int n_active = (int)a.header[kHdrNActive];
    if (u >= n_active) return false;
    const int e = a.active[u];
    bk.blob = a.blobs[e];
    bk.begin = a.offsets[e];
    bk.count = a.offsets[e + 1] - bk.begin;
    if (bk.blob == nullptr) {
        set_status(a.header + kHdrStatus, MOE_ERR_DEVICE_FAULT);
        return false;
    }
    return true;
}

template <int FMT, bool SHARED>
__global__ void __launch_bounds__(256) k_gateup(ExpertArgs a)
{
    const int FF = SHARED ? a.SFF : a.FF;
    const int lane = threadIdx.x & 31;
    const int64_t task = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int u = (int)(task / FF), f = (int)(task % FF);
    Bucket bk;
    if (!get_bucket<SHARED>(a, u, bk)) return;
    const int64_t rb = RowFmt<FMT>::row_bytes(a.H);
    const uint8_t *grow = bk.blob + (int64_t)f * rb;
    const uint8_t *urow = bk.blob + ((int64_t)FF + f) * rb;
    float *act = SHARED ? a.sh_act : a.act;
    for (int c0 = 0; c0 < bk.count; c0 += kChunk) {
        const int nt = min(kChunk, bk.count - c0);
        int tok[kChunk];
#pragma unroll
        for (int j = 0; j < kChunk; ++j)
            tok[j] = j < nt ? (SHARED ? c0 + j : a.assign[bk.begin + c0 + j] / a.k) : 0;
        float ag[kChunk], au[kChunk];
#pragma unroll
        for (int j = 0; j < kChunk; ++j) ag[j] = au[j] = 0.0f;
        for (int h = lane * 8; h < a.H; h += 256) {
            float wg[8], wu[8];
            RowFmt<FMT>::load8(grow, h, wg);
            RowFmt<FMT>::load8(urow, h, wu);
#pragma unroll
            for (int j = 0; j < kChunk; ++j) {
                if (j < nt) {
                    float xv[8];
                    load_x8(a.x + (int64_t)tok[j] * a.H + h, xv);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        ag[j] = fmaf(wg[i], xv[i], ag[j]);
                        au[j] = fmaf(wu[i], xv[i], au[j]);
                    }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
            const float g = warp_sum(ag[j]), uu = warp_sum(au[j]);
            if (lane == j && j < nt) act[(int64_t)(bk.begin + c0 + j) * FF + f] = silu_mul(g, uu);
        }
    }
}

template <int FMT, bool SHARED>
__global__ void __launch_bounds__(256) k_down(ExpertArgs a)
{
    const int FF = SHARED ? a.SFF : a.FF;
    const int lane = threadIdx.x & 31;
    const int nhb = a.H / 256;                       // 256-column groups
    const int64_t task = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int u = (int)(task / nhb), hb = (int)(task % nhb);
    Bucket bk;
    if (!get_bucket<SHARED>(a, u, bk)) return;
    const int64_t rb = RowFmt<FMT>::row_bytes(a.H);
    const uint8_t *dbase = bk.blob + 2 * (int64_t)FF * rb;
    const float *act = SHARED ? a.sh_act : a.act;
    const int h0 = hb * 256 + lane * 8;
    for (int c0 = 0; c0 < bk.count; c0 += kChunk) {
        const int nt = min(kChunk, bk.count - c0);
        float acc[kChunk][8];
#pragma unroll
        for (int j = 0; j < kChunk; ++j)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[j][i] = 0.0f;
        for (int f = 0; f < FF; ++f) {
            float wv[8];
            RowFmt<FMT>::load8(dbase + (int64_t)f * rb, h0, wv);
#pragma unroll
            for (int j = 0; j < kChunk; ++j) {
                if (j < nt) {
                    const float av = act[(int64_t)(bk.begin + c0 + j) * FF + f];
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[j][i] = fmaf(av, wv[i], acc[j][i]);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
            if (j < nt) {
                float *dst;
                float wt = 1.0f;
                if (SHARED) {
                    dst = a.sh_out + (int64_t)(c0 + j) * a.H + h0;
                } else {
                    const int asg = a.assign[bk.begin + c0 + j];
                    wt = a.w[asg];
                    dst = a.slots + (int64_t)asg * a.H + h0;
                }
                float4 *d4 = reinterpret_cast<float4 *>(dst);
                d4[0] = make_float4(wt * acc[j][0], wt * acc[j][1], wt * acc[j][2], wt * acc[j][3]);
                d4[1] = make_float4(wt * acc[j][4], wt * acc[j][5], wt * acc[j][6], wt * acc[j][7]);
            }
        }
    }
}

static unsigned blocks_for_warps(int64_t warps) { return (unsigned)((warps + 7) / 8); }

// Shared-expert down projection: warp (256-column block hb, ff segment fs)
// accumulates sum_f sh_act[t][f] * Wd[f][h] over its FR rows for every token,
// lane l owning columns 256 hb + 8 l .. + 7 (a quarter of one Q8_0 block), and
// adds the result into sh_out (zeroed by the routing kernel); with one
// segment (deterministic mode) it stores instead.
__global__ void __launch_bounds__(256) k_shared_down(ExpertArgs a, int nfs)
{
    const int lane = threadIdx.x & 31;
    const int64_t task = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nhb = a.H / 256;
    if (task >= (int64_t)nhb * nfs) return;
    const int hb = (int)(task % nhb), fs = (int)(task / nhb);
    const int FR = a.SFF / nfs, T = a.T;
    const int64_t rb = RowFmt<kFmtQ80>::row_bytes(a.H);
    const uint8_t *dbase = a.shared_blob + 2 * (int64_t)a.SFF * rb;
    const int h0 = hb * 256 + lane * 8;
    float acc[kChunk][8];
#pragma unroll
    for (int j = 0; j < kChunk; ++j)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[j][i] = 0.0f;
    for (int r = 0; r < FR; ++r) {
        const int f = fs * FR + r;
        float wv[8];
        RowFmt<kFmtQ80>::load8(dbase + (int64_t)f * rb, h0, wv);
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
            if (j < T) {
                const float av = __ldg(a.sh_act + (int64_t)j * a.SFF + f);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[j][i] = fmaf(av, wv[i], acc[j][i]);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
        if (j < T) {
            float *dst = a.sh_out + (int64_t)j * a.H + h0;
            if (nfs == 1) {
                reinterpret_cast<float4 *>(dst)[0] = make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
                reinterpret_cast<float4 *>(dst)[1] = make_float4(acc[j][4], acc[j][5], acc[j][6], acc[j][7]);
            } else {
                asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(acc[j][0]), "f"(acc[j][1]),
                             "f"(acc[j][2]), "f"(acc[j][3]) : "memory");
                asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 4), "f"(acc[j][4]),
                             "f"(acc[j][5]), "f"(acc[j][6]), "f"(acc[j][7]) : "memory");
            }
        }
    }
}

// The shared expert of a decode window (every token, weight 1): gate/up into
// sh_act, down into sh_out; the finish kernel adds sh_out to y.
cudaError_t launch_shared_gemv(const DecArgs &d, cudaStream_t s)
{
    ExpertArgs a{};
    a.H = d.H;
    a.E = d.E;
    a.FF = d.FF;
    a.k = d.k;
    a.T = d.T;
    a.SFF = d.SFF;
    a.x = d.x;
    a.shared_blob = d.shared_blob;
    a.sh_act = d.sh_act;
    a.sh_out = d.sh_out;
    a.header = d.header;
    prof_begin(kPhGateUpShared, s);
    k_gateup<kFmtQ80, true><<<blocks_for_warps(a.SFF), 256, 0, s>>>(a);
    prof_end(kPhGateUpShared, s);
    int nfs = 1;
    if (!d.det)
        while (nfs < 64 && a.SFF % (2 * nfs) == 0 && a.SFF / (2 * nfs) >= 32) nfs *= 2;
    prof_begin(kPhDownShared, s);
    k_shared_down<<<blocks_for_warps((int64_t)(a.H / 256) * nfs), 256, 0, s>>>(a, nfs);
    prof_end(kPhDownShared, s);
    return cudaGetLastError();
}

}  // namespace moe
