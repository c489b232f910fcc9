// pack.cu -- device-side Q4_K / Q5_K / Q8_0 quantisers and the dequantisation test
// hooks.  Every fp32 step uses the explicitly rounded intrinsics (__fadd_rn,
// __fmul_rn, __fdiv_rn, ...) so that no multiply-add is fused and the bytes
// equal those of the quantiser's definition (stated in include/moe.h).
//
// The pages name Q4_K for the routed experts and Q8_0 for the shared expert
// ("Strata 改源码去跑 DeepSeek V4 Flash？", lcz.me/post/23082, section 二,
// GGUF anatomy table) and a pack step that converts tensors before serving
// ("Qwen3.8-Flash-Next UD-Q4_K_XL 引擎对比", lcz.me/user/wml-ai/posts,
// section 一, pack conversions); the quantiser itself is not on the pages.
#include "moe_internal.cuh"
#include "dequant_f16.cuh"

namespace moe {

// One warp per 256-weight super-block; lane l owns weights 8l .. 8l+7, which
// lie in sub-block l/4 and, in the packed quants, in chunk c = l/8 as the
// low (l%8 < 4) or high (l%8 >= 4) nibbles of bytes 32c + 8(l%4) .. +7.
// Q5 = true: the Q5_K layout -- 31 levels, the quants' low four bits packed as
// above at byte 48, their fifth bits in qh[32] at byte 16 (bit j of qh[e] = the
// fifth bit of element e of sub-block j).
template <bool Q5>
__global__ void __launch_bounds__(256) k_pack_qk(const float *__restrict__ w, int64_t nblocks,
                                                 uint8_t *__restrict__ out, uint32_t *status)
{
    constexpr float kLevels = Q5 ? 31.0f : 15.0f;
    constexpr int kBytes = Q5 ? kQ5KBytes : kQ4KBytes, kQsAt = Q5 ? 48 : 16;
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < nblocks; b += nwarps) {
        const float4 *src = reinterpret_cast<const float4 *>(w + b * kQK + lane * 8);
        const float4 v0 = src[0], v1 = src[1];
        const float x[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};

        bool bad = false;
        float mn = x[0], mx = x[0];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            bad |= !isfinite(x[i]);
            mn = x[i] < mn ? x[i] : mn;
            mx = x[i] > mx ? x[i] : mx;
        }
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {       // the 4 lanes of one sub-block
            const float omn = __shfl_xor_sync(0xffffffffu, mn, off);
            const float omx = __shfl_xor_sync(0xffffffffu, mx, off);
            mn = omn < mn ? omn : mn;
            mx = omx > mx ? omx : mx;
        }
        if (mn > 0.0f) mn = 0.0f;
        const float scale = __fdiv_rn(__fsub_rn(mx, mn), kLevels);
        const float nmin = -mn;

        // max over the 8 sub-blocks, starting from +0 like a running maximum
        float ms = scale > 0.0f ? scale : 0.0f, mm = nmin > 0.0f ? nmin : 0.0f;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            const float os = __shfl_xor_sync(0xffffffffu, ms, off);
            const float om = __shfl_xor_sync(0xffffffffu, mm, off);
            ms = os > ms ? os : ms;
            mm = om > mm ? om : mm;
        }
        const unsigned short d_h = __half_as_ushort(__float2half_rn(__fdiv_rn(ms, 63.0f)));
        const unsigned short dm_h = __half_as_ushort(__float2half_rn(__fdiv_rn(mm, 63.0f)));
        const float d = f16_bits_to_f32(d_h), dmin = f16_bits_to_f32(dm_h);
        bad |= !isfinite(d) || !isfinite(dmin);

        const int sc = d > 0.0f ? (int)fminf(63.0f, rintf(__fdiv_rn(scale, d))) : 0;
        const int m = dmin > 0.0f ? (int)fminf(63.0f, rintf(__fdiv_rn(nmin, dmin))) : 0;
        const float s = __fmul_rn(d, (float)sc), z = __fmul_rn(dmin, (float)m);

        uint32_t packed = 0;                        // my 8 quants, 4 bits each
        uint64_t fifth = 0;                         // Q5_K: their fifth bits, as qh bytes 8 (lane % 4) .. + 7
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int q = 0;
            if (s > 0.0f) {
                const float v = rintf(__fdiv_rn(__fadd_rn(x[i], z), s));
                q = v < 0.0f ? 0 : (v > kLevels ? (int)kLevels : (int)v);
            }
            packed |= (uint32_t)(q & 15) << (4 * i);
            if (Q5) fifth |= (uint64_t)(q >> 4) << (8 * i + (lane >> 2));   // qh byte i, bit = sub-block
        }
        const uint32_t hi = __shfl_down_sync(0xffffffffu, packed, 4);   // lane l+4: high nibbles
        uint8_t *blk = out + b * kBytes;
        if (Q5) {
            // the 8 sub-blocks' fifth bits of elements 8 (lane % 4) .. + 7: OR over lanes l % 4
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) fifth |= __shfl_xor_sync(0xffffffffu, fifth, off);
            if (lane < 4)
                *reinterpret_cast<uint2 *>(blk + 16 + 8 * lane) = make_uint2((uint32_t)fifth, (uint32_t)(fifth >> 32));
        }
        if ((lane & 7) < 4) {
            uint32_t lo_word = 0, hi_word = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                lo_word |= (((packed >> (4 * i)) & 15u) | (((hi >> (4 * i)) & 15u) << 4)) << (8 * i);
                hi_word |= (((packed >> (4 * (i + 4))) & 15u) | (((hi >> (4 * (i + 4))) & 15u) << 4)) << (8 * i);
            }
            const int c = lane >> 3;
            *reinterpret_cast<uint2 *>(blk + kQsAt + 32 * c + 8 * (lane & 3)) = make_uint2(lo_word, hi_word);
        }

        // header: gather the 8 (sc, m) pairs from lanes 0, 4, ..., 28
        int scj[8], mj[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            scj[j] = __shfl_sync(0xffffffffu, sc, 4 * j);
            mj[j] = __shfl_sync(0xffffffffu, m, 4 * j);
        }
        if (lane == 0) {
            uint8_t sb[12];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                sb[j] = (uint8_t)(scj[j] | ((scj[j + 4] >> 4) << 6));
                sb[j + 4] = (uint8_t)(mj[j] | ((mj[j + 4] >> 4) << 6));
                sb[j + 8] = (uint8_t)((scj[j + 4] & 15) | ((mj[j + 4] & 15) << 4));
            }
            uint4 hdr;
            hdr.x = (uint32_t)d_h | ((uint32_t)dm_h << 16);
            hdr.y = sb[0] | (sb[1] << 8) | (sb[2] << 16) | ((uint32_t)sb[3] << 24);
            hdr.z = sb[4] | (sb[5] << 8) | (sb[6] << 16) | ((uint32_t)sb[7] << 24);
            hdr.w = sb[8] | (sb[9] << 8) | (sb[10] << 16) | ((uint32_t)sb[11] << 24);
            *reinterpret_cast<uint4 *>(blk) = hdr;
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(status, MOE_ERR_DEVICE_FAULT);
    }
}

// One warp per 32-weight Q8_0 block, one lane per weight.
__global__ void __launch_bounds__(256) k_pack_q8_0(const float *__restrict__ w, int64_t nblocks,
                                                   uint8_t *__restrict__ out, uint32_t *status)
{
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < nblocks; b += nwarps) {
        const float x = w[b * kQK8 + lane];
        bool bad = !isfinite(x);
        float a = fabsf(x);
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, a, off);
            a = o > a ? o : a;
        }
        const unsigned short d_h = __half_as_ushort(__float2half_rn(__fdiv_rn(a, 127.0f)));
        const float d = f16_bits_to_f32(d_h);
        bad |= !isfinite(d);
        int q = 0;
        if (d > 0.0f) {
            const float v = rintf(__fdiv_rn(x, d));
            q = v < -127.0f ? -127 : (v > 127.0f ? 127 : (int)v);
        }
        uint8_t *blk = out + b * kQ8Bytes;
        blk[2 + lane] = (uint8_t)(int8_t)q;
        if (lane == 0) {
            blk[0] = (uint8_t)(d_h & 0xff);
            blk[1] = (uint8_t)(d_h >> 8);
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(status, MOE_ERR_DEVICE_FAULT);
    }
}

// Thread per 8 weights: same lane <-> weight mapping as the quantiser.
__global__ void __launch_bounds__(256) k_dequant_q4k(const uint8_t *__restrict__ blocks, int64_t nblocks,
                                                     float *__restrict__ out)
{
    const int64_t n = nblocks * 32;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = i >> 5;
        const int l = (int)(i & 31);
        const uint8_t *blk = blocks + b * kQ4KBytes;
        const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
        const float d = f16_bits_to_f32(hdr.x & 0xffff), dmin = f16_bits_to_f32(hdr.x >> 16);
        uint8_t scales[12];
        *reinterpret_cast<uint32_t *>(scales) = hdr.y;
        *reinterpret_cast<uint32_t *>(scales + 4) = hdr.z;
        *reinterpret_cast<uint32_t *>(scales + 8) = hdr.w;
        int sc, m;
        q4k_scale_min(scales, l >> 2, sc, m);
        const float s = __fmul_rn(d, (float)sc), z = __fmul_rn(dmin, (float)m);
        const uint2 qv = *reinterpret_cast<const uint2 *>(blk + 16 + 32 * (l >> 3) + 8 * (l & 3));
        const int shift = (l & 7) < 4 ? 0 : 4;
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint32_t word = e < 4 ? qv.x : qv.y;
            const int q = (word >> (8 * (e & 3) + shift)) & 15;
            y[e] = __fsub_rn(__fmul_rn(s, (float)q), z);
        }
        float4 *dst = reinterpret_cast<float4 *>(out + b * kQK + 8 * l);
        dst[0] = make_float4(y[0], y[1], y[2], y[3]);
        dst[1] = make_float4(y[4], y[5], y[6], y[7]);
    }
}

// Q5_K: thread per 8 weights, as k_dequant_q4k; the fifth bit of element
// 64c + 32h + l is bit 2c + h of qh[l].
__global__ void __launch_bounds__(256) k_dequant_q5k(const uint8_t *__restrict__ blocks, int64_t nblocks,
                                                     float *__restrict__ out)
{
    const int64_t n = nblocks * 32;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = i >> 5;
        const int l = (int)(i & 31), j = l >> 2;             // weights 8l .. 8l + 7: sub-block j
        const int c = j >> 1, h = j & 1, l0 = 8 * (l & 3);  // elements 64c + 32h + l0 ..
        const uint8_t *blk = blocks + b * kQ5KBytes;
        const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
        const float d = f16_bits_to_f32(hdr.x & 0xffff), dmin = f16_bits_to_f32(hdr.x >> 16);
        uint8_t scales[12];
        *reinterpret_cast<uint32_t *>(scales) = hdr.y;
        *reinterpret_cast<uint32_t *>(scales + 4) = hdr.z;
        *reinterpret_cast<uint32_t *>(scales + 8) = hdr.w;
        int sc, m;
        q4k_scale_min(scales, j, sc, m);
        const float s = __fmul_rn(d, (float)sc), z = __fmul_rn(dmin, (float)m);
        const uint2 qv = *reinterpret_cast<const uint2 *>(blk + 48 + 32 * c + l0);
        const uint2 hv = *reinterpret_cast<const uint2 *>(blk + 16 + l0);
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint32_t word = e < 4 ? qv.x : qv.y, hw = e < 4 ? hv.x : hv.y;
            const int lo = (word >> (8 * (e & 3) + 4 * h)) & 15;
            const int q = lo | (((hw >> (8 * (e & 3) + 2 * c + h)) & 1) << 4);
            y[e] = __fsub_rn(__fmul_rn(s, (float)q), z);
        }
        float4 *dst = reinterpret_cast<float4 *>(out + b * kQK + 8 * l);
        dst[0] = make_float4(y[0], y[1], y[2], y[3]);
        dst[1] = make_float4(y[4], y[5], y[6], y[7]);
    }
}

__global__ void __launch_bounds__(256) k_dequant_q8_0(const uint8_t *__restrict__ blocks, int64_t nblocks,
                                                      float *__restrict__ out)
{
    const int64_t n = nblocks * kQK8;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint8_t *blk = blocks + (i >> 5) * kQ8Bytes;
        const float d = f16_bits_to_f32((uint32_t)blk[0] | ((uint32_t)blk[1] << 8));
        out[i] = __fmul_rn(d, (float)(int8_t)blk[2 + (i & 31)]);
    }
}

// The fp16 operand rounding of the tensor-core paths, through the very
// functions their fused kernels call (dequant_f16.cuh): thread per (block,
// 4-byte word of the quants) -> 8 fp16 weights.
__global__ void __launch_bounds__(256) k_dequant_q4k_f16(const uint8_t *__restrict__ blocks, int64_t nblocks,
                                                         uint16_t *__restrict__ out)
{
    const int64_t n = nblocks * 32;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = i >> 5;
        const int wi = (int)(i & 31), c = wi >> 3, i4 = wi & 7;     // chunk c (sub-blocks 2c, 2c+1), word i4
        const uint8_t *blk = blocks + b * kQ4KBytes;
        const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
        __half2 S, NZ;
        q4k_pair_scales_h(hdr, c, S, NZ);
        uint32_t o[4];
        q4k_word_f16(*reinterpret_cast<const uint32_t *>(blk + 16 + 32 * c + 4 * i4), __low2half2(S), __low2half2(NZ),
                     __high2half2(S), __high2half2(NZ), o);
        uint32_t *dst = reinterpret_cast<uint32_t *>(out + b * kQK + 64 * c + 4 * i4);
        dst[0] = o[0];
        dst[1] = o[1];
        dst[16] = o[2];            // elements 64c + 32 + 4 i4 ...
        dst[17] = o[3];
    }
}

__global__ void __launch_bounds__(256) k_dequant_q5k_f16(const uint8_t *__restrict__ blocks, int64_t nblocks,
                                                         uint16_t *__restrict__ out)
{
    const int64_t n = nblocks * 32;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = i >> 5;
        const int wi = (int)(i & 31), c = wi >> 3, i4 = wi & 7;
        const uint8_t *blk = blocks + b * kQ5KBytes;
        const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
        __half2 S, NZ;
        q4k_pair_scales_h(hdr, c, S, NZ);
        const uint32_t hb = *reinterpret_cast<const uint32_t *>(blk + 16 + 4 * i4) >> (2 * c);
        uint32_t o[4];
        q5k_word_f16(*reinterpret_cast<const uint32_t *>(blk + 48 + 32 * c + 4 * i4), hb, __low2half2(S),
                     __low2half2(NZ), __high2half2(S), __high2half2(NZ), o);
        uint32_t *dst = reinterpret_cast<uint32_t *>(out + b * kQK + 64 * c + 4 * i4);
        dst[0] = o[0];
        dst[1] = o[1];
        dst[16] = o[2];
        dst[17] = o[3];
    }
}

__global__ void __launch_bounds__(256) k_dequant_q8_0_f16(const uint8_t *__restrict__ blocks, int64_t nblocks,
                                                          uint16_t *__restrict__ out)
{
    const int64_t n = nblocks * 16;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint8_t *blk = blocks + (i >> 4) * kQ8Bytes;
        const int p = (int)(i & 15);
        const __half2 D = __half2half2(__ushort_as_half((unsigned short)(blk[0] | (blk[1] << 8))));
        const uint32_t pair = (uint32_t)blk[2 + 2 * p] | ((uint32_t)blk[3 + 2 * p] << 8);
        reinterpret_cast<uint32_t *>(out)[i] = q80_pair_f16(pair, D);
    }
}

static unsigned grid_for(int64_t work_items, int per_block)
{
    int64_t g = (work_items + per_block - 1) / per_block;
    const int64_t cap = 148 * 32;   // grid-stride beyond this
    if (g > cap) g = cap;
    return (unsigned)(g > 0 ? g : 1);
}

cudaError_t launch_pack_q4k(const float *w, int64_t nblocks, uint8_t *out, uint32_t *status, cudaStream_t s)
{
    if (nblocks > 0) k_pack_qk<false><<<grid_for(nblocks, 8), 256, 0, s>>>(w, nblocks, out, status);
    return cudaGetLastError();
}

cudaError_t launch_pack_q5k(const float *w, int64_t nblocks, uint8_t *out, uint32_t *status, cudaStream_t s)
{
    if (nblocks > 0) k_pack_qk<true><<<grid_for(nblocks, 8), 256, 0, s>>>(w, nblocks, out, status);
    return cudaGetLastError();
}

cudaError_t launch_pack_q8_0(const float *w, int64_t nblocks, uint8_t *out, uint32_t *status, cudaStream_t s)
{
    if (nblocks > 0) k_pack_q8_0<<<grid_for(nblocks, 8), 256, 0, s>>>(w, nblocks, out, status);
    return cudaGetLastError();
}

cudaError_t launch_dequant_q4k(const uint8_t *blk, int64_t nblocks, float *out, cudaStream_t s)
{
    if (nblocks > 0) k_dequant_q4k<<<grid_for(nblocks * 32, 256), 256, 0, s>>>(blk, nblocks, out);
    return cudaGetLastError();
}

cudaError_t launch_dequant_q5k(const uint8_t *blk, int64_t nblocks, float *out, cudaStream_t s)
{
    if (nblocks > 0) k_dequant_q5k<<<grid_for(nblocks * 32, 256), 256, 0, s>>>(blk, nblocks, out);
    return cudaGetLastError();
}

cudaError_t launch_dequant_q5k_f16(const uint8_t *blk, int64_t nblocks, uint16_t *out, cudaStream_t s)
{
    if (nblocks > 0) k_dequant_q5k_f16<<<grid_for(nblocks * 32, 256), 256, 0, s>>>(blk, nblocks, out);
    return cudaGetLastError();
}

cudaError_t launch_dequant_q8_0(const uint8_t *blk, int64_t nblocks, float *out, cudaStream_t s)
{
    if (nblocks > 0) k_dequant_q8_0<<<grid_for(nblocks * 32, 256), 256, 0, s>>>(blk, nblocks, out);
    return cudaGetLastError();
}

cudaError_t launch_dequant_q4k_f16(const uint8_t *blk, int64_t nblocks, uint16_t *out, cudaStream_t s)
{
    if (nblocks > 0) k_dequant_q4k_f16<<<grid_for(nblocks * 32, 256), 256, 0, s>>>(blk, nblocks, out);
    return cudaGetLastError();
}

cudaError_t launch_dequant_q8_0_f16(const uint8_t *blk, int64_t nblocks, uint16_t *out, cudaStream_t s)
{
    if (nblocks > 0) k_dequant_q8_0_f16<<<grid_for(nblocks * 16, 256), 256, 0, s>>>(blk, nblocks, out);
    return cudaGetLastError();
}

}  // namespace moe
