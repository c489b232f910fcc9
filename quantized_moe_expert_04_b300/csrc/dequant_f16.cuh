// dequant_f16.cuh -- the fp16 operand dequantisation of the tensor-core
// paths (decode windows and prefill), in one place so that the fused kernels
// and the test hooks moe_dequant_q4k_f16 / moe_dequant_q8_0_f16 run the same
// code.
//
// The pages name Q4_K for the routed experts and Q8_0 for the shared expert
// ("Strata 改源码去跑 DeepSeek V4 Flash？", lcz.me/post/23082, section 二,
// GGUF anatomy table) but fix no arithmetic precision.  The MMAs multiply fp16
// weights, rounded as follows:
//   Q4_K  S_j = fp16(d * sc_j), NZ_j = fp16(-(dmin * m_j)) (exact products,
//         one rounding each), then w = fp16(q * S_j + NZ_j) with one rounding
//         (a fused fp16 multiply-add on the exact integer q);
//   Q5_K  as Q4_K, q the 5-bit quant (0..31): exact in fp16 too;
//   Q8_0  w = fp16(d * q) (exact product, one rounding).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace moe {

__device__ __forceinline__ __half2 dq_u2h2(uint32_t u)
{
    __half2 h;
    memcpy(&h, &u, 4);
    return h;
}

__device__ __forceinline__ uint32_t dq_h22u(__half2 h)
{
    uint32_t u;
    memcpy(&u, &h, 4);
    return u;
}

// 4-bit quants of 4 consecutive bytes b0..b3 of a 32-bit word -> fp16 pairs
// of exact integers: lo01 = (low nibble of b0, of b1), lo23 = (b2, b3); hi01,
// hi23 the high nibbles.  1024 + q through the fp16 exponent field, then the
// offset removed (the high nibble in place gives 1024 + 16q: * 1/16 - 64).
__device__ __forceinline__ void nibbles_to_q(uint32_t w, __half2 &lo01, __half2 &lo23, __half2 &hi01, __half2 &hi23)
{
    const uint32_t p01 = __byte_perm(w, 0, 0x4140);   // bytes b0, b1 into the two halves
    const uint32_t p23 = __byte_perm(w, 0, 0x4342);   // b2, b3
    const __half2 k1024 = __float2half2_rn(1024.0f);
    const __half2 k16th = __float2half2_rn(0.0625f);
    const __half2 km64 = __float2half2_rn(-64.0f);
    lo01 = __hsub2(dq_u2h2((p01 & 0x000F000Fu) | 0x64006400u), k1024);
    lo23 = __hsub2(dq_u2h2((p23 & 0x000F000Fu) | 0x64006400u), k1024);
    hi01 = __hfma2(dq_u2h2((p01 & 0x00F000F0u) | 0x64006400u), k16th, km64);
    hi23 = __hfma2(dq_u2h2((p23 & 0x00F000F0u) | 0x64006400u), k16th, km64);
}

// Q4_K block header -> fp16 (scale, -min) of the sub-block pair (2g, 2g+1):
// S = (fp16(d sc_2g), fp16(d sc_2g+1)), NZ likewise with -dmin m.  The 6-bit
// values are exact fp16 integers and each product rounds once, as
// fp16(fp32(d) * sc) does.
__device__ __forceinline__ void q4k_pair_scales_h(uint4 hdr, int g, __half2 &S, __half2 &NZ)
{
    const uint32_t scw = g < 2 ? (hdr.y & 0x3F3F3F3Fu) : ((hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u));
    const uint32_t mw = g < 2 ? (hdr.z & 0x3F3F3F3Fu) : (((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u));
    const uint32_t sel = (g & 1) ? 0x5342u : 0x5140u;
    const __half2 k1024 = __float2half2_rn(1024.0f);
    const __half2 dd = dq_u2h2(__byte_perm(hdr.x, 0, 0x1010)), mm = dq_u2h2(__byte_perm(hdr.x, 0, 0x3232) ^ 0x80008000u);
    S = __hmul2(dd, __hsub2(dq_u2h2(__byte_perm(scw, 0x64646464u, sel)), k1024));
    NZ = __hmul2(mm, __hsub2(dq_u2h2(__byte_perm(mw, 0x64646464u, sel)), k1024));
}

// One word of Q4_K quant bytes of sub-block pair (2g, 2g+1) -> 8 fp16
// weights: out[0] = elements (4i, 4i+1) of the low sub-block, out[1] =
// (4i+2, 4i+3); out[2], out[3] the same elements of the high sub-block.
// S_lo/NZ_lo (S_hi/NZ_hi): the pair's scale and negated min broadcast for the
// low (high) sub-block.
__device__ __forceinline__ void q4k_word_f16(uint32_t w, __half2 S_lo, __half2 NZ_lo, __half2 S_hi, __half2 NZ_hi,
                                             uint32_t (&out)[4])
{
    __half2 l01, l23, h01, h23;
    nibbles_to_q(w, l01, l23, h01, h23);
    out[0] = dq_h22u(__hfma2(l01, S_lo, NZ_lo));
    out[1] = dq_h22u(__hfma2(l23, S_lo, NZ_lo));
    out[2] = dq_h22u(__hfma2(h01, S_hi, NZ_hi));
    out[3] = dq_h22u(__hfma2(h23, S_hi, NZ_hi));
}

// Q5_K: 4-bit parts w as nibbles_to_q, and hb the fifth bits of the same 4
// elements: bit 0 of byte i for the low sub-block's element, bit 1 for the
// high one's.  The fifth bit enters the fp16 mantissa next to the nibble: at
// bit 4 of 1024 + q (low), at bit 8 of 1024 + 16 q (high); both stay exact
// integers below 2048.
__device__ __forceinline__ void nibbles5_to_q(uint32_t w, uint32_t hb, __half2 &lo01, __half2 &lo23, __half2 &hi01,
                                              __half2 &hi23)
{
    const uint32_t p01 = __byte_perm(w, 0, 0x4140), p23 = __byte_perm(w, 0, 0x4342);
    const uint32_t h01 = __byte_perm(hb, 0, 0x4140), h23 = __byte_perm(hb, 0, 0x4342);
    const __half2 k1024 = __float2half2_rn(1024.0f);
    const __half2 k16th = __float2half2_rn(0.0625f);
    const __half2 km64 = __float2half2_rn(-64.0f);
    lo01 = __hsub2(dq_u2h2((p01 & 0x000F000Fu) | ((h01 << 4) & 0x00100010u) | 0x64006400u), k1024);
    lo23 = __hsub2(dq_u2h2((p23 & 0x000F000Fu) | ((h23 << 4) & 0x00100010u) | 0x64006400u), k1024);
    hi01 = __hfma2(dq_u2h2((p01 & 0x00F000F0u) | ((h01 << 7) & 0x01000100u) | 0x64006400u), k16th, km64);
    hi23 = __hfma2(dq_u2h2((p23 & 0x00F000F0u) | ((h23 << 7) & 0x01000100u) | 0x64006400u), k16th, km64);
}

// One word of Q5_K quants (4-bit parts w, fifth bits hb as nibbles5_to_q) of
// the sub-block pair -> 8 fp16 weights, laid out as q4k_word_f16's.  The
// header (d, dmin, scales) is Q4_K's: q4k_pair_scales_h gives S and NZ.
__device__ __forceinline__ void q5k_word_f16(uint32_t w, uint32_t hb, __half2 S_lo, __half2 NZ_lo, __half2 S_hi,
                                             __half2 NZ_hi, uint32_t (&out)[4])
{
    __half2 l01, l23, h01, h23;
    nibbles5_to_q(w, hb, l01, l23, h01, h23);
    out[0] = dq_h22u(__hfma2(l01, S_lo, NZ_lo));
    out[1] = dq_h22u(__hfma2(l23, S_lo, NZ_lo));
    out[2] = dq_h22u(__hfma2(h01, S_hi, NZ_hi));
    out[3] = dq_h22u(__hfma2(h23, S_hi, NZ_hi));
}

// int8 pair (the two low bytes of a 32-bit word) -> exact fp16 pair.
__device__ __forceinline__ __half2 i8pair_to_h2(uint32_t pair16)
{
    const uint32_t p = (__byte_perm(pair16, 0, 0x4140) ^ 0x00800080u) & 0x00FF00FFu;   // q + 128
    return __hsub2(dq_u2h2(p | 0x64006400u), __float2half2_rn(1152.0f));               // 1024 + q + 128 - 1152
}

// Two consecutive Q8_0 weights (int8 pair in the low half of `pair16`)
// scaled by the block's d (broadcast in D): fp16(d * q) each.
__device__ __forceinline__ uint32_t q80_pair_f16(uint32_t pair16, __half2 D)
{
    return dq_h22u(__hmul2(i8pair_to_h2(pair16), D));
}

}  // namespace moe
