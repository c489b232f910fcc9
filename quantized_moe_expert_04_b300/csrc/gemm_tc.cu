// gemm_tc.cu -- grouped expert GEMM on the 5th-generation tensor cores
// (tcgen05 MMA, fp32 accumulators in tensor memory), with the Q4_K / Q8_0
// dequantisation fused into the operand pipeline.
//
// The pages' engine has dedicated Q4_K expert "prompt" (prefill) kernels on
// NVIDIA GPUs ("Qwen3.8-Flash-Next UD-Q4_K_XL 引擎对比", lcz.me/user/wml-ai/posts,
// section 一); its kernels target sm_86/sm_120 (mma.sync generation).  Here a
// persistent CTA per SM walks a device-built list of work tiles; each tile is
// one expert's 128 weight rows x up to kGemmMaxN of its tokens:
//
//   gate/up  A = 64 gate rows and the 64 up rows of the same ff indices,
//              interleaved (row 2i = gate f0+i, row 2i+1 = up f0+i), K = H;
//            B = the tile's token rows of x (fp16);
//            epilogue: lanes 2i / 2i+1 hold g / u of one ff index ->
//              a = SiLU(g) * u, stored fp16 at the assignment's bucket position.
//   down     A = Wd^T tile (128 hidden rows, K = FF; Wd is stored [FF][H], so the
//              dequantiser writes it transposed), B = the tile's rows of a;
//            epilogue: * routing weight, atomically added into y (fp32), or
//              stored to the assignment's slot when the call is deterministic.
//
// Warp roles (16 warps): 0-3 epilogue (tensor-memory lane quarters 0-3),
// 4 MMA issue + tensor-memory allocation, 5 raw weight bytes (16-byte cp.async
// pieces into a ring, completion counted on its mbarrier), 6-7 token rows
// (16-byte cp.async gathers into 128-byte-swizzled tiles, completion counted
// on the B ring's mbarriers),
// 8-15 dequantisation (raw ring -> fp16 A ring).  All hand-offs are mbarriers;
// every wait is bounded and sets MOE_ERR_TIMEOUT instead of hanging.
//
// Operand precision: fp16 A and B (sub-block scale and min rounded to fp16,
// one fused multiply-add per weight), fp32 accumulation.
#include <algorithm>
#include <cmath>

#include "moe_internal.cuh"
#include "tc_ptx.cuh"

namespace moe {

using namespace ptx;

enum GemmOp { kOpGateUp = 0, kOpDown = 1 };
enum WFmt { kWQ4K = 0, kWQ80 = 1 };

constexpr int kGemmThreads = 512;
constexpr int kDeqThreads = 256;           // warps 8-15: dequantisation
constexpr int kABytes = 128 * 128;          // 128 rows x 64 fp16
constexpr long long kWaitCycles = 1ll << 32; // ~2 s at 2 GHz

struct GemmArgs {
    int H, FF, SFF, k, T, det, splits;
    const uint8_t *const *blobs;
    const uint8_t *shared_blob;
    const int32_t *offsets, *assign;
    const float *w;
    const __half *x16;       // [T][H]
    __half *act16;           // [T*k][FF] by bucket position
    __half *sh_act16;        // [T][SFF]
    float *yacc;             // [T][H]
    float *slots, *sh_out;   // deterministic combine
    const int4 *tiles;       // {expert (-1 shared), m tile | k split << 16, n0, n}
    const uint32_t *n_tiles; // device count
    float *gu;               // split-K gate/up partial sums [rows][2 FF] (splits > 1)
    uint32_t *split_cnt;     // split-K arrival counters, one per (expert, m, n) group
    uint32_t *status;
};

struct TileInfo {
    int e, m, ks, n0, n, nmma, bb, ksteps, k0;   // k0: first K-step of this split
    const uint8_t *blob;
};

template <int OP, int FMT>
__device__ __forceinline__ TileInfo tile_info(const GemmArgs &g, int idx)
{
    const int4 t = g.tiles[idx];
    TileInfo ti;
    ti.e = t.x;
    ti.m = t.y & 0xffff;
    ti.ks = t.y >> 16;
    ti.n0 = t.z;
    ti.n = t.w;
    ti.nmma = (t.w + 15) & ~15;
    ti.bb = t.x >= 0 ? g.offsets[t.x] : 0;
    ti.blob = t.x >= 0 ? g.blobs[t.x] : g.shared_blob;
    ti.ksteps = (OP == kOpGateUp ? g.H : (FMT == kWQ4K ? g.FF : g.SFF)) / 64 / g.splits;
    ti.k0 = ti.ks * ti.ksteps;
    return ti;
}

// Bounded wait on an mbarrier phase; false on abort (another role gave up) or
// on timeout (this call records MOE_ERR_TIMEOUT and raises the abort flag).
// Waiting warps sleep in the try_wait (hardware suspend, up to ~20 us per
// try) rather than spin, so they do not take issue slots from the working
// warps.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort, uint32_t *status)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (*abort) return false;
        if (clock64() - t0 > kWaitCycles) {
            *abort = 1;
            set_status(status, MOE_ERR_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ __half2 u2h2(uint32_t u)
{
    __half2 h;
    memcpy(&h, &u, 4);
    return h;
}

__device__ __forceinline__ uint32_t h22u(__half2 h)
{
    uint32_t u;
    memcpy(&u, &h, 4);
    return u;
}

// ---------------------------------------------------------------- dequant

// 4-bit quants of 4 consecutive bytes -> fp16 pairs (exact integers), low and
// high nibbles: 1024 + q via the fp16 exponent trick, then remove the offset.
__device__ __forceinline__ void nibbles_to_q(uint32_t w, __half2 &lo01, __half2 &lo23, __half2 &hi01, __half2 &hi23)
{
    const uint32_t p01 = __byte_perm(w, 0, 0x4140);   // bytes b0, b1 into the two halves
    const uint32_t p23 = __byte_perm(w, 0, 0x4342);   // b2, b3
    const __half2 k1024 = __float2half2_rn(1024.0f);
    const __half2 k16th = __float2half2_rn(0.0625f);
    const __half2 km64 = __float2half2_rn(-64.0f);
    lo01 = __hsub2(u2h2((p01 & 0x000F000Fu) | 0x64006400u), k1024);          // q
    lo23 = __hsub2(u2h2((p23 & 0x000F000Fu) | 0x64006400u), k1024);
    hi01 = __hfma2(u2h2((p01 & 0x00F000F0u) | 0x64006400u), k16th, km64);    // (1024 + 16q)/16 - 64 = q
    hi23 = __hfma2(u2h2((p23 & 0x00F000F0u) | 0x64006400u), k16th, km64);
}

__device__ __forceinline__ void q4k_subblock_scales(uint4 hdr, int j, __half &s, __half &nz)
{
    const float d = f16_bits_to_f32(hdr.x & 0xffff), dmin = f16_bits_to_f32(hdr.x >> 16);
    uint8_t scales[12];
    memcpy(scales, &hdr.y, 4);
    memcpy(scales + 4, &hdr.z, 4);
    memcpy(scales + 8, &hdr.w, 4);
    int sc, m;
    q4k_scale_min(scales, j, sc, m);
    s = __float2half_rn(__fmul_rn(d, (float)sc));
    nz = __float2half_rn(-__fmul_rn(dmin, (float)m));
}

// Q4_K block header -> fp16 (scale, -min) pairs of its eight sub-blocks:
// S[i] = (fp16(d sc_2i), fp16(d sc_2i+1)), NZ[i] likewise with -dmin m.  The
// 6-bit values are exact fp16 integers and each product rounds once, as
// fp16(fp32(d) * sc) does.
__device__ __forceinline__ void q4k_block_scales_h(uint4 hdr, uint32_t (&S)[4], uint32_t (&NZ)[4])
{
    const uint32_t sc_lo = hdr.y & 0x3F3F3F3Fu, m_lo = hdr.z & 0x3F3F3F3Fu;
    const uint32_t sc_hi = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
    const uint32_t m_hi = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
    const __half2 k1024 = __float2half2_rn(1024.0f);
    const __half2 dd = u2h2(__byte_perm(hdr.x, 0, 0x1010)), mm = u2h2(__byte_perm(hdr.x, 0, 0x3232) ^ 0x80008000u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t scw = i < 2 ? sc_lo : sc_hi, mw = i < 2 ? m_lo : m_hi;
        const uint32_t sel = (i & 1) ? 0x5342u : 0x5140u;
        S[i] = h22u(__hmul2(dd, __hsub2(u2h2(__byte_perm(scw, 0x64646464u, sel)), k1024)));
        NZ[i] = h22u(__hmul2(mm, __hsub2(u2h2(__byte_perm(mw, 0x64646464u, sel)), k1024)));
    }
}

// gate/up, Q4_K: thread (row, h) dequantises half h of row `row` of K-step
// `sub` of the raw block column (16 quant bytes: 16 low-nibble weights of
// sub-block 2 sub and 16 high-nibble weights of sub-block 2 sub + 1) into the
// swizzled fp16 A tile, with the block's scales decoded beforehand.
__device__ __forceinline__ void dequant_gu_q4k(const uint8_t *raw, uint32_t a_tile, int row, int h, int sub,
                                               const uint32_t (&S)[4], const uint32_t (&NZ)[4])
{
    const uint8_t *rr = raw + row * 144;
    const uint4 q = *reinterpret_cast<const uint4 *>(rr + 16 + 32 * sub + 16 * h);
    // sub is a runtime value: select, so that S and NZ stay in registers
    const uint32_t sp = sub == 0 ? S[0] : sub == 1 ? S[1] : sub == 2 ? S[2] : S[3];
    const uint32_t np = sub == 0 ? NZ[0] : sub == 1 ? NZ[1] : sub == 2 ? NZ[2] : NZ[3];
    const __half2 S_lo = __low2half2(u2h2(sp)), S_hi = __high2half2(u2h2(sp));
    const __half2 NZ_lo = __low2half2(u2h2(np)), NZ_hi = __high2half2(u2h2(np));
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        __half2 l0, l1, h0, h1, l2, l3, h2, h3;
        nibbles_to_q(words[2 * p], l0, l1, h0, h1);
        nibbles_to_q(words[2 * p + 1], l2, l3, h2, h3);
        st_shared_v4(a_tile + sw128_off(row, 2 * h + p), h22u(__hfma2(l0, S_lo, NZ_lo)), h22u(__hfma2(l1, S_lo, NZ_lo)),
                     h22u(__hfma2(l2, S_lo, NZ_lo)), h22u(__hfma2(l3, S_lo, NZ_lo)));
        st_shared_v4(a_tile + sw128_off(row, 4 + 2 * h + p), h22u(__hfma2(h0, S_hi, NZ_hi)),
                     h22u(__hfma2(h1, S_hi, NZ_hi)), h22u(__hfma2(h2, S_hi, NZ_hi)), h22u(__hfma2(h3, S_hi, NZ_hi)));
    }
}

// int8 pair (two bytes of a 16-bit word) -> exact fp16 pair
__device__ __forceinline__ __half2 i8pair_to_h2(uint32_t pair16)
{
    const uint32_t p = (__byte_perm(pair16, 0, 0x4140) ^ 0x00800080u) & 0x00FF00FFu;   // q + 128
    return __hsub2(u2h2(p | 0x64006400u), __float2half2_rn(1152.0f));                  // 1024 + q + 128 - 1152
}

// gate/up, Q8_0: thread (row, blk), K-step s: block blk of the two 34-byte
// blocks at offset (68 s) mod 16 of the 80-byte raw row.
__device__ __forceinline__ void dequant_gu_q80(const uint8_t *raw, uint32_t a_tile, int row, int blk, int s)
{
    const uint8_t *rr = raw + row * 80 + ((68 * s) & 15);
    const uint16_t *r16 = reinterpret_cast<const uint16_t *>(rr);   // offset is a multiple of 4
    {
        const __half2 D = __half2half2(__ushort_as_half(r16[17 * blk]));
#pragma unroll
        for (int cq = 0; cq < 4; ++cq) {          // 4 chunks of 8 weights per block
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] = h22u(__hmul2(i8pair_to_h2(r16[17 * blk + 1 + 4 * cq + i]), D));
            st_shared_v4(a_tile + sw128_off(row, 4 * blk + cq), o[0], o[1], o[2], o[3]);
        }
    }
}

// down, Q4_K: A[h][f] = Wd[f][h0 + h] for the tile's 128 hidden columns and
// the K-step's 64 ff rows.  Raw row i (f = 64 s + i) holds the block header
// and the 64 quant bytes of this half block (80 bytes).  Item = (row, group of
// 8 quant bytes): 8 low-nibble weights at h = 64 c + l .. +7 and 8 high-nibble
// weights at h + 32, stored as 16-bit values into their transposed places.
__device__ __forceinline__ void dequant_dn_q4k(const uint8_t *raw, uint32_t a_tile, int dt, int half)
{
#pragma unroll
    for (int it4 = 0; it4 < 512 / kDeqThreads; ++it4) {
        const int it = dt + kDeqThreads * it4;
        const int row = it & 63, bg = it >> 6;           // bg 0..7
        const uint8_t *rr = raw + row * 80;
        const uint4 hdr = *reinterpret_cast<const uint4 *>(rr);
        const int c_loc = bg >> 2, l0 = (8 * bg) & 31;
        const int jsb = 2 * (2 * half + c_loc);
        __half s_lo, nz_lo, s_hi, nz_hi;
        q4k_subblock_scales(hdr, jsb, s_lo, nz_lo);
        q4k_subblock_scales(hdr, jsb + 1, s_hi, nz_hi);
        const __half2 S_lo = __half2half2(s_lo), NZ_lo = __half2half2(nz_lo);
        const __half2 S_hi = __half2half2(s_hi), NZ_hi = __half2half2(nz_hi);
        const uint2 q8 = *reinterpret_cast<const uint2 *>(rr + 16 + 8 * bg);
        const int h_lo = 64 * c_loc + l0;
        const uint32_t kchunk = (uint32_t)row >> 3, kbyte = ((uint32_t)row & 7) * 2;
#pragma unroll
        for (int wsel = 0; wsel < 2; ++wsel) {
            __half2 l01, l23, h01, h23;
            nibbles_to_q(wsel ? q8.y : q8.x, l01, l23, h01, h23);
            const __half2 vl01 = __hfma2(l01, S_lo, NZ_lo), vl23 = __hfma2(l23, S_lo, NZ_lo);
            const __half2 vh01 = __hfma2(h01, S_hi, NZ_hi), vh23 = __hfma2(h23, S_hi, NZ_hi);
            const int hb = h_lo + 4 * wsel;
            st_shared_u16(a_tile + sw128_off(hb + 0, kchunk) + kbyte, __half_as_ushort(__low2half(vl01)));
            st_shared_u16(a_tile + sw128_off(hb + 1, kchunk) + kbyte, __half_as_ushort(__high2half(vl01)));
            st_shared_u16(a_tile + sw128_off(hb + 2, kchunk) + kbyte, __half_as_ushort(__low2half(vl23)));
            st_shared_u16(a_tile + sw128_off(hb + 3, kchunk) + kbyte, __half_as_ushort(__high2half(vl23)));
            st_shared_u16(a_tile + sw128_off(hb + 32, kchunk) + kbyte, __half_as_ushort(__low2half(vh01)));
            st_shared_u16(a_tile + sw128_off(hb + 33, kchunk) + kbyte, __half_as_ushort(__high2half(vh01)));
            st_shared_u16(a_tile + sw128_off(hb + 34, kchunk) + kbyte, __half_as_ushort(__low2half(vh23)));
            st_shared_u16(a_tile + sw128_off(hb + 35, kchunk) + kbyte, __half_as_ushort(__high2half(vh23)));
        }
    }
}

// down, Q8_0: raw row i (f = 64 s + i) is a 144-byte window holding the 4
// blocks of this tile's 128 hidden columns at offset o8 (0 or 8).
__device__ __forceinline__ void dequant_dn_q80(const uint8_t *raw, uint32_t a_tile, int dt, int o8)
{
#pragma unroll
    for (int it8 = 0; it8 < 1024 / kDeqThreads; ++it8) {
        const int it = dt + kDeqThreads * it8;
        const int row = it & 63, g = it >> 6;            // g 0..15: 8 columns each
        const int b = g >> 2, hh0 = 8 * (g & 3);
        const uint16_t *blk = reinterpret_cast<const uint16_t *>(raw + row * 144 + o8 + 34 * b);
        const __half2 D = __half2half2(__ushort_as_half(blk[0]));
        const uint32_t kchunk = (uint32_t)row >> 3, kbyte = ((uint32_t)row & 7) * 2;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 v = __hmul2(i8pair_to_h2(blk[1 + hh0 / 2 + i]), D);
            const int h = 32 * b + hh0 + 2 * i;
            st_shared_u16(a_tile + sw128_off(h, kchunk) + kbyte, __half_as_ushort(__low2half(v)));
            st_shared_u16(a_tile + sw128_off(h + 1, kchunk) + kbyte, __half_as_ushort(__high2half(v)));
        }
    }
}

// ---------------------------------------------------------------- the kernel

template <int OP, int FMT>
__host__ __device__ constexpr int raw_stage_bytes()
{
    return OP == kOpGateUp ? (FMT == kWQ4K ? 128 * 144 : 128 * 80) : (FMT == kWQ4K ? 64 * 80 : 64 * 144);
}

// K-steps covered by one raw stage: a whole Q4_K block column (4 K-steps) for
// gate/up, one K-step otherwise.
template <int OP, int FMT>
__host__ __device__ constexpr int ksteps_per_raw()
{
    return (OP == kOpGateUp && FMT == kWQ4K) ? 4 : 1;
}

template <int OP, int FMT, int NMAX, int SA, int SB, int RAW>
struct GemmCfg {
    static constexpr int kRawStage = raw_stage_bytes<OP, FMT>();
    static constexpr int RS = RAW / kRawStage;           // raw ring depth
    static constexpr int kBBytes = NMAX * 128;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + SA * kABytes;
    static constexpr int kOffRaw = kOffB + SB * kBBytes;
    static constexpr int kOffBar = kOffRaw + ((RS * kRawStage + 1023) & ~1023);
    static constexpr int kNumBars = 2 * RS + 2 * SA + 2 * SB + 6;
    static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
    static constexpr int kOffMeta = kOffMisc + 16;              // [2][NMAX] token, weight, slot
    static constexpr int kBytes = kOffMeta + 2 * NMAX * 12 + 1024;
    static_assert(RS >= 2, "raw ring too shallow");
    static_assert(kBytes <= 232448, "shared memory budget");
};

template <int OP, int FMT, int NMAX, int SA, int SB, int RAW>
__global__ void __launch_bounds__(kGemmThreads, 1) k_moe_gemm(GemmArgs g)
{
    using C = GemmCfg<OP, FMT, NMAX, SA, SB, RAW>;
    constexpr int RS = C::RS;
    constexpr int KPR = ksteps_per_raw<OP, FMT>();
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_dyn + 1023) & ~(uintptr_t)1023);
    const uint32_t sA = smem_addr(smem + C::kOffA), sB = smem_addr(smem + C::kOffB);
    uint8_t *raw_base = smem + C::kOffRaw;
    const uint32_t bar0 = smem_addr(smem + C::kOffBar);
    auto full_raw = [&](int i) { return bar0 + 8 * i; };
    auto empty_raw = [&](int i) { return bar0 + 8 * (RS + i); };
    auto full_a = [&](int i) { return bar0 + 8 * (2 * RS + i); };
    auto empty_a = [&](int i) { return bar0 + 8 * (2 * RS + SA + i); };
    auto full_b = [&](int i) { return bar0 + 8 * (2 * RS + 2 * SA + i); };
    auto empty_b = [&](int i) { return bar0 + 8 * (2 * RS + 2 * SA + SB + i); };
    const uint32_t bx = bar0 + 8 * (2 * RS + 2 * SA + 2 * SB);
    auto acc_full = [&](int i) { return bx + 8 * i; };
    auto acc_empty = [&](int i) { return bx + 8 * (2 + i); };
    const uint32_t final_bar = bx + 8 * 4, epi_bar = bx + 8 * 5;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
    volatile int *last_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 8);
    int32_t *meta_tok = reinterpret_cast<int32_t *>(smem + C::kOffMeta);           // [2][NMAX]
    float *meta_w = reinterpret_cast<float *>(smem + C::kOffMeta + 2 * NMAX * 4);   // [2][NMAX]
    int32_t *meta_slot = reinterpret_cast<int32_t *>(smem + C::kOffMeta + 2 * NMAX * 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < RS; ++i) {
            mbar_init(full_raw(i), 32);          // the 32 lanes of the raw-byte warp
            mbar_init(empty_raw(i), kDeqThreads);
        }
        for (int i = 0; i < SA; ++i) {
            mbar_init(full_a(i), kDeqThreads);
            mbar_init(empty_a(i), 1);
        }
        for (int i = 0; i < SB; ++i) {
            mbar_init(full_b(i), 64);
            mbar_init(empty_b(i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(acc_full(i), 1);
            mbar_init(acc_empty(i), 128);
        }
        mbar_init(final_bar, 1);
        mbar_init(epi_bar, 128);
        *abort_flag = 0;
        *last_flag = 0;
        fence_mbar_init();
    }
    if (warp == 4) {
        tmem_alloc(smem_addr(tmem_slot), 2 * NMAX);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int n_tiles = (int)*g.n_tiles;

    if (warp < 4) {
        // ------------------------------------------------------------ epilogue
        uint32_t t_it = 0, epi_it = 0;
        const int et = threadIdx.x;          // 0..127 = tensor-memory lane
        auto epi_sync = [&]() -> bool {      // the 4 epilogue warps only, bounded
            mbar_arrive(epi_bar);
            return wait_bar(epi_bar, (epi_it++) & 1, abort_flag, g.status);
        };
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
            const TileInfo ti = tile_info<OP, FMT>(g, tile);
            if (!ti.blob) {
                if (et == 0) set_status(g.status, MOE_ERR_DEVICE_FAULT);
                continue;
            }
            const int acc = t_it & 1;
            if (OP == kOpDown) {
                // column metadata: token, routing weight and slot of each column
                for (int j = et; j < ti.n; j += 128) {
                    int tok, slot;
                    float wt;
                    if (FMT == kWQ4K) {
                        slot = g.assign[ti.bb + ti.n0 + j];
                        tok = slot / g.k;
                        wt = g.w[slot];
                    } else {
                        tok = slot = ti.n0 + j;
                        wt = 1.0f;
                    }
                    meta_tok[acc * NMAX + j] = tok;
                    meta_w[acc * NMAX + j] = wt;
                    meta_slot[acc * NMAX + j] = slot;
                }
                if (!(ok = epi_sync())) break;
            }
            if (!(ok = wait_bar(acc_full(acc), (t_it >> 1) & 1, abort_flag, g.status))) break;
            tc_fence_after();
            const int ffop = FMT == kWQ4K ? g.FF : g.SFF;
            for (int cc = 0; cc < ti.nmma / 16; ++cc) {
                uint32_t v[16];
                tmem_ld16(tmem_base + ((uint32_t)(32 * warp) << 16) + acc * NMAX + cc * 16, v);
                tmem_wait_ld();
                if (OP == kOpGateUp) {
                    const int f = ti.m * 64 + (et >> 1);
                    if (g.splits == 1) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float val = __uint_as_float(v[i]);
                            const float other = __shfl_xor_sync(0xffffffffu, val, 1);
                            const int j = cc * 16 + i;
                            if (!(lane & 1) && j < ti.n) {
                                const float a = val / (1.0f + expf(-val)) * other;
                                __half *dst = FMT == kWQ4K ? g.act16 + (int64_t)(ti.bb + ti.n0 + j) * ffop + f
                                                           : g.sh_act16 + (int64_t)(ti.n0 + j) * ffop + f;
                                *dst = __float2half_rn(a);
                            }
                        }
                    } else {
                        // partial sums of this K split: g into [row][f], u into [row][FF + f]
                        const int col = (et & 1) ? ffop + f : f;
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int j = cc * 16 + i;
                            const int rowi = FMT == kWQ4K ? ti.bb + ti.n0 + j : ti.n0 + j;
                            if (j < ti.n) red_add_f32(g.gu + (int64_t)rowi * 2 * ffop + col, __uint_as_float(v[i]));
                        }
                    }
                } else {
                    // 4x4 transposes within lane quads: lane (q, r) ends with the
                    // values of hidden rows 4q..4q+3 for column 4b + r
                    const int hq = ti.m * 128 + 32 * warp + (lane & ~3);
                    const int r = lane & 3;
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        float a0 = __uint_as_float(v[4 * b]), a1 = __uint_as_float(v[4 * b + 1]);
                        float a2 = __uint_as_float(v[4 * b + 2]), a3 = __uint_as_float(v[4 * b + 3]);
                        float t0 = __shfl_xor_sync(0xffffffffu, (r & 2) ? a0 : a2, 2);
                        float t1 = __shfl_xor_sync(0xffffffffu, (r & 2) ? a1 : a3, 2);
                        if (r & 2) { a0 = t0; a1 = t1; } else { a2 = t0; a3 = t1; }
                        t0 = __shfl_xor_sync(0xffffffffu, (r & 1) ? a0 : a1, 1);
                        t1 = __shfl_xor_sync(0xffffffffu, (r & 1) ? a2 : a3, 1);
                        if (r & 1) { a0 = t0; a2 = t1; } else { a1 = t0; a3 = t1; }
                        const int j = cc * 16 + 4 * b + r;
                        if (j < ti.n) {
                            const float wt = meta_w[acc * NMAX + j];
                            if (g.det) {
                                float *dst = FMT == kWQ4K ? g.slots + (int64_t)meta_slot[acc * NMAX + j] * g.H + hq
                                                          : g.sh_out + (int64_t)meta_tok[acc * NMAX + j] * g.H + hq;
                                *reinterpret_cast<float4 *>(dst) = make_float4(wt * a0, wt * a1, wt * a2, wt * a3);
                            } else {
                                red_add_v4_f32(g.yacc + (int64_t)meta_tok[acc * NMAX + j] * g.H + hq, wt * a0,
                                               wt * a1, wt * a2, wt * a3);
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(acc_empty(acc));
            ++t_it;
            if (OP == kOpGateUp && g.splits > 1) {
                // the last split of this (expert, m, n) group turns g, u into a
                __threadfence();
                if (!(ok = epi_sync())) break;
                if (et == 0) {
                    const uint32_t old = atomicAdd(g.split_cnt + tile / g.splits, 1u);
                    *last_flag = old == (uint32_t)(g.splits - 1);
                }
                if (!(ok = epi_sync())) break;
                if (*last_flag) {
                    __threadfence();
                    const int f = ti.m * 64 + (et >> 1);
                    if (!(et & 1)) {
                        for (int j = 0; j < ti.n; ++j) {
                            const int rowi = FMT == kWQ4K ? ti.bb + ti.n0 + j : ti.n0 + j;
                            const float gg = ld_cg_f32(g.gu + (int64_t)rowi * 2 * ffop + f);
                            const float uu = ld_cg_f32(g.gu + (int64_t)rowi * 2 * ffop + ffop + f);
                            __half *dst = FMT == kWQ4K ? g.act16 + (int64_t)rowi * ffop + f
                                                       : g.sh_act16 + (int64_t)rowi * ffop + f;
                            *dst = __float2half_rn(gg / (1.0f + expf(-gg)) * uu);
                        }
                    }
                    if (et == 0) g.split_cnt[tile / g.splits] = 0;
                }
                if (!(ok = epi_sync())) break;     // last_flag is rewritten by the next group
            }
        }
    } else if (warp == 4) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            uint32_t sa_it = 0, sb_it = 0, t_it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
                const TileInfo ti = tile_info<OP, FMT>(g, tile);
                if (!ti.blob) continue;
                const int acc = t_it & 1;
                if (!(ok = wait_bar(acc_empty(acc), ((t_it >> 1) & 1) ^ 1, abort_flag, g.status))) break;
                tc_fence_after();
                const uint32_t idesc = idesc_f16_f32(128, ti.nmma);
                const uint32_t d_tmem = tmem_base + acc * NMAX;
                for (int s = 0; s < ti.ksteps; ++s, ++sa_it, ++sb_it) {
                    const int slot_a = sa_it % SA, slot_b = sb_it % SB;
                    if (!(ok = wait_bar(full_a(slot_a), (sa_it / SA) & 1, abort_flag, g.status))) break;
                    if (!(ok = wait_bar(full_b(slot_b), (sb_it / SB) & 1, abort_flag, g.status))) break;
                    fence_proxy_async();   // the token rows were written by cp.async (generic proxy)
                    tc_fence_after();
                    const uint32_t a0 = sA + slot_a * kABytes, b0 = sB + slot_b * C::kBBytes;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_f16(d_tmem, sdesc_kmajor_sw128(a0 + 32 * kk), sdesc_kmajor_sw128(b0 + 32 * kk), idesc,
                                (s | kk) != 0);
                    mma_commit(empty_a(slot_a));
                    mma_commit(empty_b(slot_b));
                }
                if (!ok) break;
                mma_commit(acc_full(acc));
                ++t_it;
            }
            // every issued MMA must be complete before the tensor memory is freed
            mma_commit(final_bar);
            const long long t0 = clock64();
            while (!mbar_try_wait(final_bar, 0) && clock64() - t0 < kWaitCycles) {
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        // ------------------------------------------------------------ raw weight bytes
        uint32_t rs_it = 0;
        const int H = g.H;
        const int64_t rb = FMT == kWQ4K ? (int64_t)(H / 256) * 144 : (int64_t)(H / 32) * 34;   // row bytes
        const int ffop = FMT == kWQ4K ? g.FF : g.SFF;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
            const TileInfo ti = tile_info<OP, FMT>(g, tile);
            if (!ti.blob) continue;
            const int nraw = ti.ksteps / KPR, r0 = ti.k0 / KPR;
            for (int rr = 0; rr < nraw; ++rr, ++rs_it) {
                const int r = r0 + rr;                    // raw stage (block column / K-step) index
                const int slot = rs_it % RS;
                if (!(ok = wait_bar(empty_raw(slot), ((rs_it / RS) & 1) ^ 1, abort_flag, g.status))) break;
                uint8_t *dst0 = raw_base + slot * C::kRawStage;
                // 16-byte asynchronous copies; each lane's completion arrives on full_raw
                // consecutive lanes take consecutive 16-byte pieces (coalesced requests);
                // piece p = lane + 32 j is (row p / P, piece p % P), stepped incrementally
                if (OP == kOpGateUp) {
                    // 128 rows: row 2i = gate f0+i, row 2i+1 = up f0+i
                    constexpr int kPieces = FMT == kWQ4K ? 9 : 5;           // 144 or 80 bytes per row
                    int i = lane / kPieces, pc = lane % kPieces;
                    const int64_t col = FMT == kWQ4K ? (int64_t)r * 144 : (int64_t)((68 * r) & ~15);
                    const uint8_t *gbase = ti.blob + (int64_t)ti.m * 64 * rb + col;
                    const uint8_t *ubase = gbase + (int64_t)ffop * rb;
                    for (int j = 0; j < (128 * kPieces) / 32; ++j) {
                        const uint8_t *src = ((i & 1) ? ubase : gbase) + (int64_t)(i >> 1) * rb + pc * 16;
                        cp_async16(smem_addr(dst0 + i * (16 * kPieces) + pc * 16), src);
                        i += 32 / kPieces;
                        pc += 32 % kPieces;
                        if (pc >= kPieces) {
                            pc -= kPieces;
                            ++i;
                        }
                    }
                } else {
                    // 64 ff rows of Wd for this K-step, this tile's 128 hidden columns
                    const int h0 = ti.m * 128;
                    constexpr int kPieces = FMT == kWQ4K ? 5 : 9;           // 16 + 64 or 144 bytes per row
                    const uint8_t *base = ti.blob + ((int64_t)2 * ffop + 64 * r) * rb;
                    const int64_t blk = FMT == kWQ4K ? (int64_t)(h0 / 256) * 144 : (int64_t)((34 * (h0 / 32)) & ~15);
                    const int qoff = 16 + 64 * ((h0 / 128) & 1);
                    int i = lane / kPieces, pc = lane % kPieces;
                    for (int j = 0; j < (64 * kPieces) / 32; ++j) {
                        const uint8_t *rowp = base + (int64_t)i * rb + blk;
                        const uint8_t *src = FMT == kWQ4K ? (pc == 0 ? rowp : rowp + qoff + (pc - 1) * 16) : rowp + pc * 16;
                        cp_async16(smem_addr(dst0 + i * (16 * kPieces) + pc * 16), src);
                        i += 32 / kPieces;
                        pc += 32 % kPieces;
                        if (pc >= kPieces) {
                            pc -= kPieces;
                            ++i;
                        }
                    }
                }
                cp_async_arrive_noinc(full_raw(slot));
            }
        }
        // copies still in flight (an early exit) must land before the CTA ends
        for (uint32_t i = rs_it > (uint32_t)RS ? rs_it - RS : 0; i < rs_it; ++i) {
            const long long t0 = clock64();
            while (!mbar_try_wait(full_raw(i % RS), (i / RS) & 1) && clock64() - t0 < kWaitCycles) {
            }
        }
    } else if (warp < 8) {
        // ------------------------------------------------------------ token rows (B)
        // thread bt copies 16-byte chunk (bt & 7) of rows j = (bt >> 3) + 8 i;
        // each thread's copies of a stage arrive on full_b when they land, so
        // the gatherers run up to SB stages ahead of the MMAs
        const int bt = threadIdx.x - 192;   // 0..63
        const int c = bt & 7, r0 = bt >> 3;
        const __half *srcbase = OP == kOpGateUp ? g.x16 : (FMT == kWQ4K ? g.act16 : g.sh_act16);
        const int ld = OP == kOpGateUp ? g.H : (FMT == kWQ4K ? g.FF : g.SFF);
        uint32_t sb_it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
            const TileInfo ti = tile_info<OP, FMT>(g, tile);
            if (!ti.blob) continue;
            int src[NMAX / 8];
#pragma unroll
            for (int i = 0; i < NMAX / 8; ++i) {
                const int j = r0 + 8 * i;
                src[i] = 0;
                if (j < ti.n) {
                    if (OP == kOpGateUp) src[i] = FMT == kWQ4K ? g.assign[ti.bb + ti.n0 + j] / g.k : ti.n0 + j;
                    else src[i] = FMT == kWQ4K ? ti.bb + ti.n0 + j : ti.n0 + j;
                }
            }
            for (int s = 0; s < ti.ksteps; ++s, ++sb_it) {
                const int slot = sb_it % SB;
                if (!(ok = wait_bar(empty_b(slot), ((sb_it / SB) & 1) ^ 1, abort_flag, g.status))) break;
                const uint32_t b_tile = sB + slot * C::kBBytes;
                const int kcol = (ti.k0 + s) * 64 + c * 8;
#pragma unroll
                for (int i = 0; i < NMAX / 8; ++i) {
                    const int j = r0 + 8 * i;
                    if (j < ti.n) cp_async16(b_tile + sw128_off(j, c), srcbase + (int64_t)src[i] * ld + kcol);
                }
                cp_async_arrive_noinc(full_b(slot));
            }
        }
        cp_async_wait<0>();   // nothing may still be writing shared memory when the CTA ends
    } else {
        // ------------------------------------------------------------ dequantisation (A)
        const int dt = threadIdx.x - 256;   // 0..255
        uint32_t sa_it = 0, rs_it = 0;
        uint32_t S[4], NZ[4];
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
            const TileInfo ti = tile_info<OP, FMT>(g, tile);
            if (!ti.blob) continue;
            for (int s = 0; s < ti.ksteps; ++s, ++sa_it) {
                const int sg = ti.k0 + s;                 // global K-step
                const int sub = sg % KPR;
                const bool first = s == 0 || sub == 0, last = s == ti.ksteps - 1 || sub == KPR - 1;
                const int rslot = rs_it % RS;
                if (first && !(ok = wait_bar(full_raw(rslot), (rs_it / RS) & 1, abort_flag, g.status))) break;
                const int slot = sa_it % SA;
                if (!(ok = wait_bar(empty_a(slot), ((sa_it / SA) & 1) ^ 1, abort_flag, g.status))) break;
                const uint8_t *raw = raw_base + rslot * C::kRawStage;
                const uint32_t a_tile = sA + slot * kABytes;
                if (OP == kOpGateUp) {
                    // thread dt = (row dt & 127, half dt >> 7): a warp covers 32 consecutive
                    // rows (conflict-free shared-memory accesses)
                    if (FMT == kWQ4K) {
                        if (first) q4k_block_scales_h(*reinterpret_cast<const uint4 *>(raw + (dt & 127) * 144), S, NZ);
                        dequant_gu_q4k(raw, a_tile, dt & 127, dt >> 7, sub, S, NZ);
                    } else {
                        dequant_gu_q80(raw, a_tile, dt & 127, dt >> 7, sg);
                    }
                } else {
                    if (FMT == kWQ4K) dequant_dn_q4k(raw, a_tile, dt, ti.m & 1);
                    else dequant_dn_q80(raw, a_tile, dt, (34 * (ti.m * 128 / 32)) & 15);
                }
                fence_proxy_async();
                mbar_arrive(full_a(slot));
                if (last) {
                    mbar_arrive(empty_raw(rslot));
                    ++rs_it;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 2 * NMAX);
    }
}

// ---------------------------------------------------------------- helpers

// x -> fp16 operand copy; zero the fp32 output accumulator, the split-K
// partial sums and their counters.
__global__ void __launch_bounds__(256) k_gemm_prep(const uint16_t *__restrict__ x, __half *__restrict__ x16,
                                                   float *__restrict__ yacc, int64_t n, float *__restrict__ gu,
                                                   int64_t n_gu, uint32_t *__restrict__ cnt, int64_t n_cnt,
                                                   uint32_t *status)
{
    bool bad = false;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float v = bf16_bits_to_f32(x[i]);
        const __half hv = __float2half_rn(v);
        bad |= isfinite(v) && !isfinite(__half2float(hv));    // beyond the fp16 range
        x16[i] = hv;
        if (yacc) yacc[i] = 0.0f;
    }
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_gu; i += stride) gu[i] = 0.0f;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_cnt; i += stride) cnt[i] = 0u;
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) set_status(status, MOE_ERR_DEVICE_FAULT);
}

struct PlanArgs {
    int H, FF, SFF, T, split_gu, split_dn, split_gus, split_dns;
    const int32_t *offsets, *active;
    uint32_t *header;
    int4 *gu, *dn, *gus, *dns;
};

__device__ __forceinline__ void split_tokens(int n_e, int &tn, int &nt)
{
    const int nt0 = (n_e + kGemmMaxN - 1) / kGemmMaxN;
    tn = (((n_e + nt0 - 1) / nt0) + 15) & ~15;
    nt = (n_e + tn - 1) / tn;
}

// Work tiles of the routed experts (both projections) and of the shared
// expert; one CTA, one thread per active expert, block-wide prefix sums.
// Tile (e, m | ks << 16, n0, n): expert e (-1 = shared), weight tile m, K
// split ks, tokens n0 .. n0+n-1 of the expert's bucket.  The splits of one
// (e, m, n0) group are consecutive.
__global__ void __launch_bounds__(1024) k_gemm_plan(PlanArgs p)
{
    __shared__ int scan_gu[1024], scan_dn[1024];
    const int u = threadIdx.x;
    const int n_active = (int)p.header[kHdrNActive];
    const int mt_gu = p.FF / 64, mt_dn = p.H / 128;
    int e = -1, n_e = 0, tn = 0, nt = 0;
    if (u < n_active) {
        e = p.active[u];
        n_e = p.offsets[e + 1] - p.offsets[e];
        split_tokens(n_e, tn, nt);
    }
    scan_gu[u] = nt * mt_gu * p.split_gu;
    scan_dn[u] = nt * mt_dn * p.split_dn;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
        const int a = u >= off ? scan_gu[u - off] : 0, b = u >= off ? scan_dn[u - off] : 0;
        __syncthreads();
        scan_gu[u] += a;
        scan_dn[u] += b;
        __syncthreads();
    }
    int at_gu = scan_gu[u] - nt * mt_gu * p.split_gu, at_dn = scan_dn[u] - nt * mt_dn * p.split_dn;
    for (int j = 0; j < nt; ++j) {
        const int n0 = j * tn, n = min(tn, n_e - n0);
        for (int m = 0; m < mt_gu; ++m)
            for (int ks = 0; ks < p.split_gu; ++ks) p.gu[at_gu++] = make_int4(e, m | (ks << 16), n0, n);
        for (int m = 0; m < mt_dn; ++m)
            for (int ks = 0; ks < p.split_dn; ++ks) p.dn[at_dn++] = make_int4(e, m | (ks << 16), n0, n);
    }
    if (u == 1023) {
        p.header[kHdrTilesGU] = (uint32_t)scan_gu[1023];
        p.header[kHdrTilesDN] = (uint32_t)scan_dn[1023];
    }
    if (p.SFF > 0) {
        int stn, snt;
        split_tokens(p.T, stn, snt);
        const int smt_gu = p.SFF / 64;
        const int n_gus = snt * smt_gu * p.split_gus, n_dns = snt * mt_dn * p.split_dns;
        for (int i = u; i < n_gus; i += 1024) {
            const int ks = i % p.split_gus, grp = i / p.split_gus, j = grp / smt_gu, m = grp % smt_gu;
            p.gus[i] = make_int4(-1, m | (ks << 16), j * stn, min(stn, p.T - j * stn));
        }
        for (int i = u; i < n_dns; i += 1024) {
            const int ks = i % p.split_dns, grp = i / p.split_dns, j = grp / mt_dn, m = grp % mt_dn;
            p.dns[i] = make_int4(-1, m | (ks << 16), j * stn, min(stn, p.T - j * stn));
        }
        if (u == 0) {
            p.header[kHdrTilesGUS] = (uint32_t)n_gus;
            p.header[kHdrTilesDNS] = (uint32_t)n_dns;
        }
    } else if (u == 0) {
        p.header[kHdrTilesGUS] = 0;
        p.header[kHdrTilesDNS] = 0;
    }
}

// y = bf16(accumulated y) (atomic path) or the fixed-order sum of the slots.
__global__ void __launch_bounds__(256) k_gemm_finish(const float *__restrict__ yacc, const float *__restrict__ slots,
                                                     const float *__restrict__ sh_out, int T, int H, int k,
                                                     uint16_t *__restrict__ y, float *__restrict__ y_f32)
{
    const int64_t n = (int64_t)T * H;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        float acc;
        if (slots) {
            const int64_t t = i / H, h = i % H;
            acc = 0.0f;
            for (int r = 0; r < k; ++r) acc += slots[(t * k + r) * H + h];
            if (sh_out) acc += sh_out[i];
        } else {
            acc = yacc[i];
        }
        y[i] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
        if (y_f32) y_f32[i] = acc;
    }
}

// ---------------------------------------------------------------- launch

template <int OP, int FMT, int NMAX, int SA, int SB, int RAW>
static cudaError_t launch_gemm(const GemmArgs &g, int grid, cudaStream_t s)
{
    using C = GemmCfg<OP, FMT, NMAX, SA, SB, RAW>;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(k_moe_gemm<OP, FMT, NMAX, SA, SB, RAW>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kBytes);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    k_moe_gemm<OP, FMT, NMAX, SA, SB, RAW><<<grid, kGemmThreads, C::kBytes, s>>>(g);
    return cudaGetLastError();
}

// Configurations: small buckets (every token tile <= 16 wide: decode windows)
// keep deep A and raw rings; large buckets (prefill) use token tiles of
// kGemmMaxN with A, B and raw rings of 4, 6 and 3 stages.
template <int OP, int FMT>
static cudaError_t launch_gemm_cfg(const GemmArgs &g, int grid, bool small, cudaStream_t s)
{
    if (small) return launch_gemm<OP, FMT, 16, 6, 8, 92160>(g, grid, s);
    return launch_gemm<OP, FMT, kGemmMaxN, 4, 6, 55296>(g, grid, s);
}

static int num_sms()
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

size_t gemm_tile_capacity(int mt, int64_t TK, int E)
{
    return (size_t)mt * (size_t)(TK / kGemmMaxN + 1 + std::min<int64_t>(E, TK));
}

// K split for `tiles` work tiles of `ksteps` K-steps: the smallest divisor d
// of `units` (K-steps come in units: Q4_K blocks or 64-row groups) whose waves
// over the SMs are at least 85% full, keeping >= 4 K-steps per tile; the best
// wave fill among the allowed divisors otherwise.
static int pick_split(int64_t tiles, int units, int ksteps, int sms)
{
    int best = 1;
    double best_eff = 0.0;
    for (int d = 1; d <= units; ++d) {
        if (units % d || (d > 1 && ksteps / d < 4)) continue;
        const double waves = (double)(tiles * d) / sms;
        const double eff = waves / std::ceil(waves);
        if (eff >= 0.85) return d;
        if (eff > best_eff + 1e-9) {
            best_eff = eff;
            best = d;
        }
    }
    return best;
}

GemmSplits gemm_splits(const moe_config &c, int32_t T)
{
    GemmSplits sp{1, 1, 1, 1};
    if (T > kGemmSmallTokens) return sp;                  // prefill: enough tiles without splitting K
    const int sms = num_sms();
    const int64_t active = std::min<int64_t>(c.n_experts, (int64_t)T * c.top_k);
    sp.gu = pick_split(active * (c.ff / 64), c.hidden / 256, c.hidden / 64, sms);
    sp.dn = pick_split(active * (c.hidden / 128), c.ff / 64, c.ff / 64, sms);
    if (c.shared_ff) {
        sp.gus = pick_split(c.shared_ff / 64, c.hidden / 256, c.hidden / 64, sms);
        sp.dns = pick_split(c.hidden / 128, c.shared_ff / 64, c.shared_ff / 64, sms);
    }
    if (c.flags & MOE_FLAG_DETERMINISTIC) {
        // the deterministic down epilogue stores each slot once: no K split there
        sp.dn = 1;
        sp.dns = 1;
    }
    return sp;
}

cudaError_t launch_experts_gemm(const ExpertArgs &a, const GemmWs &w, cudaStream_t s)
{
    const int64_t n = (int64_t)a.T * a.H;
    const int det = w.det;
    const bool small = a.T <= kGemmSmallTokens;
    const GemmSplits sp = w.splits;
    prof_begin(kPhGemmPrep, s);
    k_gemm_prep<<<(unsigned)std::min<int64_t>((std::max<int64_t>(n, w.n_gu) + 255) / 256, 148 * 8), 256, 0, s>>>(
        a.x, w.x16, det ? nullptr : w.yacc, n, w.gu, w.n_gu, w.split_cnt, w.n_cnt, a.header + kHdrStatus);
    PlanArgs p{a.H, a.FF, a.SFF, a.T, sp.gu, sp.dn, sp.gus, sp.dns, a.offsets, a.active, a.header,
               w.tiles_gu, w.tiles_dn, w.tiles_gus, w.tiles_dns};
    k_gemm_plan<<<1, 1024, 0, s>>>(p);
    prof_end(kPhGemmPrep, s);

    GemmArgs g{};
    g.H = a.H;
    g.FF = a.FF;
    g.SFF = a.SFF;
    g.k = a.k;
    g.T = a.T;
    g.det = det;
    g.blobs = a.blobs;
    g.shared_blob = a.shared_blob;
    g.offsets = a.offsets;
    g.assign = a.assign;
    g.w = a.w;
    g.x16 = w.x16;
    g.act16 = w.act16;
    g.sh_act16 = w.sh_act16;
    g.yacc = w.yacc;
    g.slots = a.slots;
    g.sh_out = a.sh_out;
    g.status = a.header + kHdrStatus;
    const int grid = num_sms();
    cudaError_t e;

    prof_begin(kPhGemmGateUp, s);
    g.tiles = w.tiles_gu;
    g.n_tiles = a.header + kHdrTilesGU;
    g.splits = sp.gu;
    g.gu = w.gu;
    g.split_cnt = w.split_cnt;
    e = launch_gemm_cfg<kOpGateUp, kWQ4K>(g, grid, small, s);
    if (e == cudaSuccess && a.shared_blob) {
        g.tiles = w.tiles_gus;
        g.n_tiles = a.header + kHdrTilesGUS;
        g.splits = sp.gus;
        g.gu = w.sh_gu;
        g.split_cnt = w.split_cnt + w.n_cnt_routed;
        e = launch_gemm_cfg<kOpGateUp, kWQ80>(g, grid, small, s);
    }
    prof_end(kPhGemmGateUp, s);
    if (e != cudaSuccess) return e;

    prof_begin(kPhGemmDown, s);
    g.tiles = w.tiles_dn;
    g.n_tiles = a.header + kHdrTilesDN;
    g.splits = sp.dn;
    e = launch_gemm_cfg<kOpDown, kWQ4K>(g, grid, small, s);
    if (e == cudaSuccess && a.shared_blob) {
        g.tiles = w.tiles_dns;
        g.n_tiles = a.header + kHdrTilesDNS;
        g.splits = sp.dns;
        e = launch_gemm_cfg<kOpDown, kWQ80>(g, grid, small, s);
    }
    prof_end(kPhGemmDown, s);
    if (e != cudaSuccess) return e;

    prof_begin(kPhGemmFinish, s);
    k_gemm_finish<<<(unsigned)std::min<int64_t>((n + 255) / 256, 148 * 8), 256, 0, s>>>(
        w.yacc, det ? a.slots : nullptr, det ? a.sh_out : nullptr, a.T, a.H, a.k, a.y, a.y_f32);
    prof_end(kPhGemmFinish, s);
    return cudaGetLastError();
}

}  // namespace moe
