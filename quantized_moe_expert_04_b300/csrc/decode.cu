// decode.cu -- the layer for decode / MTP-verify windows (T <= 8 tokens).
//
// The teardown page ("Strata 引擎深度拆解", lcz.me/topic/2098/5, section 一,
// CPU ledger) computes each selected expert once for all tokens of a 3-token
// verify window, and the decode critical path there is the expert arithmetic
// (section 二 item 5).  One layer call is two kernels here, chained with
// programmatic dependent launch:
//
//   k_dec_route  router logits over the grid (each router row read once per
//                window, held in registers: with static weights the rows are
//                loaded before the previous call has finished); the window's
//                x as fp16 MMA fragments; zeroes the fp32 accumulator of y.
//   k_dec_layer  one persistent CTA per SM.  Every CTA routes the window
//                itself (one warp per token: top-k by warp arg-max rounds;
//                bitmap bucketing of the selected experts), then takes an
//                equal share of the window's "units": 8 consecutive ff rows
//                of one selected expert -- its 8 gate, 8 up and 8 down rows
//                (the down matrix is stored [FF][H], so down row f needs only
//                a[f]) -- followed by the shared expert's 4-row units.
//                Consumer warp w owns a column block of H (256 columns, or
//                128 for layers without a shared expert) and stages only its
//                block of every slab into a private ring with 16-byte
//                cp.async.  Gate/up are fp16 warp MMAs (8 gate + 8 up rows =
//                the 16 MMA rows, the window's tokens = the 8 MMA columns);
//                the warps' partial sums meet in shared memory; a = w SiLU(g)
//                u in fp16 is the B operand of the down MMAs (the unit's 8
//                rows = K), which run one unit late so that one barrier per
//                unit orders both.  Down results stay in registers across all
//                the CTA's units and are added into the fp32 accumulator
//                once; the last CTA to finish writes y in bf16.
//
// k_dec_stack runs the same layer body for a window through a whole stack of
// layers in one cooperative launch (see there).  Every selected expert's
// bytes (and the shared expert's) are read once per window.
#include <algorithm>
#include <mutex>

#include "moe_internal.cuh"
#include "dequant_f16.cuh"

namespace moe {

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint32_t sm_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(1000000u)
        : "memory");
    return ok != 0;
}

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_poll(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// 1-D bulk copy global -> shared, completing `bytes` of the mbarrier's transaction count.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void red_add_v4(float *p, float a, float b, float c, float d)
{
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// Bounded wait on an mbarrier phase.  Gives up (false) when another thread of
// the CTA has raised the abort flag, or after `limit` clock cycles, in which
// case it records MOE_ERR_TIMEOUT and raises the flag itself.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int *abort, uint32_t *status,
                                           long long limit)
{
    if (mbar_test(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_test(bar, parity)) return true;
        if (*abort) return false;
        if (clock64() - t0 > limit) {
            *abort = 1;
            set_status(status, MOE_ERR_TIMEOUT);
            return false;
        }
    }
}

// ---------------------------------------------------------------- routing

// Order-preserving map of an fp32 key to uint32 (larger float -> larger
// integer); NaN maps to 0, below every number, and is never selected.
__device__ __forceinline__ uint32_t key_bits(float f)
{
    if (isnan(f)) return 0u;
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Top-k of one token by one warp.  keys[e] (shared memory) holds the
// order-preserving integer of expert e's selection score (0 = not
// selectable).  Lane l keeps the keys of experts l, l + 32, ... (NPER) in
// registers and its best one (a reduction tree, equal keys to the lower id);
// each round takes the warp maximum (redux), the lowest expert id among equal
// keys, and only the winning lane clears that key and recomputes its best.
// Weights: softmax over the k selected logits (= the full softmax
// renormalised over the k) or s / sum of the selected s; vals[e] holds the
// logit (softmax) or s = sigmoid(logit).  Lane r < k receives selection r.
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
// zeroes the fp32 accumulator of y.
constexpr int kRouteThreads = 256;

// 88 registers a thread: a CTA of this kernel (8 warps) fits on an SM beside
// the 11-warp layer kernel of the previous call, so that its router rows load
// while that call streams its experts.
__global__ void __maxnreg__(88) k_dec_route(DecArgs a)
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
    // the next kernel (the layer) may launch now: it reads nothing of ours
    // before its own dependency wait except static weights
    griddep_launch();

    {
        const int nvec = T * H / 8;
        const uint4 *src = reinterpret_cast<const uint4 *>(a.x);
        uint4 *dst = reinterpret_cast<uint4 *>(s_x);
        for (int i0 = threadIdx.x; i0 < nvec; i0 += 8 * kRouteThreads) {   // 8 loads in flight
            uint4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (i0 + j * kRouteThreads < nvec) v[j] = __ldcg(src + i0 + j * kRouteThreads);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (i0 + j * kRouteThreads < nvec) dst[i0 + j * kRouteThreads] = v[j];
        }
    }
    const int gtid = blockIdx.x * kRouteThreads + threadIdx.x, gthreads = gridDim.x * kRouteThreads;
    for (int i = gtid; i < T * H / 4; i += gthreads)
        reinterpret_cast<float4 *>(a.yacc)[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    __syncthreads();
    // x -> fp16 MMA B fragments, once for the window (every layer CTA copies them whole):
    // xf[((cb*16 + s)*4 + tq)*T + g] = x[g][e .. e+3], e = 256 cb + 64 tq + (s < 8 ? 4 s : 32 + 4 (s - 8))
    {
        bool bad = false;
        const int n = (H / 256) * 64 * T;
        for (int i = gtid; i < n; i += gthreads) {
            const int g = i % T, r = i / T, tq = r & 3, sx = (r >> 2) & 15, cb = r >> 6;
            const int e = 256 * cb + 64 * tq + (sx < 8 ? 4 * sx : 32 + 4 * (sx - 8));
            const uint2 xb = *reinterpret_cast<const uint2 *>(s_x + g * H + e);
            const float x0 = bf16_bits_to_f32(xb.x & 0xffff), x1 = bf16_bits_to_f32(xb.x >> 16);
            const float x2 = bf16_bits_to_f32(xb.y & 0xffff), x3 = bf16_bits_to_f32(xb.y >> 16);
            const float m = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
            bad |= !(m < 65504.0f);      // beyond the fp16 range, or NaN
            a.xfrag[i] = make_uint2(dq_h22u(__floats2half2_rn(x0, x1)), dq_h22u(__floats2half2_rn(x2, x3)));
        }
        if (bad) set_status(a.header + kHdrStatus, MOE_ERR_DEVICE_FAULT);
    }

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
}

// ---------------------------------------------------------------- the layer

constexpr int kUnitRows = 8;            // ff rows of a routed unit (the 8 MMA rows of each of gate, up)
constexpr int kSharedRows = 4;          // ff rows of a shared-expert unit
constexpr int kPieceQ4K = 144;          // bytes of one row's 256-column block: one Q4_K super-block
constexpr int kPieceQ5K = 176;          // ... in Q5_K
constexpr int kPieceQ80 = 272;          // the same block in Q8_0: eight 34-byte blocks
constexpr uint32_t kSlotBytes = 1152;   // one stage of one warp: 8 x 144 (>= 4 x 272)
constexpr uint32_t kSlotHalf = 640;     // ... of a half-block warp: 8 x 64 quant bytes, then 8 x 16 header bytes
constexpr uint32_t kSlotQ5K = 1408;     // ... of a Q5_K warp: 8 x 176
constexpr int kMaxCons = 16;            // consumer warps of 256 columns
constexpr int kMaxConsHalf = 20;        // consumer warps of 128 columns (96 registers a thread)

// Shared-memory carve of k_dec_layer (byte offsets).
struct LayerSmem {
    uint32_t tab, xf, ids, w, pe, ptok, tmask, bits, pre, red, sa, bar, misc, ring, ring_bytes, total;
};

__host__ __device__ inline uint32_t al16(uint32_t v) { return (v + 15u) & ~15u; }

__host__ __device__ inline LayerSmem layer_smem(int E, int T, int H, int nc, uint32_t ring_bytes)
{
    LayerSmem L{};
    uint32_t o = 0;
    L.tab = o;   o = al16(o + 8u * E);                           // expert table
    L.xf = o;    o = al16(o + 2u * T * H);                       // fp16 MMA B fragments of x
    L.ids = o;   o = al16(o + 4u * kDecMaxAssign);
    L.w = o;     o = al16(o + 4u * kDecMaxAssign);
    L.pe = o;    o = al16(o + 2u * kDecMaxAssign);               // active expert ids
    L.ptok = o;  o = al16(o + 2u * kDecMaxAssign * kDecTok);     // [u][t] assignment of token t, -1 if none
    L.tmask = o; o = al16(o + 4u * kDecMaxAssign);               // [u] tokens routed to active expert u
    L.bits = o;  o = al16(o + 4u * 32);
    L.pre = o;   o = al16(o + 4u * 32);
    L.red = o;   o = al16(o + 2u * 8u * nc * kDecTok * kUnitRows); // [2][warp][token][f] (g, u) partial sums
    L.sa = o;    o = al16(o + 2u * 2u * kDecTok * kUnitRows);      // [2][token][f] weighted activations (fp16)
    L.bar = o;   o = al16(o + 8u);                                 // the prologue's mbarrier
    L.misc = o;  o = al16(o + 64u);
    o = (o + 127u) & ~127u;
    L.ring = o;
    L.ring_bytes = ring_bytes;
    L.total = o + ring_bytes;
    return L;
}

// Unit geometry of a window: Nr routed units (8 ff rows of one active expert)
// then Ns shared-expert units (4 rows), split over the CTAs in equal counts.
// A unit's time is set by its instructions, not its bytes: a 4-row Q8_0 unit
// of the shared expert (52 KB at H = 4096) took as long as an 8-row Q4_K
// unit (55 KB) -- the same MMA and dequantisation steps a warp, half of the
// shared unit's MMA rows idle -- so a split by bytes left the CTAs holding
// shared units about 7% behind the rest.
struct Units {
    int64_t nr, ns;          // unit counts
    int rb, rbs;             // row bytes: routed (Q4_K or Q5_K), Q8_0 shared
    const uint8_t *shared;   // the shared expert's blob, or null
};

struct UnitInfo {
    const uint8_t *blob;
    int fmt;                 // 0: routed (the kernel's codec), 1: Q8_0 shared
    int u;                   // active-expert index (routed), -1 shared
    int f0;                  // first ff row
    int ffm;                 // rows of one matrix in the blob (FF or SFF)
    int rowb;                // row bytes
    int rows;                // ff rows of the unit
};

// Unit i of the window.
__device__ __forceinline__ UnitInfo unit_info(const DecArgs &a, const Units &un, const int16_t *pe,
                                              const uint8_t *const *tab, int i)
{
    UnitInfo ui;
    if (i < (int)un.nr) {
        const int mt = a.FF / kUnitRows;
        ui.u = i / mt;
        ui.rows = kUnitRows;
        ui.f0 = (i - ui.u * mt) * kUnitRows;
        ui.blob = tab[pe[ui.u]];
        ui.fmt = 0;
        ui.ffm = a.FF;
        ui.rowb = un.rb;
    } else {
        ui.u = -1;
        ui.rows = kSharedRows;
        ui.f0 = (i - (int)un.nr) * kSharedRows;
        ui.blob = un.shared;
        ui.fmt = 1;
        ui.ffm = a.SFF;
        ui.rowb = un.rbs;
    }
    return ui;
}

// The unit after c.i (c.ui describes unit c.i): consecutive routed units walk an
// expert's ff rows 8 at a time, then the next active expert's; the shared expert's
// units follow the routed ones.  No division: this runs once per stage.
struct UnitCursor {
    UnitInfo ui;
    int i;
};

__device__ __forceinline__ void unit_next(UnitCursor &c, const DecArgs &a, const Units &un, const int16_t *pe,
                                          const uint8_t *const *tab)
{
    ++c.i;
    if (c.i < (int)un.nr) {
        c.ui.f0 += kUnitRows;
        if (c.ui.f0 == a.FF) {
            c.ui.f0 = 0;
            ++c.ui.u;
            c.ui.blob = tab[pe[c.ui.u]];
        }
    } else if (c.i == (int)un.nr) {
        c.ui = unit_info(a, un, pe, tab, c.i);
    } else {
        c.ui.f0 += kSharedRows;
    }
}

__device__ __forceinline__ void mma16808(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t b0)
{
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(b0));
}

// fp16 pair (row r0, row r1) of the nibbles at byte b (0..3) of words w0 (row
// r0) and w1 (row r1): low nibbles -> q_lo, high nibbles -> q_hi (exact).
__device__ __forceinline__ void nib_pair(uint32_t w0, uint32_t w1, int b, __half2 &q_lo, __half2 &q_hi)
{
    const uint32_t p = __byte_perm(w0, w1, (uint32_t)b | ((uint32_t)(4 + b) << 8));
    q_lo = __hsub2(dq_u2h2((p & 0x000F000Fu) | 0x64006400u), __float2half2_rn(1024.0f));
    q_hi = __hfma2(dq_u2h2((p & 0x00F000F0u) | 0x64006400u), __float2half2_rn(0.0625f), __float2half2_rn(-64.0f));
}

// Q5_K: as nib_pair, with the fifth bits in bit 0 (low nibble's element) and
// bit 1 (high nibble's) of byte b of h0 (row r0) and h1 (row r1).
__device__ __forceinline__ void nib5_pair(uint32_t w0, uint32_t w1, uint32_t h0, uint32_t h1, int b, __half2 &q_lo,
                                          __half2 &q_hi)
{
    const uint32_t sel = (uint32_t)b | ((uint32_t)(4 + b) << 8);
    const uint32_t p = __byte_perm(w0, w1, sel), f = __byte_perm(h0, h1, sel);
    q_lo = __hsub2(dq_u2h2((p & 0x000F000Fu) | ((f << 4) & 0x00100010u) | 0x64006400u), __float2half2_rn(1024.0f));
    q_hi = __hfma2(dq_u2h2((p & 0x00F000F0u) | ((f << 7) & 0x01000100u) | 0x64006400u), __float2half2_rn(0.0625f),
                   __float2half2_rn(-64.0f));
}

// int8 pair (row r0, row r1) at byte b of words w0 and w1 -> exact fp16 pair.
__device__ __forceinline__ __half2 i8_pair(uint32_t w0, uint32_t w1, int b)
{
    const uint32_t p = __byte_perm(w0, w1, (uint32_t)b | ((uint32_t)(4 + b) << 8));
    return __hsub2(dq_u2h2(((p ^ 0x00800080u) & 0x00FF00FFu) | 0x64006400u), __float2half2_rn(1152.0f));
}

__device__ __forceinline__ void cp16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp8(uint32_t dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// One warp copies its column block (P 16-byte pieces) of ROWS consecutive rows
// (`rowb` bytes apart in global memory) into a packed [ROWS][16 P] slab: piece
// i = lane + 32 k (ROWS * P <= 96 pieces).
template <int P, int ROWS>
__device__ __forceinline__ void copy_block(uint32_t dst, const uint8_t *src, int rowb, int lane)
{
    static_assert(ROWS * P <= 96, "three pieces a lane");
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const int i = lane + 32 * k;
        if (i < ROWS * P) {
            const int r = i / P, p = i - r * P;
            cp16(dst + (uint32_t)(r * 16 * P + 16 * p), src + r * rowb + 16 * p);
        }
    }
}

// Variants of the layer kernel: Q4_K routed rows with 256-column warps, with
// 128-column warps, or Q5_K routed rows with 256-column warps.
constexpr int kVarQ4K = 0, kVarHalf = 1, kVarQ5K = 2;

// One layer of a window, in every CTA (the body of the layer kernel and of
// the stack kernel): the routing of the window from the logits in shared
// memory (the ring's first 4 T E bytes), then this CTA's share of the units,
// whose down projections are added into yacc; CTA 0 publishes the routing to
// the workspace when `publish` is set.  On entry the expert table
// and the x fragments are in shared memory, the abort flag is settled, and
// every thread that reads the logits has seen them land.  S stages per
// consumer warp.  HALF: each consumer warp owns 128 columns (half a Q4_K
// super-block) instead of 256, for twice the warps; only for layers without a
// shared expert.  Q5: the routed rows are Q5_K blocks (the layout of Q4_K's
// plus 32 bytes of fifth bits, qh, before the nibbles).
template <int S, int V>
__device__ __forceinline__ void dec_window(const DecArgs &a, uint8_t *smem, const float *bias,
                                           const uint8_t *shared_blob, float *yacc, bool publish)
{
    static_assert(S >= 4, "the lagging down projection keeps 3 stages busy");
    constexpr bool HALF = V == kVarHalf, Q5 = V == kVarQ5K;
    constexpr int PIECE = Q5 ? kPieceQ5K : kPieceQ4K;   // bytes of a routed row's 256-column block
    constexpr int QS = Q5 ? 48 : 16;                     // offset of its nibbles
    const int T = a.T, H = a.H, E = a.E, k = a.k, nb = H / 256, NC = a.nc;
    const LayerSmem L = layer_smem(E, T, H, NC, a.ring_bytes);
    const uint8_t **s_tab = reinterpret_cast<const uint8_t **>(smem + L.tab);
    uint2 *s_xf = reinterpret_cast<uint2 *>(smem + L.xf);
    int32_t *s_ids = reinterpret_cast<int32_t *>(smem + L.ids);
    float *s_w = reinterpret_cast<float *>(smem + L.w);
    int16_t *s_pe = reinterpret_cast<int16_t *>(smem + L.pe);
    int16_t(*s_ptok)[kDecTok] = reinterpret_cast<int16_t(*)[kDecTok]>(smem + L.ptok);
    uint32_t *s_tmask = reinterpret_cast<uint32_t *>(smem + L.tmask);
    uint32_t *s_bits = reinterpret_cast<uint32_t *>(smem + L.bits);
    int32_t *s_pre = reinterpret_cast<int32_t *>(smem + L.pre);
    float2 *s_red = reinterpret_cast<float2 *>(smem + L.red);     // [2][NC][window token][8]
    __half *s_wa = reinterpret_cast<__half *>(smem + L.sa);       // [2][kDecTok][8]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.misc);
    int *s_nact = reinterpret_cast<int *>(smem + L.misc + 4);
    uint8_t *ring = smem + L.ring;
    uint32_t *status = a.header + kHdrStatus;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nthr = blockDim.x;

    // selection keys and values beside the logits (the ring is not in use yet)
    const float *s_lg = reinterpret_cast<const float *>(ring);
    uint32_t *s_key = reinterpret_cast<uint32_t *>(ring + 4 * T * E);
    float *s_val = reinterpret_cast<float *>(ring + 8 * T * E);
    {
        const bool sig = a.score_fn != MOE_SCORE_SOFTMAX;
        for (int i = threadIdx.x; i < T * E; i += nthr) {
            const float l = s_lg[i];
            const float sv = sig ? 1.0f / (1.0f + expf(-l)) : l;
            const float b = (sig && bias) ? __ldg(bias + i % E) : 0.0f;
            s_val[i] = sv;
            s_key[i] = key_bits(sig ? sv + b : sv);
        }
    }
    if (threadIdx.x < 32) s_bits[threadIdx.x] = 0u;
    for (int i = threadIdx.x; i < 2 * kDecTok * kUnitRows; i += nthr) s_wa[i] = __float2half_rn(0.0f);
    __syncthreads();
    if (warp < T) {
        int id;
        float wt;
        bool f;
        const uint32_t *kr = s_key + warp * E;
        const float *vr = s_val + warp * E;
        if (E <= 256) warp_topk<8>(kr, vr, E, k, a.score_fn, lane, id, wt, f);
        else if (E <= 512) warp_topk<16>(kr, vr, E, k, a.score_fn, lane, id, wt, f);
        else warp_topk<32>(kr, vr, E, k, a.score_fn, lane, id, wt, f);
        if (lane < k) {
            s_ids[warp * k + lane] = id;
            s_w[warp * k + lane] = wt;
            atomicOr(&s_bits[id >> 5], 1u << (id & 31));
        }
        if (f && lane == 0 && blockIdx.x == 0) set_status(status, MOE_ERR_DEVICE_FAULT);
    }
    __syncthreads();
    if (warp == 0) {
        // active experts in id order: bitmap word l covers experts 32 l .. 32 l + 31
        const uint32_t word = s_bits[lane];
        const int c = __popc(word);
        int incl = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        s_pre[lane] = incl - c;
        uint32_t wd = word;
        int j = incl - c;
        while (wd) {
            const int b = __ffs(wd) - 1;
            wd &= wd - 1;
            s_pe[j++] = (int16_t)(32 * lane + b);
        }
        if (lane == 31) *s_nact = incl;
    }
    __syncthreads();
    const int U = *s_nact, TK = T * k;
    auto rank_of = [&](int e) { return s_pre[e >> 5] + __popc(s_bits[e >> 5] & ((1u << (e & 31)) - 1u)); };
    for (int i = threadIdx.x; i < U * kDecTok; i += nthr) s_ptok[i / kDecTok][i % kDecTok] = -1;
    for (int i = threadIdx.x; i < U; i += nthr) s_tmask[i] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < TK; i += nthr) {
        const int u = rank_of(s_ids[i]), t = i / k;
        s_ptok[u][t] = (int16_t)i;
        atomicOr(&s_tmask[u], 1u << t);
    }
    __syncthreads();
    if (publish && blockIdx.x == 0) {
        // publish the routing: ids, w, counts, offsets, assign, active list
        for (int i = threadIdx.x; i < TK; i += nthr) {
            a.ids[i] = s_ids[i];
            a.w[i] = s_w[i];
        }
        if (warp == 0) {
            // exclusive scan of the active experts' token counts, in id order
            const int per = (U + 31) / 32;
            int tot = 0;
            for (int j = 0; j < per; ++j) {
                const int u = lane * per + j;
                if (u < U) tot += __popc(s_tmask[u]);
            }
            int incl = tot;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            int run = incl - tot;
            for (int j = 0; j < per; ++j) {
                const int u = lane * per + j;
                if (u < U) {
                    const uint32_t m = s_tmask[u];
                    for (int t = 0; t < T; ++t)
                        if ((m >> t) & 1u) a.assign[run + __popc(m & ((1u << t) - 1u))] = s_ptok[u][t];
                    a.active[u] = s_pe[u];
                    reinterpret_cast<int32_t *>(ring)[u] = run;   // scratch (the keys are dead): offset of u
                    run += __popc(m);
                }
            }
        }
        __syncthreads();
        for (int e = threadIdx.x; e < E; e += nthr) {
            const uint32_t wd = s_bits[e >> 5];
            const int u = rank_of(e);
            const bool sel = (wd >> (e & 31)) & 1u;
            a.counts[e] = sel ? __popc(s_tmask[u]) : 0;
            a.offsets[e] = u < U ? reinterpret_cast<const int32_t *>(ring)[u] : TK;
        }
        if (threadIdx.x == 0) {
            a.offsets[E] = TK;
            a.header[kHdrNActive] = (uint32_t)U;
        }
        __syncthreads();
    }

    // ---- this CTA's share of the window's units
    Units un;
    un.rb = nb * PIECE;
    un.rbs = nb * kPieceQ80;
    un.nr = (int64_t)U * (a.FF / kUnitRows);
    un.shared = shared_blob;
    un.ns = shared_blob ? a.SFF / kSharedRows : 0;
    const int64_t total = un.nr + un.ns;
    const int64_t u_begin = total * blockIdx.x / gridDim.x;
    const int64_t u_end = total * (blockIdx.x + 1) / gridDim.x;
    __syncthreads();   // the routing scratch in the ring is free from here on; the abort flag is settled

    if (warp < NC && !*abort_flag) {
        // ------------------------------------------------------------ consumers
        // Warp w owns the 256-column block w of H, and reads nothing else of a
        // row: of every slab (8 rows of gate, up or down of a unit) it stages its
        // own block -- 144 bytes a Q4_K row, 272 a Q8_0 row -- into its own ring
        // of S stages with 16-byte cp.async, so the warps stream independently and
        // no copy is issued on another warp's behalf.  Stage j (unit j / 3, matrix
        // j % 3) sits in slot j % S.  The down projection of unit u runs one unit
        // late, after the gate/up of unit u + 1, so one barrier per unit orders
        // both the partial sums (gate/up) and the activations (down).
        // (HALF: warp w owns the 128-column half w % 2 of block w / 2, and stages the
        // row headers and its half of the quant bytes.)
        constexpr uint32_t SLOT = HALF ? kSlotHalf : Q5 ? kSlotQ5K : kSlotBytes;
        constexpr int NT = HALF ? 8 : 16;                // down tiles of 16 columns (x 2) per warp
        const int g = lane >> 2, tq = lane & 3;
        const int cb = HALF ? warp >> 1 : warp, hh = HALF ? warp & 1 : 0;
        const int n_unit = (int)(u_end - u_begin), n_stage = 3 * n_unit;
        const uint32_t wring = sm_addr(ring) + (uint32_t)(warp * S) * SLOT;
        const uint8_t *wring_p = ring + (size_t)warp * S * SLOT;
        // the next stage to copy: stage js, matrix im of the unit under the cursor ic
        const UnitInfo ui0 = unit_info(a, un, s_pe, s_tab, (int)u_begin);
        UnitCursor ic{ui0, (int)u_begin};
        int js = 0, im = 0;
        // HALF: this lane's pieces of every slab, fixed for the whole stream: piece i
        // (lane, and lane + 32 for lanes < 8) = (offset in the slab << 10) | offset in
        // the slot (the slab offset is < 8 rows x 1440 bytes, the slot offset < 640)
        uint32_t hp0 = 0, hp1 = 0;
        if (HALF) {
            auto piece = [&](int i) {
                const int r = i / 5, p = i - r * 5;
                const uint32_t d = p == 0 ? 512u + 16u * r : (uint32_t)(64 * r + 16 * (p - 1));
                const uint32_t o = (uint32_t)(r * un.rb + (p == 0 ? 0 : 16 + 64 * hh + 16 * (p - 1)));
                return (o << 10) | d;
            };
            hp0 = piece(lane);
            hp1 = lane < kUnitRows * 5 - 32 ? piece(lane + 32) : 0u;
        }
        auto issue = [&]() {
            if (js < n_stage && ic.ui.blob) {
                const uint8_t *src = ic.ui.blob + ((int64_t)im * ic.ui.ffm + ic.ui.f0) * ic.ui.rowb;
                const uint32_t dst = wring + (uint32_t)(js % S) * SLOT;
                if (HALF) {                              // routed units only
                    const uint8_t *sb = src + cb * kPieceQ4K;
                    cp16(dst + (hp0 & 1023u), sb + (hp0 >> 10));
                    if (lane < kUnitRows * 5 - 32) cp16(dst + (hp1 & 1023u), sb + (hp1 >> 10));
                } else if (ic.ui.fmt == 0) copy_block<PIECE / 16, kUnitRows>(dst, src + cb * PIECE, ic.ui.rowb, lane);
                else copy_block<kPieceQ80 / 16, kSharedRows>(dst, src + cb * kPieceQ80, ic.ui.rowb, lane);
            }
            cp_commit();                                 // one group a stage, empty or not
            ++js;
            if (++im == 3) {
                im = 0;
                if (js < n_stage) unit_next(ic, a, un, s_pe, s_tab);
            }
        };
        for (int j = 0; j < S - 1; ++j) issue();
        // B fragment x[token g][e .. e+3] in fp16 (zero for g >= T), e = 256 cb + 64 c +
        // (s < 8 ? 4 s : 32 + 4 (s - 8)): sub-block pair c, word s of its quant bytes
        auto xb = [&](int s, int c) { return g < T ? s_xf[((cb * 16 + s) * 4 + c) * T + g] : make_uint2(0u, 0u); };
        // down accumulators: tile i (16 hidden rows x the 8 window tokens): d0/d1 =
        // columns hl(g, i) for tokens 2tq, 2tq+1, d2/d3 = columns hl(g, i) + 32, with
        // hl(g, i) = 256 cb + 64 (g / 2) + 16 (g % 2) + i, or (HALF) 256 cb + 64 c +
        // 8 (g % 4) + i with c = 2 hh + g / 4
        float D[NT][4];
#pragma unroll
        for (int i4 = 0; i4 < NT; ++i4) D[i4][0] = D[i4][1] = D[i4][2] = D[i4][3] = 0.0f;
        auto down = [&](const UnitInfo &ui, const uint8_t *dn, const __half *wa) {
            // B fragment: rows f = 2tq, 2tq + 1 of token g
            const uint32_t bfr = *reinterpret_cast<const uint32_t *>(wa + g * kUnitRows + 2 * tq);
            // rows 2tq, 2tq + 1 (K of the MMA); beyond a short unit they read row 0, whose
            // product with the zero activations of those rows adds nothing
            if (HALF) {
                // lane g takes quant bytes 8 (g % 4) .. + 7 of pair c = 2 hh + g / 4, i.e. bytes
                // 8 g .. 8 g + 7 of the staged half: columns 64 c + 8 (g % 4) + i (low
                // nibbles) and + 32 (high)
                const uint8_t *q0p = dn + (2 * tq) * 64, *q1p = q0p + 64;
                const uint8_t *h0p = dn + 512 + (2 * tq) * 16, *h1p = h0p + 16;
                const int c = 2 * hh + (g >> 2);
                __half2 S0, N0, S1, N1;
                q4k_pair_scales_h(*reinterpret_cast<const uint4 *>(h0p), c, S0, N0);
                q4k_pair_scales_h(*reinterpret_cast<const uint4 *>(h1p), c, S1, N1);
                const __half2 Slo = __lows2half2(S0, S1), Shi = __highs2half2(S0, S1);
                const __half2 Nlo = __lows2half2(N0, N1), Nhi = __highs2half2(N0, N1);
                const uint2 q0 = *reinterpret_cast<const uint2 *>(q0p + 8 * g);
                const uint2 q1 = *reinterpret_cast<const uint2 *>(q1p + 8 * g);
                const uint32_t w0[2] = {q0.x, q0.y}, w1[2] = {q1.x, q1.y};
#pragma unroll
                for (int t8 = 0; t8 < NT; ++t8) {
                    __half2 ql, qh;
                    nib_pair(w0[(t8 >> 2) & 1], w1[(t8 >> 2) & 1], t8 & 3, ql, qh);
                    mma16808(D[t8], dq_h22u(__hfma2(ql, Slo, Nlo)), dq_h22u(__hfma2(qh, Shi, Nhi)), bfr);
                }
            } else if (ui.fmt == 0) {
                const uint8_t *r0 = dn + (2 * tq) * PIECE, *r1 = r0 + PIECE;
                // lane g takes quant bytes 16 g .. 16 g + 15 of the block: chunk c = g / 2
                // (sub-blocks 2c low nibbles, 2c + 1 high), columns hl(g, i)
                const int c = g >> 1;
                __half2 S0, N0, S1, N1;
                q4k_pair_scales_h(*reinterpret_cast<const uint4 *>(r0), c, S0, N0);
                q4k_pair_scales_h(*reinterpret_cast<const uint4 *>(r1), c, S1, N1);
                const __half2 Slo = __lows2half2(S0, S1), Shi = __highs2half2(S0, S1);
                const __half2 Nlo = __lows2half2(N0, N1), Nhi = __highs2half2(N0, N1);
                const uint4 q0 = *reinterpret_cast<const uint4 *>(r0 + QS + 16 * g);
                const uint4 q1 = *reinterpret_cast<const uint4 *>(r1 + QS + 16 * g);
                const uint32_t w0[4] = {q0.x, q0.y, q0.z, q0.w}, w1[4] = {q1.x, q1.y, q1.z, q1.w};
                uint32_t f0[4] = {0u, 0u, 0u, 0u}, f1[4] = {0u, 0u, 0u, 0u};
                if (Q5) {
                    // the fifth bits of the same 16 elements: qh bytes 16 (g % 2) .. + 15, bits
                    // 2c (low sub-block) and 2c + 1 (high) moved to bits 0 and 1
                    const uint4 h0 = *reinterpret_cast<const uint4 *>(r0 + 16 + 16 * (g & 1));
                    const uint4 h1 = *reinterpret_cast<const uint4 *>(r1 + 16 + 16 * (g & 1));
                    const int sh = 2 * c;
                    f0[0] = h0.x >> sh; f0[1] = h0.y >> sh; f0[2] = h0.z >> sh; f0[3] = h0.w >> sh;
                    f1[0] = h1.x >> sh; f1[1] = h1.y >> sh; f1[2] = h1.z >> sh; f1[3] = h1.w >> sh;
                }
#pragma unroll
                for (int t16 = 0; t16 < NT; ++t16) {
                    __half2 ql, qh;
                    if (Q5) nib5_pair(w0[(t16 >> 2) & 3], w1[(t16 >> 2) & 3], f0[(t16 >> 2) & 3], f1[(t16 >> 2) & 3],
                                      t16 & 3, ql, qh);
                    else nib_pair(w0[(t16 >> 2) & 3], w1[(t16 >> 2) & 3], t16 & 3, ql, qh);
                    mma16808(D[t16], dq_h22u(__hfma2(ql, Slo, Nlo)), dq_h22u(__hfma2(qh, Shi, Nhi)), bfr);
                }
            } else {
                const uint8_t *r0 = dn + (2 * tq < ui.rows ? 2 * tq : 0) * kPieceQ80;
                const uint8_t *r1 = dn + (2 * tq + 1 < ui.rows ? 2 * tq + 1 : 0) * kPieceQ80;
                // Q8_0: the same columns: hl(g, i) lies in block 2c of this 256-column
                // window at position 16 (g % 2) + i, hl + 32 in block 2c + 1
                const int c = g >> 1, h1 = g & 1;
                const uint32_t *p0 = reinterpret_cast<const uint32_t *>(r0 + 68 * c);   // block 2c (2c + 1 at + 34)
                const uint32_t *p1 = reinterpret_cast<const uint32_t *>(r1 + 68 * c);
                const __half2 dlo = __halves2half2(__ushort_as_half((unsigned short)(p0[0] & 0xffff)),
                                                   __ushort_as_half((unsigned short)(p1[0] & 0xffff)));
                const __half2 dhi = __halves2half2(__ushort_as_half((unsigned short)(p0[8] >> 16)),
                                                   __ushort_as_half((unsigned short)(p1[8] >> 16)));
#pragma unroll
                for (int wq = 0; wq < 4; ++wq) {
                    // block 2c bytes 2 + 16 h1 + 4 wq ..: words (16 h1 + 4 wq) / 4 .. shifted 16
                    const int wl = 4 * h1 + wq;
                    const uint32_t l0 = __funnelshift_r(p0[wl], p0[wl + 1], 16);
                    const uint32_t l1 = __funnelshift_r(p1[wl], p1[wl + 1], 16);
                    // block 2c + 1 bytes 36 + 16 h1 + 4 wq: word 9 + 4 h1 + wq (aligned)
                    const uint32_t u0 = p0[9 + wl], u1 = p1[9 + wl];
#pragma unroll
                    for (int b = 0; b < 4; ++b)
                        mma16808(D[(4 * wq + b) % NT], dq_h22u(__hmul2(i8_pair(l0, l1, b), dlo)),
                                 dq_h22u(__hmul2(i8_pair(u0, u1, b), dhi)), bfr);
                }
            }
        };
        uint32_t touched = 0;                             // window tokens this CTA's units served
        UnitInfo prev{};
        bool prev_live = false;
        UnitCursor cc{ui0, (int)u_begin};                   // the unit being computed
        for (int u = 0; u < n_unit; ++u) {
            if (u > 0) unit_next(cc, a, un, s_pe, s_tab);
            const UnitInfo ui = cc.ui;
            const bool live = ui.blob != nullptr;
            if (!live && warp == 0 && lane == 0) set_status(status, MOE_ERR_DEVICE_FAULT);
            // tokens of this unit: the expert's, or every token (shared)
            const uint32_t tmask = live ? (ui.u >= 0 ? s_tmask[ui.u] : ((1u << T) - 1u)) : 0u;
            touched |= tmask;
            cp_wait<S - 3>();                            // stages up to 3u + 1 have landed
            __syncwarp();
            // ---- gate / up over this warp's block
            float c4[2][4];
#pragma unroll
            for (int i2 = 0; i2 < 2; ++i2) c4[i2][0] = c4[i2][1] = c4[i2][2] = c4[i2][3] = 0.0f;
            if (live) {
                const uint8_t *gst = wring_p + (uint32_t)((3 * u) % S) * SLOT;
                const uint8_t *ust = wring_p + (uint32_t)((3 * u + 1) % S) * SLOT;
                if (HALF) {
                    // lane tq takes quant bytes 16 tq .. 16 tq + 15 of the staged half: words
                    // 4 (tq % 2) .. + 3 of pair c = 2 hh + tq / 2
                    const uint8_t *gr = gst + g * 64, *ur = ust + g * 64;
                    const int c = 2 * hh + (tq >> 1);
                    __half2 Sg, NZg, Su, NZu;
                    q4k_pair_scales_h(*reinterpret_cast<const uint4 *>(gst + 512 + g * 16), c, Sg, NZg);
                    q4k_pair_scales_h(*reinterpret_cast<const uint4 *>(ust + 512 + g * 16), c, Su, NZu);
                    const uint4 ga = *reinterpret_cast<const uint4 *>(gr + 16 * tq);
                    const uint4 ua = *reinterpret_cast<const uint4 *>(ur + 16 * tq);
                    const uint32_t gq[4] = {ga.x, ga.y, ga.z, ga.w};
                    const uint32_t uq[4] = {ua.x, ua.y, ua.z, ua.w};
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        uint32_t og[4], ou[4];
                        q4k_word_f16(gq[s], __low2half2(Sg), __low2half2(NZg), __high2half2(Sg), __high2half2(NZg), og);
                        q4k_word_f16(uq[s], __low2half2(Su), __low2half2(NZu), __high2half2(Su), __high2half2(NZu), ou);
                        const int w = 4 * (tq & 1) + s;
                        const uint2 xl = xb(w, c), xh = xb(8 + w, c);
                        mma16816(c4[0], og[0], ou[0], og[1], ou[1], xl.x, xl.y);
                        mma16816(c4[1], og[2], ou[2], og[3], ou[3], xh.x, xh.y);
                    }
                } else if (ui.fmt == 0) {
                    const uint8_t *gr = gst + g * PIECE, *ur = ust + g * PIECE;
                    __half2 Sg, NZg, Su, NZu;
                    q4k_pair_scales_h(*reinterpret_cast<const uint4 *>(gr), tq, Sg, NZg);
                    q4k_pair_scales_h(*reinterpret_cast<const uint4 *>(ur), tq, Su, NZu);
                    const uint4 ga = *reinterpret_cast<const uint4 *>(gr + QS + 32 * tq);
                    const uint4 gb = *reinterpret_cast<const uint4 *>(gr + QS + 16 + 32 * tq);
                    const uint4 ua = *reinterpret_cast<const uint4 *>(ur + QS + 32 * tq);
                    const uint4 ub = *reinterpret_cast<const uint4 *>(ur + QS + 16 + 32 * tq);
                    const uint32_t gq[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
                    const uint32_t uq[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
                    // Q5_K: the fifth bits of quant byte l of chunk tq are bits 2 tq, 2 tq + 1
                    // of qh[l]; word s of qh covers the bytes of word s of the chunk
                    const uint32_t *gqh = reinterpret_cast<const uint32_t *>(gr + 16);
                    const uint32_t *uqh = reinterpret_cast<const uint32_t *>(ur + 16);
#pragma unroll
                    for (int s = 0; s < 8; ++s) {
                        uint32_t og[4], ou[4];
                        if (Q5) {
                            q5k_word_f16(gq[s], gqh[s] >> (2 * tq), __low2half2(Sg), __low2half2(NZg), __high2half2(Sg),
                                         __high2half2(NZg), og);
                            q5k_word_f16(uq[s], uqh[s] >> (2 * tq), __low2half2(Su), __low2half2(NZu), __high2half2(Su),
                                         __high2half2(NZu), ou);
                        } else {
                            q4k_word_f16(gq[s], __low2half2(Sg), __low2half2(NZg), __high2half2(Sg), __high2half2(NZg), og);
                            q4k_word_f16(uq[s], __low2half2(Su), __low2half2(NZu), __high2half2(Su), __high2half2(NZu), ou);
                        }
                        const uint2 xl = xb(s, tq), xh = xb(8 + s, tq);
                        mma16816(c4[0], og[0], ou[0], og[1], ou[1], xl.x, xl.y);
                        mma16816(c4[1], og[2], ou[2], og[3], ou[3], xh.x, xh.y);
                    }
                } else {
                    // units shorter than 8 rows: MMA rows g >= rows read row 0 (their
                    // outputs are not used)
                    const int gr_ = g < ui.rows ? g : 0;
                    const uint32_t *gw = reinterpret_cast<const uint32_t *>(gst + gr_ * kPieceQ80 + 68 * tq);
                    const uint32_t *uw = reinterpret_cast<const uint32_t *>(ust + gr_ * kPieceQ80 + 68 * tq);
                    const __half2 Dg0 = __half2half2(__ushort_as_half((unsigned short)(gw[0] & 0xffff)));
                    const __half2 Dg1 = __half2half2(__ushort_as_half((unsigned short)(gw[8] >> 16)));
                    const __half2 Du0 = __half2half2(__ushort_as_half((unsigned short)(uw[0] & 0xffff)));
                    const __half2 Du1 = __half2half2(__ushort_as_half((unsigned short)(uw[8] >> 16)));
#pragma unroll
                    for (int s = 0; s < 8; ++s) {
                        // block 2tq: q8 bytes 2 + 4s .. 5 + 4s; block 2tq + 1: bytes 36 + 4s ..
                        const uint32_t gl = __funnelshift_r(gw[s], gw[s + 1], 16);
                        const uint32_t ul = __funnelshift_r(uw[s], uw[s + 1], 16);
                        const uint32_t gh = gw[9 + s], uh = uw[9 + s];
                        const uint2 xl = xb(s, tq), xh = xb(8 + s, tq);
                        mma16816(c4[0], q80_pair_f16(gl, Dg0), q80_pair_f16(ul, Du0), q80_pair_f16(gl >> 16, Dg0),
                                 q80_pair_f16(ul >> 16, Du0), xl.x, xl.y);
                        mma16816(c4[1], q80_pair_f16(gh, Dg1), q80_pair_f16(uh, Du1), q80_pair_f16(gh >> 16, Dg1),
                                 q80_pair_f16(uh >> 16, Du1), xh.x, xh.y);
                    }
                }
            }
            // partial sums of this warp: (g, u) of ff row f0 + g for window token n
            const int buf = u & 1;
            {
                float2 *red = s_red + (size_t)buf * NC * kDecTok * kUnitRows;
                const float c0 = c4[0][0] + c4[1][0], c1 = c4[0][1] + c4[1][1];
                const float c2 = c4[0][2] + c4[1][2], c3 = c4[0][3] + c4[1][3];
                if (g < ui.rows) {
                    if ((tmask >> (2 * tq)) & 1u) red[(warp * kDecTok + 2 * tq) * kUnitRows + g] = make_float2(c0, c2);
                    if ((tmask >> (2 * tq + 1)) & 1u)
                        red[(warp * kDecTok + 2 * tq + 1) * kUnitRows + g] = make_float2(c1, c3);
                }
            }
            // every warp's partial sums of unit u, and the activations of unit u - 1, are
            // complete past this barrier
            __syncwarp();
            asm volatile("bar.sync 1, %0;" ::"r"(NC * 32) : "memory");
            // B operand of the down projection of unit u: w_{n,e} * SiLU(g) * u in fp16, [token n][ff row f],
            // for the window's tokens (the MMA columns of absent tokens hold zeros)
            // (half-block warps: 8 threads an activation, each adding every 8th warp's partial
            // sums, then the 8 added across lanes in a fixed order; otherwise one thread an
            // activation: the other warps go on to their down rows meanwhile)
            {
                const float2 *red = s_red + (size_t)buf * NC * kDecTok * kUnitRows;
                auto finish = [&](int n, int f, bool act, float gs, float us) {
                    float v = 0.0f;
                    if (act) {
                        const float wt = ui.u >= 0 ? s_w[s_ptok[ui.u][n]] : 1.0f;
                        v = silu_mul(gs, us) * wt;
                        if (!(fabsf(v) <= 65504.0f)) set_status(status, MOE_ERR_DEVICE_FAULT);
                    }
                    s_wa[buf * kDecTok * kUnitRows + n * kUnitRows + f] = __float2half_rn(v);
                };
                if (HALF && NC >= 16) {
                    const int ct = warp * 32 + lane;
                    if (ct < 8 * kUnitRows * T) {                   // whole warps (T of them)
                        const int item = ct >> 3, sl = ct & 7, f = item & 7, n = item >> 3;
                        const bool act = ((tmask >> n) & 1u) && f < ui.rows;
                        float gs = 0.0f, us = 0.0f;
                        if (act)
                            for (int w2 = sl; w2 < NC; w2 += 8) {
                                const float2 pv = red[(w2 * kDecTok + n) * kUnitRows + f];
                                gs += pv.x;
                                us += pv.y;
                            }
#pragma unroll
                        for (int off = 1; off < 8; off <<= 1) {
                            gs += __shfl_xor_sync(0xffffffffu, gs, off);
                            us += __shfl_xor_sync(0xffffffffu, us, off);
                        }
                        if (sl == 0) finish(n, f, act, gs, us);
                    }
                } else {
                    for (int ct = warp * 32 + lane; ct < kUnitRows * T; ct += NC * 32) {
                        const int f = ct & 7, n = ct >> 3;
                        const bool act = ((tmask >> n) & 1u) && f < ui.rows;
                        float gs = 0.0f, us = 0.0f;
                        if (act)
                            for (int w2 = 0; w2 < NC; ++w2) {
                                const float2 pv = red[(w2 * kDecTok + n) * kUnitRows + f];
                                gs += pv.x;
                                us += pv.y;
                            }
                        finish(n, f, act, gs, us);
                    }
                }
            }
            // ---- down rows of unit u - 1 (the 8 rows are the MMA K), for this warp's block
            if (u > 0 && prev_live)
                down(prev, wring_p + (uint32_t)((3 * u - 1) % S) * SLOT, s_wa + (buf ^ 1) * kDecTok * kUnitRows);
            // the slots of stages 3u - 1, 3u and 3u + 1 are read: refill them
            __syncwarp();
            issue();                                     // stages 3u - 1 + S .. 3u + 1 + S
            issue();
            issue();
            prev = ui;
            prev_live = live;
        }
        if (n_unit > 0) {
            cp_wait<0>();
            __syncwarp();
            asm volatile("bar.sync 1, %0;" ::"r"(NC * 32) : "memory");   // the last activations
            if (prev_live)
                down(prev, wring_p + (uint32_t)((3 * n_unit - 1) % S) * SLOT,
                     s_wa + ((n_unit - 1) & 1) * kDecTok * kUnitRows);
        }
        // ---- this CTA's share of y, for the window tokens its units served
        {
            const int hl = HALF ? 256 * cb + 64 * (2 * hh + (g >> 2)) + 8 * (g & 3)
                                : 256 * cb + 64 * (g >> 1) + 16 * (g & 1);
#pragma unroll
            for (int half = 0; half < 2; ++half)
#pragma unroll
                for (int tk = 0; tk < 2; ++tk) {
                    const int n = 2 * tq + tk;
                    if ((touched >> n) & 1u) {
                        float *dst = yacc + (int64_t)n * H + hl + 32 * half;
#pragma unroll
                        for (int v = 0; v < NT / 4; ++v)
                            red_add_v4(dst + 4 * v, D[4 * v][2 * half + tk], D[4 * v + 1][2 * half + tk],
                                       D[4 * v + 2][2 * half + tk], D[4 * v + 3][2 * half + tk]);
                    }
                }
        }
    }
}

// y = bf16(acc) (and y_f32 = acc when given) over float4 items i0, i0 + step, ...
// below n4; the loads of a batch are issued before its stores.
__device__ __forceinline__ void y_from_acc(const float *acc_, uint16_t *y_, float *y_f32_, int i0, int n4, int step)
{
    const float4 *__restrict__ acc = reinterpret_cast<const float4 *>(acc_);
    uint2 *__restrict__ yb = reinterpret_cast<uint2 *>(y_);
    float4 *__restrict__ yf = reinterpret_cast<float4 *>(y_f32_);
    constexpr int kBatch = 8;
    for (; i0 < n4; i0 += kBatch * step) {
        float4 v[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
            if (i0 + j * step < n4) v[j] = __ldcg(acc + i0 + j * step);
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int i = i0 + j * step;
            if (i < n4) {
                const uint32_t lo = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[j].x)) |
                                    ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[j].y)) << 16);
                const uint32_t hi = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[j].z)) |
                                    ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[j].w)) << 16);
                yb[i] = make_uint2(lo, hi);
                if (yf) yf[i] = v[j];
            }
        }
    }
}

// The layer kernel of one window: one persistent CTA per SM, S stages per
// consumer warp.  128 registers a thread at 256 columns (16 warps, 4 on each
// SM sub-partition, fit one SM), 96 for half-block warps (20 warps).
template <int S, int V>
__global__ void __maxnreg__(V == kVarHalf ? 96 : 128) k_dec_layer(const __grid_constant__ DecArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int T = a.T, H = a.H, E = a.E;
    const LayerSmem L = layer_smem(E, T, H, a.nc, a.ring_bytes);
    const uint8_t **s_tab = reinterpret_cast<const uint8_t **>(smem + L.tab);
    uint2 *s_xf = reinterpret_cast<uint2 *>(smem + L.xf);
    const uint32_t bx = sm_addr(smem + L.bar);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.misc);
    int *s_is_last = reinterpret_cast<int *>(smem + L.misc + 8);
    uint8_t *ring = smem + L.ring;
    uint32_t *status = a.header + kHdrStatus;
    const long long limit = a.wait_cycles;
    const int nthr = blockDim.x;

    if (threadIdx.x == 0) {
        mbar_init(bx, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // no thread may touch the barrier (or the abort flag) before they are initialised:
    // warps start independently, and a wait on an uninitialised barrier is undefined
    __syncthreads();
    // the expert table: before the dependency wait when the weights are static
    if (a.overlap_prev)
        for (int e = threadIdx.x; e < E; e += nthr) s_tab[e] = a.blobs[e];
    // the next call's router kernel may launch now and load its (static) rows
    // while this window streams
    griddep_launch();
    griddep_wait();
    if (!a.overlap_prev)
        for (int e = threadIdx.x; e < E; e += nthr) s_tab[e] = a.blobs[e];

    // ---- the window's x fragments (built by the router kernel) and logits: one bulk
    //      copy each (every CTA reads the same bytes: whole copies keep that cheap)
    {
        const uint32_t xbytes = 2u * T * H, lbytes = (4u * T * E + 15u) & ~15u;
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(bx, xbytes + lbytes);
            if ((int)blockIdx.x != a.skip_cta) {      // test hook: never issued, so the wait runs out
                bulk_g2s(sm_addr(s_xf), a.xfrag, xbytes, bx);
                bulk_g2s(sm_addr(ring), a.logits, lbytes, bx);
            }
        }
        if (!wait_phase(bx, 0u, abort_flag, status, limit) && threadIdx.x == 0) {
            *abort_flag = 1;
            // copies in flight must land before the CTA ends (bounded)
            const long long t0 = clock64();
            while ((int)blockIdx.x != a.skip_cta && !mbar_poll(bx, 0u) && clock64() - t0 < limit) {
            }
        }
    }
    dec_window<S, V>(a, smem, a.bias, a.shared_blob, a.yacc, true);

    // ---- the last CTA to finish writes y
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t ticket = atomicAdd(a.header + kHdrTicketDown, 1u);
        *s_is_last = ticket == gridDim.x - 1;
    }
    __syncthreads();
    if (*s_is_last) {
        __threadfence();
        y_from_acc(a.yacc, a.y, a.y_f32, threadIdx.x, T * H / 4, nthr);
        if (threadIdx.x == 0) a.header[kHdrTicketDown] = 0u;
    }
}

// ---------------------------------------------------------------- the layer stack

constexpr int kStackMaxRows = 8;        // router rows a CTA of the stack kernel holds

// Bounded grid-wide barrier n (0, 1, ...) of a cooperative launch: thread 0 of
// every CTA adds one to *count with release semantics (publishing the CTA's
// writes), then polls it with acquire loads until all CTAs have arrived at
// barrier n.  A wait that runs out records
// MOE_ERR_TIMEOUT and raises the grid's abort word, which ends every other
// CTA's wait as well.  arrive == false is the test hook of a CTA that never
// arrives.
__device__ __forceinline__ bool grid_barrier(uint32_t *count, uint32_t *gabort, uint32_t n, bool arrive,
                                             long long limit, uint32_t *status, volatile int *abort)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        // release: the CTA's writes (ordered before this thread by the CTA barrier) before the arrival
        if (arrive) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(count) : "memory");
        const uint32_t target = (n + 1u) * gridDim.x;
        const long long t0 = clock64();
        while (true) {
            uint32_t c;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(c) : "l"(count) : "memory");
            if (c >= target) break;
            if (*reinterpret_cast<volatile uint32_t *>(gabort)) {
                *abort = 1;
                break;
            }
            if (clock64() - t0 > limit) {
                set_status(status, MOE_ERR_TIMEOUT);
                atomicExch(gabort, 1u);
                *abort = 1;
                break;
            }
        }
        __threadfence();
    }
    __syncthreads();
    return !*abort;
}

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi)
{
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}

// The input of layer l, in every CTA: x of the window as fp16 MMA fragments
// (s_xf, the layout k_dec_route writes), and the logits of this CTA's router
// rows (r0 .. r0 + nr - 1, held in shared memory at s_wr) written to the
// workspace.  From layer 1 on it first finishes layer l - 1: y = bf16 of its
// accumulator, written by this CTA for the float4 items [q0, q1).  With the
// residual stream the input is bf16(x[l - 1] + y[l - 1]) (an fp32 sum of the
// two bf16 values, rounded once), also written for [q0, q1); otherwise it is
// x[l].  Every CTA reads the accumulator whole in the residual case, so no
// barrier separates y from the next layer's logits.  x is staged in bf16 at
// s_x (the ring's head) with its loads in flight together; each router row's
// T logits are one warp's dot products over it.
__device__ __noinline__ void stack_input(const StackArgs &sa, int l, uint8_t *smem, const LayerSmem &L, const float *s_wr,
                            int r0, int nr, int q0, int q1)
{
    const DecArgs &d = sa.d;
    const int T = d.T, H = d.H, E = d.E, H4 = H / 4, n4 = T * H4, nthr = blockDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarp = nthr >> 5;
    uint2 *s_xf = reinterpret_cast<uint2 *>(smem + L.xf);
    uint2 *s_x = reinterpret_cast<uint2 *>(smem + L.ring);           // bf16 [T][H], 4 a uint2
    const size_t TH = (size_t)T * H;
    const bool res = sa.residual && l > 0;
    const float4 *yprev = reinterpret_cast<const float4 *>(sa.yacc + (size_t)((l + 1) & 1) * TH);  // layer l - 1's
    uint2 *yout = reinterpret_cast<uint2 *>(sa.y + (size_t)(l > 0 ? l - 1 : 0) * TH);
    float4 *yfout = sa.y_f32 ? reinterpret_cast<float4 *>(sa.y_f32 + (size_t)(l > 0 ? l - 1 : 0) * TH) : nullptr;
    if (!res) {
        // x[l] as it is: one cp.async group; y of layer l - 1 for this CTA's items meanwhile
        const uint16_t *xin = sa.x + (size_t)l * TH;
        const uint32_t dst = sm_addr(s_x);
        for (int i = threadIdx.x; i < n4 / 2; i += nthr) cp16(dst + 16u * i, xin + 8 * i);
        cp_commit();
        if (l > 0)
            for (int q = q0 + threadIdx.x; q < q1; q += nthr) {
                const float4 v = __ldcg(yprev + q);
                yout[q] = make_uint2(bf16x2_rn(v.x, v.y), bf16x2_rn(v.z, v.w));
                if (yfout) yfout[q] = v;
            }
        cp_wait<0>();
    } else {
        // x[l] = bf16(x[l - 1] + bf16(acc)), one item at a time (deeper batches here cost the
        // streaming loop registers)
        const uint2 *xin = reinterpret_cast<const uint2 *>(sa.x + (size_t)(l - 1) * TH);
        uint2 *xout = reinterpret_cast<uint2 *>(sa.x + (size_t)l * TH);
        constexpr int kB = 1;
        for (int i0 = threadIdx.x; i0 < n4; i0 += kB * nthr) {
            float4 yv[kB];
            uint2 xv[kB];
#pragma unroll
            for (int j = 0; j < kB; ++j)
                if (i0 + j * nthr < n4) {
                    yv[j] = __ldcg(yprev + i0 + j * nthr);
                    xv[j] = __ldcg(xin + i0 + j * nthr);
                }
#pragma unroll
            for (int j = 0; j < kB; ++j) {
                const int q = i0 + j * nthr;
                if (q < n4) {
                    const uint32_t ylo = bf16x2_rn(yv[j].x, yv[j].y), yhi = bf16x2_rn(yv[j].z, yv[j].w);
                    uint2 xb = xv[j];
                    xb.x = bf16x2_rn(__fadd_rn(bf16_bits_to_f32(xb.x & 0xffff), bf16_bits_to_f32(ylo & 0xffff)),
                                     __fadd_rn(bf16_bits_to_f32(xb.x >> 16), bf16_bits_to_f32(ylo >> 16)));
                    xb.y = bf16x2_rn(__fadd_rn(bf16_bits_to_f32(xb.y & 0xffff), bf16_bits_to_f32(yhi & 0xffff)),
                                     __fadd_rn(bf16_bits_to_f32(xb.y >> 16), bf16_bits_to_f32(yhi >> 16)));
                    s_x[q] = xb;
                    if (q >= q0 && q < q1) {
                        yout[q] = make_uint2(ylo, yhi);
                        if (yfout) yfout[q] = yv[j];
                        xout[q] = xb;
                    }
                }
            }
        }
    }
    __syncthreads();
    // fp16 MMA fragments: item q = (token g, elements e .. e + 3), e = 4 (q % H4), to slot
    // ((cb * 16 + s) * 4 + tq) * T + g with e = 256 cb + 64 tq + (s < 8 ? 4 s : 32 + 4 (s - 8))
    bool bad = false;
    for (int q = threadIdx.x; q < n4; q += nthr) {
        const int g = q / H4, e = 4 * (q - g * H4);
        const uint2 xb = s_x[q];
        const float x0 = bf16_bits_to_f32(xb.x & 0xffff), x1 = bf16_bits_to_f32(xb.x >> 16);
        const float x2 = bf16_bits_to_f32(xb.y & 0xffff), x3 = bf16_bits_to_f32(xb.y >> 16);
        const float m = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
        bad |= !(m < 65504.0f);      // beyond the fp16 range, or NaN
        const int cb = e >> 8, rem = e & 255, tq = rem >> 6, r2 = rem & 63;
        const int sx = r2 < 32 ? r2 >> 2 : 8 + ((r2 - 32) >> 2);
        s_xf[((cb * 16 + sx) * 4 + tq) * T + g] =
            make_uint2(dq_h22u(__floats2half2_rn(x0, x1)), dq_h22u(__floats2half2_rn(x2, x3)));
    }
    if (bad) set_status(d.header + kHdrStatus, MOE_ERR_DEVICE_FAULT);
    // logits: warp p takes (row r, token g) pairs, lanes along H in float4 steps
    for (int p = warp; p < nr * T; p += nwarp) {
        const int r = p / T, g = p - r * T;
        const float4 *w4 = reinterpret_cast<const float4 *>(s_wr + (size_t)r * H);
        const uint2 *x4 = s_x + (size_t)g * H4;
        float acc = 0.0f;
        for (int j = lane; j < H4; j += 32) {
            const float4 w = w4[j];
            const uint2 xb = x4[j];
            acc = fmaf(w.x, bf16_bits_to_f32(xb.x & 0xffff), acc);
            acc = fmaf(w.y, bf16_bits_to_f32(xb.x >> 16), acc);
            acc = fmaf(w.z, bf16_bits_to_f32(xb.y & 0xffff), acc);
            acc = fmaf(w.w, bf16_bits_to_f32(xb.y >> 16), acc);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) d.logits[(size_t)g * E + r0 + r] = acc;
    }
}

// A decode window through a stack of L layers in one launch: one persistent
// CTA per SM (a cooperative launch), the layers in order, each between two
// grid-wide barriers -- after its router logits (each CTA computes those of
// its share of the router rows, kept in shared memory), and after its experts
// (every contribution to its accumulator added).  The two accumulators
// alternate: layer l + 1's is zeroed while layer l streams, and layer l's is
// read whole by every CTA to build layer l + 1's input.  A CTA that has
// finished its units loads the next layer's router rows into the tail of its
// ring while it waits for the rest of the grid.
template <int S, int V>
__global__ void __maxnreg__(V == kVarHalf ? 96 : 128) k_dec_stack(const __grid_constant__ StackArgs sa)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const DecArgs &d = sa.d;
    const int T = d.T, H = d.H, E = d.E, G = gridDim.x, b = blockIdx.x, nthr = blockDim.x;
    const LayerSmem L = layer_smem(E, T, H, d.nc, d.ring_bytes);
    const uint8_t **s_tab = reinterpret_cast<const uint8_t **>(smem + L.tab);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.misc);
    float *s_lg = reinterpret_cast<float *>(smem + L.ring);
    const float *s_wr = reinterpret_cast<const float *>(smem + L.ring + L.ring_bytes - (uint32_t)sa.rows * H * 4);
    uint32_t *status = d.header + kHdrStatus;
    uint32_t *gbar = d.header + kHdrGridBar, *gabort = d.header + kHdrGridAbort;
    const int r0 = (int)((int64_t)E * b / G), nr = (int)((int64_t)E * (b + 1) / G) - r0;
    const int n4 = T * H / 4;
    const int q0 = (int)((int64_t)n4 * b / G), q1 = (int)((int64_t)n4 * (b + 1) / G);
    const size_t TH = (size_t)T * H;

    if (threadIdx.x == 0) *abort_flag = 0;
    // one cp.async group: this CTA's router rows of layer l -> the ring's tail, and the
    // layer's expert table -> s_tab (both free once the previous layer's units are done)
    auto load_rows = [&](int l) {
        const float *wr = sa.wr[l] + (size_t)r0 * H;
        const uint32_t dst = sm_addr(s_wr);
        for (int i = threadIdx.x; i < nr * H / 4; i += nthr) cp16(dst + 16u * i, wr + 4 * i);
        const uint8_t *const *blobs = sa.blobs + (size_t)l * E;
        for (int e = threadIdx.x; e < E; e += nthr) cp8(sm_addr(s_tab + e), blobs + e);
        cp_commit();
    };
    load_rows(0);
    for (int i = q0 + threadIdx.x; i < q1; i += nthr) reinterpret_cast<float4 *>(sa.yacc)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    uint32_t nbar = 0;
    bool ok = true;
    for (int l = 0; l < sa.L && ok; ++l) {
        cp_wait<0>();
        __syncthreads();
        stack_input(sa, l, smem, L, s_wr, r0, nr, q0, q1);
        // ---- every CTA's logits of layer l are in place
        ok = grid_barrier(gbar, gabort, nbar++, !(l == 0 && b == d.skip_cta), d.wait_cycles, status, abort_flag);
        if (!ok) break;
        for (int i = threadIdx.x; i < T * E; i += nthr) s_lg[i] = __ldcg(d.logits + i);
        // nobody reads the other accumulator past that barrier: this CTA's share of it, zeroed for layer l + 1
        if (l + 1 < sa.L) {
            float4 *nxt = reinterpret_cast<float4 *>(sa.yacc + (size_t)((l + 1) & 1) * TH);
            for (int i = q0 + threadIdx.x; i < q1; i += nthr) nxt[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        __syncthreads();
        dec_window<S, V>(d, smem, sa.bias ? sa.bias[l] : nullptr, sa.shared ? sa.shared[l] : nullptr,
                         sa.yacc + (size_t)(l & 1) * TH, l == sa.L - 1);
        // ---- the ring is free: the next layer's router rows
        __syncthreads();
        if (l + 1 < sa.L) load_rows(l + 1);
        ok = grid_barrier(gbar, gabort, nbar++, true, d.wait_cycles, status, abort_flag);
    }
    // y of the last layer (the earlier layers' were written while building the next input)
    if (ok) {
        const size_t lo = (size_t)(sa.L - 1) * TH;
        const float4 *acc = reinterpret_cast<const float4 *>(sa.yacc + (size_t)((sa.L - 1) & 1) * TH);
        uint2 *yo = reinterpret_cast<uint2 *>(sa.y + lo);
        float4 *yf = sa.y_f32 ? reinterpret_cast<float4 *>(sa.y_f32 + lo) : nullptr;
        for (int q = q0 + threadIdx.x; q < q1; q += nthr) {
            const float4 v = __ldcg(acc + q);
            yo[q] = make_uint2(bf16x2_rn(v.x, v.y), bf16x2_rn(v.z, v.w));
            if (yf) yf[q] = v;
        }
    }
    cp_wait<0>();           // no copy outlives the CTA (an aborted stack may leave the next rows in flight)
}

// ---------------------------------------------------------------- launch

static int dec_sms()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    return n;
}

int dec_route_parts(int H)
{
    for (int P = 1; P <= 8; P *= 2)
        if (H % (128 * P) == 0 && H / (128 * P) <= kRouteMaxVec) return P;
    return 0;   // unsupported
}

// Half-block warps (128 columns each) for Q4_K layers without a shared expert
// whose 128-column blocks fit kMaxConsHalf warps; 256-column warps otherwise.
bool dec_half(const moe_config &c)
{
    return c.codec == MOE_CODEC_Q4K && c.shared_ff == 0 && c.hidden / 128 <= kMaxConsHalf;
}

static uint32_t dec_slot(const moe_config &c)
{
    return dec_half(c) ? kSlotHalf : c.codec == MOE_CODEC_Q5K ? kSlotQ5K : kSlotBytes;
}

int dec_consumers(const moe_config &c) { return dec_half(c) ? c.hidden / 128 : c.hidden / 256; }

// The staging rings take all the shared memory the rest of the kernel leaves.
static int64_t dec_base_ring(const moe_config &c, int32_t T)
{
    const LayerSmem base = layer_smem(c.n_experts, T, c.hidden, dec_consumers(c), 0);
    return ((int64_t)kDecSmemBudget - (int64_t)base.total) & ~(int64_t)127;
}

uint32_t dec_ring_bytes(const moe_config &c, int32_t T) { return (uint32_t)dec_base_ring(c, T); }

// Stages of each consumer warp's ring: the largest of the compiled counts that
// fits (0: none does, or the routing scratch does not fit the ring).
static const int kStageCounts[] = {16, 14, 12, 10, 8, 7, 6};

using LayerFn = void (*)(DecArgs);
using StackFn = void (*)(StackArgs);

template <int V>
static LayerFn layer_fn(int S)
{
    switch (S) {
    case 16: return k_dec_layer<16, V>;
    case 14: return k_dec_layer<14, V>;
    case 12: return k_dec_layer<12, V>;
    case 10: return k_dec_layer<10, V>;
    case 8: return k_dec_layer<8, V>;
    case 7: return k_dec_layer<7, V>;
    case 6: return k_dec_layer<6, V>;
    }
    return nullptr;
}

template <int V>
static StackFn stack_fn(int S)
{
    switch (S) {
    case 16: return k_dec_stack<16, V>;
    case 14: return k_dec_stack<14, V>;
    case 12: return k_dec_stack<12, V>;
    case 10: return k_dec_stack<10, V>;
    case 8: return k_dec_stack<8, V>;
    case 7: return k_dec_stack<7, V>;
    case 6: return k_dec_stack<6, V>;
    }
    return nullptr;
}

int dec_stages(const moe_config &c, int32_t T)
{
    const int64_t ring = dec_base_ring(c, T);
    const int nc = dec_consumers(c);
    if (nc <= 0 || ring < (int64_t)T * c.n_experts * 12 + 16) return 0;
    const int64_t per = ring / ((int64_t)nc * dec_slot(c));
    for (int s : kStageCounts)
        if (per >= s) return s;
    return 0;
}

bool dec_supported(const moe_config &c, int32_t T)
{
    return T >= 0 && T <= kDecTok && dec_route_parts(c.hidden) != 0 && (dec_half(c) || c.hidden / 256 <= kMaxCons) &&
           c.ff % kUnitRows == 0 && c.shared_ff % kSharedRows == 0 && dec_stages(c, T) > 0;
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

// Function attributes (dynamic shared-memory limits) are per device: set once
// for each device this process launches on.
static cudaError_t dec_set_attributes()
{
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(k_dec_route, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kDecTok * 8192 * (int)sizeof(uint16_t));
    for (int S : kStageCounts)
        for (LayerFn f : {layer_fn<kVarQ4K>(S), layer_fn<kVarHalf>(S), layer_fn<kVarQ5K>(S)})
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmemBudget);
    for (int S : kStageCounts)
        for (StackFn f : {stack_fn<kVarQ4K>(S), stack_fn<kVarHalf>(S), stack_fn<kVarQ5K>(S)})
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmemBudget);
    if (e == cudaSuccess) done[dev] = true;
    return e;
}

cudaError_t launch_decode(const DecArgs &a0, cudaStream_t s)
{
    DecArgs a = a0;
    if (a.T <= 0) return cudaSuccess;
    cudaError_t e = dec_set_attributes();
    if (e != cudaSuccess) return e;
    const int rpc = 8 / a.route_parts;
    prof_begin(kPhDecRoute, s);
    e = launch_pdl(k_dec_route, dim3((a.E + rpc - 1) / rpc), dim3(kRouteThreads), (size_t)a.T * a.H * 2, s,
                   a.overlap_prev != 0, a);
    prof_end(kPhDecRoute, s);
    if (e != cudaSuccess) return e;
    const LayerSmem L = layer_smem(a.E, a.T, a.H, a.nc, a.ring_bytes);
    const dim3 grid(dec_sms()), block(32 * std::max(a.nc, kDecTok));   // at least one warp per token
    prof_begin(kPhDecLayer, s);
    const LayerFn fn = a.half ? layer_fn<kVarHalf>(a.stages)
                       : a.codec == MOE_CODEC_Q5K ? layer_fn<kVarQ5K>(a.stages) : layer_fn<kVarQ4K>(a.stages);
    e = fn ? launch_pdl(fn, grid, block, L.total, s, true, a) : cudaErrorInvalidValue;
    prof_end(kPhDecLayer, s);
    return e;
}

// The stack kernel needs the decode path's layer kernel configuration, and
// room in the ring for a CTA's router rows (tail) beside the staged x (head);
// both are live only between a layer's experts.
int stack_grid() { return dec_sms(); }

bool stack_supported(const moe_config &c, int32_t T)
{
    if (T < 1 || !dec_supported(c, T)) return false;
    const int G = dec_sms();
    const int rows = (c.n_experts + G - 1) / G;
    if (rows > kStackMaxRows) return false;
    // x staged in bf16 at the ring's head, the router rows at its tail
    return 2ll * T * c.hidden + (int64_t)rows * c.hidden * 4 <= (int64_t)dec_ring_bytes(c, T);
}

cudaError_t launch_stack(const StackArgs &a, cudaStream_t s)
{
    if (a.d.T <= 0 || a.L <= 0) return cudaSuccess;
    cudaError_t e = dec_set_attributes();
    if (e != cudaSuccess) return e;
    // the grid barriers count from zero in every launch
    e = cudaMemsetAsync(a.d.header + kHdrGridBar, 0, 2 * sizeof(uint32_t), s);
    if (e != cudaSuccess) return e;
    const LayerSmem L = layer_smem(a.d.E, a.d.T, a.d.H, a.d.nc, a.d.ring_bytes);
    const StackFn fn = a.d.half ? stack_fn<kVarHalf>(a.d.stages)
                       : a.d.codec == MOE_CODEC_Q5K ? stack_fn<kVarQ5K>(a.d.stages) : stack_fn<kVarQ4K>(a.d.stages);
    if (!fn) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(dec_sms());
    cfg.blockDim = dim3(32 * std::max(a.d.nc, kDecTok));
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;     // every CTA resident at once: the grid barriers need it
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    prof_begin(kPhDecStack, s);
    e = cudaLaunchKernelEx(&cfg, fn, a);
    prof_end(kPhDecStack, s);
    return e;
}

}  // namespace moe
