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
//              interleaved (row 2i = gate f0+i, row 2i+1 = up f0+i), K = H,
//              dequantised by the dequantisation warps straight into tensor
//              memory (thread = tensor-memory lane = weight row) and read from
//              there by the MMA;
//            B = the tile's rows of xg (x in fp16, permuted into bucket order,
//              so a tile's token rows are consecutive);
//            epilogue: lanes 2i / 2i+1 hold g / u of one ff index ->
//              a = SiLU(g) * u, stored fp16 at the assignment's bucket position.
//   down     A = Wd^T tile (128 hidden rows, K = FF), written MN-major into
//              shared memory (Wd is stored [FF][H]: eight consecutive weights
//              of a row are eight consecutive M indices), B = the tile's rows of a;
//            epilogue: * routing weight, atomically added into y (fp32), or
//              stored to the assignment's slot when the call is deterministic.
//
// Warp roles (16 warps): 0-3 epilogue (tensor-memory lane quarters 0-3; down
// projections short along K add warps 12-15), 4 MMA issue + tensor-memory
// allocation, 5 raw weight bytes (2-D tensor copies of 144-byte x 64-row boxes
// of the expert blob, through a per-CTA tensor map rewritten for each expert),
// 6-7 B rows (2-D tensor copies, one per 64-wide K sub-tile), 8-15 (or 8-11)
// dequantisation.  All hand-offs are mbarriers: per pipeline stage one "full"
// (dequantised A and B rows in place) and one "empty" (the stage's MMAs done);
// every wait is bounded and sets MOE_ERR_TIMEOUT instead of hanging.
//
// Operand precision: fp16 A and B (sub-block scale and min rounded to fp16,
// one fused multiply-add per weight), fp32 accumulation.
#include <atomic>
#include <mutex>
#include <algorithm>
#include <cmath>

#include <cuda.h>

#include "moe_internal.cuh"
#include "debug_hooks.cuh"
#include "tc_ptx.cuh"
#include "dequant_f16.cuh"

namespace moe {

using namespace ptx;

enum GemmOp { kOpGateUp = 0, kOpDown = 1 };
enum WFmt { kWQ4K = 0, kWQ80 = 1 };

constexpr int kGemmThreads = 512;
// Warp roles: the epilogue runs on warps 0-3, the dequantisation on warps
// 8-15, unless EW = 8 (down projections whose tiles are short along K, where
// the epilogue's additions into y outweigh the dequantisation): then warps
// 12-15 join the epilogue (two groups taking alternate 16-column chunks) and
// warps 8-11 dequantise.
template <int EW>
__host__ __device__ constexpr int deq_threads()
{
    return EW == 8 ? 128 : 256;
}

constexpr int kABytes = 128 * 128;          // 128 rows x 64 fp16
constexpr long long kWaitCycles = 1ll << 32; // ~2 s at 2 GHz

struct GemmArgs {
    int H, FF, SFF, k, T, det, splits;
    const uint8_t *const *blobs;
    const uint8_t *shared_blob;
    const int32_t *offsets, *assign;
    const float *w;
    const __half *xg;        // [T*k][H] x rows in bucket order (routed gate/up operand)
    const __half *x16;       // [T][H] (shared expert's gate/up operand; null without one)
    __half *act16;           // [T*k][FF] by bucket position
    __half *sh_act16;        // [T][SFF]
    float *yacc;             // [T][H]
    float *slots, *sh_out;   // deterministic combine
    const int4 *tiles;       // {expert (-1 shared), m tile | k split << 16 | no blob << 30, first row, n}
    const uint32_t *n_tiles; // device count
    float *gu;               // split-K gate/up partial sums [rows][2 FF] (splits > 1)
    uint32_t *split_cnt;     // split-K arrival counters, one per (expert, m, n) group
    uint32_t *status;
    CUtensorMap *tmaps;      // [grid][2] per-CTA tensor maps of the current expert's blob
    long long wait_cycles;   // limit of the bounded waits
    int skip_cta;            // test hook: this CTA never issues its first token-row copy (-1: none)
};

// A work tile.  The record holds everything the roles need but the blob's
// address (read by the raw-weight copier alone): row0 is the first row of the
// tile's tokens in the operand (the expert's bucket offset + the tile's
// position in it, or the token index for the shared expert), live is false
// when the expert's blob pointer is null.
struct TileInfo {
    int e, m, ks, row0, n, nmma, ksteps, k0;   // k0: first K-step of this split
    bool live;
};

constexpr int kTileNoBlob = 1 << 30;         // record flag: the expert's blob pointer is null

template <int OP, int FMT>
__device__ __forceinline__ TileInfo tile_decode(const GemmArgs &g, int4 t)
{
    TileInfo ti;
    ti.e = t.x;
    ti.m = t.y & 0xffff;
    ti.ks = (t.y >> 16) & 0x3fff;
    ti.live = !(t.y & kTileNoBlob);
    ti.row0 = t.z;
    ti.n = t.w;
    ti.nmma = (t.w + 15) & ~15;
    ti.ksteps = (OP == kOpGateUp ? g.H : (FMT == kWQ4K ? g.FF : g.SFF)) / 64 / g.splits;
    ti.k0 = ti.ks * ti.ksteps;
    return ti;
}

// Record of tile idx (zeros past the list): each role reads the next tile's
// record one tile ahead, so the load is in flight while the current tile runs.
__device__ __forceinline__ int4 tile_fetch(const GemmArgs &g, int idx, int n_tiles)
{
    return idx < n_tiles ? __ldg(g.tiles + idx) : make_int4(0, 0, 0, 0);
}

// a = SiLU(g) * u as the fp16 operand of the down projection.  A value
// beyond the fp16 range (it would become +-inf, or NaN) is a device fault:
// the call reports MOE_ERR_DEVICE_FAULT rather than a silently infinite y.
__device__ __forceinline__ __half act_to_f16(float a, uint32_t *status)
{
    if (!(fabsf(a) <= 65504.0f)) set_status(status, MOE_ERR_DEVICE_FAULT);
    return __float2half_rn(a);
}

// Bounded wait on an mbarrier phase; false on abort (another role gave up) or
// on timeout (this call records MOE_ERR_TIMEOUT and raises the abort flag).
// Waiting warps sleep in the try_wait (hardware suspend, up to ~20 us per
// try) rather than spin, so they do not take issue slots from the working
// warps.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort, uint32_t *status,
                                         long long limit)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (*abort) return false;
        if (clock64() - t0 > limit) {
            *abort = 1;
            set_status(status, MOE_ERR_TIMEOUT);
            return false;
        }
    }
}

// ---------------------------------------------------------------- dequant
// (the fp16 operand recipe lives in dequant_f16.cuh, shared with the decode
// kernel and the test hooks)

// gate/up, Q4_K, one 128-wide K stage: thread (row, half h) turns group g of
// the row's super-block (32 quant bytes at q: 32 weights of sub-block 2g in
// the low nibbles, 32 of sub-block 2g + 1 in the high ones) into 64 fp16 A
// values, written to tensor-memory columns `taddr` + 0..31 of its lane (K
// order: low nibbles, then high nibbles).  hdr: the block's 16-byte header.
__device__ __forceinline__ void dequant_gu_q4k_tmem(const uint8_t *hdr_p, const uint8_t *q, int g, uint32_t taddr)
{
    const uint4 hdr = *reinterpret_cast<const uint4 *>(hdr_p);
    const uint4 qa = *reinterpret_cast<const uint4 *>(q);
    const uint4 qb = *reinterpret_cast<const uint4 *>(q + 16);
    __half2 S, NZ;
    q4k_pair_scales_h(hdr, g, S, NZ);
    const __half2 S_lo = __low2half2(S), S_hi = __high2half2(S);
    const __half2 NZ_lo = __low2half2(NZ), NZ_hi = __high2half2(NZ);
    const uint32_t words[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
    uint32_t lo[16], hi[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t o[4];
        q4k_word_f16(words[i], S_lo, NZ_lo, S_hi, NZ_hi, o);
        lo[2 * i] = o[0];
        lo[2 * i + 1] = o[1];
        hi[2 * i] = o[2];
        hi[2 * i + 1] = o[3];
    }
    tmem_st16(taddr, lo);
    tmem_st16(taddr + 16, hi);
}

// gate/up, Q8_0, one 128-wide K stage: thread (row, half h) turns blocks 2h and
// 2h + 1 of the stage's four into 64 fp16 A values (tensor-memory columns
// `taddr` + 0..31).  rr: the row's 144-byte window holding the stage's 136
// bytes at offset o (0 or 8).
__device__ __forceinline__ void dequant_gu_q80_tmem(const uint8_t *rr, int o, int h, uint32_t taddr)
{
    const uint16_t *r16 = reinterpret_cast<const uint16_t *>(rr + o);
#pragma unroll
    for (int bi = 0; bi < 2; ++bi) {
        const int b = 2 * h + bi;
        const __half2 D = __half2half2(__ushort_as_half(r16[17 * b]));
        uint32_t v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = q80_pair_f16(r16[17 * b + 1 + i], D);
        tmem_st16(taddr + 16 * bi, v);
    }
}

// Byte offset of element (m, k) in an MN-major 128-byte-swizzled tile of 128
// M x 64 K fp16: atoms of 64 M x 8 K, 1024 bytes apart along M and 2048 along K.
__device__ __forceinline__ uint32_t mn_off(uint32_t m, uint32_t k)
{
    return ((k >> 3) << 11) + ((m >> 6) << 10) + ((k & 7) << 7) + ((((m & 63) >> 3) ^ (k & 7)) << 4) + ((m & 7) << 1);
}

// down, Q4_K: A[h][f] = Wd[f][h0 + h] for the tile's 128 hidden columns and
// the stage's 64 ff rows, stored MN-major (h contiguous), so eight consecutive
// weights of a raw row land in one 16-byte chunk.  Raw row i (f = 64 s + i)
// is the 144-byte block holding the tile's columns; `half` selects its 64
// quant bytes: group c (32 bytes) holds 32 low-nibble weights at h = 64 c + l
// and 32 high-nibble ones at h = 64 c + 32 + l.  Thread (row, c, part) takes
// 32 / P bytes of group c (P = NT / 128 parts), so one scale decode serves all
// its weights; lanes take consecutive rows (conflict-free stores).
template <int NT>
__device__ __forceinline__ void dequant_dn_q4k(const uint8_t *raw, uint32_t a_tile, int dt, int half)
{
    constexpr int P = NT / 128, NB = 32 / P;            // parts per group, bytes per thread
    const int row = dt & 63, c = (dt >> 6) / P, part = (dt >> 6) % P;
    const uint8_t *rr = raw + row * 144;
    __half2 S, NZ;
    q4k_pair_scales_h(*reinterpret_cast<const uint4 *>(rr), 2 * half + c, S, NZ);
    const __half2 S_lo = __low2half2(S), S_hi = __high2half2(S);
    const __half2 NZ_lo = __low2half2(NZ), NZ_hi = __high2half2(NZ);
    const uint8_t *q = rr + 16 + 64 * half + 32 * c + NB * part;
#pragma unroll
    for (int u = 0; u < NB / 16; ++u) {
        const uint4 w = *reinterpret_cast<const uint4 *>(q + 16 * u);
        const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int p = 0; p < 2; ++p) {                   // 8 bytes: 8 low and 8 high weights
            uint32_t a[4], b[4];
            q4k_word_f16(words[2 * p], S_lo, NZ_lo, S_hi, NZ_hi, a);
            q4k_word_f16(words[2 * p + 1], S_lo, NZ_lo, S_hi, NZ_hi, b);
            const int h_lo = 64 * c + NB * part + 16 * u + 8 * p;
            st_shared_v4(a_tile + mn_off(h_lo, row), a[0], a[1], b[0], b[1]);
            st_shared_v4(a_tile + mn_off(h_lo + 32, row), a[2], a[3], b[2], b[3]);
        }
    }
}

// down, Q8_0: raw row i (f = 64 s + i) is a 144-byte window holding the 4
// blocks of this tile's 128 hidden columns at offset o8 (0 or 8); item
// (row, group g of 8 hidden columns) -> one 16-byte chunk of the MN-major tile.
template <int NT>
__device__ __forceinline__ void dequant_dn_q80(const uint8_t *raw, uint32_t a_tile, int dt, int o8)
{
#pragma unroll
    for (int it8 = 0; it8 < 1024 / NT; ++it8) {
        const int it = dt + NT * it8;
        const int row = it & 63, g = it >> 6;            // g 0..15: 8 columns each
        const int b = g >> 2, hh0 = 8 * (g & 3);
        const uint16_t *blk = reinterpret_cast<const uint16_t *>(raw + row * 144 + o8 + 34 * b);
        const __half2 D = __half2half2(__ushort_as_half(blk[0]));
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = q80_pair_f16(blk[1 + hh0 / 2 + i], D);
        st_shared_v4(a_tile + mn_off(32 * b + hh0, row), o[0], o[1], o[2], o[3]);
    }
}

// ---------------------------------------------------------------- the kernel

// K-steps (64 wide) per pipeline stage: gate/up stages are 128 wide (8 MMAs
// per hand-off), down stages 64 (its K, FF, is short).
template <int OP>
__host__ __device__ constexpr int kstep_per_stage()
{
    return OP == kOpGateUp ? 2 : 1;
}

// Raw bytes of one raw-ring slot, filled by 2-D tensor copies of 144-byte x
// 64-row boxes of the expert blob: gate/up 64 gate rows then the 64 up rows
// (Q4_K: a whole block column, the raw of two stages; Q8_0: a 16-byte aligned
// window over one stage's 136 bytes); down 64 ff rows (Q4_K: the block
// holding the tile's 128 hidden columns; Q8_0: a window over its 4 blocks).
template <int OP, int FMT>
__host__ __device__ constexpr int raw_stage_bytes()
{
    return OP == kOpGateUp ? 128 * 144 : 64 * 144;
}

// pipeline stages served by one raw slot
template <int OP, int FMT>
__host__ __device__ constexpr int stages_per_raw()
{
    return (OP == kOpGateUp && FMT == kWQ4K) ? 2 : 1;
}

template <int OP, int FMT, int NMAX, int S, int RAW>
struct GemmCfg {
    static constexpr int KS = kstep_per_stage<OP>();
    static constexpr int kRawStage = raw_stage_bytes<OP, FMT>();
    static constexpr int RS = RAW / kRawStage;           // raw ring depth
    static constexpr int SPR = stages_per_raw<OP, FMT>();
    static constexpr int kBSub = NMAX * 128;             // one 64-wide K sub-tile of token rows
    static constexpr int kBStage = KS * kBSub;
    static constexpr int kAStage = OP == kOpGateUp ? 0 : kABytes;   // down: A in shared memory
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + S * kAStage;
    static constexpr int kOffRaw = kOffB + S * kBStage;
    static constexpr int kOffBar = kOffRaw + ((RS * kRawStage + 1023) & ~1023);
    static constexpr int kNumBars = 2 * S + 2 * RS + 6;
    static constexpr int kOffTmap = (kOffBar + 8 * kNumBars + 127) & ~127;   // 128-byte tensor map
    static constexpr int kOffMisc = kOffTmap + 128;
    static constexpr int kOffMeta = kOffMisc + 16;              // [2][NMAX] token, weight, slot
    static constexpr int kBytes = kOffMeta + 2 * NMAX * 12 + 1024;
    // tensor memory: two accumulators of NMAX columns; gate/up adds S A stages
    // of 64 columns (128 rows x 128 K fp16)
    static constexpr int kColA = 2 * NMAX;
    static constexpr int kCols = OP == kOpGateUp ? 512 : (2 * NMAX < 32 ? 32 : 2 * NMAX);
    static_assert(RS >= 2, "raw ring too shallow");
    static_assert(kBytes <= 227 * 1024, "shared memory budget");
    static_assert(OP != kOpGateUp || kColA + 64 * S <= 512, "tensor memory budget");
    static_assert((kCols & (kCols - 1)) == 0, "tensor-memory allocations are powers of two");
};

// Bounded wait of a whole warp: every lane polls, and the lanes agree on the
// outcome (false if any lane saw an abort or a timeout).
__device__ __forceinline__ bool warp_wait_bar(uint32_t bar, uint32_t parity, volatile int *abort, uint32_t *status,
                                              long long limit)
{
    const bool ok = wait_bar(bar, parity, abort, status, limit);
    return __all_sync(0xffffffffu, ok);
}

template <int OP, int FMT, int NMAX, int S, int RAW, int EW>
__global__ void __launch_bounds__(kGemmThreads, 1) k_moe_gemm(GemmArgs g, const __grid_constant__ CUtensorMap tmap_b,
                                                          const __grid_constant__ CUtensorMap tmap_w)
{
    using C = GemmCfg<OP, FMT, NMAX, S, RAW>;
    constexpr int RS = C::RS;
    constexpr int KS = C::KS;
    constexpr int SPR = C::SPR;
    static_assert(EW == 4 || (EW == 8 && OP == kOpDown), "8 epilogue warps: down only");
    constexpr int kDeq = deq_threads<EW>(), kEpi = 32 * EW;
    constexpr int kEG = kEpi / 128;          // epilogue groups (alternate 16-column chunks)
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_dyn + 1023) & ~(uintptr_t)1023);
    const uint32_t sA = smem_addr(smem + C::kOffA), sB = smem_addr(smem + C::kOffB);
    uint8_t *raw_base = smem + C::kOffRaw;
    const uint32_t bar0 = smem_addr(smem + C::kOffBar);
    // stage ring: `full` completes when the stage's A (dequantised weights) and
    // B (token rows) are in place, `empty` when its MMAs have read them
    auto full = [&](int i) { return bar0 + 8 * i; };
    auto empty = [&](int i) { return bar0 + 8 * (S + i); };
    auto full_raw = [&](int i) { return bar0 + 8 * (2 * S + i); };
    auto empty_raw = [&](int i) { return bar0 + 8 * (2 * S + RS + i); };
    const uint32_t bx = bar0 + 8 * (2 * S + 2 * RS);
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
        for (int i = 0; i < S; ++i) {
            mbar_init(full(i), kDeq + KS);          // dequantisers + one expect_tx per B sub-tile
            mbar_init(empty(i), 1);
        }
        for (int i = 0; i < RS; ++i) {
            mbar_init(full_raw(i), 1);              // the raw copies' expect_tx
            mbar_init(empty_raw(i), kDeq);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(acc_full(i), 1);
            mbar_init(acc_empty(i), kEpi);
        }
        mbar_init(final_bar, 1);
        mbar_init(epi_bar, kEpi);
        *abort_flag = 0;
        *last_flag = 0;
        fence_mbar_init();
    }
    if (warp == 4) {
        tmem_alloc(smem_addr(tmem_slot), C::kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int n_tiles = (int)*g.n_tiles;

    if (warp < 4 || (kEG == 2 && warp >= 12)) {
        // ------------------------------------------------------------ epilogue
        uint32_t t_it = 0, epi_it = 0;
        const int wq = warp & 3;             // tensor-memory lane quarter of this warp
        const int et = 32 * wq + lane;       // 0..127 = tensor-memory lane (row of the tile)
        const int eg = warp < 4 ? 0 : 1;     // epilogue group
        const int ei = eg * 128 + et;        // 0 .. kEpi-1
        auto epi_sync = [&]() -> bool {      // the epilogue warps only, bounded
            mbar_arrive(epi_bar);
            return wait_bar(epi_bar, (epi_it++) & 1, abort_flag, g.status, g.wait_cycles);
        };
        bool ok = true;
        // routed down: each thread owns column ei of every tile (kEpi >= NMAX); its
        // slot and routing weight are loaded a tile ahead (the slot once the next
        // tile's record is in, the weight after this tile's sums)
        static_assert(kEpi >= NMAX, "one column of metadata per epilogue thread");
        constexpr bool kMeta = OP == kOpDown && FMT == kWQ4K;
        int4 tnext = tile_fetch(g, blockIdx.x, n_tiles);
        int pslot = 0;
        float pw = 0.0f;
        if (kMeta && (int)blockIdx.x < n_tiles && ei < tnext.w && !(tnext.y & kTileNoBlob)) {
            pslot = __ldg(g.assign + tnext.z + ei);
            pw = __ldg(g.w + pslot);
        }
        for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
            const TileInfo ti = tile_decode<OP, FMT>(g, tnext);
            tnext = tile_fetch(g, tile + (int)gridDim.x, n_tiles);
            const int cslot = pslot;
            const float cw = pw;
            const bool nmeta = kMeta && tile + (int)gridDim.x < n_tiles;   // the next tile's column, if any
            if (!ti.live) {
                if (ei == 0) set_status(g.status, MOE_ERR_DEVICE_FAULT);
                if (nmeta && ei < tnext.w && !(tnext.y & kTileNoBlob)) {
                    pslot = __ldg(g.assign + tnext.z + ei);
                    pw = __ldg(g.w + pslot);
                }
                continue;
            }
            const int acc = t_it & 1;
            if (OP == kOpDown) {
                // column metadata: token, routing weight and slot of each column
                if (ei < ti.n) {
                    int tok, slot;
                    float wt;
                    if (FMT == kWQ4K) {
                        slot = cslot;
                        tok = slot / g.k;
                        wt = cw;
                    } else {
                        tok = slot = ti.row0 + ei;
                        wt = 1.0f;
                    }
                    meta_tok[acc * NMAX + ei] = tok;
                    meta_w[acc * NMAX + ei] = wt;
                    meta_slot[acc * NMAX + ei] = slot;
                }
                if (!(ok = epi_sync())) break;
            }
            if (!(ok = wait_bar(acc_full(acc), (t_it >> 1) & 1, abort_flag, g.status, g.wait_cycles))) break;
            tc_fence_after();
            int nslot = 0;
            const bool nload = nmeta && ei < tnext.w && !(tnext.y & kTileNoBlob);
            if (nload) nslot = __ldg(g.assign + tnext.z + ei);
            const int ffop = FMT == kWQ4K ? g.FF : g.SFF;
            for (int cc = eg; cc < ti.nmma / 16; cc += kEG) {
                uint32_t v[16];
                tmem_ld16(tmem_base + ((uint32_t)(32 * wq) << 16) + acc * NMAX + cc * 16, v);
                tmem_wait_ld();
                if (OP == kOpGateUp) {
                    const int f = ti.m * 64 + (et >> 1);
                    if (g.splits == 1) {
                        // lanes 2i (gate row) and 2i+1 (up row) of ff index f split the
                        // columns: the even lane takes the even ones, the odd lane the odd
                        // ones, after one exchange per column pair
                        const int par = lane & 1;
#pragma unroll
                        for (int pp = 0; pp < 8; ++pp) {
                            const float own = __uint_as_float(v[2 * pp + par]);
                            const float recv = __shfl_xor_sync(0xffffffffu, __uint_as_float(v[2 * pp + 1 - par]), 1);
                            const float gg = par ? recv : own, uu = par ? own : recv;
                            const int j = cc * 16 + 2 * pp + par;
                            if (j < ti.n) {
                                const float a = __fdividef(gg, 1.0f + __expf(-gg)) * uu;
                                __half *dst = FMT == kWQ4K ? g.act16 + (int64_t)(ti.row0 + j) * ffop + f
                                                           : g.sh_act16 + (int64_t)(ti.row0 + j) * ffop + f;
                                *dst = act_to_f16(a, g.status);
                            }
                        }
                    } else {
                        // partial sums of this K split: g into [row][f], u into [row][FF + f]
                        const int col = (et & 1) ? ffop + f : f;
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int j = cc * 16 + i;
                            const int rowi = ti.row0 + j;
                            if (j < ti.n) red_add_f32(g.gu + (int64_t)rowi * 2 * ffop + col, __uint_as_float(v[i]));
                        }
                    }
                } else {
                    // 4x4 transposes within lane quads: lane (q, r) ends with the
                    // values of hidden rows 4q..4q+3 for column 4b + r, added as one
                    // 16-byte vector
                    const int hq = ti.m * 128 + 32 * wq + (lane & ~3);
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
            if (nload) {
                pslot = nslot;
                pw = __ldg(g.w + nslot);
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
                            const int rowi = ti.row0 + j;
                            const float gg = ld_cg_f32(g.gu + (int64_t)rowi * 2 * ffop + f);
                            const float uu = ld_cg_f32(g.gu + (int64_t)rowi * 2 * ffop + ffop + f);
                            __half *dst = FMT == kWQ4K ? g.act16 + (int64_t)rowi * ffop + f
                                                       : g.sh_act16 + (int64_t)rowi * ffop + f;
                            *dst = act_to_f16(__fdividef(gg, 1.0f + __expf(-gg)) * uu, g.status);
                        }
                    }
                    if (et == 0) g.split_cnt[tile / g.splits] = 0;
                }
                if (!(ok = epi_sync())) break;     // last_flag is rewritten by the next group
            }
        }
    } else if (warp == 4) {
        // ------------------------------------------------------------ MMA issue
        // the whole warp walks the stages (waits are warp-wide); lane 0 issues
        // every MMA and every commit (a commit tracks the issuing thread's MMAs)
        uint32_t st_it = 0, t_it = 0;
        bool ok = true;
        int4 tnext = tile_fetch(g, blockIdx.x, n_tiles);
        for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
            const TileInfo ti = tile_decode<OP, FMT>(g, tnext);
            tnext = tile_fetch(g, tile + (int)gridDim.x, n_tiles);
            if (!ti.live) continue;
            const int acc = t_it & 1;
            if (!(ok = warp_wait_bar(acc_empty(acc), ((t_it >> 1) & 1) ^ 1, abort_flag, g.status, g.wait_cycles))) break;
            tc_fence_after();
            const uint32_t idesc = idesc_f16_f32(128, ti.nmma) | (OP == kOpDown ? kIdescAMnMajor : 0u);
            const uint32_t d_tmem = tmem_base + acc * NMAX;
            const int nst = (ti.ksteps + KS - 1) / KS;
            for (int st = 0; st < nst; ++st, ++st_it) {
                const int slot = st_it % S;
                if (!(ok = warp_wait_bar(full(slot), (st_it / S) & 1, abort_flag, g.status, g.wait_cycles))) break;
                tc_fence_after();
                // straight-line issue: no branch between the MMAs of a stage (the
                // issue rate halves otherwise); gate/up stages always hold 8 K16 steps
                // (tiles cover whole Q4_K block columns), down stages 4
                if (lane == 0) {
                    const uint64_t bdesc0 = sdesc_kmajor_sw128(sB + slot * C::kBStage);
                    const uint32_t acc0 = st != 0;
                    if (OP == kOpGateUp) {
                        const uint32_t a0 = tmem_base + C::kColA + 64 * slot;
#pragma unroll
                        for (int kk = 0; kk < 4 * KS; ++kk)
                            mma_f16_ta(d_tmem, a0 + 8 * kk,
                                       bdesc0 + (uint64_t)(((kk >> 2) * C::kBSub + 32 * (kk & 3)) >> 4), idesc,
                                       kk == 0 ? acc0 : 1u);
                    } else {
                        const uint64_t adesc0 = sdesc_mnmajor_sw128(sA + slot * C::kAStage, 1024, 2048);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_f16(d_tmem, adesc0 + (uint64_t)((4096 * kk) >> 4),
                                    bdesc0 + (uint64_t)((32 * kk) >> 4), idesc, kk == 0 ? acc0 : 1u);
                    }
                    mma_commit(empty(slot));
                }
                __syncwarp();
            }
            if (!ok) break;
            if (lane == 0) mma_commit(acc_full(acc));
            __syncwarp();
            ++t_it;
        }
        // every issued MMA must be complete before the tensor memory is freed
        if (lane == 0) {
            mma_commit(final_bar);
            const long long t0 = clock64();
            while (!mbar_try_wait(final_bar, 0) && clock64() - t0 < kWaitCycles) {
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        // ------------------------------------------------------------ raw weight bytes
        // 2-D tensor copies of 144-byte x 64-row boxes of the blob, issued by
        // lane 0.  Q8_0 (the shared expert) copies through the launch's map;
        // Q4_K through a per-CTA map whose global address is rewritten for
        // each new expert (two global slots used in turn: a slot is reused only
        // once the copies that named it have landed).
        uint32_t rs_it = 0;
        const int ffop = FMT == kWQ4K ? g.FF : g.SFF;
        const void *tm = &tmap_w;
        const uint32_t s_tmap = smem_addr(smem + C::kOffTmap);
        int cur_e = -2, nmaps = 0;
        uint32_t last_rs0 = 0, last_rs1 = 0;   // raw index after the last copy that named slot 0 / 1
        if (FMT == kWQ4K) {
            reinterpret_cast<uint32_t *>(smem + C::kOffTmap)[lane] = reinterpret_cast<const uint32_t *>(&tmap_w)[lane];
            __syncwarp();
        }
        bool ok = true;
        // the next tile's record and (once that is in) its blob address, a tile ahead
        int4 tnext = tile_fetch(g, blockIdx.x, n_tiles);
        const uint8_t *bnext = FMT == kWQ4K && (int)blockIdx.x < n_tiles && tnext.x >= 0 ? g.blobs[tnext.x]
                                                                                       : nullptr;
        for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
            const TileInfo ti = tile_decode<OP, FMT>(g, tnext);
            const uint8_t *blob = bnext;
            tnext = tile_fetch(g, tile + (int)gridDim.x, n_tiles);
            if (!ti.live) {
                if (FMT == kWQ4K)
                    bnext = tnext.x >= 0 && tile + (int)gridDim.x < n_tiles ? g.blobs[tnext.x] : nullptr;
                continue;
            }
            if (FMT == kWQ4K && ti.e != cur_e) {
                const int ms = nmaps & 1;
                // the copies that last named this slot must have landed (a raw slot is
                // refilled only after it was consumed, which settles every older copy)
                const uint32_t lr = ms ? last_rs1 : last_rs0;
                if (nmaps >= 2 && lr > 0 && rs_it < lr - 1 + RS && lane == 0) {
                    const uint32_t i = lr - 1;
                    const long long t0 = clock64();
                    while (!mbar_try_wait(full_raw(i % RS), (i / RS) & 1) && clock64() - t0 < kWaitCycles) {
                    }
                }
                __syncwarp();
                CUtensorMap *gslot = g.tmaps + 2 * blockIdx.x + ms;
                if (lane == 0) tmap_set_addr_smem(s_tmap, blob);
                __syncwarp();
                tmap_copy_release(gslot, s_tmap);
                if (lane == 0) tmap_acquire(gslot);
                __syncwarp();
                tm = gslot;
                cur_e = ti.e;
                ++nmaps;
            }
            const int nrs = ((ti.ksteps + KS - 1) / KS + SPR - 1) / SPR;
            for (int rsi = 0; rsi < nrs; ++rsi, ++rs_it) {
                const int slot = rs_it % RS;
                if (!(ok = warp_wait_bar(empty_raw(slot), ((rs_it / RS) & 1) ^ 1, abort_flag, g.status, g.wait_cycles))) break;
                if (lane == 0) {
                    const uint32_t dst0 = smem_addr(raw_base + slot * C::kRawStage);
                    mbar_arrive_expect_tx(full_raw(slot), C::kRawStage);
                    if (OP == kOpGateUp) {
                        const int kst0 = ti.k0 / KS + rsi * SPR;               // first 128-wide K stage
                        const int x = FMT == kWQ4K ? (kst0 >> 1) * 144 : (136 * kst0) & ~15;
                        tma_load_2d(dst0, tm, x, ti.m * 64, full_raw(slot));
                        tma_load_2d(dst0 + 64 * 144, tm, x, ffop + ti.m * 64, full_raw(slot));
                    } else {
                        const int h0 = ti.m * 128;
                        const int x = FMT == kWQ4K ? (h0 / 256) * 144 : (34 * (h0 / 32)) & ~15;
                        tma_load_2d(dst0, tm, x, 2 * ffop + 64 * (ti.k0 + rsi), full_raw(slot));
                    }
                }
                __syncwarp();
            }
            if (FMT == kWQ4K) {
                if ((nmaps - 1) & 1) last_rs1 = rs_it;
                else last_rs0 = rs_it;
                bnext = tnext.x >= 0 && tile + (int)gridDim.x < n_tiles ? g.blobs[tnext.x] : nullptr;
            }
        }
        // copies still in flight (an early exit) must land before the CTA ends
        if (lane == 0) {
            for (uint32_t i = rs_it > (uint32_t)RS ? rs_it - RS : 0; i < rs_it; ++i) {
                const long long t0 = clock64();
                while (!mbar_try_wait(full_raw(i % RS), (i / RS) & 1) && clock64() - t0 < kWaitCycles) {
                }
            }
        }
        __syncwarp();
    } else if (warp < 8) {
        // ------------------------------------------------------------ token rows (B)
        // the tile's rows are consecutive (xg and a are in bucket order): one
        // tensor box of NMAX rows per 64-wide K sub-tile, sub-tile i issued by
        // lane 0 of warp 6 + i (two issuing warps keep two copies in flight)
        const int sub = warp - 6;
        uint32_t st_it = 0;
        bool ok = true;
        if (sub < KS) {
            int4 tnext = tile_fetch(g, blockIdx.x, n_tiles);
            for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
                const TileInfo ti = tile_decode<OP, FMT>(g, tnext);
                tnext = tile_fetch(g, tile + (int)gridDim.x, n_tiles);
                if (!ti.live) continue;
                const int row0 = ti.row0;
                const int nst = (ti.ksteps + KS - 1) / KS;
                for (int st = 0; st < nst; ++st, ++st_it) {
                    const int slot = st_it % S;
                    if (!(ok = warp_wait_bar(empty(slot), ((st_it / S) & 1) ^ 1, abort_flag, g.status, g.wait_cycles))) break;
                    if (lane == 0) {
                        const bool has = st * KS + sub < ti.ksteps;
                        mbar_arrive_expect_tx(full(slot), has ? (uint32_t)C::kBSub : 0u);
                        // test hook: the first copy of this CTA is armed but never issued,
                        // so the waits for its stage run out
                        const bool skip = (int)blockIdx.x == g.skip_cta && st_it == 0 && sub == 0;
                        if (has && !skip)
                            tma_load_2d(sB + slot * C::kBStage + sub * C::kBSub, &tmap_b,
                                        (ti.k0 + st * KS + sub) * 64, row0, full(slot));
                    }
                    __syncwarp();
                }
            }
            // tensor copies still in flight (an early exit) must land before the
            // CTA ends; they complete within microseconds, so a short bounded wait
            if (lane == 0) {
                for (uint32_t i = st_it > (uint32_t)S ? st_it - S : 0; i < st_it; ++i) {
                    const long long t0 = clock64();
                    while (!mbar_try_wait(full(i % S), (i / S) & 1) && clock64() - t0 < (1 << 21)) {
                    }
                }
            }
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------ dequantisation (A)
        const int dt = threadIdx.x - 256;   // 0 .. kDeq-1
        // gate/up: thread (row, half) with row = tensor-memory lane 32 (warp % 4) + lane
        const int q_lane = 32 * (warp & 3), row = q_lane + lane, hh = (warp - 8) >> 2;
        uint32_t st_it = 0, rs_it = 0;
        bool ok = true;
        int4 tnext = tile_fetch(g, blockIdx.x, n_tiles);
        for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
            const TileInfo ti = tile_decode<OP, FMT>(g, tnext);
            tnext = tile_fetch(g, tile + (int)gridDim.x, n_tiles);
            if (!ti.live) continue;
            const int nst = (ti.ksteps + KS - 1) / KS;
            for (int st = 0; st < nst; ++st, ++st_it) {
                // warp-wide waits: the tensor-memory stores below are warp-collective
                const int kst = ti.k0 / KS + st;                  // global stage index along K
                const bool first = SPR == 1 || (kst & 1) == 0, last = SPR == 1 || (kst & 1) == 1;
                const int rslot = rs_it % RS;
                if (first && !(ok = warp_wait_bar(full_raw(rslot), (rs_it / RS) & 1, abort_flag, g.status, g.wait_cycles))) break;
                const int slot = st_it % S;
                if (!(ok = warp_wait_bar(empty(slot), ((st_it / S) & 1) ^ 1, abort_flag, g.status, g.wait_cycles))) break;
                const uint8_t *raw = raw_base + rslot * C::kRawStage;
                if (OP == kOpGateUp) {
                    tc_fence_after();
                    const uint32_t taddr = tmem_base + ((uint32_t)q_lane << 16) + C::kColA + 64 * slot + 32 * hh;
                    const uint8_t *rr = raw + ((row & 1) * 64 + (row >> 1)) * 144;   // lane 2i: gate, 2i+1: up
                    if (FMT == kWQ4K) dequant_gu_q4k_tmem(rr, rr + 16 + 64 * (kst & 1) + 32 * hh, 2 * (kst & 1) + hh, taddr);
                    else dequant_gu_q80_tmem(rr, (136 * kst) & 15, hh, taddr);
                    tmem_wait_st();
                    tc_fence_before();
                } else {
                    const uint32_t a_tile = sA + slot * C::kAStage;
                    if (FMT == kWQ4K) dequant_dn_q4k<kDeq>(raw, a_tile, dt, ti.m & 1);
                    else dequant_dn_q80<kDeq>(raw, a_tile, dt, (34 * (ti.m * 128 / 32)) & 15);
                    fence_proxy_async();
                }
                mbar_arrive(full(slot));
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
        tmem_dealloc(tmem_base, C::kCols);
    }
}

// ---------------------------------------------------------------- helpers

struct PlanArgs {
    int H, FF, SFF, T, split_gu, split_dn, split_gus, split_dns;
    const int32_t *offsets, *active;
    const uint8_t *const *blobs;   // routed experts' blobs (a null one is flagged in its tiles)
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
// expert, by one CTA of 1024 threads (block 0 of k_gemm_prep, beside the
// permutation): one thread per active expert, block-wide prefix sums.
// Tile (e, m | ks << 16 | no blob << 30, row0, n): expert e (-1 = shared),
// weight tile m, K split ks, tokens n0 .. n0+n-1 of the expert's bucket, whose
// rows start at row0 = the bucket's offset + n0 (the shared expert: row0 =
// n0, a token index).  The splits of one (e, m, n0) group are consecutive.
__device__ __forceinline__ void plan_tiles(const PlanArgs &p)
{
    __shared__ int scan_gu[1024], scan_dn[1024];
    __shared__ int s_e[1024], s_n[1024], s_tn[1024], s_bb[1024], s_flag[1024];
    const int u = threadIdx.x;
    const int n_active = (int)p.header[kHdrNActive];
    const int mt_gu = p.FF / 64, mt_dn = p.H / 128;
    int e = -1, n_e = 0, tn = 0, nt = 0, bb = 0, flag = 0;
    if (u < n_active) {
        e = p.active[u];
        bb = p.offsets[e];
        n_e = p.offsets[e + 1] - bb;
        split_tokens(n_e, tn, nt);
        flag = p.blobs[e] ? 0 : kTileNoBlob;
    }
    s_e[u] = e;
    s_n[u] = n_e;
    s_tn[u] = tn;
    s_bb[u] = bb;
    s_flag[u] = flag;
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
    // every thread writes tiles: tile i of a list belongs to the expert whose
    // inclusive prefix first exceeds i (binary search); within an expert the
    // order is token tile j, then weight tile m, then K split ks
    auto fill = [&](const int *scan, int mt, int split, int4 *out) {
        const int total = scan[1023];
        for (int i = u; i < total; i += 1024) {
            int lo = 0, hi = 1023;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (scan[mid] > i) hi = mid;
                else lo = mid + 1;
            }
            const int l = i - (lo ? scan[lo - 1] : 0);
            const int ks = l % split, m = (l / split) % mt, j = l / (split * mt);
            const int n0 = j * s_tn[lo];
            out[i] = make_int4(s_e[lo], m | (ks << 16) | s_flag[lo], s_bb[lo] + n0, min(s_tn[lo], s_n[lo] - n0));
        }
    };
    fill(scan_gu, mt_gu, p.split_gu, p.gu);
    fill(scan_dn, mt_dn, p.split_dn, p.dn);
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

// fp16 operand copies of x: xg, the rows in bucket order (row p holds token
// assign[p] / k), and x16 in token order when a shared expert needs it; zero
// the fp32 output accumulator, the split-K partial sums and their counters.
// Eight elements per item (16-byte loads and stores).  Block 0 plans the
// GEMMs' work tiles meanwhile (plan_tiles); the other blocks do the rest.
__global__ void __launch_bounds__(1024) k_gemm_prep(const uint16_t *__restrict__ x, const int32_t *__restrict__ assign,
                                                    int k, int T, int H, __half *__restrict__ xg,
                                                    __half *__restrict__ x16, float *__restrict__ yacc,
                                                    float *__restrict__ gu, int64_t n_gu, uint32_t *__restrict__ cnt,
                                                    int64_t n_cnt, uint32_t *status, const __grid_constant__ PlanArgs plan)
{
    if (blockIdx.x == 0) {
        plan_tiles(plan);
        return;
    }
    bool bad = false;
    const int64_t stride = (int64_t)(gridDim.x - 1) * blockDim.x;
    const int64_t tid = (int64_t)(blockIdx.x - 1) * blockDim.x + threadIdx.x;
    const int cpr = H / 8;                               // 8-element chunks per row
    // bf16 pairs -> fp16 pairs (each rounded once); |x| >= 65504 -- for a bf16
    // value, magnitude bits >= 0x4780 (2^16; the bf16 below it, 65280, is an
    // fp16 number), infinities and NaN included -- flags the call
    auto convert_v = [&](const uint4 v, __half *dst) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
        const uint32_t mag = __vmaxu2(__vmaxu2(v.x & 0x7fff7fffu, v.y & 0x7fff7fffu),
                                      __vmaxu2(v.z & 0x7fff7fffu, v.w & 0x7fff7fffu));
        bad |= __vcmpgeu2(mag, 0x47804780u) != 0u;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 h = __floats2half2_rn(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
            memcpy(&o[i], &h, 4);
        }
        *reinterpret_cast<uint4 *>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
    };
    auto convert = [&](const uint16_t *src, __half *dst) { convert_v(__ldg(reinterpret_cast<const uint4 *>(src)), dst); };
    // one warp per row: lanes take consecutive 16-byte chunks, four loads in flight
    const int lane = threadIdx.x & 31;
    const int64_t gwarp = tid >> 5, nwarps = stride >> 5;
    for (int64_t p = gwarp; p < (int64_t)T * k; p += nwarps) {
        const int t = assign[p] / k;
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (int64_t)t * H);
        __half *dst = xg + p * H;
        for (int c0 = lane; c0 < cpr; c0 += 4 * 32) {
            uint4 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (c0 + 32 * j < cpr) v[j] = __ldg(src + c0 + 32 * j);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (c0 + 32 * j < cpr) convert_v(v[j], dst + 8 * (c0 + 32 * j));
        }
    }
    const int64_t n_x = (int64_t)T * cpr;
    if (x16)
        for (int64_t i = tid; i < n_x; i += stride) convert(x + 8 * i, x16 + 8 * i);
    if (yacc)
        for (int64_t i = tid; i < 2 * n_x; i += stride)
            reinterpret_cast<float4 *>(yacc)[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int64_t i = tid; i < n_gu; i += stride) gu[i] = 0.0f;
    for (int64_t i = tid; i < n_cnt; i += stride) cnt[i] = 0u;
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) set_status(status, MOE_ERR_DEVICE_FAULT);
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

// ---------------------------------------------------------------- router logits on tcgen05

// logits[T][E] = x[T][H] * Wr[E][H]^T for the tensor-core routing path.  The
// fp32 router matrix arrives split into three bf16 planes (w = w1 + w2 + w3
// exactly: each bf16 x bf16 product is exact), stacked as [3E][H].  CTA tile:
// 128 tokens (MMA M) x N experts; K stages of 64 (one 128-byte swizzle row of
// bf16), kRtStages in flight.  The 24 MMAs of every two stages (128 of K x
// 3 planes) sum into a fresh accumulator in tensor memory (two, used in turn),
// and the epilogue warps add those partial sums into fp32 registers: no long
// chain runs inside the tensor-memory accumulator (one chain over all of K
// drifted by ~2e-6 on logits of ~2.5, beyond the 1e-6 near-tie band of the
// selection).
// Warp 0 issues the 2-D tensor copies, warp 1 owns the tensor memory and
// issues the MMAs, warps 2-5 add and store (one lane quadrant each).
constexpr int kRtM = 128, kRtK = 64, kRtStages = 3, kRtThreads = 192, kRtEpi = 4;
constexpr int kRtKpb = 2;               // K stages summed in one tensor-memory accumulator

template <int N>
struct RtSmem {
    static constexpr uint32_t kX = kRtM * kRtK * 2;       // x rows of a stage
    static constexpr uint32_t kW = N * kRtK * 2;          // one plane's rows of a stage
    static constexpr uint32_t kStage = kX + 3 * kW;
    static constexpr uint32_t kBytes = kRtStages * kStage + 1024 /* alignment */ + 256 /* barriers, slots */;
};

template <int N>
__global__ void __launch_bounds__(kRtThreads, 1) k_router_tc(const __grid_constant__ CUtensorMap tmap_x,
                                                            const __grid_constant__ CUtensorMap tmap_w, int T, int H,
                                                            int E, float *__restrict__ logits, uint32_t *status,
                                                            long long limit, int skip_cta)
{
    using C = RtSmem<N>;
    extern __shared__ uint8_t rt_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(rt_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sX = smem_addr(smem), sW = sX + kRtStages * C::kX;   // x stages, then [stage][plane] rows
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kRtStages * C::kStage);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * kRtStages + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * kRtM, e0 = blockIdx.y * N, nk = H / kRtK;
    auto full = [&](int s) { return smem_addr(bars + s); };
    auto empty = [&](int s) { return smem_addr(bars + kRtStages + s); };
    auto acc_full = [&](int b) { return smem_addr(bars + 2 * kRtStages + b); };
    auto acc_empty = [&](int b) { return smem_addr(bars + 2 * kRtStages + 2 + b); };
    const uint32_t done = smem_addr(bars + 2 * kRtStages + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRtStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full(b), 1);
            mbar_init(acc_empty(b), kRtEpi);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), 2 * N);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // test hook: this tile never issues (nor arms) its first stage
            const bool skip0 = skip_cta == (int)(blockIdx.y * gridDim.x + blockIdx.x);
            int issued = 0;
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % kRtStages;
                if (kb >= kRtStages && !wait_bar(empty(s), ((kb / kRtStages) - 1) & 1, abort_flag, status, limit))
                    break;
                if (kb == 0 && skip0) {
                    ++issued;
                    continue;
                }
                mbar_arrive_expect_tx(full(s), C::kStage);
                tma_load_2d(sX + s * C::kX, &tmap_x, kb * kRtK, t0, full(s));
#pragma unroll
                for (int sp = 0; sp < 3; ++sp)
                    tma_load_2d(sW + (s * 3 + sp) * C::kW, &tmap_w, kb * kRtK, sp * E + e0, full(s));
                ++issued;
            }
            // copies in flight must land before the CTA ends (only left after an abort)
            for (int kb = issued > kRtStages ? issued - kRtStages : 0; kb < issued; ++kb) {
                if (kb == 0 && skip0) continue;
                const long long c0 = clock64();
                while (!mbar_try_wait(full(kb % kRtStages), (kb / kRtStages) & 1) && clock64() - c0 < limit) {
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kRtM, N);
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % kRtStages, pb = kb / kRtKpb, b = pb & 1;
                const bool first = kb % kRtKpb == 0, last = kb % kRtKpb == kRtKpb - 1 || kb == nk - 1;
                if (!wait_bar(full(s), (kb / kRtStages) & 1, abort_flag, status, limit)) break;
                if (first && pb >= 2 && !wait_bar(acc_empty(b), ((pb >> 1) - 1) & 1, abort_flag, status, limit))
                    break;
                tc_fence_after();
                const uint64_t a0 = sdesc_kmajor_sw128(sX + s * C::kX);
#pragma unroll
                for (int kk = 0; kk < kRtK / 16; ++kk)
#pragma unroll
                    for (int sp = 0; sp < 3; ++sp)
                        mma_f16(tmem + b * N, a0 + (uint64_t)((32 * kk) >> 4),
                                sdesc_kmajor_sw128(sW + (s * 3 + sp) * C::kW) + (uint64_t)((32 * kk) >> 4), idesc,
                                !first || (kk | sp) != 0);
                mma_commit(empty(s));
                if (last) mma_commit(acc_full(b));
            }
            mma_commit(done);           // every MMA issued (all of them, or those before an abort)
        }
        __syncwarp();
    } else {
        const int q = warp & 3;         // the lane quadrant this warp may read
        float acc[N];
#pragma unroll
        for (int c = 0; c < N; ++c) acc[c] = 0.0f;
        bool ok = true;
        const int np = (nk + kRtKpb - 1) / kRtKpb;
        for (int pb = 0; pb < np && ok; ++pb) {
            const int b = pb & 1;
            if (lane == 0) ok = wait_bar(acc_full(b), (pb >> 1) & 1, abort_flag, status, limit);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            // 64 columns a round: four loads in flight, then the adds
#pragma unroll
            for (int c = 0; c < N; c += 64) {
                uint32_t v[4][16];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (c + 16 * i < N) tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + b * N + c + 16 * i, v[i]);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c + 16 * i < N) acc[c + 16 * i + j] += __uint_as_float(v[i][j]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(b));
        }
        const int t = t0 + 32 * q + lane;
        if (ok && t < T) {
            float *row = logits + (int64_t)t * E + e0;
#pragma unroll
            for (int c = 0; c < N; ++c)
                if (e0 + c < E) row[c] = acc[c];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        // every issued MMA has completed before the tensor memory is freed
        if (lane == 0) {
            const long long c0 = clock64();
            while (!mbar_try_wait(done, 0) && clock64() - c0 < limit) {
            }
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 2 * N);
    }
}

// ---------------------------------------------------------------- launch

// cuTensorMapEncodeTiled, fetched from the driver through the runtime (no
// link against the driver library)
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// Tensor map of an fp16 matrix [rows][cols] (row-major, cols % 8 == 0, base
// 16-byte aligned): boxes of 64 columns x box_rows rows, 128-byte swizzle
// (the K-major layout the MMA descriptors expect), zero fill past the edges.
static bool make_tmap_f16(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int box_rows)
{
    EncodeTiledFn fn = encode_tiled();
    if (!fn || rows <= 0 || cols <= 0) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of the raw bytes of a blob of 3 matrices [rows][row_bytes]
// (uint8 elements, no swizzle): boxes of 144 bytes x 64 rows.
static bool make_tmap_raw(CUtensorMap *m, const void *base, int64_t rows, int64_t row_bytes)
{
    EncodeTiledFn fn = encode_tiled();
    if (!fn || rows <= 0 || row_bytes <= 0) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {144, 64};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The weight tensor map of one launch: the shared expert's blob (Q8_0), or
// for the routed experts (Q4_K) a template whose address each CTA rewrites.
template <int FMT>
static bool make_tmap_w(CUtensorMap *m, const GemmArgs &g)
{
    if (FMT == kWQ80) return make_tmap_raw(m, g.shared_blob, 3 * (int64_t)g.SFF, (int64_t)(g.H / 32) * 34);
    return make_tmap_raw(m, g.tmaps, 3 * (int64_t)g.FF, (int64_t)(g.H / 256) * 144);
}

// The B operand's tensor map of one launch: boxes of NMAX consecutive rows of
// xg (routed gate/up), x16 (shared gate/up) or a (down).
template <int OP, int FMT, int NMAX>
static bool make_tmap_b(CUtensorMap *m, const GemmArgs &g)
{
    if (OP == kOpGateUp) {
        if (FMT == kWQ4K) return make_tmap_f16(m, g.xg, (int64_t)g.T * g.k, g.H, NMAX);
        return make_tmap_f16(m, g.x16, g.T, g.H, NMAX);
    }
    if (FMT == kWQ4K) return make_tmap_f16(m, g.act16, (int64_t)g.T * g.k, g.FF, NMAX);
    return make_tmap_f16(m, g.sh_act16, g.T, g.SFF, NMAX);
}

template <int OP, int FMT, int NMAX, int S, int RAW, int EW>
static cudaError_t launch_gemm(const GemmArgs &g, int grid, cudaStream_t s)
{
    using C = GemmCfg<OP, FMT, NMAX, S, RAW>;
    {
        // function attributes are per device: set once for each device this process uses
        static std::mutex mu;
        static bool done[64] = {};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev]) {
            e = cudaFuncSetAttribute(k_moe_gemm<OP, FMT, NMAX, S, RAW, EW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     C::kBytes);
            if (e != cudaSuccess) return e;
            done[dev] = true;
        }
    }
    CUtensorMap tmap_b, tmap_w;
    if (!make_tmap_b<OP, FMT, NMAX>(&tmap_b, g) || !make_tmap_w<FMT>(&tmap_w, g)) return cudaErrorInvalidValue;
    k_moe_gemm<OP, FMT, NMAX, S, RAW, EW><<<grid, kGemmThreads, C::kBytes, s>>>(g, tmap_b, tmap_w);
    return cudaGetLastError();
}

// Configurations: small buckets (every token tile <= 16 wide) keep a 6-stage
// ring; large buckets (prefill) use token tiles of kGemmMaxN and 4 stages
// (gate/up: the A stages fill the tensor memory beside the two accumulators).
// The raw-byte rings take what shared memory is left.  Down projections with
// few 64-row K-steps per token column (ff / tokens per expert below 8) give
// the epilogue 8 warps.
template <int OP, int FMT>
static cudaError_t launch_gemm_cfg(const GemmArgs &g, int grid, bool small, bool epi8, cudaStream_t s)
{
    if constexpr (OP == kOpDown) {
        if (epi8) {
            if (small) return launch_gemm<OP, FMT, 16, 6, 98304, 8>(g, grid, s);
            return launch_gemm<OP, FMT, kGemmMaxN, 4, 81920, 8>(g, grid, s);
        }
    }
    if (small) return launch_gemm<OP, FMT, 16, 6, OP == kOpGateUp ? 163840 : 98304, 4>(g, grid, s);
    return launch_gemm<OP, FMT, kGemmMaxN, 4, 81920, 4>(g, grid, s);
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

size_t gemm_tmap_bytes() { return (size_t)num_sms() * 2 * sizeof(CUtensorMap); }

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
        // no K split anywhere: the split gate/up sums meet through atomic additions
        // (their order varies), and the deterministic down epilogue stores each slot once
        sp = GemmSplits{1, 1, 1, 1};
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
    const int64_t items = std::max<int64_t>((int64_t)a.T * a.k * (a.H / 8), w.n_gu);
    PlanArgs p{a.H, a.FF, a.SFF, a.T, sp.gu, sp.dn, sp.gus, sp.dns, a.offsets, a.active, a.blobs, a.header,
               w.tiles_gu, w.tiles_dn, w.tiles_gus, w.tiles_dns};
    // one wave: the planning CTA and as many grid-stride CTAs as stay resident beside it
    static std::atomic<int> prep_per_sm{0};
    if (prep_per_sm.load() == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemm_prep, 1024, 0) != cudaSuccess || n < 1) n = 1;
        prep_per_sm.store(n);
    }
    const int64_t prep_workers = std::max<int64_t>(1, (int64_t)prep_per_sm.load() * num_sms() - 1);
    k_gemm_prep<<<1 + (unsigned)std::min<int64_t>((items + 1023) / 1024, prep_workers), 1024, 0, s>>>(
        a.x, a.assign, a.k, a.T, a.H, w.xg, a.shared_blob ? w.x16 : nullptr, det ? nullptr : w.yacc, w.gu, w.n_gu,
        w.split_cnt, w.n_cnt, a.header + kHdrStatus, p);
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
    g.xg = w.xg;
    g.x16 = w.x16;
    g.act16 = w.act16;
    g.sh_act16 = w.sh_act16;
    g.yacc = w.yacc;
    g.slots = a.slots;
    g.sh_out = a.sh_out;
    g.status = a.header + kHdrStatus;
    g.tmaps = reinterpret_cast<CUtensorMap *>(w.tmaps);
    g.wait_cycles = a.wait_cycles;
    g.skip_cta = a.skip_cta;                 // the routed gate/up launch only
    const int grid = num_sms();
    cudaError_t e;

    prof_begin(kPhGemmGateUp, s);
    g.tiles = w.tiles_gu;
    g.n_tiles = a.header + kHdrTilesGU;
    g.splits = sp.gu;
    g.gu = w.gu;
    g.split_cnt = w.split_cnt;
    e = launch_gemm_cfg<kOpGateUp, kWQ4K>(g, grid, small, false, s);
    g.skip_cta = -1;
    if (e == cudaSuccess && a.shared_blob) {
        g.tiles = w.tiles_gus;
        g.n_tiles = a.header + kHdrTilesGUS;
        g.splits = sp.gus;
        g.gu = w.sh_gu;
        g.split_cnt = w.split_cnt + w.n_cnt_routed;
        e = launch_gemm_cfg<kOpGateUp, kWQ80>(g, grid, small, false, s);
    }
    prof_end(kPhGemmGateUp, s);
    if (e != cudaSuccess) return e;

    prof_begin(kPhGemmDown, s);
    g.tiles = w.tiles_dn;
    g.n_tiles = a.header + kHdrTilesDN;
    g.splits = sp.dn;
    // a tile's K against its token columns (tokens per expert on average, at
    // most kGemmMaxN)
    const int64_t n_avg = std::min<int64_t>((int64_t)a.T * a.k / std::max(1, a.E), kGemmMaxN);
    e = launch_gemm_cfg<kOpDown, kWQ4K>(g, grid, small, a.FF < 8 * n_avg, s);
    if (e == cudaSuccess && a.shared_blob) {
        g.tiles = w.tiles_dns;
        g.n_tiles = a.header + kHdrTilesDNS;
        g.splits = sp.dns;
        e = launch_gemm_cfg<kOpDown, kWQ80>(g, grid, small, a.SFF < 8 * std::min<int64_t>(a.T, kGemmMaxN), s);
    }
    prof_end(kPhGemmDown, s);
    if (e != cudaSuccess) return e;

    prof_begin(kPhGemmFinish, s);
    k_gemm_finish<<<(unsigned)std::min<int64_t>((n + 255) / 256, 148 * 8), 256, 0, s>>>(
        w.yacc, det ? a.slots : nullptr, det ? a.sh_out : nullptr, a.T, a.H, a.k, a.y, a.y_f32);
    prof_end(kPhGemmFinish, s);
    return cudaGetLastError();
}

// Tensor map of a bf16 matrix [rows][cols] (row-major, base 16-byte aligned,
// cols % 8 == 0): boxes of 64 columns x box_rows rows, 128-byte swizzle, zero
// fill past the edges.
static bool make_tmap_bf16(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int box_rows)
{
    EncodeTiledFn fn = encode_tiled();
    if (!fn || rows <= 0 || cols <= 0) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int N>
static cudaError_t launch_router_tc_n(const uint16_t *x, const uint16_t *planes, int T, int H, int E, float *logits,
                                      uint32_t *status, long long limit, int skip_cta, cudaStream_t s)
{
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev]) {
            e = cudaFuncSetAttribute(k_router_tc<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)RtSmem<N>::kBytes);
            if (e != cudaSuccess) return e;
            done[dev] = true;
        }
    }
    CUtensorMap tx, tw;
    if (!make_tmap_bf16(&tx, x, T, H, kRtM) || !make_tmap_bf16(&tw, planes, 3 * (int64_t)E, H, N))
        return cudaErrorInvalidValue;
    const dim3 grid((T + kRtM - 1) / kRtM, (E + N - 1) / N);
    k_router_tc<N><<<grid, kRtThreads, RtSmem<N>::kBytes, s>>>(tx, tw, T, H, E, logits, status, limit, skip_cta);
    return cudaGetLastError();
}

// 128-expert tiles when they fill most SMs, else 64
cudaError_t launch_router_tc(const uint16_t *x, const uint16_t *planes, int T, int H, int E, float *logits,
                             uint32_t *status, long long limit, cudaStream_t s)
{
    const int64_t tiles128 = (int64_t)((T + kRtM - 1) / kRtM) * ((E + 127) / 128);
    const int skip = debug_take_skip_router();
    if (E % 128 == 0 && tiles128 >= 120)
        return launch_router_tc_n<128>(x, planes, T, H, E, logits, status, limit, skip, s);
    return launch_router_tc_n<64>(x, planes, T, H, E, logits, status, limit, skip, s);
}

}  // namespace moe
