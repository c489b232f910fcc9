// moe_internal.cuh -- internal declarations shared by the CUDA translation
// units of libmoe.so (kernels + C ABI).  Nothing here is part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "../../include/moe.h"

namespace moe {

// ---- block formats (GGUF layouts; the pages name Q4_K / Q8_0 for the expert
// ---- tensors in the DeepSeek-V4-Flash GGUF anatomy table, section 二)
constexpr int kQK = 256;          // weights per Q4_K super-block
constexpr int kQ4KBytes = 144;    // fp16 d, fp16 dmin, scales[12], qs[128]
constexpr int kQ5KBytes = 176;    // fp16 d, fp16 dmin, scales[12], qh[32], qs[128]
constexpr int kQK8 = 32;          // weights per Q8_0 block
constexpr int kQ8Bytes = 34;      // fp16 d, int8 qs[32]

constexpr int kHeaderBytes = 256; // workspace header (status word, counters)
constexpr int kGemvMaxTokens = 8; // decode windows: MTP verify windows of 1-8 tokens

// Header words of the workspace.
enum HeaderWord : int {
    kHdrStatus = 0,       // first device-side fault (moe_status), sticky until read
    kHdrNActive = 1,      // number of experts with at least one token
    kHdrTilesGU = 2,      // GEMM path: work tiles of the routed gate/up projection
    kHdrTilesDN = 3,      //            routed down projection
    kHdrTilesGUS = 4,     //            shared expert gate/up
    kHdrTilesDNS = 5,     //            shared expert down
    kHdrTicketRoute = 6,  // decode path: CTAs done with the router logits (last one routes)
    kHdrTicketDown = 7,   // decode path: CTAs done with the down projection (last one writes y)
    kHdrCounter0 = 8,     // completion counters, reset by their last user
    kHdrGridBar = 56,     // layer stack: arrivals at its grid-wide barriers (zeroed before each launch)
    kHdrGridAbort = 57,   //              raised by a CTA whose barrier wait ran out
};

__device__ __forceinline__ void set_status(uint32_t *status, uint32_t code)
{
    if (status) atomicCAS(status, 0u, code);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ float f16_bits_to_f32(uint32_t h)
{
    return __half2float(__ushort_as_half((unsigned short)h));
}

// 6-bit scale / min of sub-block j from the 12 packed bytes.
__device__ __forceinline__ void q4k_scale_min(const uint8_t *scales, int j, int &sc, int &m)
{
    if (j < 4) {
        sc = scales[j] & 63;
        m = scales[j + 4] & 63;
    } else {
        sc = (scales[j + 4] & 15) | ((scales[j - 4] >> 6) << 4);
        m = (scales[j + 4] >> 4) | ((scales[j] >> 6) << 4);
    }
}

// Kernels counted / timed by the diagnostics API (moe_profile_*).
enum Phase : int {
    kPhRouterLogits = 0, kPhTopk, kPhBucket, kPhGemmPrep, kPhGemmGateUp, kPhGemmDown, kPhGemmFinish,
    kPhDecRoute, kPhDecLayer, kPhDecStack, kNumPhases
};
void prof_begin(int phase, cudaStream_t s);   // no-ops unless profiling is enabled
void prof_end(int phase, cudaStream_t s);

// Workspace regions (byte offsets from the workspace base) for one call shape.
struct WsLayout {
    size_t header, logits, ids, w, counts, offsets, assign, active;
    size_t slots, yacc, xg, x16, sh_out, bhist, xfrag, wsplit;
    size_t act16, sh_act16, tiles_gu, tiles_dn, tiles_gus, tiles_dns, tmaps, gu, sh_gu, split_cnt;
    size_t total;
};

moe_status forward_checks(const moe_config *cfg, const uint16_t *x, const float *router_w, const float *router_bias,
                          const uint8_t *const *expert_blobs, const uint8_t *shared_blob, int32_t T, uint16_t *y,
                          float *y_f32, void *ws, size_t ws_bytes);

// Routing path choice for T tokens under cfg flags.
bool use_gemv(const moe_config &c, int32_t T);
WsLayout ws_layout(const moe_config &c, int32_t T);

// ---- launchers (each returns cudaGetLastError() of its launches) ----------
cudaError_t launch_pack_q5k(const float *w, int64_t nblocks, uint8_t *out, uint32_t *status, cudaStream_t s);
cudaError_t launch_pack_q4k(const float *w, int64_t nblocks, uint8_t *out, uint32_t *status,
                            cudaStream_t s);
cudaError_t launch_pack_q8_0(const float *w, int64_t nblocks, uint8_t *out, uint32_t *status,
                             cudaStream_t s);
cudaError_t launch_dequant_q4k(const uint8_t *blk, int64_t nblocks, float *out, cudaStream_t s);
cudaError_t launch_dequant_q8_0(const uint8_t *blk, int64_t nblocks, float *out, cudaStream_t s);
cudaError_t launch_dequant_q4k_f16(const uint8_t *blk, int64_t nblocks, uint16_t *out, cudaStream_t s);
cudaError_t launch_dequant_q5k(const uint8_t *blk, int64_t nblocks, float *out, cudaStream_t s);
cudaError_t launch_dequant_q5k_f16(const uint8_t *blk, int64_t nblocks, uint16_t *out, cudaStream_t s);
cudaError_t launch_dequant_q8_0_f16(const uint8_t *blk, int64_t nblocks, uint16_t *out, cudaStream_t s);

struct RouteArgs {
    int H, E, k, T, score_fn;
    const uint16_t *x;
    const float *wr, *bias;
    float *logits;
    int32_t *ids;
    float *w;
    int32_t *counts, *offsets, *assign, *active;
    int32_t *bhist;                      // bucketing: [ceil(T*k / kBucketItems)][E] per-CTA counts
    uint16_t *wsplit;                    // [3][E][H] bf16 parts of the router matrix (tensor-core logits)
    uint32_t *header;
};
size_t router_split_bytes(int E, int H, int T);
// Router logits on tcgen05 from the split planes (gemm_tc.cu).
cudaError_t launch_router_tc(const uint16_t *x, const uint16_t *planes, int T, int H, int E, float *logits,
                             uint32_t *status, long long limit, cudaStream_t s);
constexpr int kBucketItems = 1024;       // assignments per CTA of the parallel bucketing
cudaError_t launch_route(const RouteArgs &a, cudaStream_t s);

struct ExpertArgs {
    int H, E, FF, k, T, SFF;
    const uint16_t *x;                  // bf16 [T][H]
    const uint8_t *const *blobs;        // device table [E]
    const uint8_t *shared_blob;         // Q8_0 or null
    const int32_t *offsets, *assign, *active;
    const float *w;                     // routing weights [T*k]
    float *slots;                       // [T*k][H] (deterministic combine)
    float *sh_out;                      // [T][H] (deterministic combine)
    uint16_t *y;                        // bf16 [T][H]
    float *y_f32;                       // optional
    uint32_t *header;
    long long wait_cycles;              // limit of every bounded wait
    int skip_cta;                       // test hook: the routed gate/up kernel's CTA that never issues its first copy
};

// ---- decode path (T <= kDecTok): router logits, then one persistent kernel
// ---- (routing, gate/up + SiLU*mul, down, combine), chained with PDL
constexpr int kDecTok = 8;                         // window tokens = MMA N columns
constexpr int kDecMaxAssign = kDecTok * 32;        // T * k
constexpr int kRouteMaxVec = 10;                   // router float4 per lane and warp
constexpr int kDecSmemBudget = 232448;             // dynamic shared memory of the layer kernel (227 KB)
constexpr int kSmemPerSM = 233472;                 // shared memory of one SM (228 KB)
constexpr long long kDefaultWaitCycles = 1ll << 32; // bounded device waits: ~2 s at 2 GHz

struct DecArgs {
    int H, E, FF, k, T, SFF, score_fn;
    int route_parts;             // router row split per CTA (1, 2, 4 or 8)
    int nc;                      // consumer warps of the layer kernel
    int half;                    // they own 128 columns each (else 256)
    int codec;                   // routed experts' blocks (moe_codec); Q5_K: 256-column warps
    uint32_t ring_bytes;         // their staging rings
    int stages;                  // stages of each consumer warp's ring
    int overlap_prev;            // weights may be read before the previous kernel ends
    long long wait_cycles;       // limit of every bounded wait
    int skip_cta;                // test hook: this CTA never issues its first bulk copy (-1: none)
    const uint16_t *x;
    const float *wr, *bias;
    const uint8_t *const *blobs;
    const uint8_t *shared_blob;
    float *logits;
    uint2 *xfrag;                // [H/256][16][4][T] fp16 MMA B fragments of x (built by the router kernel)
    int32_t *ids;
    float *w;
    int32_t *counts, *offsets, *assign, *active;
    float *yacc;                 // [T][H] fp32 accumulator
    uint16_t *y;
    float *y_f32;
    uint32_t *header;
};
int dec_route_parts(int H);
bool dec_half(const moe_config &c);
int dec_consumers(const moe_config &c);
uint32_t dec_ring_bytes(const moe_config &c, int32_t T);
int dec_stages(const moe_config &c, int32_t T);
bool dec_supported(const moe_config &c, int32_t T);
cudaError_t launch_decode(const DecArgs &a, cudaStream_t s);

// A window through a stack of layers in one cooperative launch (moe_forward_stack).
struct StackArgs {
    DecArgs d;                          // shapes, ring, hooks, workspace views (logits, routing, header)
    int L;                              // layers
    int residual;                       // x[l + 1] = bf16(x[l] + y[l]) written by the kernel
    int rows;                           // router rows a CTA holds: ceil(E / CTAs)
    const float *const *wr;             // device [L] router matrices
    const float *const *bias;           // device [L] or null
    const uint8_t *const *blobs;        // device [L][E] expert blobs
    const uint8_t *const *shared;       // device [L] or null
    uint16_t *x;                        // bf16 [L][T][H]
    uint16_t *y;                        // bf16 [L][T][H]
    float *y_f32;                       // [L][T][H] or null
    float *yacc;                        // [2][T][H] fp32 accumulators (alternating layers)
};
bool stack_supported(const moe_config &c, int32_t T);
int stack_grid();                       // CTAs of the stack kernel: one per SM
cudaError_t launch_stack(const StackArgs &a, cudaStream_t s);

// Test hooks (moe_debug_set): limit of the bounded device waits, and a CTA of
// the next call's main kernel that never issues its first bulk copy.
long long debug_wait_cycles();
int debug_take_skip_copy();

// Tensor-core (tcgen05) grouped GEMM path: its workspace regions.
constexpr int kGemmSmallTokens = 16;   // calls with T <= 16 use the small-bucket GEMM configuration
constexpr int kGemmMaxN = 128;         // tokens per work tile of the large-bucket configuration
struct GemmSplits {
    int gu, dn, gus, dns;                // K splits: routed gate/up, down; shared gate/up, down
};
struct GemmWs {
    __half *xg, *x16, *act16, *sh_act16;
    float *yacc;
    float *gu, *sh_gu;                   // split-K partial sums of g and u
    int64_t n_gu;                        // floats to zero in gu and sh_gu (contiguous)
    uint32_t *split_cnt;                 // split-K counters (routed groups, then shared groups)
    int64_t n_cnt, n_cnt_routed;
    int4 *tiles_gu, *tiles_dn, *tiles_gus, *tiles_dns;
    void *tmaps;                         // two 128-byte tensor-map slots per GEMM CTA
    GemmSplits splits;
    int det;
};
size_t gemm_tile_capacity(int mt, int64_t TK, int E);
size_t gemm_tmap_bytes();
GemmSplits gemm_splits(const moe_config &c, int32_t T);
cudaError_t launch_experts_gemm(const ExpertArgs &a, const GemmWs &w, cudaStream_t s);

}  // namespace moe
