// abi.cu -- the extern "C" entry points of libmoe.so: host-side argument
// checks, workspace layout, and the sequence of kernel launches of a call.
// The ABI itself (argument meaning, layouts, ownership, errors) is specified
// in include/moe.h.
#include <algorithm>
#include <atomic>

#include "moe_internal.cuh"
#include "debug_hooks.cuh"

namespace moe {

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

static bool cfg_valid(const moe_config *c)
{
    if (!c) return false;
    if (c->hidden < 256 || c->hidden > 8192 || c->hidden % 256) return false;
    if (c->n_experts < 1 || c->n_experts > 1024) return false;
    if (c->ff < 64 || c->ff > 8192 || c->ff % 64) return false;
    if (c->top_k < 1 || c->top_k > 32 || c->top_k > c->n_experts) return false;
    if (c->score_fn != MOE_SCORE_SOFTMAX && c->score_fn != MOE_SCORE_SIGMOID_BIAS) return false;
    if (c->shared_ff != 0 && (c->shared_ff < 64 || c->shared_ff > 8192 || c->shared_ff % 64)) return false;
    if (c->codec != MOE_CODEC_Q4K && c->codec != MOE_CODEC_Q5K) return false;
    return true;
}

// Decode path (windows of up to kDecTok tokens) unless the tensor-core GEMM
// is forced, the call is deterministic (the decode kernel combines with
// atomic additions; the GEMM path has the fixed-order slots), or the shape
// does not fit the decode kernel.
bool use_gemv(const moe_config &c, int32_t T)
{
    if (c.flags & (MOE_FLAG_FORCE_GEMM | MOE_FLAG_DETERMINISTIC)) return false;
    if (T > kDecTok || !dec_supported(c, T)) return false;
    if (c.flags & MOE_FLAG_FORCE_GEMV) return true;
    return T <= kGemvMaxTokens;
}

// ---- test hooks of the bounded device waits (moe_debug_set)
static std::atomic<long long> g_wait_cycles{kDefaultWaitCycles};
static std::atomic<int> g_skip_copy{-1};
static std::atomic<int> g_skip_router{-1};
long long debug_wait_cycles() { return g_wait_cycles.load(); }
int debug_take_skip_copy() { return g_skip_copy.exchange(-1); }
int debug_take_skip_router() { return g_skip_router.exchange(-1); }

WsLayout ws_layout(const moe_config &c, int32_t T)
{
    WsLayout L{};
    const size_t TK = (size_t)T * c.top_k, E = c.n_experts, H = c.hidden;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    L.header = take(kHeaderBytes);
    L.logits = take((size_t)T * E * 4);
    L.ids = take(TK * 4);
    L.w = take(TK * 4);
    L.counts = take(E * 4);
    L.offsets = take((E + 1) * 4);
    L.assign = take(TK * 4);
    L.active = take((E + 1) * 4);
    L.bhist = take((TK + kBucketItems - 1) / kBucketItems * E * 4);
    L.wsplit = take(router_split_bytes(c.n_experts, c.hidden, T));
    const bool gemv = use_gemv(c, T), det = (c.flags & MOE_FLAG_DETERMINISTIC) != 0;
    L.slots = take(det ? TK * H * 4 : 0);
    L.yacc = take((size_t)T * H * 4 * (gemv ? 2 : 1));   // decode: two (the layer stack alternates them)
    L.xfrag = take(gemv ? (size_t)T * H * 2 : 0);
    L.xg = take(gemv ? 0 : TK * H * 2);
    L.x16 = take(gemv || !c.shared_ff ? 0 : (size_t)T * H * 2);
    L.sh_out = take(!gemv && c.shared_ff && det ? (size_t)T * H * 4 : 0);
    L.act16 = take(gemv ? 0 : TK * c.ff * 2);
    L.sh_act16 = take(!gemv && c.shared_ff ? (size_t)T * c.shared_ff * 2 : 0);
    const size_t sh_tiles = (size_t)((T + kGemmMaxN - 1) / kGemmMaxN + 1);
    const GemmSplits sp = gemv ? GemmSplits{1, 1, 1, 1} : gemm_splits(c, T);
    const size_t cap_gu = gemv ? 0 : gemm_tile_capacity(c.ff / 64, (int64_t)TK, c.n_experts);
    const size_t cap_dn = gemv ? 0 : gemm_tile_capacity(c.hidden / 128, (int64_t)TK, c.n_experts);
    const size_t cap_gus = !gemv && c.shared_ff ? sh_tiles * (c.shared_ff / 64) : 0;
    const size_t cap_dns = !gemv && c.shared_ff ? sh_tiles * (c.hidden / 128) : 0;
    L.tiles_gu = take(cap_gu * sp.gu * 16);
    L.tiles_dn = take(cap_dn * sp.dn * 16);
    L.tiles_gus = take(cap_gus * sp.gus * 16);
    L.tiles_dns = take(cap_dns * sp.dns * 16);
    L.tmaps = take(gemv ? 0 : gemm_tmap_bytes());
    L.gu = take(sp.gu > 1 ? TK * 2 * c.ff * 4 : 0);
    L.sh_gu = take(sp.gus > 1 ? (size_t)T * 2 * c.shared_ff * 4 : 0);
    L.split_cnt = take(((sp.gu > 1 ? cap_gu : 0) + (sp.gus > 1 ? cap_gus : 0)) * 4);
    L.total = off;
    return L;
}

static moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

static moe_status check_call(const moe_config *cfg, const uint16_t *x, const float *router_w,
                             const float *router_bias, int32_t T, void *ws, size_t ws_bytes)
{
    if (!cfg_valid(cfg)) {
        if (!cfg) return MOE_ERR_INVALID_ARG;
        if (cfg->score_fn != MOE_SCORE_SOFTMAX && cfg->score_fn != MOE_SCORE_SIGMOID_BIAS)
            return MOE_ERR_INVALID_ARG;
        if ((cfg->codec != MOE_CODEC_Q4K && cfg->codec != MOE_CODEC_Q5K) || cfg->top_k < 1 ||
            cfg->top_k > cfg->n_experts)
            return MOE_ERR_INVALID_ARG;
        return MOE_ERR_UNSUPPORTED_SHAPE;
    }
    if (T < 0) return MOE_ERR_INVALID_ARG;
    if (!ws) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!x || !router_w)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(ws) || (x && !aligned16(x)) || (router_w && !aligned16(router_w)))
        return MOE_ERR_MISALIGNED;
    (void)router_bias;
    if (ws_bytes < ws_layout(*cfg, T).total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    return MOE_OK;
}

// Every host-side check of moe_forward (also run by moe_forward_static_ws
// before it touches its array): nothing is enqueued when one fails.
moe_status forward_checks(const moe_config *cfg, const uint16_t *x, const float *router_w, const float *router_bias,
                          const uint8_t *const *expert_blobs, const uint8_t *shared_blob, int32_t T, uint16_t *y,
                          float *y_f32, void *ws, size_t ws_bytes)
{
    moe_status st = check_call(cfg, x, router_w, router_bias, T, ws, ws_bytes);
    if (st != MOE_OK) return st;
    if (T > 0 && (!y || !expert_blobs)) return MOE_ERR_INVALID_ARG;
    if (cfg->shared_ff > 0 && T > 0 && !shared_blob) return MOE_ERR_INVALID_ARG;
    if ((y && !aligned16(y)) || (y_f32 && !aligned16(y_f32)) || (shared_blob && !aligned16(shared_blob)))
        return MOE_ERR_MISALIGNED;
    if (T > 0 && (cfg->flags & MOE_FLAG_FORCE_GEMV) && !use_gemv(*cfg, T)) return MOE_ERR_UNSUPPORTED_SHAPE;
    // Q5_K experts: the decode path only
    if (T > 0 && cfg->codec == MOE_CODEC_Q5K && !use_gemv(*cfg, T)) return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_q4k_bytes(int64_t rows, int64_t cols)
{
    if (rows < 0 || cols <= 0 || cols % kQK) return 0;
    return (size_t)rows * (size_t)(cols / kQK) * kQ4KBytes;
}

size_t moe_q5k_bytes(int64_t rows, int64_t cols)
{
    if (rows < 0 || cols <= 0 || cols % kQK) return 0;
    return (size_t)rows * (size_t)(cols / kQK) * kQ5KBytes;
}

size_t moe_q8_0_bytes(int64_t rows, int64_t cols)
{
    if (rows < 0 || cols <= 0 || cols % kQK8) return 0;
    return (size_t)rows * (size_t)(cols / kQK8) * kQ8Bytes;
}

size_t moe_expert_bytes(const moe_config *cfg)
{
    if (!cfg_valid(cfg)) return 0;
    return 3 * (cfg->codec == MOE_CODEC_Q5K ? moe_q5k_bytes(cfg->ff, cfg->hidden) : moe_q4k_bytes(cfg->ff, cfg->hidden));
}

size_t moe_shared_bytes(const moe_config *cfg)
{
    if (!cfg_valid(cfg) || cfg->shared_ff == 0) return 0;
    return 3 * moe_q8_0_bytes(cfg->shared_ff, cfg->hidden);
}

moe_status moe_pack_q4k(const float *w, int64_t rows, int64_t cols, uint8_t *out, uint32_t *dev_status,
                        moe_stream_t stream)
{
    if (rows < 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
    if (cols % kQK) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!w || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(out)) return MOE_ERR_MISALIGNED;
    return cuda_status(launch_pack_q4k(w, rows * (cols / kQK), out, dev_status, (cudaStream_t)stream));
}

moe_status moe_pack_q5k(const float *w, int64_t rows, int64_t cols, uint8_t *out, uint32_t *dev_status,
                        moe_stream_t stream)
{
    if (rows < 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
    if (cols % kQK) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!w || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(out)) return MOE_ERR_MISALIGNED;
    return cuda_status(launch_pack_q5k(w, rows * (cols / kQK), out, dev_status, (cudaStream_t)stream));
}

moe_status moe_pack_q8_0(const float *w, int64_t rows, int64_t cols, uint8_t *out, uint32_t *dev_status,
                         moe_stream_t stream)
{
    if (rows < 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
    if (cols % kQK8) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!w || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(out)) return MOE_ERR_MISALIGNED;
    return cuda_status(launch_pack_q8_0(w, rows * (cols / kQK8), out, dev_status, (cudaStream_t)stream));
}

moe_status moe_dequant_q4k(const uint8_t *blocks, int64_t rows, int64_t cols, float *out, moe_stream_t stream)
{
    if (rows < 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
    if (cols % kQK) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!blocks || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(blocks) || !aligned16(out)) return MOE_ERR_MISALIGNED;
    return cuda_status(launch_dequant_q4k(blocks, rows * (cols / kQK), out, (cudaStream_t)stream));
}

moe_status moe_dequant_q5k(const uint8_t *blocks, int64_t rows, int64_t cols, float *out, moe_stream_t stream)
{
    if (rows < 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
    if (cols % kQK) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!blocks || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(blocks) || !aligned16(out)) return MOE_ERR_MISALIGNED;
    return cuda_status(launch_dequant_q5k(blocks, rows * (cols / kQK), out, (cudaStream_t)stream));
}

moe_status moe_dequant_q5k_f16(const uint8_t *blocks, int64_t rows, int64_t cols, uint16_t *out, moe_stream_t stream)
{
    if (rows < 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
    if (cols % kQK) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!blocks || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(blocks) || !aligned16(out)) return MOE_ERR_MISALIGNED;
    return cuda_status(launch_dequant_q5k_f16(blocks, rows * (cols / kQK), out, (cudaStream_t)stream));
}

moe_status moe_dequant_q8_0(const uint8_t *blocks, int64_t rows, int64_t cols, float *out, moe_stream_t stream)
{
    if (rows < 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
    if (cols % kQK8) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!blocks || !out) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_dequant_q8_0(blocks, rows * (cols / kQK8), out, (cudaStream_t)stream));
}

moe_status moe_dequant_q4k_f16(const uint8_t *blocks, int64_t rows, int64_t cols, uint16_t *out, moe_stream_t stream)
{
    if (rows < 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
    if (cols % kQK) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!blocks || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(blocks) || !aligned16(out)) return MOE_ERR_MISALIGNED;
    return cuda_status(launch_dequant_q4k_f16(blocks, rows * (cols / kQK), out, (cudaStream_t)stream));
}

moe_status moe_dequant_q8_0_f16(const uint8_t *blocks, int64_t rows, int64_t cols, uint16_t *out,
                                moe_stream_t stream)
{
    if (rows < 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
    if (cols % kQK8) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!blocks || !out) return MOE_ERR_INVALID_ARG;
    if (((uintptr_t)out & 3u) != 0) return MOE_ERR_MISALIGNED;
    return cuda_status(launch_dequant_q8_0_f16(blocks, rows * (cols / kQK8), out, (cudaStream_t)stream));
}

size_t moe_workspace_bytes(const moe_config *cfg, int32_t max_tokens)
{
    if (!cfg_valid(cfg) || max_tokens < 0) return 0;
    return ws_layout(*cfg, max_tokens).total;
}

moe_status moe_workspace_init(void *ws, size_t ws_bytes, moe_stream_t stream)
{
    if (!ws || ws_bytes < (size_t)kHeaderBytes) return MOE_ERR_INVALID_ARG;
    return cuda_status(cudaMemsetAsync(ws, 0, kHeaderBytes, (cudaStream_t)stream));
}


static RouteArgs route_args(const moe_config *cfg, const uint16_t *x, const float *router_w,
                            const float *router_bias, int32_t T, void *ws)
{
    const WsLayout L = ws_layout(*cfg, T);
    char *base = (char *)ws;
    RouteArgs r{};
    r.H = cfg->hidden;
    r.E = cfg->n_experts;
    r.k = cfg->top_k;
    r.T = T;
    r.score_fn = cfg->score_fn;
    r.x = x;
    r.wr = router_w;
    r.bias = router_bias;
    r.logits = (float *)(base + L.logits);
    r.ids = (int32_t *)(base + L.ids);
    r.w = (float *)(base + L.w);
    r.counts = (int32_t *)(base + L.counts);
    r.offsets = (int32_t *)(base + L.offsets);
    r.assign = (int32_t *)(base + L.assign);
    r.active = (int32_t *)(base + L.active);
    r.bhist = (int32_t *)(base + L.bhist);
    r.wsplit = (uint16_t *)(base + L.wsplit);
    r.header = (uint32_t *)(base + L.header);
    return r;
}

moe_status moe_route(const moe_config *cfg, const uint16_t *x, const float *router_w,
                     const float *router_bias, int32_t T, int32_t *topk_ids, float *topk_w,
                     int32_t *expert_offsets, int32_t *assign, void *ws, size_t ws_bytes,
                     moe_stream_t stream)
{
    moe_status st = check_call(cfg, x, router_w, router_bias, T, ws, ws_bytes);
    if (st != MOE_OK) return st;
    if (!expert_offsets || (T > 0 && (!topk_ids || !topk_w || !assign))) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    RouteArgs r = route_args(cfg, x, router_w, router_bias, T, ws);
    cudaError_t e = launch_route(r, s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    const size_t TK = (size_t)T * cfg->top_k;
    if (TK) {
        e = cudaMemcpyAsync(topk_ids, r.ids, TK * 4, cudaMemcpyDeviceToDevice, s);
        if (e == cudaSuccess) e = cudaMemcpyAsync(topk_w, r.w, TK * 4, cudaMemcpyDeviceToDevice, s);
        if (e == cudaSuccess) e = cudaMemcpyAsync(assign, r.assign, TK * 4, cudaMemcpyDeviceToDevice, s);
    }
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(expert_offsets, r.offsets, (cfg->n_experts + 1) * 4, cudaMemcpyDeviceToDevice, s);
    return cuda_status(e);
}


moe_status moe_forward_stack(const moe_config *cfg, int32_t n_layers, uint16_t *x, const float *const *router_w,
                             const float *const *router_bias, const uint8_t *const *expert_blobs,
                             const uint8_t *const *shared_blobs, int32_t T, uint16_t *y, float *y_f32, void *ws,
                             size_t ws_bytes, moe_stream_t stream)
{
    if (n_layers < 0 || T < 0) return MOE_ERR_INVALID_ARG;
    // configuration, workspace and x as for one layer call (the router matrices come from a table here)
    moe_status st = check_call(cfg, x, nullptr, nullptr, 0, ws, ws_bytes);
    if (st != MOE_OK) return st;
    if (n_layers == 0 || T == 0) return MOE_OK;
    if (!x || !router_w || !y || !expert_blobs || (cfg->shared_ff > 0 && !shared_blobs)) return MOE_ERR_INVALID_ARG;
    auto al8 = [](const void *p) { return ((uintptr_t)p & 7u) == 0; };
    if (!aligned16(y) || (y_f32 && !aligned16(y_f32)) || !al8(router_w) || !al8(expert_blobs) ||
        (router_bias && !al8(router_bias)) || (shared_blobs && !al8(shared_blobs)))
        return MOE_ERR_MISALIGNED;
    if (!use_gemv(*cfg, T) || !stack_supported(*cfg, T)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (ws_bytes < ws_layout(*cfg, T).total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    const WsLayout L = ws_layout(*cfg, T);
    char *base = (char *)ws;
    RouteArgs r = route_args(cfg, x, nullptr, nullptr, T, ws);
    StackArgs a{};
    DecArgs &d = a.d;
    d.H = cfg->hidden;
    d.E = cfg->n_experts;
    d.FF = cfg->ff;
    d.k = cfg->top_k;
    d.T = T;
    d.SFF = cfg->shared_ff;
    d.score_fn = cfg->score_fn;
    d.route_parts = dec_route_parts(cfg->hidden);
    d.nc = dec_consumers(*cfg);
    d.half = dec_half(*cfg) ? 1 : 0;
    d.codec = cfg->codec;
    d.ring_bytes = dec_ring_bytes(*cfg, T);
    d.stages = dec_stages(*cfg, T);
    d.wait_cycles = debug_wait_cycles();
    d.skip_cta = debug_take_skip_copy();
    d.logits = r.logits;
    d.ids = r.ids;
    d.w = r.w;
    d.counts = r.counts;
    d.offsets = r.offsets;
    d.assign = r.assign;
    d.active = r.active;
    d.header = r.header;
    a.L = n_layers;
    a.residual = (cfg->flags & MOE_FLAG_RESIDUAL) != 0;
    a.rows = (cfg->n_experts + stack_grid() - 1) / stack_grid();
    a.wr = router_w;
    a.bias = cfg->score_fn == MOE_SCORE_SIGMOID_BIAS ? router_bias : nullptr;
    a.blobs = expert_blobs;
    a.shared = cfg->shared_ff > 0 ? shared_blobs : nullptr;
    a.x = x;
    a.y = y;
    a.y_f32 = y_f32;
    a.yacc = (float *)(base + L.yacc);
    return cuda_status(launch_stack(a, (cudaStream_t)stream));
}

moe_status moe_forward(const moe_config *cfg, const uint16_t *x, const float *router_w,
                       const float *router_bias, const uint8_t *const *expert_blobs,
                       const uint8_t *shared_blob, int32_t T, uint16_t *y, float *y_f32, void *ws,
                       size_t ws_bytes, moe_stream_t stream)
{
    moe_status st = forward_checks(cfg, x, router_w, router_bias, expert_blobs, shared_blob, T, y, y_f32, ws, ws_bytes);
    if (st != MOE_OK) return st;
    if (T == 0) return MOE_OK;
    cudaStream_t s = (cudaStream_t)stream;
    const WsLayout L = ws_layout(*cfg, T);
    char *base = (char *)ws;
    RouteArgs r = route_args(cfg, x, router_w, router_bias, T, ws);
    if (use_gemv(*cfg, T)) {
        DecArgs d{};
        d.H = cfg->hidden;
        d.E = cfg->n_experts;
        d.FF = cfg->ff;
        d.k = cfg->top_k;
        d.T = T;
        d.SFF = cfg->shared_ff;
        d.score_fn = cfg->score_fn;
        d.route_parts = dec_route_parts(cfg->hidden);
        d.nc = dec_consumers(*cfg);
        d.half = dec_half(*cfg) ? 1 : 0;
        d.codec = cfg->codec;
        d.ring_bytes = dec_ring_bytes(*cfg, T);
        d.stages = dec_stages(*cfg, T);
        d.overlap_prev = (cfg->flags & MOE_FLAG_STATIC_WEIGHTS) != 0;
        d.wait_cycles = debug_wait_cycles();
        d.skip_cta = debug_take_skip_copy();
        d.x = x;
        d.wr = router_w;
        d.bias = cfg->score_fn == MOE_SCORE_SIGMOID_BIAS ? router_bias : nullptr;
        d.blobs = expert_blobs;
        d.shared_blob = cfg->shared_ff > 0 ? shared_blob : nullptr;
        d.logits = r.logits;
        d.xfrag = (uint2 *)(base + L.xfrag);
        d.ids = r.ids;
        d.w = r.w;
        d.counts = r.counts;
        d.offsets = r.offsets;
        d.assign = r.assign;
        d.active = r.active;
        d.yacc = (float *)(base + L.yacc);
        d.y = y;
        d.y_f32 = y_f32;
        d.header = r.header;
        return cuda_status(launch_decode(d, s));
    }
    cudaError_t e = launch_route(r, s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;

    ExpertArgs a{};
    a.H = cfg->hidden;
    a.E = cfg->n_experts;
    a.FF = cfg->ff;
    a.k = cfg->top_k;
    a.T = T;
    a.SFF = cfg->shared_ff;
    a.x = x;
    a.blobs = expert_blobs;
    a.shared_blob = cfg->shared_ff > 0 ? shared_blob : nullptr;
    a.offsets = r.offsets;
    a.assign = r.assign;
    a.active = r.active;
    a.w = r.w;
    a.slots = (float *)(base + L.slots);
    a.sh_out = cfg->shared_ff ? (float *)(base + L.sh_out) : nullptr;
    a.y = y;
    a.y_f32 = y_f32;
    a.header = r.header;
    a.wait_cycles = debug_wait_cycles();
    a.skip_cta = debug_take_skip_copy();
    {
        GemmWs gw{};
        gw.xg = (__half *)(base + L.xg);
        gw.x16 = (__half *)(base + L.x16);
        gw.act16 = (__half *)(base + L.act16);
        gw.sh_act16 = (__half *)(base + L.sh_act16);
        gw.yacc = (float *)(base + L.yacc);
        gw.tiles_gu = (int4 *)(base + L.tiles_gu);
        gw.tiles_dn = (int4 *)(base + L.tiles_dn);
        gw.tiles_gus = (int4 *)(base + L.tiles_gus);
        gw.tiles_dns = (int4 *)(base + L.tiles_dns);
        gw.tmaps = base + L.tmaps;
        gw.splits = gemm_splits(*cfg, T);
        gw.gu = (float *)(base + L.gu);
        gw.sh_gu = (float *)(base + L.sh_gu);
        gw.n_gu = gw.splits.gu > 1 || gw.splits.gus > 1 ? (int64_t)((L.split_cnt - L.gu) / 4) : 0;
        gw.split_cnt = (uint32_t *)(base + L.split_cnt);
        gw.n_cnt_routed = gw.splits.gu > 1 ? (int64_t)gemm_tile_capacity(cfg->ff / 64, (int64_t)T * cfg->top_k,
                                                                             cfg->n_experts)
                                           : 0;
        gw.n_cnt = (int64_t)((L.total - L.split_cnt) / 4);
        gw.det = (cfg->flags & MOE_FLAG_DETERMINISTIC) != 0;
        e = launch_experts_gemm(a, gw, s);
    }
    return cuda_status(e);
}

moe_status moe_workspace_routing(const moe_config *cfg, int32_t T, const void *ws, size_t ws_bytes,
                                 const int32_t **ids, const float **w, const int32_t **offsets,
                                 const int32_t **assign)
{
    if (!cfg_valid(cfg) || !ws || T < 0) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(*cfg, T);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    const char *base = (const char *)ws;
    if (ids) *ids = (const int32_t *)(base + L.ids);
    if (w) *w = (const float *)(base + L.w);
    if (offsets) *offsets = (const int32_t *)(base + L.offsets);
    if (assign) *assign = (const int32_t *)(base + L.assign);
    return MOE_OK;
}

moe_status moe_last_device_status(void *ws, moe_stream_t stream)
{
    if (!ws) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (v != 0) {
        e = cudaMemsetAsync(ws, 0, sizeof(uint32_t), s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    return (moe_status)v;
}

moe_status moe_debug_set(int32_t what, int64_t value)
{
    switch (what) {
    case MOE_DEBUG_WAIT_CYCLES:
        if (value < 0) return MOE_ERR_INVALID_ARG;
        g_wait_cycles.store(value == 0 ? kDefaultWaitCycles : (long long)value);
        return MOE_OK;
    case MOE_DEBUG_SKIP_COPY:
        if (value < -1 || value > (1 << 20)) return MOE_ERR_INVALID_ARG;
        g_skip_copy.store((int)value);
        return MOE_OK;
    case MOE_DEBUG_SKIP_ROUTER:
        if (value < -1 || value > (1 << 20)) return MOE_ERR_INVALID_ARG;
        g_skip_router.store((int)value);
        return MOE_OK;
    }
    return MOE_ERR_INVALID_ARG;
}

const char *moe_status_string(moe_status status)
{
    switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_DEVICE_FAULT: return "device found invalid data";
    }
    return "unknown status";
}

}  // extern "C"
