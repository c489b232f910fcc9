/*
 * moe.h -- C ABI of the single-GPU (B300, sm_103a) sparse mixture-of-experts
 * layer over Q4_K block-quantised experts.
 *
 * The layer (pages cited by title and section):
 *   "Strata 改源码去跑 DeepSeek V4 Flash？要不就试试！" (lcz.me/post/23082),
 *     section 二 (GGUF anatomy table): routed experts are the fused tensors
 *     ffn_{gate,up,down}_exps in Q4_K; the always-on shared expert is Q8_0;
 *     256 routed experts, 6 active, "router bias" on most layers.
 *     section 三 item 4: one expert is a 1,382,400-byte blob at width 2560.
 *   "Strata 引擎深度拆解：125B MoE 跑进 2×3090 + EPYC" (lcz.me/topic/2098/5),
 *     section 二: 48 layers x 512 experts, ~10 active per token, MTP verify
 *     windows of 3-5 tokens run as one forward; section 一 (CPU ledger): the
 *     multi-token expert kernel reads an expert's bytes once per window.
 *   "Qwen3.8-Flash-Next UD-Q4_K_XL 引擎对比：llama.cpp 与 Strata"
 *     (lcz.me/user/wml-ai/posts), section 一 (部署): Q4_K expert prompt
 *     (prefill) kernels.
 *
 * For each token t with hidden state x_t (bf16, length H):
 *   1. router logits l_e = sum_h x_t[h] * Wr[e][h]                 (Wr fp32 [E][H])
 *   2. scores: softmax p = softmax(l), or sigmoid s_e = 1/(1+exp(-l_e));
 *      the k experts with the largest p (softmax) or s_e + b_e (sigmoid with
 *      per-expert bias b) are selected, largest first, equal scores to the
 *      lower id; weights w_r = p_{e_r} / sum_sel p  or  s_{e_r} / sum_sel s.
 *   3. bucketing: stable counting sort of the T*k assignments a = t*k + r by
 *      expert id -> expert_offsets[E+1], assign[T*k] (ascending t in an expert).
 *   4. per assignment: g = Wg x_t, u = Wu x_t, a = SiLU(g) * u   (Wg, Wu [FF][H])
 *   5. o = sum_f a_f * Wd[f][:]   (Wd stored [FF][H], super-blocks along H)
 *   6. y_t = sum_r w_r * o_{t,r} (+ the shared expert's FFN of x_t, weight 1).
 *
 * Data formats (the pages name Q4_K and Q8_0 but print no layout; the GGUF
 * layouts are used):
 *   Q4_K  144 bytes per 256 weights along a row: fp16 d, fp16 dmin,
 *         12 bytes of packed 6-bit sub-block scales/mins, 128 bytes of 4-bit
 *         quants; weight = (d*sc_j)*q - dmin*m_j.
 *   Q8_0  34 bytes per 32 weights: fp16 d then 32 int8; weight = d*q.
 *   Expert blob  [gate FF x H][up FF x H][down FF x H], each row-major with
 *         its blocks along H: 3*FF*(H/256)*144 bytes (1,382,400 at H=2560,
 *         FF=320).  The shared blob has the same order in Q8_0.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers unless stated otherwise; the
 *     caller owns every buffer.  The library never allocates device memory
 *     and never synchronises the stream, except moe_last_device_status().
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default).
 *   - Arguments are checked on the host before anything is launched; a
 *     failing check returns its status and enqueues nothing.
 *   - Faults found on the device (non-finite pack input, router id out of
 *     range, a bounded wait that gave up) are recorded in a status word
 *     and read with moe_last_device_status() (pack calls take their own
 *     status word).  Nothing traps and nothing throws.
 *   - Calls sharing one workspace must not overlap on the device (same
 *     stream, or ordered by events); distinct workspaces are independent.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

/* == cudaStream_t */
typedef struct CUstream_st *moe_stream_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,         /* null pointer, negative size, bad enum value      */
    MOE_ERR_UNSUPPORTED_SHAPE = 2,   /* a shape the kernels do not handle (see moe_config) */
    MOE_ERR_MISALIGNED = 3,          /* a pointer that must be 16-byte aligned is not    */
    MOE_ERR_WORKSPACE_TOO_SMALL = 4, /* ws_bytes < moe_workspace_bytes(cfg, T)           */
    MOE_ERR_CUDA = 5,                /* a CUDA runtime call or launch failed             */
    MOE_ERR_TIMEOUT = 6,             /* a device-side bounded wait gave up               */
    MOE_ERR_DEVICE_FAULT = 7         /* the device found invalid data (non-finite input,
                                        an expert id out of range, a null expert blob)   */
} moe_status;

typedef enum {
    MOE_SCORE_SOFTMAX = 0,           /* softmax over all E logits, renormalised over k   */
    MOE_SCORE_SIGMOID_BIAS = 1       /* sigmoid scores; selection by score + bias        */
} moe_score_fn;

enum {
    MOE_FLAG_DETERMINISTIC = 1,      /* combine through per-assignment slots in a fixed
                                        order on every path (bit-identical reruns)        */
    MOE_FLAG_FORCE_GEMV = 2,         /* use the decode (grouped GEMV) path; T <= 8 only  */
    MOE_FLAG_FORCE_GEMM = 4,         /* use the prefill (tensor-core GEMM) path at any T */
    MOE_FLAG_STATIC_WEIGHTS = 8,     /* the caller guarantees that router_w, router_bias,
                                        the expert table and the expert blobs are not
                                        written by the work enqueued just before this call
                                        on the stream: a decode call may then start
                                        reading the router rows and the expert table
                                        while that work is still running (its other
                                        inputs are read only after it has finished)     */
    MOE_FLAG_RESIDUAL = 16           /* moe_forward_stack: the layers' inputs form a
                                        residual stream (see there)                      */
};

/* Block format of the routed experts (the shared expert is always Q8_0).
 * Q5_K experts run on the decode path only (T <= 8): a call that would take
 * the tensor-core path returns MOE_ERR_UNSUPPORTED_SHAPE. */
typedef enum {
    MOE_CODEC_Q4K = 0,               /* 144 bytes per 256 weights (4-bit)                */
    MOE_CODEC_Q5K = 1                /* 176 bytes per 256 weights (5-bit, fifth bits in qh) */
} moe_codec;

/*
 * Layer shape.  Limits: hidden % 256 == 0 and 256 <= hidden <= 8192;
 * 1 <= n_experts <= 1024; ff % 64 == 0 and 64 <= ff <= 8192;
 * 1 <= top_k <= min(n_experts, 32); shared_ff == 0 (no shared expert) or
 * shared_ff % 64 == 0 and <= 8192.
 */
typedef struct {
    int32_t hidden;      /* H                                   */
    int32_t n_experts;   /* E routed experts                    */
    int32_t ff;          /* expert intermediate width FF        */
    int32_t top_k;       /* k experts per token                 */
    int32_t score_fn;    /* moe_score_fn                        */
    int32_t shared_ff;   /* shared expert width, 0 = none       */
    int32_t flags;       /* MOE_FLAG_*                          */
    int32_t codec;       /* routed experts' blocks: moe_codec   */
} moe_config;

/* ---------------------------------------------------------------- sizes */

/* Bytes of a [rows][cols] matrix in Q4_K (cols % 256 == 0): rows*cols/256*144.
 * Returns 0 for an invalid shape. */
MOE_API size_t moe_q4k_bytes(int64_t rows, int64_t cols);
/* Bytes of a [rows][cols] matrix in Q5_K (cols % 256 == 0): rows*cols/256*176. */
MOE_API size_t moe_q5k_bytes(int64_t rows, int64_t cols);
/* Bytes of a [rows][cols] matrix in Q8_0 (cols % 32 == 0): rows*cols/32*34. */
MOE_API size_t moe_q8_0_bytes(int64_t rows, int64_t cols);
/* Bytes of one routed-expert blob, 3*moe_q4k_bytes(ff, hidden) (Q5_K:
 * 3*moe_q5k_bytes); 0 if cfg invalid. */
MOE_API size_t moe_expert_bytes(const moe_config *cfg);
/* Bytes of the shared-expert blob, 3*moe_q8_0_bytes(shared_ff, hidden); 0 if none. */
MOE_API size_t moe_shared_bytes(const moe_config *cfg);

/* ---------------------------------------------------------------- packing */

/*
 * Quantise a row-major fp32 matrix w[rows][cols] (device) to Q4_K, written
 * to out (device, moe_q4k_bytes(rows, cols) bytes, 16-byte aligned).  The
 * quantiser is deterministic (fp32 IEEE, round half to even) and gives the
 * same bytes as its definition everywhere:
 *   per 32-weight sub-block: mn = min(0, min x), mx = max x,
 *     scale_j = (mx - mn)/15, nmin_j = -mn;
 *   d = fp16(max_j scale_j / 63), dmin = fp16(max_j nmin_j / 63);
 *   sc_j = d > 0 ? min(63, rint(scale_j / d)) : 0  (m_j alike with dmin);
 *   q = d*sc_j > 0 ? clamp(rint((x + dmin*m_j) / (d*sc_j)), 0, 15) : 0.
 * Non-finite input, or a d / dmin that overflows fp16, sets *dev_status
 * (device uint32, may be NULL) to MOE_ERR_DEVICE_FAULT; the block is still
 * written.  Errors: INVALID_ARG (null, rows < 0), UNSUPPORTED_SHAPE
 * (cols % 256), MISALIGNED (out or w not 16-byte aligned), CUDA.
 */
MOE_API moe_status moe_pack_q4k(const float *w, int64_t rows, int64_t cols, uint8_t *out,
                        uint32_t *dev_status, moe_stream_t stream);

/*
 * Quantise w[rows][cols] (device fp32) to Q5_K blocks (GGUF layout: fp16 d,
 * fp16 dmin, scales[12] packed as Q4_K's, qh[32], qs[128]; the quant of
 * element 64c + 32h + l keeps its low four bits in the low (h = 0) or high
 * (h = 1) nibble of qs[32c + l] and its fifth bit in bit 2c + h of qh[l]).
 * The quantiser is moe_pack_q4k's with 31 levels: scale_j = (mx - mn)/31 and
 * q clamped to 0..31.  out gets moe_q5k_bytes(rows, cols) bytes; errors as
 * moe_pack_q4k.
 */
MOE_API moe_status moe_pack_q5k(const float *w, int64_t rows, int64_t cols, uint8_t *out,
                        uint32_t *dev_status, moe_stream_t stream);

/*
 * Quantise w[rows][cols] (device fp32) to Q8_0: d = fp16(max|x|/127),
 * q = d > 0 ? clamp(rint(x/d), -127, 127) : 0.  cols % 32 == 0; out gets
 * moe_q8_0_bytes(rows, cols) bytes.  cols*34/32 must be a multiple of 16 for
 * rows to stay 16-byte aligned (cols % 256 == 0 always satisfies it); errors
 * as moe_pack_q4k.
 */
MOE_API moe_status moe_pack_q8_0(const float *w, int64_t rows, int64_t cols, uint8_t *out,
                         uint32_t *dev_status, moe_stream_t stream);

/* Test hooks: dequantise a Q4_K / Q5_K / Q8_0 matrix to fp32
 * out[rows][cols] (device).  Bit-exact with the format definition (each
 * product and the difference rounded to fp32 separately). */
MOE_API moe_status moe_dequant_q4k(const uint8_t *blocks, int64_t rows, int64_t cols, float *out,
                           moe_stream_t stream);
MOE_API moe_status moe_dequant_q5k(const uint8_t *blocks, int64_t rows, int64_t cols, float *out,
                           moe_stream_t stream);
MOE_API moe_status moe_dequant_q8_0(const uint8_t *blocks, int64_t rows, int64_t cols, float *out,
                            moe_stream_t stream);

/* Test hooks of the tensor-core operand rounding: the fp16 weights that the
 * fused decode and prefill kernels multiply, produced by the same device
 * functions those kernels call, as binary16 bit patterns out[rows][cols]
 * (device).  Q4_K: S_j = fp16(d*sc_j), NZ_j = fp16(-(dmin*m_j)),
 * w = fp16(q*S_j + NZ_j) rounded once; Q8_0: w = fp16(d*q).  The pages fix no
 * precision; this rounding is the library's (see moe_forward).  Errors as
 * moe_dequant_q4k (Q8_0: out 4-byte aligned). */
MOE_API moe_status moe_dequant_q5k_f16(const uint8_t *blocks, int64_t rows, int64_t cols, uint16_t *out,
                               moe_stream_t stream);   /* Q5_K: as Q4_K, q in 0..31 */
MOE_API moe_status moe_dequant_q4k_f16(const uint8_t *blocks, int64_t rows, int64_t cols, uint16_t *out,
                               moe_stream_t stream);
MOE_API moe_status moe_dequant_q8_0_f16(const uint8_t *blocks, int64_t rows, int64_t cols, uint16_t *out,
                                moe_stream_t stream);

/* ---------------------------------------------------------------- workspace */

/*
 * Device workspace bytes for calls with up to max_tokens tokens (0 if cfg is
 * invalid).  The workspace holds routing results, intermediate activations,
 * accumulators and the device status word.  Before its first use, a
 * workspace must be initialised with moe_workspace_init (it zeroes the
 * 256-byte header that holds the status word and the completion counters).
 */
MOE_API size_t moe_workspace_bytes(const moe_config *cfg, int32_t max_tokens);
MOE_API moe_status moe_workspace_init(void *ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------- the layer */

/*
 * Steps 1-3 only.  x: bf16 [T][H] (16-byte aligned); router_w: fp32 [E][H];
 * router_bias: fp32 [E] (required for MOE_SCORE_SIGMOID_BIAS, may be NULL
 * there to mean zero; ignored for softmax).  Outputs (device): topk_ids
 * int32 [T][k], topk_w fp32 [T][k], expert_offsets int32 [E+1],
 * assign int32 [T*k].  T may be 0 (offsets become all zero).
 */
MOE_API moe_status moe_route(const moe_config *cfg, const uint16_t *x, const float *router_w,
                     const float *router_bias, int32_t T, int32_t *topk_ids, float *topk_w,
                     int32_t *expert_offsets, int32_t *assign, void *ws, size_t ws_bytes,
                     moe_stream_t stream);

/*
 * The whole layer.  expert_blobs: DEVICE array of E device pointers, each to
 * a 16-byte aligned expert blob (moe_expert_bytes); an expert that no token
 * selects may be NULL.  shared_blob: the shared expert's blob
 * (moe_shared_bytes) when cfg->shared_ff > 0, else ignored.  Output y:
 * bf16 [T][H]; y_f32: optional fp32 [T][H] copy before rounding (may be NULL).
 * The routing of the call stays readable in the workspace
 * (moe_workspace_routing) until the next call.
 * Path: T <= 8 (or MOE_FLAG_FORCE_GEMV) runs the decode path: each selected
 * expert's bytes are streamed once per window; both projections multiply
 * fp16 dequantised weights by fp16 operands (x; the weighted activations
 * w * SiLU(g) * u) with fp32 accumulation (warp MMAs).  Larger T runs the
 * tensor-core grouped GEMM with fp16 operands and fp32 accumulation.  Both
 * paths need |x| < 65504 (fp16 range; larger values set MOE_ERR_DEVICE_FAULT)
 * and an fp16-representable activation (a larger one sets
 * MOE_ERR_DEVICE_FAULT).  On the decode path an expert blob may live in
 * pinned, mapped host memory (its device-usable address in the table): the
 * kernels then read it from there (see the expert cache below); the
 * tensor-core path needs every blob in device memory.
 */
MOE_API moe_status moe_forward(const moe_config *cfg, const uint16_t *x, const float *router_w,
                       const float *router_bias, const uint8_t *const *expert_blobs,
                       const uint8_t *shared_blob, int32_t T, uint16_t *y, float *y_f32,
                       void *ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Device pointers, inside ws, to the routing of the last moe_forward with
 * this workspace and T tokens: ids [T][k], w [T][k], offsets [E+1],
 * assign [T*k].  Any out pointer may be NULL.  No device work.
 */
MOE_API moe_status moe_workspace_routing(const moe_config *cfg, int32_t T, const void *ws, size_t ws_bytes,
                                 const int32_t **ids, const float **w, const int32_t **offsets,
                                 const int32_t **assign);

/*
 * Synchronises `stream`, then returns the first device-side fault recorded
 * in the workspace's status word since the last call of this function
 * (MOE_OK if none) and clears it.
 */
MOE_API moe_status moe_last_device_status(void *ws, moe_stream_t stream);

/* ---------------------------------------------------------------- host tier of the experts */

/*
 * A device cache of expert blobs over pinned host memory: every expert has a
 * copy in pinned, mapped host memory, a part of them also in device slots.
 * Host-side bookkeeping only; the copies are cudaMemcpyAsync on a stream the
 * caller names.  One cache serves one table of n_experts entries (a layer, or
 * the experts of several layers numbered as the caller likes).  Not
 * thread-safe.
 *
 * moe_cache_create: host_blobs is a HOST array of n_experts device-usable
 * addresses (cudaHostAlloc(..., cudaHostAllocMapped) + cudaHostGetDevicePointer),
 * each 16-byte aligned and blob_bytes long; slot_memory is DEVICE memory of
 * n_slots * blob_bytes bytes (16-byte aligned; n_slots may be 0).  The caller
 * owns both and keeps them alive until moe_cache_destroy.
 * Errors: MOE_ERR_INVALID_ARG (null or non-positive arguments),
 * MOE_ERR_MISALIGNED.
 */
typedef struct moe_cache moe_cache;
MOE_API moe_status moe_cache_create(int32_t n_experts, int64_t blob_bytes, const uint8_t *const *host_blobs,
                                    uint8_t *slot_memory, int32_t n_slots, moe_cache **out);
/* Frees the bookkeeping (not the memory the caller owns).  NULL is a no-op. */
MOE_API void moe_cache_destroy(moe_cache *cache);
/*
 * Host only, no CUDA call.  ids: HOST array of the window's selected expert
 * ids (any order, repeats allowed).  Marks them used and gives each missed
 * expert a slot -- a free one, or the least recently used slot whose expert
 * this window does not select -- with a fill planned for moe_cache_issue.
 * Writes the HOST array table[n_experts] (to be copied to the device table
 * moe_forward reads): the slot address of every expert that has a slot
 * (resident, or filled by this window's moe_cache_issue), else its host
 * address (a missed expert that found no slot is read from host memory by
 * the decode kernels).  *n_fills (may be NULL) = fills planned.
 * Errors: MOE_ERR_INVALID_ARG (null pointers, an id out of range).
 */
MOE_API moe_status moe_cache_plan(moe_cache *cache, const int32_t *ids, int32_t n_ids, const uint8_t **table,
                                  int32_t *n_fills);
/*
 * Queues the planned fills on copy_stream (one cudaMemcpyAsync per expert
 * blob) behind the work queued so far on compute_stream -- a refilled slot may
 * still be read by a queued kernel -- and makes compute_stream wait for them:
 * call it after moe_cache_plan and before queueing the window's moe_forward
 * on compute_stream.  Errors: MOE_ERR_CUDA (the window's fills are then
 * dropped: do not run the window with that plan's table).
 */
MOE_API moe_status moe_cache_issue(moe_cache *cache, moe_stream_t compute_stream, moe_stream_t copy_stream);
/* Kept for callers that poll: every fill is ordered by moe_cache_issue, so
 * there is nothing to collect (MOE_OK). */
MOE_API moe_status moe_cache_poll(moe_cache *cache);
/* out[4] = {hits, misses, fills issued, bytes filled} since creation. */
MOE_API moe_status moe_cache_stats(const moe_cache *cache, int64_t *out);
/* The device-usable address of pinned, mapped host memory (a CUDA call).
 * Errors: MOE_ERR_INVALID_ARG when host_ptr is not such memory. */
MOE_API moe_status moe_host_address(const void *host_ptr, const uint8_t **device_ptr);

/* ---------------------------------------------------------------- no-allocation variant */

/*
 * moe_forward for callers that cannot allocate device memory where they run
 * the layer (a runtime that only hands out pre-registered buffers, a plugin
 * inside another framework's allocator, a hot path that must not call
 * cudaMalloc).  There is no counterpart on the source pages: it is a
 * convenience of this library.
 *
 * Same arguments and results as moe_forward, without the workspace: the
 * scratch is a file-scope device array of MOE_STATIC_WS_BYTES bytes inside
 * the library, which every GPU that loads the library holds until the
 * process exits.  Calls whose moe_workspace_bytes(cfg, T) exceeds it return
 * MOE_ERR_WORKSPACE_TOO_SMALL; with the default flags 4 MiB fits decode
 * windows of up to 8 tokens of both the 2560x512x320 and the 4096x256x2048
 * + shared layer shapes (MOE_FLAG_DETERMINISTIC needs more: see
 * moe_workspace_bytes).  Nothing is allocated: no cudaMalloc, cudaFree or
 * allocating library call.
 *
 * Every argument is checked before the array is touched; a rejected call
 * enqueues nothing and leaves *dev_status as it was.  Otherwise dev_status
 * (device uint32, 4-byte aligned, may be NULL) receives the call's
 * device-side status (0 = MOE_OK, else a moe_status), as
 * moe_last_device_status reports it for an ordinary workspace; a call with
 * T == 0 writes MOE_OK there.
 *
 * Every call on a device shares the one array, which keeps the previous
 * call's contents (the call clears its header itself).  Calls that overlap on
 * the GPU -- different streams without ordering, or several host threads --
 * race on it: order them.  The first call on each device looks up the
 * array's device address (cudaGetSymbolAddress, with that device current)
 * and keeps it for the life of the process; make that first call before any
 * stream capture, and do not call cudaDeviceReset on a device after it (the
 * kept address would then be stale).
 */
#define MOE_STATIC_WS_BYTES (4u << 20)
MOE_API moe_status moe_forward_static_ws(const moe_config *cfg, const uint16_t *x, const float *router_w,
                                         const float *router_bias, const uint8_t *const *expert_blobs,
                                         const uint8_t *shared_blob, int32_t T, uint16_t *y, float *y_f32,
                                         uint32_t *dev_status, moe_stream_t stream);

/* ---------------------------------------------------------------- layer stack */

/*
 * One decode window through a stack of n_layers MoE layers in one launch:
 * every layer computes what moe_forward computes on the decode path, with
 * its own router, experts and shared expert, and the layers run in order --
 * layer l + 1 reads its input only once y of layer l is complete.  One
 * persistent CTA per SM (a cooperative launch: the call fails with
 * MOE_ERR_CUDA if the GPU cannot hold them all at once) takes the layers one
 * after the other with two grid-wide barriers each, instead of two kernels
 * per layer.  The barriers' waits are bounded (MOE_ERR_TIMEOUT, see
 * moe_debug_set).  This follows the verify-window forward of the teardown page
 * ("Strata 引擎深度拆解", lcz.me/topic/2098/5, section 二 item 1: the 3-5
 * drafted tokens verified in one forward; item 2: a window crosses the layer
 * stack with one hand-off between the halves of the stack).
 *
 *   x      device bf16 [n_layers][T][hidden].  Without MOE_FLAG_RESIDUAL
 *          every x[l] is an input.  With it only x[0] is read, and the call
 *          writes the residual stream x[l + 1] = bf16(x[l] + y[l]) (the fp32
 *          sum of the two bf16 values, rounded to nearest even once) for
 *          l + 1 < n_layers.
 *   router_w      device array of n_layers device pointers, each to a
 *                 16-byte aligned [E][H] fp32 matrix.
 *   router_bias   device array of n_layers pointers ([E] fp32), or NULL; read
 *                 for MOE_SCORE_SIGMOID_BIAS only.
 *   expert_blobs  device array [n_layers][n_experts] of blob pointers (as
 *                 moe_forward's, layer after layer; blobs in device memory).
 *   shared_blobs  device array of n_layers 16-byte aligned shared-expert
 *                 blobs when cfg->shared_ff > 0, else ignored.
 *   The pointer arrays themselves must be 8-byte aligned (else
 *   MOE_ERR_MISALIGNED); the pointers in them are not read on the host.
 *   y      device bf16 [n_layers][T][hidden]; y_f32 optional fp32, same shape.
 *   ws     as moe_forward's (moe_workspace_bytes(cfg, T)); its routing views
 *          hold the last layer's routing afterwards.
 * T in 1..8 with a configuration the decode path runs (not
 * MOE_FLAG_DETERMINISTIC or MOE_FLAG_FORCE_GEMM), and each CTA must hold
 * ceil(n_experts / SMs) <= 8 router rows beside its staging ring; otherwise
 * MOE_ERR_UNSUPPORTED_SHAPE.  n_layers == 0 or T == 0 is a no-op.  Host
 * checks as moe_forward; nothing is enqueued when one fails.
 */
MOE_API moe_status moe_forward_stack(const moe_config *cfg, int32_t n_layers, uint16_t *x,
                                     const float *const *router_w, const float *const *router_bias,
                                     const uint8_t *const *expert_blobs, const uint8_t *const *shared_blobs,
                                     int32_t T, uint16_t *y, float *y_f32, void *ws, size_t ws_bytes,
                                     moe_stream_t stream);

/* ---------------------------------------------------------------- diagnostics */

/*
 * Per-kernel timing for benchmarks.  While enabled, every kernel launch made
 * by moe_forward / moe_route is bracketed by two CUDA events recorded on the
 * call's stream (not while the stream is being captured into a graph), and
 * the launches are counted per kernel.  Enabling (on != 0) or disabling
 * resets the counters.  Host-global state: use from one host thread.
 */
typedef struct {
    const char *name;     /* kernel name (static string)                    */
    int64_t launches;     /* launches counted since the last reset          */
    int64_t timed;        /* launches with an event pair (<= launches)      */
    double total_ms;      /* sum of event-measured durations of those       */
} moe_profile_entry;

MOE_API moe_status moe_profile_enable(int32_t on);
/* Waits for the recorded events, fills up to max_entries entries (kernels
 * with at least one launch) and returns how many it filled. */
MOE_API int32_t moe_profile_read(moe_profile_entry *out, int32_t max_entries);

/*
 * Test hooks of the bounded device waits (host-global; use from one thread).
 *   MOE_DEBUG_WAIT_CYCLES  value > 0: every bounded wait of the kernels
 *                          launched afterwards gives up after `value` clock
 *                          cycles (0 restores the default, ~2 s).
 *   MOE_DEBUG_SKIP_COPY    value >= 0: in the next call, CTA `value` of its
 *                          main kernel never issues one bulk copy that it
 *                          waits for -- on the decode path the layer kernel's
 *                          copy of the window's x fragments and logits, on the
 *                          tensor-core path the routed gate/up kernel's first
 *                          token-row copy; in moe_forward_stack that CTA never
 *                          arrives at the first grid-wide barrier -- so that wait runs out: the call
 *                          then ends with MOE_ERR_TIMEOUT in its status word
 *                          (the context stays usable; a value past the grid
 *                          does nothing).  -1 clears it.
 *   MOE_DEBUG_SKIP_ROUTER  value >= 0: in the next call whose router logits
 *                          run on the tensor cores (more than 8 tokens,
 *                          hidden a multiple of 64), router tile `value`
 *                          (tiles of 128 tokens; index = token tile + expert
 *                          tile * token tiles) never issues the copies of its
 *                          first stage, so its MMA warp's wait runs out and
 *                          the call ends with MOE_ERR_TIMEOUT; the logits of
 *                          that tile are left unwritten.  A value past the
 *                          grid does nothing; -1 clears it.
 * Errors: MOE_ERR_INVALID_ARG for an unknown `what` or a value out of range.
 */
enum { MOE_DEBUG_WAIT_CYCLES = 1, MOE_DEBUG_SKIP_COPY = 2, MOE_DEBUG_SKIP_ROUTER = 3 };
MOE_API moe_status moe_debug_set(int32_t what, int64_t value);

/* Static string for a status code. */
MOE_API const char *moe_status_string(moe_status status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
