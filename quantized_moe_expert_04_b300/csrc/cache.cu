// cache.cu -- host tier of the experts: a device cache of expert blobs over
// pinned host memory.
//
// The teardown page ("Strata 引擎深度拆解", lcz.me/topic/2098/5, section 一, RAM
// ledger, and section 二 items 1 and 4) keeps every expert in pinned host RAM
// and only a part of them in device memory, an adaptive cache deciding which;
// the engine-compare page ("Qwen3.8-Flash-Next UD-Q4_K_XL 引擎对比", section 一,
// 部署) runs the same split.  Here the tier is device-side only: a missed expert
// is copied by the copy engine into a device slot before the window's kernels
// run (a whole blob per cudaMemcpyAsync), or, when no slot is free, read by the
// layer kernels straight from pinned, mapped host memory (its table entry
// points there).  Nothing runs on the CPU besides the bookkeeping below.
//
// Per window (see moe.h): moe_cache_plan (host only) marks the window's experts
// used, picks slots for the missed ones -- evicting the least recently used
// experts the window does not need -- and writes the pointer table (slot
// address, or host address for a missed expert without a slot);
// moe_cache_issue queues the fills on the copy stream behind an event of the
// compute stream (a refilled slot may still be read by a queued kernel) and
// makes the compute stream wait for them before the window's forward.
#include <cstdint>
#include <cstring>
#include <vector>

#include <cuda_runtime.h>

#include "moe_internal.cuh"

struct moe_cache {
    int32_t n_experts = 0, n_slots = 0;
    int64_t blob_bytes = 0;
    std::vector<const uint8_t *> host;        // [E] device-usable address of the host copy
    uint8_t *slots = nullptr;                 // n_slots * blob_bytes of device memory
    std::vector<int32_t> slot_of;             // [E] resident slot, or -1
    std::vector<int32_t> expert_in;           // [n_slots] expert held (or being filled), or -1
    std::vector<uint8_t> ready;               // [n_slots] filled, or its fill issued (stream-ordered)
    std::vector<int64_t> last_use;            // [n_slots] window counter of the last use
    std::vector<int32_t> pending;             // slots whose fill is planned but not issued
    cudaEvent_t order = nullptr;              // compute-stream point the fills must follow
    cudaEvent_t filled = nullptr;             // copy-stream point the compute stream must follow
    int64_t clock = 0, hits = 0, misses = 0, fills = 0, bytes = 0;
};

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

moe_status moe_cache_create(int32_t n_experts, int64_t blob_bytes, const uint8_t *const *host_blobs,
                            uint8_t *slot_memory, int32_t n_slots, moe_cache **out)
{
    if (!out) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    if (n_experts <= 0 || blob_bytes <= 0 || n_slots < 0 || !host_blobs || (n_slots > 0 && !slot_memory))
        return MOE_ERR_INVALID_ARG;
    if (blob_bytes % 16 != 0) return MOE_ERR_MISALIGNED;
    if (n_slots > 0 && !aligned16(slot_memory)) return MOE_ERR_MISALIGNED;
    for (int32_t e = 0; e < n_experts; ++e) {
        if (!host_blobs[e]) return MOE_ERR_INVALID_ARG;
        if (!aligned16(host_blobs[e])) return MOE_ERR_MISALIGNED;
    }
    moe_cache *c = new moe_cache;
    c->n_experts = n_experts;
    c->n_slots = n_slots;
    c->blob_bytes = blob_bytes;
    c->host.assign(host_blobs, host_blobs + n_experts);
    c->slots = slot_memory;
    c->slot_of.assign(n_experts, -1);
    c->expert_in.assign(n_slots, -1);
    c->ready.assign(n_slots, 0);
    c->last_use.assign(n_slots, -1);
    *out = c;
    return MOE_OK;
}

void moe_cache_destroy(moe_cache *c)
{
    if (!c) return;
    if (c->order) cudaEventDestroy(c->order);
    if (c->filled) cudaEventDestroy(c->filled);
    delete c;
}

moe_status moe_cache_plan(moe_cache *c, const int32_t *ids, int32_t n_ids, const uint8_t **table, int32_t *n_fills)
{
    if (!c || !table || n_ids < 0 || (n_ids > 0 && !ids)) return MOE_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n_ids; ++i)
        if (ids[i] < 0 || ids[i] >= c->n_experts) return MOE_ERR_INVALID_ARG;
    const int64_t now = ++c->clock;
    // the window's experts, once each; their slots (resident or being filled) are in use
    std::vector<int32_t> want;
    std::vector<uint8_t> seen(c->n_experts, 0);
    for (int32_t i = 0; i < n_ids; ++i)
        if (!seen[ids[i]]) {
            seen[ids[i]] = 1;
            want.push_back(ids[i]);
        }
    for (int32_t e : want) {
        const int32_t s = c->slot_of[e];
        if (s >= 0) c->last_use[s] = now;
    }
    int32_t planned = 0;
    for (int32_t e : want) {
        const int32_t s = c->slot_of[e];
        if (s >= 0 && c->ready[s]) {
            ++c->hits;
            continue;
        }
        ++c->misses;
        if (s >= 0) continue;                   // its fill is planned already
        // a slot for e: a free one, else the least recently used one that holds a
        // resident expert this window does not need
        int32_t best = -1;
        for (int32_t t = 0; t < c->n_slots; ++t) {
            if (c->expert_in[t] < 0) {
                best = t;
                break;
            }
            if (!c->ready[t] || c->last_use[t] == now) continue;   // being filled, or used now
            if (best < 0 || c->last_use[t] < c->last_use[best]) best = t;
        }
        if (best < 0) continue;                 // every slot busy: e stays in host memory
        if (c->expert_in[best] >= 0) c->slot_of[c->expert_in[best]] = -1;
        c->expert_in[best] = e;
        c->slot_of[e] = best;
        c->ready[best] = 0;
        c->last_use[best] = now;
        c->pending.push_back(best);
        ++planned;
    }
    // resident experts and the ones filled before this window's forward: their slot
    for (int32_t e = 0; e < c->n_experts; ++e) {
        const int32_t s = c->slot_of[e];
        table[e] = s >= 0 ? c->slots + (int64_t)s * c->blob_bytes : c->host[e];
    }
    if (n_fills) *n_fills = planned;
    return MOE_OK;
}

moe_status moe_cache_issue(moe_cache *c, moe_stream_t compute_stream, moe_stream_t copy_stream)
{
    if (!c) return MOE_ERR_INVALID_ARG;
    if (c->pending.empty()) return MOE_OK;
    cudaError_t e = cudaSuccess;
    if (!c->order) e = cudaEventCreateWithFlags(&c->order, cudaEventDisableTiming);
    if (e == cudaSuccess && !c->filled) e = cudaEventCreateWithFlags(&c->filled, cudaEventDisableTiming);
    // the fills follow everything queued so far on the compute stream: a refilled
    // slot may hold an expert a queued kernel still reads
    if (e == cudaSuccess) e = cudaEventRecord(c->order, (cudaStream_t)compute_stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent((cudaStream_t)copy_stream, c->order, 0);
    for (size_t i = 0; e == cudaSuccess && i < c->pending.size(); ++i) {
        const int32_t s = c->pending[i];
        e = cudaMemcpyAsync(c->slots + (int64_t)s * c->blob_bytes, c->host[c->expert_in[s]], (size_t)c->blob_bytes,
                            cudaMemcpyDefault, (cudaStream_t)copy_stream);
        if (e == cudaSuccess) {
            c->ready[s] = 1;                    // everything queued later on the compute stream sees it
            ++c->fills;
            c->bytes += c->blob_bytes;
        }
    }
    // the window's forward (queued next on the compute stream) waits for the fills
    if (e == cudaSuccess) e = cudaEventRecord(c->filled, (cudaStream_t)copy_stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent((cudaStream_t)compute_stream, c->filled, 0);
    if (e != cudaSuccess) {
        // the window's fills are not all issued and ordered: their slots go back to the
        // free pool (the caller must not queue the window's forward with this plan)
        for (const int32_t t : c->pending) {
            if (c->expert_in[t] >= 0) c->slot_of[c->expert_in[t]] = -1;
            c->expert_in[t] = -1;
            c->ready[t] = 0;
        }
    }
    c->pending.clear();
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_cache_poll(moe_cache *c)
{
    // fills are ordered before the compute stream's later work by moe_cache_issue;
    // nothing is left to collect
    return c ? MOE_OK : MOE_ERR_INVALID_ARG;
}

moe_status moe_host_address(const void *host_ptr, const uint8_t **device_ptr)
{
    if (!host_ptr || !device_ptr) return MOE_ERR_INVALID_ARG;
    *device_ptr = nullptr;
    void *d = nullptr;
    const cudaError_t e = cudaHostGetDevicePointer(&d, const_cast<void *>(host_ptr), 0);
    if (e != cudaSuccess) {
        cudaGetLastError();                     // not pinned and mapped: not a CUDA failure to keep
        return MOE_ERR_INVALID_ARG;
    }
    *device_ptr = static_cast<const uint8_t *>(d);
    return MOE_OK;
}

moe_status moe_cache_stats(const moe_cache *c, int64_t *out4)
{
    if (!c || !out4) return MOE_ERR_INVALID_ARG;
    out4[0] = c->hits;
    out4[1] = c->misses;
    out4[2] = c->fills;
    out4[3] = c->bytes;
    return MOE_OK;
}
