// topk_warp.cuh -- the selection step of a token's top-k by one warp (the
// prefill top-k kernel, many tokens at once: uniform code keeps the issue
// slots busy; the decode window's few tokens are routed in the layer kernel).
//
// Lane l holds the selection keys of experts l, l + 32, ... (NPER of them):
// order-preserving integers of the scores, 0 = never selected.  It packs them
// as 64-bit words key << 32 | (0xffff - e), so that a larger word is the larger
// key and, among equal keys, the lower expert id, and sorts them once in
// registers with Batcher's odd-even merge network (uniform code, every lane
// busy).  Each round then takes the warp maximum of the lanes' first words
// (the key, then the lowest id among equal keys: two reductions) and the lane
// that held it shifts its words by one.  The selection is the k largest keys,
// ties to the lower id: the router's ~10 of 512 experts a token ("Strata
// 引擎深度拆解", lcz.me/topic/2098/5, section 二) or 6 of 256 with the router
// bias ("Strata 改源码去跑 DeepSeek V4 Flash？", lcz.me/post/23082, section 二,
// anatomy table).
#pragma once

#include <stdint.h>

namespace moe {

// Batcher's odd-even merge sort of N words into descending order (N a power
// of two): for p = 1, 2, 4, ... < N: for k = p, p/2, ..., 1: compare-exchange
// elements i + j and i + j + k (j from k mod p in steps of 2k, i < k) when
// both lie in the same block of 2p.  19 / 63 / 191 comparators for 8 / 16 /
// 32.  One pass (p, k) per instantiation, so that every loop bound is a
// constant and the words stay in registers.
template <int N, int P, int K>
struct OddEvenPass {
    static __device__ __forceinline__ void run(uint64_t (&v)[N])
    {
#pragma unroll
        for (int j = K % P; j + K < N; j += 2 * K)
#pragma unroll
            for (int i = 0; i < K; ++i) {
                const int lo = i + j, hi = i + j + K;
                if (hi < N && lo / (2 * P) == hi / (2 * P)) {
                    const uint64_t x = v[lo], y = v[hi];
                    const bool sw = y > x;
                    v[lo] = sw ? y : x;
                    v[hi] = sw ? x : y;
                }
            }
        if constexpr (K > 1) OddEvenPass<N, P, K / 2>::run(v);
        else if constexpr (2 * P < N) OddEvenPass<N, 2 * P, 2 * P>::run(v);
    }
};

template <int N>
__device__ __forceinline__ void sort_desc(uint64_t (&v)[N])
{
    OddEvenPass<N, 1, 1>::run(v);
}

// The k selections of the warp's token (k <= 32): lane r < k receives
// selection r (in descending key order) as out_id and its key as out_key.
// Fewer than k selectable keys (non-zero) set fault; the missing selections
// are then id r with key 0.  All 32 lanes take part.
template <int NPER>
__device__ __forceinline__ void warp_select(const uint32_t (&key)[NPER], int k, int lane, int &out_id,
                                            uint32_t &out_key, bool &fault)
{
    uint64_t v[NPER];
#pragma unroll
    for (int i = 0; i < NPER; ++i) v[i] = ((uint64_t)key[i] << 32) | (uint32_t)(0xffff - (lane + 32 * i));
    sort_desc<NPER>(v);
    out_id = 0;
    out_key = 0u;
    fault = false;
    for (int r = 0; r < k; ++r) {
        const uint32_t hk = (uint32_t)(v[0] >> 32);
        const uint32_t mk = __reduce_max_sync(0xffffffffu, hk);
        const uint32_t ml = __reduce_max_sync(0xffffffffu, hk == mk ? (uint32_t)v[0] : 0u);
        const int e = 0xffff - (int)ml;                  // the lowest id among the equal keys
        if (mk == 0u) fault = true;                      // nothing selectable (non-finite scores)
        if (lane == r) {
            out_id = mk == 0u ? r : e;
            out_key = mk;
        }
        const bool pop = mk != 0u && lane == (e & 31);
#pragma unroll
        for (int i = 0; i + 1 < NPER; ++i) v[i] = pop ? v[i + 1] : v[i];
        v[NPER - 1] = pop ? 0ull : v[NPER - 1];
    }
}

}  // namespace moe
