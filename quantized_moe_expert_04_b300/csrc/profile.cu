// profile.cu -- the diagnostics API (moe_profile_enable / moe_profile_read):
// optional CUDA-event brackets around each kernel launch of a call, and
// per-kernel launch counts, for benchmarks that report a kernel's achieved
// bandwidth or throughput.
#include <vector>

#include "moe_internal.cuh"

namespace moe {

static const char *kPhaseNames[kNumPhases] = {
    "router_logits", "topk", "bucket", "gemm_prep", "gemm_gateup", "gemm_down", "gemm_finish",
    "dec_route", "dec_layer", "dec_stack",
};

namespace {
struct Pair {
    cudaEvent_t a = nullptr, b = nullptr;
    int phase = -1;
};
struct ProfState {
    bool on = false;
    std::vector<Pair> pool;
    size_t used = 0;
    long pending = -1;               // pair index opened by prof_begin
    int64_t launches[kNumPhases] = {};
    int64_t timed[kNumPhases] = {};
    double ms[kNumPhases] = {};
};
ProfState g;
constexpr size_t kMaxPairs = 1 << 16;
}  // namespace

static bool capturing(cudaStream_t s)
{
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &st) != cudaSuccess) return true;
    return st != cudaStreamCaptureStatusNone;
}

void prof_begin(int phase, cudaStream_t s)
{
    if (!g.on) return;
    g.launches[phase]++;
    g.pending = -1;
    if (capturing(s)) return;
    if (g.used == g.pool.size()) {
        if (g.pool.size() >= kMaxPairs) return;
        Pair p;
        if (cudaEventCreate(&p.a) != cudaSuccess || cudaEventCreate(&p.b) != cudaSuccess) return;
        g.pool.push_back(p);
    }
    if (cudaEventRecord(g.pool[g.used].a, s) != cudaSuccess) return;
    g.pool[g.used].phase = phase;
    g.pending = (long)g.used;
}

void prof_end(int phase, cudaStream_t s)
{
    if (!g.on || g.pending < 0) return;
    Pair &p = g.pool[(size_t)g.pending];
    g.pending = -1;
    if (p.phase != phase) return;
    if (cudaEventRecord(p.b, s) == cudaSuccess) g.used++;
}

static void reset()
{
    g.used = 0;
    g.pending = -1;
    for (int i = 0; i < kNumPhases; ++i) {
        g.launches[i] = g.timed[i] = 0;
        g.ms[i] = 0.0;
    }
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_profile_enable(int32_t on)
{
    g.on = on != 0;
    reset();
    return MOE_OK;
}

extern "C" int32_t moe_profile_read(moe_profile_entry *out, int32_t max_entries)
{
    for (size_t i = 0; i < g.used; ++i) {
        Pair &p = g.pool[i];
        float ms = 0.0f;
        if (cudaEventSynchronize(p.b) == cudaSuccess && cudaEventElapsedTime(&ms, p.a, p.b) == cudaSuccess) {
            g.ms[p.phase] += ms;
            g.timed[p.phase]++;
        }
    }
    g.used = 0;
    int32_t n = 0;
    for (int i = 0; i < kNumPhases && out && n < max_entries; ++i) {
        if (g.launches[i] == 0) continue;
        out[n].name = kPhaseNames[i];
        out[n].launches = g.launches[i];
        out[n].timed = g.timed[i];
        out[n].total_ms = g.ms[i];
        ++n;
    }
    return n;
}
