// no_alloc.cu -- moe_forward_static_ws: the whole layer with its scratch in a
// fixed, library-owned device array instead of a caller-allocated workspace.
//
// Who needs it: code that may not call cudaMalloc at the point where it runs
// the layer -- for example a host runtime that hands out only pre-registered
// buffers, a plugin living inside another framework's allocator, or a caller
// that must not allocate on its hot path.  Such callers still pass their
// inputs and outputs; the scratch comes from `g_static_ws` below, which every
// GPU that loads this library keeps (MOE_STATIC_WS_BYTES bytes) until the
// process exits.
#include <mutex>

#include "moe_internal.cuh"

namespace moe {

// The shared scratch.  One array per device, zero at module load, shared by
// every call on that device, and it keeps the previous call's contents.
static __device__ __align__(256) unsigned char g_static_ws[MOE_STATIC_WS_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_static_ws_addr[kMaxDevices] = {};
}  // namespace

// Device address of g_static_ws on the current device, looked up once per
// device.  In host code the array's name only stands in for the symbol; the
// address kernels may use comes from cudaGetSymbolAddress.
static cudaError_t static_ws_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_static_ws_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_ws);
        if (e != cudaSuccess) return e;
        g_static_ws_addr[dev] = p;
    }
    *out = g_static_ws_addr[dev];
    return cudaSuccess;
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_forward_static_ws(const moe_config *cfg, const uint16_t *x, const float *router_w,
                                           const float *router_bias, const uint8_t *const *expert_blobs,
                                           const uint8_t *shared_blob, int32_t T, uint16_t *y, float *y_f32,
                                           uint32_t *dev_status, moe_stream_t stream)
{
    // every argument check first, before the array is touched: a rejected
    // call enqueues nothing (in particular it does not clear the header of a
    // call that may still be running)
    if (dev_status && ((uintptr_t)dev_status & 3u)) return MOE_ERR_MISALIGNED;
    const size_t need = moe_workspace_bytes(cfg, T < 0 ? 0 : T);
    if (need > (size_t)MOE_STATIC_WS_BYTES) return MOE_ERR_WORKSPACE_TOO_SMALL;   // call too large for the array
    const void *const kAligned = reinterpret_cast<const void *>(256);               // stands in for the array
    moe_status st = forward_checks(cfg, x, router_w, router_bias, expert_blobs, shared_blob, T, y, y_f32,
                                   const_cast<void *>(kAligned), MOE_STATIC_WS_BYTES);
    if (st != MOE_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (T == 0) {
        if (dev_status && cudaMemsetAsync(dev_status, 0, sizeof(uint32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
        return MOE_OK;
    }
    void *ws = nullptr;
    if (static_ws_address(&ws) != cudaSuccess) return MOE_ERR_CUDA;
    // the array still holds the previous call's header: its status word and
    // counters must start at zero
    if (cudaMemsetAsync(ws, 0, kHeaderBytes, s) != cudaSuccess) return MOE_ERR_CUDA;
    st = moe_forward(cfg, x, router_w, router_bias, expert_blobs, shared_blob, T, y, y_f32, ws, MOE_STATIC_WS_BYTES,
                     stream);
    if (st == MOE_OK && dev_status) {
        if (cudaMemcpyAsync(dev_status, ws, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    return st;
}
