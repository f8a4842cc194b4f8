// Gradient entry point for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: plug-ins that receive device buffers
// from a host framework's own allocator and have no allocator of their own,
// or processes that have reserved all device memory up front.  For them
// tnd_attn_grad_static_ws runs the same gradient as tnd_attn_grad with its
// workspace taken from a fixed, file-scope device array instead of a buffer
// the caller allocates, and it uploads its plan without the library's pinned
// staging slots (which are allocated on first use), so it allocates nothing.
//
// The array is a static __device__ object: every GPU that loads this
// library holds it (kStaticWsBytes) until the process exits.  Host code
// cannot use the array's name as a device address (on the host it names a
// shadow variable), so the address is looked up with cudaGetSymbolAddress,
// with that device current, on the first call made on the device, and looked
// up again if the device's context has changed since (after cudaDeviceReset).
#include "tnd_internal.h"

#include <cudaTypedefs.h>
#include <mutex>

namespace tnd {
namespace {

constexpr uint64_t kStaticWsBytes = TND_STATIC_WS_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

std::mutex g_static_mu;
void *g_static_ptr[kMaxDevices] = {};
void *g_static_ctx[kMaxDevices] = {};

// The current context of the calling thread (nullptr if it cannot be read).
void *current_context()
{
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    });
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

// Device address of g_static_ws on the current device (nullptr on failure).
void *static_ws_address()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!g_static_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess) return nullptr;
        g_static_ptr[dev] = p;
        g_static_ctx[dev] = current_context();
        return p;
    }
    void *ctx = current_context();
    if (ctx != g_static_ctx[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess) return nullptr;
        g_static_ptr[dev] = p;
        g_static_ctx[dev] = ctx;
    }
    return g_static_ptr[dev];
}

}  // namespace
}  // namespace tnd

extern "C" {

tnd_status tnd_attn_grad_static_ws(const void *q, const void *k, const void *v, const void *dy,
                                   const uint8_t *drop_mask, const float *smax, const float *ssum, const void *o,
                                   const float *sink, tnd_dtype dtype, int64_t batch, const int64_t *cuq,
                                   const int64_t *cukv, int64_t nq, int64_t nkv, int64_t d, double scale,
                                   double keep, int64_t pre, int64_t next, int64_t mode, void *dq, void *dk, void *dv,
                                   float *dsink, void *stream)
{
    uint64_t need = 0;
    tnd_status st = tnd_attn_grad_workspace_size(dtype, batch, cuq, cukv, nullptr, nq, nkv, d, d, scale, keep, pre,
                                                 next, mode, drop_mask != nullptr, 0, sink != nullptr, &need);
    if (st != TND_OK) return st;
    if (need > tnd::kStaticWsBytes) return TND_ERR_WORKSPACE;
    void *ws = tnd::static_ws_address();
    if (!ws) return TND_ERR_CUDA;
    return tnd::grad_run(q, k, v, dy, nullptr, 0, 1, drop_mask, nullptr, smax, ssum, o, sink, dtype, batch, cuq, cukv,
                         nullptr, nq, nkv, d, d, scale, keep, pre, next, mode, dq, dk, dv, dsink, ws,
                         tnd::kStaticWsBytes, stream, false);
}

tnd_status tnd_attn_grad_static_ws_status(void *stream)
{
    void *ws = tnd::static_ws_address();
    if (!ws) return TND_ERR_CUDA;
    return tnd_attn_device_status(ws, tnd::kStaticWsBytes, stream);
}

}  // extern "C"
