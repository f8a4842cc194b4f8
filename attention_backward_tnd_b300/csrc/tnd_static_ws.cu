// Gradient entry point for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code running while a CUDA stream is
// being captured into a graph, plug-ins that receive device buffers from a
// host framework's own allocator and have no allocator of their own, or
// processes that have reserved all device memory up front.  For them
// tnd_attn_grad_static_ws runs the same gradient as tnd_attn_grad with its
// workspace taken from a fixed, file-scope device array instead of a buffer
// the caller allocates.
//
// The array is a static __device__ object: every GPU that loads this
// library holds it (kStaticWsBytes) until the process exits.  Host code
// cannot use the array's name as a device address (on the host it names a
// shadow variable), so the address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call made
// while it is current.
#include "tnd_internal.h"

#include <mutex>

namespace tnd {
namespace {

constexpr uint64_t kStaticWsBytes = TND_STATIC_WS_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

std::mutex g_static_mu;
void *g_static_ptr[kMaxDevices] = {};

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
    tnd_status st = tnd_attn_grad_workspace_size(dtype, batch, cuq, cukv, nq, nkv, d, scale, keep, pre, next, mode,
                                                 drop_mask != nullptr, sink != nullptr, &need);
    if (st != TND_OK) return st;
    if (need > tnd::kStaticWsBytes) return TND_ERR_WORKSPACE;
    void *ws = tnd::static_ws_address();
    if (!ws) return TND_ERR_CUDA;
    return tnd_attn_grad(q, k, v, dy, drop_mask, smax, ssum, o, sink, dtype, batch, cuq, cukv, nq, nkv, d, scale,
                         keep, pre, next, mode, dq, dk, dv, dsink, ws, tnd::kStaticWsBytes, stream);
}

}  // extern "C"
