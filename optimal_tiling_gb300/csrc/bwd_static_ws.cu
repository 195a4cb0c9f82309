// attn_bwd_static_workspace: the backward pass for callers that cannot
// allocate device memory.
//
// attn_bwd needs scratch (the row terms D and, for bf16, LSE log2(e) and the
// fp32 dQ accumulator) that the caller normally allocates and passes in.  Some callers
// cannot do that: code that runs inside a host framework which owns every device
// allocation through its own pool and forbids allocations made behind its back,
// or code on a latency-critical path that must not allocate after start-up
// (cudaMalloc may synchronise the device and stall the work already queued).
// This entry point takes the scratch from a fixed array compiled into the
// library instead, so the call itself allocates nothing.
//
// The array lives in device memory of every GPU that loads the library, for as
// long as the process runs.  It is shared by every call on a device and keeps
// the contents of the last call; the backward writes its row terms in full and
// zeroes the dQ accumulator before adding into it, so nothing stale is read.  Two calls
// whose work overlaps on the GPU (for example on two streams without ordering
// between them) race on the array.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/attn.h"
#include "internal.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(64) << 20;  // 64 MiB, the documented maximum

static __device__ __align__(256) unsigned char g_static_ws[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 64;
struct WsAddr {
    void *ctx;   // CUDA context the address was looked up in
    void *ptr;
};
WsAddr g_static_ws_addr[kMaxDevices];
std::mutex g_static_ws_mu;

// Device address of the array on the current device.  In host code the name
// g_static_ws is only a host-side stand-in, so the real address is looked up with
// cudaGetSymbolAddress, with the device current, on the first call on that device,
// and kept for the CUDA context it was found in: a later call in another context
// (the primary context torn down and created again, e.g. after cudaDeviceReset)
// looks it up again instead of handing the kernels a stale address.
void *static_ws_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    void *ctx = attn::current_context();
    std::lock_guard<std::mutex> lk(g_static_ws_mu);
    WsAddr &a = g_static_ws_addr[dev];
    if (ctx == nullptr || a.ctx != ctx || a.ptr == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess) return nullptr;
        a.ptr = p;
        a.ctx = attn::current_context();  // the lookup makes the device's primary context current
    }
    return a.ptr;
}

}  // namespace

extern "C" attn_status attn_bwd_static_workspace(const void *Q, const void *K, const void *V, const void *O,
                                                 const void *dO, const float *LSE, void *dQ, void *dK, void *dV,
                                                 int B, int H, int N, int d, float scale, attn_dtype dtype,
                                                 const uint8_t *block_mask, void *stream) {
    // attn_bwd's own argument checks first, so that a bad argument gets the same status as
    // from attn_bwd whatever the shape's size; then the size, then the array's address
    const attn_status s = attn::bwd_args_status(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, dtype);
    if (s != ATTN_OK) return s;
    // the shape's row terms and dQ scratch must fit the array; attn_bwd splits the last wave only
    // when the split's scratch fits as well
    if (attn::bwd_base_bytes(B, H, N, d, dtype == ATTN_DTYPE_BF16) > kStaticWorkspaceBytes)
        return ATTN_ERR_WORKSPACE;
    void *ws = static_ws_address();
    if (ws == nullptr) return ATTN_ERR_CUDA;
    return attn_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, dtype, block_mask, ws,
                    kStaticWorkspaceBytes, stream);
}
