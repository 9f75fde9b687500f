// bwd_noalloc.cu -- the backward entry point for callers that cannot allocate device memory.
//
// fibattn_bwd needs a device workspace that the caller allocates (D_i = dO_i . o_i for
// every row and, on the bf16 path, the (P, dS) pair of every diagonal entry). Some callers
// cannot call cudaMalloc at all: an operator hosted by a framework that owns the device
// allocator and hands it no workspace, or a latency-critical loop where cudaMalloc/cudaFree
// would synchronise the device. For them this file keeps the workspace in a fixed-size
// file-scope __device__ array instead, and fibattn_bwd_noalloc passes that array to
// fibattn_bwd.
//
// Properties a caller must know:
//   - The array holds FIBATTN_NOALLOC_SCRATCH_BYTES (40 MiB) on every GPU that loads the
//     library, for the life of the process. Calls whose workspace is larger are rejected
//     with FIBATTN_ERR_SCRATCH_LIMIT before anything is launched.
//   - Host code cannot use the array's name as a device address. The first call on each
//     device (that device current) looks the address up with cudaGetSymbolAddress and
//     caches it; make that first call before any stream capture begins.
//   - Every call on a device shares the one array, and it keeps the last call's contents.
//     Nothing needs clearing: the backward writes every workspace value it uses, and the
//     bytes it reads without writing (the pad rows of D and lse * log2(e) past T, the pairs
//     of queries past T) are discarded by selects, so an earlier call's contents, even
//     non-finite ones, cannot reach the outputs. Calls whose kernels overlap on the GPU
//     (different streams, no ordering between them) race on the array.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"

namespace fibattn {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_ws[FIBATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ws_ptr[kMaxDevices] = {};

// Device address of g_noalloc_ws on the current device (looked up once per device).
fibattn_status scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail((int32_t)e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return FIBATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_ws_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_ws);
        if (e != cudaSuccess || !p) return cuda_fail((int32_t)e, "cudaGetSymbolAddress (scratch)");
        g_ws_ptr[dev] = p;
    }
    *out = g_ws_ptr[dev];
    return FIBATTN_OK;
}

}  // namespace
}  // namespace fibattn

using namespace fibattn;

extern "C" FIBATTN_API fibattn_status fibattn_bwd_noalloc(
    const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
    void* dq, void* dk, void* dv, int32_t B, int32_t H, int32_t T, int32_t d, int32_t dtype,
    int32_t W, float scale, const fibattn_schedule* sched, int32_t layer0, int32_t n_layers_call,
    void* cuda_stream) {
    uint64_t need = 0;
    fibattn_status st = fibattn_bwd_workspace_size(B, H, T, d, dtype, W, sched, layer0,
                                                   n_layers_call, &need);
    if (st != FIBATTN_OK) return st;
    if (need > FIBATTN_NOALLOC_SCRATCH_BYTES) return FIBATTN_ERR_SCRATCH_LIMIT;
    void* ws = nullptr;
    st = scratch_address(&ws);
    if (st != FIBATTN_OK) return st;
    return fibattn_bwd(q, k, v, o, lse, dO, dq, dk, dv, ws, FIBATTN_NOALLOC_SCRATCH_BYTES, B, H, T,
                       d, dtype, W, scale, sched, layer0, n_layers_call, cuda_stream);
}
