// bwd_noalloc.cu -- the backward entry point for callers that cannot allocate device memory.
//
// fibattn_bwd needs a float32 scratch buffer of Lc*B*H*T entries (D_i = dO_i . o_i) that
// the caller allocates. Some callers cannot call cudaMalloc at all: an operator hosted by
// a framework that owns the device allocator and hands it no workspace, or a
// latency-critical loop where cudaMalloc/cudaFree would synchronise the device. For them
// this file keeps the scratch in a fixed-size file-scope __device__ array instead, and
// fibattn_bwd_noalloc passes that array to the same backward launcher fibattn_bwd uses.
//
// Properties a caller must know:
//   - The array holds FIBATTN_NOALLOC_MAX_ROWS floats (4 MiB) on every GPU that loads the
//     library, for the life of the process. Larger calls are rejected with
//     FIBATTN_ERR_SCRATCH_LIMIT before anything is launched.
//   - Host code cannot use the array's name as a device address. The first call on each
//     device (that device current) looks the address up with cudaGetSymbolAddress and
//     caches it; make that first call before any stream capture begins.
//   - Every call on a device shares the one array, and it keeps the last call's contents.
//     The backward overwrites every entry it reads (D is computed before it is used), so
//     nothing needs clearing; but calls whose kernels overlap on the GPU (different
//     streams, no ordering between them) race on the array.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"

namespace fibattn {
namespace {

static __device__ __align__(256) float g_noalloc_delta[FIBATTN_NOALLOC_MAX_ROWS];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_delta_ptr[kMaxDevices] = {};

// Device address of g_noalloc_delta on the current device (looked up once per device).
fibattn_status scratch_address(float** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return FIBATTN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FIBATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_delta_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_delta) != cudaSuccess || !p) return FIBATTN_ERR_CUDA;
        g_delta_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_delta_ptr[dev];
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
    if (B < 1 || H < 1 || T < 1 || n_layers_call < 1) return FIBATTN_ERR_INVALID_ARG;
    const int64_t rows = (int64_t)n_layers_call * B * H * T;
    if (rows > (int64_t)FIBATTN_NOALLOC_MAX_ROWS) return FIBATTN_ERR_SCRATCH_LIMIT;
    float* delta = nullptr;
    fibattn_status st = scratch_address(&delta);
    if (st != FIBATTN_OK) return st;
    return fibattn_bwd(q, k, v, o, lse, dO, dq, dk, dv, delta, B, H, T, d, dtype, W, scale, sched,
                       layer0, n_layers_call, cuda_stream);
}
