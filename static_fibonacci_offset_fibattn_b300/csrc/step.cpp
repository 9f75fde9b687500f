// step.cpp -- the forward and backward of a layer stack in one call (fibattn_fwd_bwd), with
// the call's layers split into contiguous groups that run on concurrent streams.
//
// Every layer of the stack is an independent problem for this path (its own q, k, v, dO and
// table), so the groups share nothing but the GPU: group g runs the forward and then the
// backward of its layers on an internal stream of the library, forked from the caller's stream
// by an event and joined back by another. Kernels of different groups then fill each other's
// gaps (a persistent kernel's tail, one kernel's wait on another), which one stream in order
// cannot. Each group's kernels are the ones fibattn_fwd_gqa / fibattn_bwd_gqa launch, on its
// own part of the workspace, so the results equal the sequential calls bit for bit.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"

namespace fibattn {
namespace {

constexpr int kMaxDevices = 64;

std::mutex g_mu;
cudaStream_t g_streams[kMaxDevices][FIBATTN_STEP_STREAMS_MAX] = {};

// The library's first n non-blocking streams on the current device (created once).
fibattn_status group_streams(int n, cudaStream_t* out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail((int32_t)e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return FIBATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> g(g_mu);
    for (int i = 0; i < n; ++i) {
        if (!g_streams[dev][i]) {
            e = cudaStreamCreateWithFlags(&g_streams[dev][i], cudaStreamNonBlocking);
            if (e != cudaSuccess) {
                g_streams[dev][i] = nullptr;
                return cuda_fail((int32_t)e, "cudaStreamCreateWithFlags");
            }
        }
        out[i] = g_streams[dev][i];
    }
    return FIBATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

uint64_t align256(uint64_t x) { return (x + 255) & ~(uint64_t)255; }

// First layer of group g of `groups` over n layers (contiguous, sizes differing by at most 1).
int32_t group_first(int32_t g, int32_t groups, int32_t n) {
    return (int32_t)((int64_t)n * g / groups);
}

}  // namespace
}  // namespace fibattn

using namespace fibattn;

extern "C" {

fibattn_status fibattn_fwd_bwd_workspace_size(int32_t B, int32_t H, int32_t T, int32_t d,
                                              int32_t dtype, int32_t W,
                                              const fibattn_schedule* sched, int32_t layer0,
                                              int32_t n_layers_call, int32_t n_streams,
                                              uint64_t* bytes) {
    if (!bytes || n_streams < 1 || n_streams > FIBATTN_STEP_STREAMS_MAX || n_layers_call < 1)
        return FIBATTN_ERR_INVALID_ARG;
    const int32_t groups = n_streams < n_layers_call ? n_streams : n_layers_call;
    uint64_t total = 0;
    for (int32_t g = 0; g < groups; ++g) {
        const int32_t a = group_first(g, groups, n_layers_call);
        const int32_t b = group_first(g + 1, groups, n_layers_call);
        uint64_t n = 0;
        const fibattn_status st =
            fibattn_bwd_workspace_size(B, H, T, d, dtype, W, sched, layer0 + a, b - a, &n);
        if (st != FIBATTN_OK) return st;
        total += align256(n);
    }
    *bytes = total;
    return FIBATTN_OK;
}

fibattn_status fibattn_fwd_bwd(const void* q, const void* k, const void* v, const void* dO,
                               void* o, float* lse, void* dq, void* dk, void* dv, void* workspace,
                               uint64_t workspace_bytes, int32_t B, int32_t H, int32_t H_kv,
                               int32_t T, int32_t d, int32_t dtype, int32_t W, float scale,
                               const fibattn_schedule* sched, int32_t layer0,
                               int32_t n_layers_call, int32_t n_streams, void* cuda_stream) {
    // everything is checked before anything is enqueued
    const void* ptrs[] = {q, k, v, dO, o, lse, dq, dk, dv};
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return FIBATTN_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return FIBATTN_ERR_INVALID_ARG;
    if (H_kv < 1 || H < 1 || H % H_kv != 0) return FIBATTN_ERR_INVALID_ARG;
    uint64_t need = 0;
    fibattn_status st = fibattn_fwd_bwd_workspace_size(B, H, T, d, dtype, W, sched, layer0,
                                                       n_layers_call, n_streams, &need);
    if (st != FIBATTN_OK) return st;
    if (workspace_bytes < need) return FIBATTN_ERR_INVALID_ARG;
    const int32_t groups = n_streams < n_layers_call ? n_streams : n_layers_call;
    if (groups == 1) {
        st = fibattn_fwd_gqa(q, k, v, o, lse, B, H, H_kv, T, d, dtype, W, scale, sched, layer0,
                             n_layers_call, cuda_stream);
        if (st != FIBATTN_OK) return st;
        return fibattn_bwd_gqa(q, k, v, o, lse, dO, dq, dk, dv, workspace, workspace_bytes, B, H,
                               H_kv, T, d, dtype, W, scale, sched, layer0, n_layers_call,
                               cuda_stream);
    }

    cudaStream_t s[FIBATTN_STEP_STREAMS_MAX];
    st = group_streams(groups, s);
    if (st != FIBATTN_OK) return st;
    cudaStream_t caller = reinterpret_cast<cudaStream_t>(cuda_stream);
    cudaEvent_t fork = nullptr;
    cudaError_t e = cudaEventCreateWithFlags(&fork, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail((int32_t)e, "cudaEventCreateWithFlags");
    e = cudaEventRecord(fork, caller);
    for (int32_t g = 0; g < groups && e == cudaSuccess; ++g) e = cudaStreamWaitEvent(s[g], fork, 0);
    cudaEventDestroy(fork);  // released once it completes
    if (e != cudaSuccess) return cuda_fail((int32_t)e, "cudaEventRecord / cudaStreamWaitEvent (fork)");

    const size_t es = dtype == FIBATTN_F32 ? 4 : 2;
    const int64_t rows = (int64_t)B * H * T, rows_kv = (int64_t)B * H_kv * T;  // per layer
    uint64_t ws_off = 0;
    fibattn_status first_err = FIBATTN_OK;
    for (int32_t g = 0; g < groups; ++g) {
        const int32_t a = group_first(g, groups, n_layers_call);
        const int32_t n = group_first(g + 1, groups, n_layers_call) - a;
        const size_t off = (size_t)a * rows * d * es, koff = (size_t)a * rows_kv * d * es;
        float* lg = lse + (size_t)a * rows;
        uint64_t need_g = 0;
        fibattn_bwd_workspace_size(B, H, T, d, dtype, W, sched, layer0 + a, n, &need_g);  // checked above
        void* wg = static_cast<char*>(workspace) + ws_off;
        ws_off += align256(need_g);
        // a group that fails to launch still joins (its stream holds no work from this call)
        if (first_err == FIBATTN_OK) {
            st = fibattn_fwd_gqa((const char*)q + off, (const char*)k + koff, (const char*)v + koff,
                                 (char*)o + off, lg, B, H, H_kv, T, d, dtype, W, scale, sched,
                                 layer0 + a, n, s[g]);
            if (st == FIBATTN_OK)
                st = fibattn_bwd_gqa((const char*)q + off, (const char*)k + koff,
                                     (const char*)v + koff, (const char*)o + off, lg,
                                     (const char*)dO + off, (char*)dq + off, (char*)dk + koff,
                                     (char*)dv + koff, wg, need_g, B, H, H_kv, T, d, dtype, W,
                                     scale, sched, layer0 + a, n, s[g]);
            if (st != FIBATTN_OK) first_err = st;
        }
        cudaEvent_t done = nullptr;
        e = cudaEventCreateWithFlags(&done, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventRecord(done, s[g]);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(caller, done, 0);
        if (done) cudaEventDestroy(done);
        if (e != cudaSuccess && first_err == FIBATTN_OK)
            first_err = cuda_fail((int32_t)e, "cudaEventRecord / cudaStreamWaitEvent (join)");
    }
    return first_err;
}

}  // extern "C"
