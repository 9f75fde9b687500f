// profile.cpp -- per-kernel timing hook and launch counter of the library.
//
// When enabled, every kernel launch of the library is bracketed by two cudaEventRecord
// calls on the stream the kernel is launched on, so that the caller can read each
// kernel's device time without a profiler. The launch counter always runs.
#include <cuda_runtime.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

namespace fibattn {
namespace {

struct Rec {
    int kernel;
    cudaEvent_t start, stop;
};

struct Profiler {
    std::mutex mu;
    bool on = false;
    std::vector<std::string> names;
    std::vector<Rec> pending;
    std::vector<cudaEvent_t> pool;
    std::vector<double> total_ms;
    std::vector<long long> launches;
};

Profiler& prof() {
    static Profiler* p = new Profiler();  // never destroyed: events may outlive static teardown
    return *p;
}

std::atomic<long long> g_launches{0};
std::atomic<int32_t> g_last_cuda_error{0};
std::atomic<const char*> g_last_cuda_where{""};

cudaEvent_t take_event(Profiler& p) {
    if (!p.pool.empty()) {
        cudaEvent_t e = p.pool.back();
        p.pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

int kernel_id(Profiler& p, const char* name) {
    for (size_t i = 0; i < p.names.size(); ++i)
        if (p.names[i] == name) return (int)i;
    p.names.emplace_back(name);
    p.total_ms.push_back(0.0);
    p.launches.push_back(0);
    return (int)p.names.size() - 1;
}

}  // namespace

fibattn_status cuda_fail(int32_t code, const char* where) {
    g_last_cuda_error.store(code, std::memory_order_relaxed);
    g_last_cuda_where.store(where, std::memory_order_relaxed);
    return FIBATTN_ERR_CUDA;
}

fibattn_status launch_status(const char* where) {
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? FIBATTN_OK : cuda_fail((int32_t)e, where);
}

KernelScope::KernelScope(const char* name, cudaStream_t st) : st_(st), rec_(-1) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    Profiler& p = prof();
    std::lock_guard<std::mutex> g(p.mu);
    if (!p.on) return;
    Rec r;
    r.kernel = kernel_id(p, name);
    r.start = take_event(p);
    r.stop = take_event(p);
    if (!r.start || !r.stop) return;
    cudaEventRecord(r.start, st);
    p.pending.push_back(r);
    rec_ = (int)p.pending.size() - 1;
}

KernelScope::~KernelScope() {
    if (rec_ < 0) return;
    Profiler& p = prof();
    std::lock_guard<std::mutex> g(p.mu);
    if (rec_ < (int)p.pending.size()) cudaEventRecord(p.pending[rec_].stop, st_);
}

}  // namespace fibattn

using namespace fibattn;

extern "C" {

FIBATTN_API fibattn_status fibattn_profile_enable(int32_t on) {
    Profiler& p = prof();
    std::lock_guard<std::mutex> g(p.mu);
    p.on = on != 0;
    return FIBATTN_OK;
}

FIBATTN_API int64_t fibattn_launch_count(void) { return g_launches.load(); }

FIBATTN_API int32_t fibattn_last_cuda_error(const char** where) {
    if (where) *where = g_last_cuda_where.load(std::memory_order_relaxed);
    return g_last_cuda_error.load(std::memory_order_relaxed);
}

FIBATTN_API int32_t fibattn_profile_read(char* names, int32_t name_len, double* total_ms,
                                         int64_t* launches, int32_t cap) {
    Profiler& p = prof();
    std::lock_guard<std::mutex> g(p.mu);
    for (Rec& r : p.pending) {
        float ms = 0.f;
        if (cudaEventSynchronize(r.stop) == cudaSuccess &&
            cudaEventElapsedTime(&ms, r.start, r.stop) == cudaSuccess) {
            p.total_ms[r.kernel] += ms;
            p.launches[r.kernel] += 1;
        }
        p.pool.push_back(r.start);
        p.pool.push_back(r.stop);
    }
    p.pending.clear();
    int32_t n = (int32_t)p.names.size();
    for (int32_t i = 0; i < n && i < cap; ++i) {
        if (names && name_len > 0) {
            strncpy(names + (size_t)i * name_len, p.names[i].c_str(), (size_t)name_len - 1);
            names[(size_t)i * name_len + name_len - 1] = 0;
        }
        if (total_ms) total_ms[i] = p.total_ms[i];
        if (launches) launches[i] = p.launches[i];
        p.total_ms[i] = 0.0;
        p.launches[i] = 0;
    }
    return n;
}

}  // extern "C"
