// offsets_device.cu -- the offset-table builder as a device kernel, the key-set
// export kernel, and the device error word.
//
// The builder repeats, in device integer arithmetic, the host rule of schedule.cpp
// ("Depth-Staggered Fibonacci Spacing for Sparse Attention", gist.science explainer,
// Metodologia: d_k = alpha * f_k with alpha from a fixed, linear-stagger or
// coprime-reassigned schedule, Fibonacci or power-of-two base). The tests compare
// its tables with the host's bit for bit.
#include <stdint.h>

#include "internal.h"

namespace fibattn {

__device__ int32_t g_device_error = 0;

int32_t* device_error_word() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    return static_cast<int32_t*>(p);
}

namespace {

struct DevSchedule {
    int32_t base, kind;
    int64_t a_num, a_den, lo_num, lo_den, hi_num, hi_den;
    int64_t n_layers, coprime_c, base_max;
};

__device__ int64_t dgcd(int64_t a, int64_t b) {
    if (a < 0) a = -a;
    if (b < 0) b = -b;
    while (b) {
        int64_t t = a % b;
        a = b;
        b = t;
    }
    return a;
}

__device__ void dev_alpha(const DevSchedule& s, int64_t layer, int64_t* num, int64_t* den) {
    if (s.kind == FIBATTN_SCHED_FIXED) {
        int64_t g = dgcd(s.a_num, s.a_den);
        *num = s.a_num / g;
        *den = s.a_den / g;
        return;
    }
    int64_t L = s.n_layers;
    int64_t l = s.kind == FIBATTN_SCHED_COPRIME ? (s.coprime_c * layer) % L : layer;
    if (L == 1) {
        *num = s.lo_num;
        *den = s.lo_den;
        return;
    }
    __int128 a = (__int128)s.lo_num * s.hi_den;
    __int128 b = (__int128)s.hi_num * s.lo_den;
    int64_t n = (int64_t)(a * (L - 1) + (b - a) * l);
    int64_t d = (int64_t)((__int128)s.lo_den * s.hi_den * (L - 1));
    int64_t g = dgcd(n, d);
    *num = n / g;
    *den = d / g;
}

// One thread per layer: the table of layer0 + blockIdx.x * blockDim.x + threadIdx.x.
__global__ void build_tables_kernel(DevSchedule s, int32_t layer0, int32_t n_layers, int32_t W,
                                    int32_t T, int32_t* tables, int32_t* counts) {
    int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= n_layers) return;
    int64_t num, den;
    dev_alpha(s, layer0 + c, &num, &den);
    const bool fib = s.base == FIBATTN_BASE_FIB;
    const int64_t fmax = s.base_max > 0 ? s.base_max : (fib ? 987 : INT64_MAX);
    int32_t* row = tables + (int64_t)c * kMaxOffsets;
    for (int e = 0; e < kMaxOffsets; ++e) row[e] = -1;
    int32_t n = 0;
    int64_t last = -1, f = 1, g = 2;
    while (f <= fmax) {
        __int128 o = ((__int128)2 * num * f + den) / ((__int128)2 * den);
        if (o > (__int128)T - 1) break;
        if (o >= W && (int64_t)o != last) {
            if (n < kMaxOffsets) row[n] = (int32_t)o;
            ++n;
            last = (int64_t)o;
        }
        if (fib) {
            int64_t h = f + g;
            f = g;
            g = h;
        } else {
            if (f > INT64_MAX / 2) break;
            f *= 2;
        }
    }
    counts[c] = n;
}

// One thread per (query i, 32-key word): bit b of mask[i][w] = [32w + b in S_i],
// by the predicate 0 <= i - j < W or (i - j) in the layer's table.
__global__ void keyset_kernel(const __grid_constant__ OffsetTables t, int32_t W, int32_t T,
                              uint32_t* mask) {
    int64_t words = (T + 31) / 32;
    int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)T * words) return;
    int32_t i = (int32_t)(idx / words);
    int32_t w = (int32_t)(idx % words);
    uint32_t bits = 0;
    for (int b = 0; b < 32; ++b) {
        int32_t j = w * 32 + b;
        if (j >= T || j > i) break;
        int32_t dist = i - j;
        bool in = dist < W;
        for (int e = 0; e < t.count[0] && !in; ++e) in = (t.off[0][e] == dist);
        if (in) bits |= 1u << b;
    }
    mask[idx] = bits;
}

}  // namespace

fibattn_status launch_offsets_device(const fibattn_schedule* s, int32_t layer0, int32_t n,
                                     int32_t W, int32_t T, int32_t* d_tables, int32_t* d_counts,
                                     cudaStream_t st) {
    DevSchedule ds;
    ds.base = s->base;
    ds.kind = s->kind;
    ds.a_num = s->alpha.num;
    ds.a_den = s->alpha.den;
    ds.lo_num = s->alpha_min.num;
    ds.lo_den = s->alpha_min.den;
    ds.hi_num = s->alpha_max.num;
    ds.hi_den = s->alpha_max.den;
    ds.n_layers = s->n_layers;
    ds.coprime_c = s->coprime_c;
    ds.base_max = s->base_max;
    int threads = 64;
    int blocks = (n + threads - 1) / threads;
    KernelScope ks("offsets_device", st);
    build_tables_kernel<<<blocks, threads, 0, st>>>(ds, layer0, n, W, T, d_tables, d_counts);
    return launch_status("launch offsets kernel");
}

fibattn_status launch_keyset(const OffsetTables& t, int32_t W, int32_t T, uint32_t* d_mask,
                             cudaStream_t st) {
    int64_t total = (int64_t)T * ((T + 31) / 32);
    int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 0x7fffffff) return FIBATTN_ERR_INVALID_ARG;
    KernelScope ks("keyset_debug", st);
    keyset_kernel<<<(unsigned)blocks, threads, 0, st>>>(t, W, T, d_mask);
    return launch_status("launch offsets kernel");
}

}  // namespace fibattn
