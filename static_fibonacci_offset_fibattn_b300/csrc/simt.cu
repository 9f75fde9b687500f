// simt.cu -- SIMT (CUDA-core) kernels: the fp32 forward and the backward.
//
// One warp owns one row; lane l holds head dims N l .. N l + N - 1 (N = d / 32: 2 at d = 64,
// 4 at d = 128), so every K/V/Q row is read by one coalesced warp access and dot products
// finish with an xor shuffle reduction (every lane receives the sum, bit-identically). The
// fractional-offset kernels are written for d = 64.
//
// Attended set ("Depth-Staggered Fibonacci Spacing for Sparse Attention", gist.science
// explainer, Metodologia / Arquitetura, "Conjunto Atendido"): query i sees keys
// i - W + 1 .. i (clipped at 0) and i - o for each table offset o <= i. Table offsets
// are >= W, so the two parts never overlap.
#include <math.h>
#include <stdint.h>

#include "internal.h"

namespace fibattn {
namespace {

constexpr int kD = 64;
constexpr int kWarpsPerBlock = 8;

template <typename E>
struct Io;

template <>
struct Io<float> {
    static __device__ __forceinline__ float2 ld(const float* p) {
        return __ldg(reinterpret_cast<const float2*>(p));
    }
    static __device__ __forceinline__ void st(float* p, float2 x) {
        *reinterpret_cast<float2*>(p) = x;
    }
};


// Element offset of the kv slice read by query slice `s` of launch layer `layer` (query head h
// of batch b reads kv head h / group of batch b; K/V hold slices_per_layer / group slices).
__device__ __forceinline__ int64_t kv_base(const AttnShape& sh, int layer, int64_t s, int d = 64) {
    return ((int64_t)layer * (sh.slices_per_layer / sh.group) + s / sh.group) * sh.T * d;
}

// N consecutive elements of a row in fp32 registers (N = 2 or 4).
template <int N>
struct Vec {
    float x[N];
};

template <typename E, int N>
struct VIo;
template <>
struct VIo<float, 2> {
    static __device__ __forceinline__ Vec<2> ld(const float* p) {
        const float2 a = __ldg(reinterpret_cast<const float2*>(p));
        return Vec<2>{{a.x, a.y}};
    }
    static __device__ __forceinline__ void st(float* p, const Vec<2>& v) {
        *reinterpret_cast<float2*>(p) = make_float2(v.x[0], v.x[1]);
    }
};
template <>
struct VIo<float, 4> {
    static __device__ __forceinline__ Vec<4> ld(const float* p) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(p));
        return Vec<4>{{a.x, a.y, a.z, a.w}};
    }
    static __device__ __forceinline__ void st(float* p, const Vec<4>& v) {
        *reinterpret_cast<float4*>(p) = make_float4(v.x[0], v.x[1], v.x[2], v.x[3]);
    }
};

// this lane's part of a . b (the N = 2 form is the two-term sum x0 y0 + x1 y1)
template <int N>
__device__ __forceinline__ float dot_part(const Vec<N>& a, const Vec<N>& b) {
    float s = a.x[0] * b.x[0] + a.x[1] * b.x[1];
#pragma unroll
    for (int t = 2; t < N; t += 2) s += a.x[t] * b.x[t] + a.x[t + 1] * b.x[t + 1];
    return s;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    return x;
}

// ---------------------------------------------------------------- forward (fp32 path)
// Online softmax over S_i in fp32: running max m, running sum l, accumulator acc.
template <typename E, int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
fwd_simt_kernel(const E* __restrict__ q, const E* __restrict__ k, const E* __restrict__ v,
                E* __restrict__ o, float* __restrict__ lse, AttnShape sh,
                const __grid_constant__ OffsetTables tab) {
    constexpr int N = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t rows = sh.slices_per_layer * sh.T;
    const int64_t row = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    const int layer = blockIdx.y;
    if (row >= rows) return;
    const int64_t slice = (int64_t)layer * sh.slices_per_layer + row / sh.T;
    const int32_t i = (int32_t)(row % sh.T);
    const int64_t base = slice * sh.T * D;
    const int64_t kbase = kv_base(sh, layer, row / sh.T, D);
    const Vec<N> qv = VIo<E, N>::ld(q + base + (int64_t)i * D + N * lane);

    float m = -INFINITY, l = 0.f;
    Vec<N> acc;
#pragma unroll
    for (int t = 0; t < N; ++t) acc.x[t] = 0.f;
    auto visit = [&](int32_t j) {
        const Vec<N> kv = VIo<E, N>::ld(k + kbase + (int64_t)j * D + N * lane);
        const float s = warp_sum(dot_part(qv, kv)) * sh.scale;
        const Vec<N> vv = VIo<E, N>::ld(v + kbase + (int64_t)j * D + N * lane);
        const float mn = fmaxf(m, s);
        const float corr = expf(m - mn);  // m = -inf on the first key: corr = 0
        const float p = expf(s - mn);
        l = l * corr + p;
#pragma unroll
        for (int t = 0; t < N; ++t) acc.x[t] = acc.x[t] * corr + p * vv.x[t];
        m = mn;
    };
    const int n_off = tab.count[layer];
    for (int e = n_off - 1; e >= 0; --e) {
        const int32_t j = i - tab.off[layer][e];
        if (j >= 0) visit(j);
    }
    const int32_t j0 = i - sh.W + 1 > 0 ? i - sh.W + 1 : 0;
    for (int32_t j = j0; j <= i; ++j) visit(j);

    const float inv = 1.f / l;
#pragma unroll
    for (int t = 0; t < N; ++t) acc.x[t] *= inv;
    VIo<E, N>::st(o + base + (int64_t)i * D + N * lane, acc);
    if (lane == 0) lse[slice * sh.T + i] = m + logf(l);
}

// Fractional offsets (the learned-alpha variant; Metodologia / Arquitetura, "Implementacao"):
// each real distance d, held as c = ceil(d) and w = c - d, contributes for i >= c one key and
// value interpolated between rows i - c and i - c + 1: x~ = (1 - w) x_{i-c} + w x_{i-c+1}.
template <typename E>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
fwd_frac_simt_kernel(const E* __restrict__ q, const E* __restrict__ k, const E* __restrict__ v,
                     E* __restrict__ o, float* __restrict__ lse, AttnShape sh,
                     const __grid_constant__ FracTables tab) {
    const int lane = threadIdx.x & 31;
    const int64_t rows = sh.slices_per_layer * sh.T;
    const int64_t row = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    const int layer = blockIdx.y;
    if (row >= rows) return;
    const int64_t slice = (int64_t)layer * sh.slices_per_layer + row / sh.T;
    const int32_t i = (int32_t)(row % sh.T);
    const int64_t base = slice * sh.T * kD;
    const float2 qv = Io<E>::ld(q + base + (int64_t)i * kD + 2 * lane);

    float m = -INFINITY, l = 0.f;
    float2 acc = make_float2(0.f, 0.f);
    auto visit = [&](float2 kv, float2 vv) {
        const float s = warp_sum(qv.x * kv.x + qv.y * kv.y) * sh.scale;
        const float mn = fmaxf(m, s);
        const float corr = expf(m - mn);  // m = -inf on the first key: corr = 0
        const float p = expf(s - mn);
        l = l * corr + p;
        acc.x = acc.x * corr + p * vv.x;
        acc.y = acc.y * corr + p * vv.y;
        m = mn;
    };
    const int64_t kbase = kv_base(sh, layer, row / sh.T);
    auto row_of = [&](const E* x, int32_t j) { return Io<E>::ld(x + kbase + (int64_t)j * kD + 2 * lane); };
    const int n_off = tab.c.count[layer];
    for (int e = n_off - 1; e >= 0; --e) {
        const int32_t j = i - tab.c.off[layer][e];
        if (j < 0) continue;
        const float w = tab.w[layer][e];
        float2 kv = row_of(k, j), vv = row_of(v, j);
        if (w != 0.f) {  // j + 1 <= i - W + 1 <= i: inside the sequence
            const float2 k1 = row_of(k, j + 1), v1 = row_of(v, j + 1);
            kv = make_float2((1.f - w) * kv.x + w * k1.x, (1.f - w) * kv.y + w * k1.y);
            vv = make_float2((1.f - w) * vv.x + w * v1.x, (1.f - w) * vv.y + w * v1.y);
        }
        visit(kv, vv);
    }
    const int32_t j0 = i - sh.W + 1 > 0 ? i - sh.W + 1 : 0;
    for (int32_t j = j0; j <= i; ++j) visit(row_of(k, j), row_of(v, j));

    const float inv = 1.f / l;
    Io<E>::st(o + base + (int64_t)i * kD + 2 * lane, make_float2(acc.x * inv, acc.y * inv));
    if (lane == 0) lse[slice * sh.T + i] = m + logf(l);
}

// ---------------------------------------------------------------- backward
// D_i = dO_i . O_i
template <typename E, int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
bwd_delta_kernel(const E* __restrict__ o, const E* __restrict__ dO, float* __restrict__ delta,
                 int64_t total_rows) {
    constexpr int N = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (row >= total_rows) return;
    const Vec<N> a = VIo<E, N>::ld(o + row * D + N * lane);
    const Vec<N> b = VIo<E, N>::ld(dO + row * D + N * lane);
    const float s = warp_sum(dot_part(a, b));
    if (lane == 0) delta[row] = s;
}

// dQ_i = scale * sum_{j in S_i} P_ij (dO_i . v_j - D_i) k_j   (query owner)
template <typename E, int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
bwd_dq_kernel(const E* __restrict__ q, const E* __restrict__ k, const E* __restrict__ v,
              const float* __restrict__ lse, const E* __restrict__ dO,
              const float* __restrict__ delta, E* __restrict__ dq, AttnShape sh,
              const __grid_constant__ OffsetTables tab) {
    constexpr int N = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t rows = sh.slices_per_layer * sh.T;
    const int64_t row = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    const int layer = blockIdx.y;
    if (row >= rows) return;
    const int64_t slice = (int64_t)layer * sh.slices_per_layer + row / sh.T;
    const int32_t i = (int32_t)(row % sh.T);
    const int64_t base = slice * sh.T * D;
    const int64_t ri = base + (int64_t)i * D + N * lane;
    const Vec<N> qv = VIo<E, N>::ld(q + ri);
    const Vec<N> gv = VIo<E, N>::ld(dO + ri);
    const float Li = lse[slice * sh.T + i];
    const float Di = delta[slice * sh.T + i];
    const int64_t kbase = kv_base(sh, layer, row / sh.T, D);
    Vec<N> acc;
#pragma unroll
    for (int t = 0; t < N; ++t) acc.x[t] = 0.f;
    auto visit = [&](int32_t j) {
        const int64_t rj = kbase + (int64_t)j * D + N * lane;
        const Vec<N> kv = VIo<E, N>::ld(k + rj);
        const Vec<N> vv = VIo<E, N>::ld(v + rj);
        const float s = warp_sum(dot_part(qv, kv));
        const float dp = warp_sum(dot_part(gv, vv));
        const float p = expf(s * sh.scale - Li);
        const float ds = p * (dp - Di);
#pragma unroll
        for (int t = 0; t < N; ++t) acc.x[t] += ds * kv.x[t];
    };
    for (int e = tab.count[layer] - 1; e >= 0; --e) {
        const int32_t j = i - tab.off[layer][e];
        if (j >= 0) visit(j);
    }
    const int32_t j0 = i - sh.W + 1 > 0 ? i - sh.W + 1 : 0;
    for (int32_t j = j0; j <= i; ++j) visit(j);
#pragma unroll
    for (int t = 0; t < N; ++t) acc.x[t] *= sh.scale;
    VIo<E, N>::st(dq + ri, acc);
}

// dK_j = scale * sum_{i : j in S_i} dS_ij q_i,  dV_j = sum_{i : j in S_i} P_ij dO_i  (key owner)
// The queries that see key j: i = j + t for 0 <= t < W, and i = j + o for table offsets o,
// each only while i < T, in each of the `group` query heads that read this kv head. One warp
// per kv row; no atomics: this warp is the only writer of row j.
template <typename E, int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
bwd_dkdv_kernel(const E* __restrict__ q, const E* __restrict__ k, const E* __restrict__ v,
                const float* __restrict__ lse, const E* __restrict__ dO,
                const float* __restrict__ delta, E* __restrict__ dk, E* __restrict__ dv,
                AttnShape sh, const __grid_constant__ OffsetTables tab) {
    constexpr int N = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t spl_kv = sh.slices_per_layer / sh.group;
    const int64_t rows = spl_kv * sh.T;
    const int64_t row = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    const int layer = blockIdx.y;
    if (row >= rows) return;
    const int64_t skv = row / sh.T;  // kv slice within the layer
    const int32_t j = (int32_t)(row % sh.T);
    const int64_t rj = ((int64_t)layer * spl_kv + skv) * sh.T * D + (int64_t)j * D + N * lane;
    const Vec<N> kv = VIo<E, N>::ld(k + rj);
    const Vec<N> vv = VIo<E, N>::ld(v + rj);
    Vec<N> ak, av;
#pragma unroll
    for (int t = 0; t < N; ++t) ak.x[t] = av.x[t] = 0.f;
    for (int g = 0; g < sh.group; ++g) {
        const int64_t slice = (int64_t)layer * sh.slices_per_layer + skv * sh.group + g;
        const int64_t base = slice * sh.T * D;
        auto visit = [&](int32_t i) {
            const int64_t ri = base + (int64_t)i * D + N * lane;
            const Vec<N> qv = VIo<E, N>::ld(q + ri);
            const Vec<N> gv = VIo<E, N>::ld(dO + ri);
            const float s = warp_sum(dot_part(qv, kv));
            const float dp = warp_sum(dot_part(gv, vv));
            const float p = expf(s * sh.scale - lse[slice * sh.T + i]);
            const float ds = p * (dp - delta[slice * sh.T + i]);
#pragma unroll
            for (int t = 0; t < N; ++t) {
                av.x[t] += p * gv.x[t];
                ak.x[t] += ds * qv.x[t];
            }
        };
        const int32_t i1 = j + sh.W - 1 < sh.T - 1 ? j + sh.W - 1 : sh.T - 1;
        for (int32_t i = j; i <= i1; ++i) visit(i);
        for (int e = 0; e < tab.count[layer]; ++e) {
            const int64_t i = (int64_t)j + tab.off[layer][e];
            if (i < sh.T) visit((int32_t)i);
        }
    }
#pragma unroll
    for (int t = 0; t < N; ++t) ak.x[t] *= sh.scale;
    VIo<E, N>::st(dk + rj, ak);
    VIo<E, N>::st(dv + rj, av);
}

// ---------------------------------------------------------------- fractional backward
// The rows interpolated at i - d (c = ceil(d), w = c - d, rows lo = i - c and lo + 1):
//   k~ = (1 - w) k_lo + w k_lo+1, v~ likewise; s = scale q.k~, P = exp(s - lse), dS = P (dO.v~ - D)
//   dq_i += scale dS k~;  dk_lo += (1 - w) scale dS q_i, dk_lo+1 += w scale dS q_i;
//   dv_lo += (1 - w) P dO_i, dv_lo+1 += w P dO_i;
//   dL/dd = dS scale q.(k_lo - k_lo+1) + P dO.(v_lo - v_lo+1)  (the segment [lo, lo+1] even
//   at w = 0), and the query's share of dL/dalpha is g_i = sum_k f_k dL/dd_k.

// Query owner: dq and g_i (into galpha).
template <typename E>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
bwd_dq_frac_kernel(const E* __restrict__ q, const E* __restrict__ k, const E* __restrict__ v,
                   const float* __restrict__ lse, const E* __restrict__ dO,
                   const float* __restrict__ delta, E* __restrict__ dq, float* __restrict__ galpha,
                   AttnShape sh, const __grid_constant__ FracTables tab) {
    const int lane = threadIdx.x & 31;
    const int64_t rows = sh.slices_per_layer * sh.T;
    const int64_t row = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    const int layer = blockIdx.y;
    if (row >= rows) return;
    const int64_t slice = (int64_t)layer * sh.slices_per_layer + row / sh.T;
    const int32_t i = (int32_t)(row % sh.T);
    const int64_t base = slice * sh.T * kD;
    const int64_t kbase = kv_base(sh, layer, row / sh.T);
    auto row_of = [&](const E* x, int32_t j) { return Io<E>::ld(x + kbase + (int64_t)j * kD + 2 * lane); };
    const float2 qv = Io<E>::ld(q + base + (int64_t)i * kD + 2 * lane);
    const float2 gv = Io<E>::ld(dO + base + (int64_t)i * kD + 2 * lane);
    const float Li = lse[slice * sh.T + i];
    const float Di = delta[slice * sh.T + i];
    // the static kernel's order (distances descending, then the window), so that an integer
    // alpha gives its results bit for bit
    float2 acc = make_float2(0.f, 0.f);
    float ga = 0.f;
    for (int e = tab.c.count[layer] - 1; e >= 0; --e) {
        const int32_t lo = i - tab.c.off[layer][e];
        if (lo < 0) continue;
        const float w = tab.w[layer][e];
        const float2 k0 = row_of(k, lo), k1 = row_of(k, lo + 1);  // lo + 1 <= i
        const float2 v0 = row_of(v, lo), v1 = row_of(v, lo + 1);
        const float2 kt = make_float2((1.f - w) * k0.x + w * k1.x, (1.f - w) * k0.y + w * k1.y);
        const float2 vt = make_float2((1.f - w) * v0.x + w * v1.x, (1.f - w) * v0.y + w * v1.y);
        const float s = warp_sum(qv.x * kt.x + qv.y * kt.y);
        const float dp = warp_sum(gv.x * vt.x + gv.y * vt.y);
        const float sdiff = warp_sum(qv.x * (k0.x - k1.x) + qv.y * (k0.y - k1.y));
        const float vdiff = warp_sum(gv.x * (v0.x - v1.x) + gv.y * (v0.y - v1.y));
        const float p = expf(s * sh.scale - Li);
        const float ds = p * (dp - Di);
        acc.x += ds * kt.x;
        acc.y += ds * kt.y;
        ga += tab.f[layer][e] * (ds * sh.scale * sdiff + p * vdiff);
    }
    const int32_t j0 = i - sh.W + 1 > 0 ? i - sh.W + 1 : 0;
    for (int32_t j = j0; j <= i; ++j) {
        const float2 kv = row_of(k, j), vv = row_of(v, j);
        const float s = warp_sum(qv.x * kv.x + qv.y * kv.y);
        const float dp = warp_sum(gv.x * vv.x + gv.y * vv.y);
        const float p = expf(s * sh.scale - Li);
        const float ds = p * (dp - Di);
        acc.x += ds * kv.x;
        acc.y += ds * kv.y;
    }
    Io<E>::st(dq + base + (int64_t)i * kD + 2 * lane, make_float2(acc.x * sh.scale, acc.y * sh.scale));
    if (lane == 0) galpha[slice * sh.T + i] = ga;
}

// Key owner: key j is row lo of the query i = j + c (weight 1 - w) and row lo + 1 of the
// query i = j + c - 1 (weight w), for every distance; plus its window queries j .. j+W-1.
template <typename E>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
bwd_dkdv_frac_kernel(const E* __restrict__ q, const E* __restrict__ k, const E* __restrict__ v,
                     const float* __restrict__ lse, const E* __restrict__ dO,
                     const float* __restrict__ delta, E* __restrict__ dk, E* __restrict__ dv,
                     AttnShape sh, const __grid_constant__ FracTables tab) {
    const int lane = threadIdx.x & 31;
    const int64_t spl_kv = sh.slices_per_layer / sh.group;
    const int64_t rows = spl_kv * sh.T;
    const int64_t row = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    const int layer = blockIdx.y;
    if (row >= rows) return;
    const int64_t skv = row / sh.T;  // kv slice within the layer
    const int32_t j = (int32_t)(row % sh.T);
    const int64_t kb = ((int64_t)layer * spl_kv + skv) * sh.T * kD;
    auto kv_row = [&](const E* x, int32_t r) { return Io<E>::ld(x + kb + (int64_t)r * kD + 2 * lane); };
    const float2 kv = kv_row(k, j);
    const float2 vv = kv_row(v, j);
    float2 ak = make_float2(0.f, 0.f), av = make_float2(0.f, 0.f);
    for (int g = 0; g < sh.group; ++g) {
        const int64_t slice = (int64_t)layer * sh.slices_per_layer + skv * sh.group + g;
        const int64_t base = slice * sh.T * kD;
        // query i sees key and value rows (kx, vx); this key's share of them is wt
        auto visit = [&](int32_t i, float2 kx, float2 vx, float wt) {
            const float2 qv = Io<E>::ld(q + base + (int64_t)i * kD + 2 * lane);
            const float2 gv = Io<E>::ld(dO + base + (int64_t)i * kD + 2 * lane);
            const float s = warp_sum(qv.x * kx.x + qv.y * kx.y);
            const float dp = warp_sum(gv.x * vx.x + gv.y * vx.y);
            const float p = expf(s * sh.scale - lse[slice * sh.T + i]);
            const float ds = p * (dp - delta[slice * sh.T + i]);
            av.x += wt * p * gv.x;
            av.y += wt * p * gv.y;
            ak.x += wt * ds * qv.x;
            ak.y += wt * ds * qv.y;
        };
        const int32_t i1 = j + sh.W - 1 < sh.T - 1 ? j + sh.W - 1 : sh.T - 1;
        for (int32_t i = j; i <= i1; ++i) visit(i, kv, vv, 1.f);
        for (int e = 0; e < tab.c.count[layer]; ++e) {
            const int64_t c = tab.c.off[layer][e];
            const float w = tab.w[layer][e];
            if ((int64_t)j + c < sh.T) {  // row lo of query j + c: the other row is j + 1 <= j + c
                const float2 k1 = kv_row(k, j + 1), v1 = kv_row(v, j + 1);
                visit((int32_t)(j + c), make_float2((1.f - w) * kv.x + w * k1.x, (1.f - w) * kv.y + w * k1.y),
                      make_float2((1.f - w) * vv.x + w * v1.x, (1.f - w) * vv.y + w * v1.y), 1.f - w);
            }
            if (w != 0.f && j >= 1 && (int64_t)j + c - 1 < sh.T) {  // row lo + 1 of query j + c - 1
                const float2 k0 = kv_row(k, j - 1), v0 = kv_row(v, j - 1);
                visit((int32_t)(j + c - 1), make_float2((1.f - w) * k0.x + w * kv.x, (1.f - w) * k0.y + w * kv.y),
                      make_float2((1.f - w) * v0.x + w * vv.x, (1.f - w) * v0.y + w * vv.y), w);
            }
        }
    }
    Io<E>::st(dk + kb + (int64_t)j * kD + 2 * lane, make_float2(ak.x * sh.scale, ak.y * sh.scale));
    Io<E>::st(dv + kb + (int64_t)j * kD + 2 * lane, av);
}

// One block per layer: a fixed-order sum (strided fp64 partials, then a tree) of its rows.
constexpr int kReduceThreads = 1024;
__global__ void __launch_bounds__(kReduceThreads)
dalpha_reduce_kernel(const float* __restrict__ galpha, float* __restrict__ dalpha, int64_t rows) {
    __shared__ double part[kReduceThreads];
    const float* g = galpha + (int64_t)blockIdx.x * rows;
    double a = 0.0;
    for (int64_t r = threadIdx.x; r < rows; r += kReduceThreads) a += (double)g[r];
    part[threadIdx.x] = a;
    __syncthreads();
    for (int s = kReduceThreads / 2; s > 0; s >>= 1) {
        if ((int)threadIdx.x < s) part[threadIdx.x] += part[threadIdx.x + s];
        __syncthreads();
    }
    if (threadIdx.x == 0) dalpha[blockIdx.x] = (float)part[0];
}

}  // namespace

fibattn_status launch_dalpha_reduce(const float* galpha, float* dalpha, int32_t n,
                                    int64_t rows_per_layer, cudaStream_t st) {
    KernelScope ks("dalpha_reduce", st);
    dalpha_reduce_kernel<<<n, kReduceThreads, 0, st>>>(galpha, dalpha, rows_per_layer);
    return launch_status("launch dalpha_reduce");
}

fibattn_status launch_bwd_frac_simt_f32(const float* q, const float* k, const float* v,
                                        const float* o, const float* lse, const float* dO,
                                        float* dq, float* dk, float* dv, float* delta,
                                        float* galpha, const AttnShape& sh, const FracTables& t,
                                        cudaStream_t st) {
    const int64_t rows = sh.slices_per_layer * sh.T;
    const int64_t blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
    const int64_t all_rows = rows * sh.n_layers;
    const int64_t dblocks = (all_rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (blocks > 0x7fffffff || dblocks > 0x7fffffff) return FIBATTN_ERR_INVALID_ARG;
    {
        KernelScope ks("bwd_delta_simt", st);
        bwd_delta_kernel<float, 64><<<(unsigned)dblocks, kWarpsPerBlock * 32, 0, st>>>(o, dO, delta, all_rows);
    }
    dim3 grid((unsigned)blocks, sh.n_layers);
    {
        KernelScope ks("bwd_dq_frac_simt", st);
        bwd_dq_frac_kernel<float><<<grid, kWarpsPerBlock * 32, 0, st>>>(q, k, v, lse, dO, delta, dq,
                                                                         galpha, sh, t);
    }
    {
        // one warp per kv row
        const int64_t kv_rows = sh.slices_per_layer / sh.group * sh.T;
        dim3 kgrid((unsigned)((kv_rows + kWarpsPerBlock - 1) / kWarpsPerBlock), sh.n_layers);
        KernelScope ks("bwd_dkdv_frac_simt", st);
        bwd_dkdv_frac_kernel<float><<<kgrid, kWarpsPerBlock * 32, 0, st>>>(q, k, v, lse, dO, delta,
                                                                            dk, dv, sh, t);
    }
    return launch_status("launch SIMT kernel");
}

fibattn_status launch_fwd_simt_f32(const float* q, const float* k, const float* v, float* o,
                                   float* lse, const AttnShape& sh, const OffsetTables& t,
                                   cudaStream_t st) {
    const int64_t rows = sh.slices_per_layer * sh.T;
    const int64_t blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (blocks > 0x7fffffff) return FIBATTN_ERR_INVALID_ARG;
    dim3 grid((unsigned)blocks, sh.n_layers);
    KernelScope ks("fwd_simt_f32", st);
    if (sh.d == 128)
        fwd_simt_kernel<float, 128><<<grid, kWarpsPerBlock * 32, 0, st>>>(q, k, v, o, lse, sh, t);
    else
        fwd_simt_kernel<float, 64><<<grid, kWarpsPerBlock * 32, 0, st>>>(q, k, v, o, lse, sh, t);
    return launch_status("launch SIMT kernel");
}


fibattn_status launch_fwd_frac_simt_f32(const float* q, const float* k, const float* v, float* o,
                                        float* lse, const AttnShape& sh, const FracTables& t,
                                        cudaStream_t st) {
    const int64_t rows = sh.slices_per_layer * sh.T;
    const int64_t blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (blocks > 0x7fffffff) return FIBATTN_ERR_INVALID_ARG;
    dim3 grid((unsigned)blocks, sh.n_layers);
    KernelScope ks("fwd_frac_simt_f32", st);
    fwd_frac_simt_kernel<float><<<grid, kWarpsPerBlock * 32, 0, st>>>(q, k, v, o, lse, sh, t);
    return launch_status("launch SIMT kernel");
}

template <typename E, int D>
static fibattn_status bwd_typed(const E* q, const E* k, const E* v, const E* o, const float* lse,
                                const E* dO, E* dq, E* dk, E* dv, float* delta,
                                const AttnShape& sh, const OffsetTables& t, cudaStream_t st) {
    const int64_t rows = sh.slices_per_layer * sh.T;
    const int64_t blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
    const int64_t all_rows = rows * sh.n_layers;
    const int64_t dblocks = (all_rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (blocks > 0x7fffffff || dblocks > 0x7fffffff) return FIBATTN_ERR_INVALID_ARG;
    {
        KernelScope ks("bwd_delta_simt", st);
        bwd_delta_kernel<E, D><<<(unsigned)dblocks, kWarpsPerBlock * 32, 0, st>>>(o, dO, delta, all_rows);
    }
    dim3 grid((unsigned)blocks, sh.n_layers);
    {
        KernelScope ks("bwd_dq_simt", st);
        bwd_dq_kernel<E, D><<<grid, kWarpsPerBlock * 32, 0, st>>>(q, k, v, lse, dO, delta, dq, sh, t);
    }
    {
        // one warp per kv row
        const int64_t kv_rows = sh.slices_per_layer / sh.group * sh.T;
        dim3 kgrid((unsigned)((kv_rows + kWarpsPerBlock - 1) / kWarpsPerBlock), sh.n_layers);
        KernelScope ks("bwd_dkdv_simt", st);
        bwd_dkdv_kernel<E, D><<<kgrid, kWarpsPerBlock * 32, 0, st>>>(q, k, v, lse, dO, delta, dk, dv, sh, t);
    }
    return launch_status("launch SIMT kernel");
}

fibattn_status launch_bwd_simt_f32(const float* q, const float* k, const float* v, const float* o,
                                   const float* lse, const float* dO, float* dq, float* dk,
                                   float* dv, float* delta, const AttnShape& sh,
                                   const OffsetTables& t, cudaStream_t st) {
    if (sh.d == 128) return bwd_typed<float, 128>(q, k, v, o, lse, dO, dq, dk, dv, delta, sh, t, st);
    return bwd_typed<float, 64>(q, k, v, o, lse, dO, dq, dk, dv, delta, sh, t, st);
}

}  // namespace fibattn
