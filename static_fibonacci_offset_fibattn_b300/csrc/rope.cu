// rope.cu -- rotary position embedding applied before the attention's gather.
//
// "Depth-Staggered Fibonacci Spacing for Sparse Attention" (gist.science explainer,
// Metodologia / Arquitetura, "Implementacao": RoPE is applied before the gather; Significancia:
// vanilla RoPE without scaling). Row i of a [T][64] slice has each pair (2p, 2p+1) rotated by
// i * theta_p, theta_p = base^(-2p/64):
//   y_2p = x_2p cos - x_2p+1 sin,  y_2p+1 = x_2p sin + x_2p+1 cos   (sin negated: inverse).
//
// The cos/sin table [T][32] (float2) is built once per (T, base) in fp64 and read through L2
// by the rotation kernel, a grid-stride stream over 16-byte chunks (one chunk = 4 pairs of
// bf16 or 2 pairs of fp32): HBM-bound, one read and one write of every row. x and y may be
// the same buffer (each chunk is read, then written, by one thread).
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "internal.h"

namespace fibattn {
namespace {

constexpr int kPairs = 32;  // d = 64

__global__ void rope_table_kernel(float2* __restrict__ table, int32_t T, double base) {
    const int64_t n = (int64_t)T * kPairs;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int32_t i = (int32_t)(e / kPairs);
        const int p = (int)(e % kPairs);
        const double theta = pow(base, -2.0 * p / (2.0 * kPairs));
        double s, c;
        sincos((double)i * theta, &s, &c);
        table[e] = make_float2((float)c, (float)s);
    }
}

__device__ __forceinline__ float2 rot(float x0, float x1, float2 cs, float sgn) {
    const float s = sgn * cs.y;
    return make_float2(x0 * cs.x - x1 * s, x0 * s + x1 * cs.x);
}

// bf16: chunk = 8 elements = 4 pairs; 8 chunks per row
__global__ void __launch_bounds__(256)
rope_bf16_kernel(const uint4* x, uint4* y, int64_t chunks, int32_t T,
                 const float4* __restrict__ table, float sgn) {
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < chunks;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = e >> 3;
        const int c = (int)(e & 7);
        const int32_t i = (int32_t)(row % T);
        const uint4 v = x[e];
        // pairs 4c .. 4c+3: two float4 of (cos, sin, cos, sin)
        const float4 t0 = __ldg(table + (int64_t)i * (kPairs / 2) + 2 * c);
        const float4 t1 = __ldg(table + (int64_t)i * (kPairs / 2) + 2 * c + 1);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        const float2 cs[4] = {make_float2(t0.x, t0.y), make_float2(t0.z, t0.w),
                              make_float2(t1.x, t1.y), make_float2(t1.z, t1.w)};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[q]);
            const float2 f = __bfloat1622float2(h);
            const __nv_bfloat162 r = __float22bfloat162_rn(rot(f.x, f.y, cs[q], sgn));
            o[q] = *reinterpret_cast<const uint32_t*>(&r);
        }
        y[e] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// fp32: chunk = 4 elements = 2 pairs; 16 chunks per row
__global__ void __launch_bounds__(256)
rope_f32_kernel(const float4* x, float4* y, int64_t chunks, int32_t T,
                const float4* __restrict__ table, float sgn) {
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < chunks;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = e >> 4;
        const int c = (int)(e & 15);
        const int32_t i = (int32_t)(row % T);
        const float4 v = x[e];
        const float4 t = __ldg(table + (int64_t)i * (kPairs / 2) + c);
        const float2 a = rot(v.x, v.y, make_float2(t.x, t.y), sgn);
        const float2 b = rot(v.z, v.w, make_float2(t.z, t.w), sgn);
        y[e] = make_float4(a.x, a.y, b.x, b.y);
    }
}

int grid_for(int64_t n, int threads) {
    static int n_sm[64] = {};
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) {
        if (n_sm[dev] == 0 && cudaDeviceGetAttribute(&n_sm[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            n_sm[dev] = 0;
        if (n_sm[dev] > 0) sms = n_sm[dev];
    }
    const int64_t want = (n + threads - 1) / threads;
    const int64_t cap = (int64_t)sms * 8;  // 8 resident blocks of 256 per SM
    return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

fibattn_status launch_rope_table(float* table, int32_t T, double base, cudaStream_t st) {
    const int64_t n = (int64_t)T * kPairs;
    {
        KernelScope ks("rope_table", st);
        rope_table_kernel<<<grid_for(n, 256), 256, 0, st>>>(reinterpret_cast<float2*>(table), T, base);
    }
    return launch_status("launch rope_table");
}

fibattn_status launch_rope(const void* x, void* y, int64_t rows, int32_t T, int32_t dtype,
                           const float* table, bool inverse, cudaStream_t st) {
    const float sgn = inverse ? -1.f : 1.f;
    const float4* t4 = reinterpret_cast<const float4*>(table);
    if (dtype == FIBATTN_BF16) {
        const int64_t chunks = rows * 8;
        KernelScope ks("rope_bf16", st);
        rope_bf16_kernel<<<grid_for(chunks, 256), 256, 0, st>>>(
            static_cast<const uint4*>(x), static_cast<uint4*>(y), chunks, T, t4, sgn);
    } else {
        const int64_t chunks = rows * 16;
        KernelScope ks("rope_f32", st);
        rope_f32_kernel<<<grid_for(chunks, 256), 256, 0, st>>>(
            static_cast<const float4*>(x), static_cast<float4*>(y), chunks, T, t4, sgn);
    }
    return launch_status("launch rope");
}

}  // namespace fibattn
