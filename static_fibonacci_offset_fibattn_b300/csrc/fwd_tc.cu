// fwd_tc.cu -- bf16 forward of Fibonacci-offset sparse attention on sm_103a tensor cores.
//
// What is computed ("Depth-Staggered Fibonacci Spacing for Sparse Attention", gist.science
// explainer, Metodologia / Arquitetura e Mecanismo de Atencao, "Conjunto Atendido"):
// query i attends the dense window i-W+1..i and the keys i-o for the layer's offsets o;
// o_i = softmax(scale * q_i . k_j over those keys) . v_j, lse_i = log sum_j exp(...).
// The pages' static variants use fused boolean masking instead of a gather (same page,
// Principais Contribuicoes 2, "Eficiencia"); here the window is a masked dense band on
// the tensor cores and each offset is a diagonal handled by CUDA-core row dot products.
//
// One CTA = one tile of 128 queries [i0, i0+128) of one (layer, batch, head) slice.
//   warps 0-3 : one thread per query row (TMEM lane = row); softmax, offsets, epilogue.
//   warp 4    : TMEM allocation, band TMA loads, tcgen05.mma issue (lane 0).
//   warp 5    : TMA loads of the shifted offset tiles into a 2-stage ring (lane 0).
// Band: keys [max(0, i0-W+1), i0+127] in 64-key chunks, up to 3 chunks per group:
//   S = Q K^T (tcgen05, M=128, N=64*chunks, K=64) -> TMEM columns [0, 192)
//   masked online softmax per row (fp32, log2 domain), P (bf16) written back over S
//   O_band += P V (tcgen05, A = P from TMEM, B = V MN-major in smem) -> TMEM [192, 256)
// Offsets: for table entry o the shifted tiles K[i0-o .. i0-o+127], V[same] arrive by TMA
//   (negative rows zero-filled); thread r takes row r of each: s = q_r . k_{i-o}, then a
//   second pass accumulates exp(s - m) v_{i-o} in registers. The band and offset parts
//   keep separate running maxima and are merged once in the epilogue.
// Epilogue: O = (O_band 2^(m_b-m) + O_off 2^(m_o-m)) / l, staged to smem, TMA-stored;
//   lse = (m + log2 l) ln 2.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "internal.h"
#include "tc_prims.cuh"
#include "tmap.h"

namespace fibattn {
namespace {

using namespace tc;

constexpr int kRows = 128;          // queries per tile
constexpr int kChunk = 64;          // keys per band chunk (one TMA box)
constexpr int kMaxGroupChunks = 3;  // band chunks per S group (N <= 192)
constexpr int kRing = 2;            // offset-tile ring stages
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTmemO = 192;    // O accumulator columns [192, 256)

constexpr uint32_t kTileBytes = kRows * 128;    // 16 KB: 128 rows x 64 bf16
constexpr uint32_t kChunkBytes = kChunk * 128;  // 8 KB
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileBytes;
constexpr uint32_t kOffV = kOffK + kMaxGroupChunks * kChunkBytes;
constexpr uint32_t kOffRing = kOffV + kMaxGroupChunks * kChunkBytes;
constexpr uint32_t kOffBar = kOffRing + kRing * kTileBytes;
// barriers: q, k, v, s, p, o, full[kRing], empty[kRing]; then the TMEM address word
constexpr uint32_t kNumBars = 6 + 2 * kRing;
constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemBytes = kOffTmemSlot + 16;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;  // slack for 1024-byte alignment

struct FwdParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_o;  // 3D {64, T, slices}, box {64, 64, 1}, 128B swizzle
    float* lse;
    int32_t* err;
    int64_t slices_per_layer;
    int32_t T, W;
    int32_t tiles_per_slice;
    float scale_log2;  // scale * log2(e)
    OffsetTables tabs;
};

__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int idx) { return base + kOffBar + 8u * idx; }

__global__ void __launch_bounds__(kThreads, 2)
fwd_tc_kernel(const __grid_constant__ FwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - smem_u32(smem_raw));

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int layer = blockIdx.y;
    const int tile = blockIdx.x % p.tiles_per_slice;
    const int64_t slice = (int64_t)layer * p.slices_per_layer + blockIdx.x / p.tiles_per_slice;
    const int32_t z = (int32_t)slice;
    const int32_t T = p.T, W = p.W;
    const int32_t i0 = tile * kRows;

    const uint32_t B_Q = bar_addr(sbase, 0), B_K = bar_addr(sbase, 1), B_V = bar_addr(sbase, 2);
    const uint32_t B_S = bar_addr(sbase, 3), B_P = bar_addr(sbase, 4), B_O = bar_addr(sbase, 5);
    auto B_FULL = [&](int s) { return bar_addr(sbase, 6 + s); };
    auto B_EMPTY = [&](int s) { return bar_addr(sbase, 6 + kRing + s); };

    // band extent (64-key chunks) and active offsets (the table is ascending)
    const int32_t kstart = i0 - W + 1 > 0 ? i0 - W + 1 : 0;
    const int32_t klast = (i0 + kRows - 1 < T - 1) ? i0 + kRows - 1 : T - 1;
    const int32_t c_lo = kstart / kChunk;
    const int32_t n_chunks = klast / kChunk - c_lo + 1;
    const int32_t n_groups = (n_chunks + kMaxGroupChunks - 1) / kMaxGroupChunks;
    const int32_t* offs = p.tabs.off[layer];
    int32_t n_act = 0;
    for (int e = 0; e < p.tabs.count[layer]; ++e)
        if (offs[e] <= klast) n_act = e + 1;

    if (tid == 0) {
        for (int b = 0; b < (int)kNumBars; ++b) {
            uint32_t cnt = 1;
            if (b == 4) cnt = kRows;                       // P written by every row thread
            if (b >= 6 + kRing) cnt = kRows;               // ring slot released by every row
            mbar_init(bar_addr(sbase, b), cnt);
        }
        fence_mbar_init();
    }
    if (warp == 4) {
        tmem_alloc(sbase + kOffTmemSlot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmemSlot);
    bool aborted = false;

    if (warp == 4) {
        // ------------------------------------------------ band loads + MMA issue
        if (lane == 0) {
            prefetch_tmap(&p.tm_q);
            prefetch_tmap(&p.tm_k);
            prefetch_tmap(&p.tm_v);
            mbar_arrive_expect_tx(B_Q, kTileBytes);
            tma_load_3d(sbase + kOffQ, &p.tm_q, B_Q, 0, i0, z);
            tma_load_3d(sbase + kOffQ + kChunkBytes, &p.tm_q, B_Q, 0, i0 + kChunk, z);
            for (int g = 0; g < n_groups; ++g) {
                const int nch = min(kMaxGroupChunks, n_chunks - g * kMaxGroupChunks);
                const int32_t ybase = (c_lo + g * kMaxGroupChunks) * kChunk;
                if (g > 0) {  // K and V buffers (and the P columns) free again
                    mbar_wait(B_S, (g - 1) & 1, aborted, p.err);
                    mbar_wait(B_O, (g - 1) & 1, aborted, p.err);
                }
                mbar_arrive_expect_tx(B_K, nch * kChunkBytes);
                for (int c = 0; c < nch; ++c)
                    tma_load_3d(sbase + kOffK + c * kChunkBytes, &p.tm_k, B_K, 0, ybase + c * kChunk, z);
                mbar_arrive_expect_tx(B_V, nch * kChunkBytes);
                for (int c = 0; c < nch; ++c)
                    tma_load_3d(sbase + kOffV + c * kChunkBytes, &p.tm_v, B_V, 0, ybase + c * kChunk, z);
                if (g == 0) mbar_wait(B_Q, 0, aborted, p.err);
                mbar_wait(B_K, g & 1, aborted, p.err);
                tc_fence_after();
                const uint32_t idesc_s = idesc_bf16(128, 64 * nch, 0, 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tmem, sdesc_sw128(sbase + kOffQ + 32 * kk, 16, 1024),
                           sdesc_sw128(sbase + kOffK + 32 * kk, 16, 1024), idesc_s, kk > 0);
                mma_commit(B_S);
                mbar_wait(B_P, g & 1, aborted, p.err);
                tc_fence_after();
                mbar_wait(B_V, g & 1, aborted, p.err);
                const uint32_t idesc_o = idesc_bf16(128, 64, 0, 1);
                for (int kk = 0; kk < nch * (kChunk / 16); ++kk)
                    mma_ts(tmem + kTmemO, tmem + 8 * kk, sdesc_sw128(sbase + kOffV + 2048 * kk, 0, 1024),
                           idesc_o, (g > 0 || kk > 0) ? 1u : 0u);
                mma_commit(B_O);
            }
            // teardown: the last commit must have landed before TMEM is released
            mbar_wait(B_O, (n_groups - 1) & 1, aborted, p.err);
        }
    } else if (warp == 5) {
        // ------------------------------------------------ offset tiles: K_o then V_o, per offset
        if (lane == 0 && n_act > 0) {
            uint32_t seq = 0;
            for (int k = 0; k < n_act; ++k) {
                const int32_t y = i0 - offs[k];
                for (int h = 0; h < 2; ++h, ++seq) {
                    const CUtensorMap* map = h == 0 ? &p.tm_k : &p.tm_v;
                    const int s = seq % kRing;
                    mbar_wait(B_EMPTY(s), ((seq / kRing) & 1) ^ 1, aborted, p.err);
                    mbar_arrive_expect_tx(B_FULL(s), kTileBytes);
                    tma_load_3d(sbase + kOffRing + s * kTileBytes, map, B_FULL(s), 0, y, z);
                    tma_load_3d(sbase + kOffRing + s * kTileBytes + kChunkBytes, map, B_FULL(s), 0,
                                y + kChunk, z);
                }
            }
            // teardown: wait for the copies still in flight (already-completed phases pass)
            for (uint32_t q = seq > kRing ? seq - kRing : 0; q < seq; ++q)
                mbar_wait(B_FULL(q % kRing), (q / kRing) & 1, aborted, p.err);
        }
    } else {
        // ------------------------------------------------ row threads
        const int r = tid;
        const int32_t i = i0 + r;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const float sl2 = p.scale_log2;

        // ---- band: masked online softmax over the S groups. Only the 32-column chunks that
        // some row of this warp can reach are read (3 of 6 at W = 64); the rest of P is zero.
        float m_b = -INFINITY, l_b = 0.f;
        for (int g = 0; g < n_groups; ++g) {
            const int nch = min(kMaxGroupChunks, n_chunks - g * kMaxGroupChunks);
            const int32_t kbase = (c_lo + g * kMaxGroupChunks) * kChunk;
            const int32_t d0 = i - kbase;  // dist(i, key kbase + c) = d0 - c
            const int32_t wrow = i0 + warp * 32 - kbase;
            const int32_t colA = max(0, wrow - W + 1);
            const int32_t colB = min(nch * kChunk - 1, wrow + 31);
            const int ccA = colA / 32;
            const int n_need = colA <= colB ? colB / 32 - ccA + 1 : 0;
            mbar_wait(B_S, g & 1, aborted, p.err);
            tc_fence_after();
            float mn = m_b;
            if (n_need <= 3) {
                uint32_t v[3][32];
#pragma unroll
                for (int j = 0; j < 3; ++j)
                    if (j < n_need) tmem_ld32(tmem + lane_base + 32 * (ccA + j), v[j]);
                tmem_ld_wait();
                float mx = -INFINITY;
#pragma unroll
                for (int j = 0; j < 3; ++j) {
                    if (j < n_need) {
                        const int32_t dj = d0 - 32 * (ccA + j);
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const bool ok = (uint32_t)(dj - e) < (uint32_t)W;
                            const float x = ok ? __uint_as_float(v[j][e]) * sl2 : -INFINITY;
                            v[j][e] = __float_as_uint(x);
                            mx = fmaxf(mx, x);
                        }
                    }
                }
                mn = fmaxf(m_b, mx);
                if (g > 0) {
                    mbar_wait(B_O, (g - 1) & 1, aborted, p.err);
                    tc_fence_after();
                    const float corr = (m_b == -INFINITY) ? 0.f : ex2(m_b - mn);
                    if (__any_sync(0xffffffffu, mn != m_b)) {
                        uint32_t o[32];
                        for (int h = 0; h < 2; ++h) {
                            tmem_ld32(tmem + lane_base + kTmemO + 32 * h, o);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
                            tmem_st32(tmem + lane_base + kTmemO + 32 * h, o);
                        }
                        tmem_st_wait();
                    }
                    l_b *= corr;
                }
                const float mu = mn == -INFINITY ? 0.f : mn;
#pragma unroll
                for (int j = 0; j < 3; ++j) {
                    if (j < n_need) {
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float p0 = ex2(__uint_as_float(v[j][e]) - mu);
                            const float p1 = ex2(__uint_as_float(v[j][e + 1]) - mu);
                            l_b += p0 + p1;
                            pk[e >> 1] = pack_bf16x2(p0, p1);
                        }
                        tmem_st16(tmem + lane_base + 16 * (ccA + j), pk);
                    }
                }
                uint32_t zero[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) zero[e] = 0u;
                for (int cc = 0; cc < nch * 2; ++cc)
                    if (cc < ccA || cc >= ccA + n_need) tmem_st16(tmem + lane_base + 16 * cc, zero);
            } else {
                // general window (more than 96 reachable columns): two passes over TMEM
                uint32_t v[32];
                float mx = -INFINITY;
                for (int j = 0; j < n_need; ++j) {
                    tmem_ld32(tmem + lane_base + 32 * (ccA + j), v);
                    tmem_ld_wait();
                    const int32_t dj = d0 - 32 * (ccA + j);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if ((uint32_t)(dj - e) < (uint32_t)W) mx = fmaxf(mx, __uint_as_float(v[e]) * sl2);
                }
                mn = fmaxf(m_b, mx);
                if (g > 0) {
                    mbar_wait(B_O, (g - 1) & 1, aborted, p.err);
                    tc_fence_after();
                    const float corr = (m_b == -INFINITY) ? 0.f : ex2(m_b - mn);
                    if (__any_sync(0xffffffffu, mn != m_b)) {
                        for (int h = 0; h < 2; ++h) {
                            tmem_ld32(tmem + lane_base + kTmemO + 32 * h, v);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * corr);
                            tmem_st32(tmem + lane_base + kTmemO + 32 * h, v);
                        }
                        tmem_st_wait();
                    }
                    l_b *= corr;
                }
                const float mu = mn == -INFINITY ? 0.f : mn;
                for (int cc = 0; cc < nch * 2; ++cc) {
                    const int j = cc - ccA;
                    uint32_t pk[16];
                    if (j >= 0 && j < n_need) {
                        tmem_ld32(tmem + lane_base + 32 * cc, v);
                        tmem_ld_wait();
                        const int32_t dj = d0 - 32 * cc;
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float p0 = (uint32_t)(dj - e) < (uint32_t)W
                                                 ? ex2(__uint_as_float(v[e]) * sl2 - mu) : 0.f;
                            const float p1 = (uint32_t)(dj - e - 1) < (uint32_t)W
                                                 ? ex2(__uint_as_float(v[e + 1]) * sl2 - mu) : 0.f;
                            l_b += p0 + p1;
                            pk[e >> 1] = pack_bf16x2(p0, p1);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) pk[e] = 0u;
                    }
                    tmem_st16(tmem + lane_base + 16 * cc, pk);
                }
            }
            m_b = mn;
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(B_P);
        }

        // ---- offsets: one pass per offset; the running max starts at the band's max and is
        // only raised when a score exceeds it by more than 2^8 (bounded growth, rare rescale)
        uint32_t qw[32];
        {
            const uint8_t* qrow = smem + kOffQ;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 w = *reinterpret_cast<const uint4*>(qrow + sw128_off(r, c));
                qw[4 * c + 0] = w.x; qw[4 * c + 1] = w.y; qw[4 * c + 2] = w.z; qw[4 * c + 3] = w.w;
            }
        }
        float m_o = m_b, l_o = 0.f;
        float oacc[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) oacc[c] = 0.f;
        uint32_t seq = 0;
#pragma unroll 1
        for (int k = 0; k < n_act; ++k) {
            const bool valid = i - offs[k] >= 0;
            int s = seq % kRing;
            mbar_wait(B_FULL(s), (seq / kRing) & 1, aborted, p.err);
            const uint8_t* krow = smem + kOffRing + s * kTileBytes;
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 w = *reinterpret_cast<const uint4*>(krow + sw128_off(r, c));
                fma2_bf16(qw[4 * c + 0], w.x, a0, a1);
                fma2_bf16(qw[4 * c + 1], w.y, a2, a3);
                fma2_bf16(qw[4 * c + 2], w.z, a0, a1);
                fma2_bf16(qw[4 * c + 3], w.w, a2, a3);
            }
            mbar_arrive(B_EMPTY(s));
            ++seq;
            const float sc = valid ? ((a0 + a1) + (a2 + a3)) * sl2 : -INFINITY;
            if (sc > m_o + 8.f) {
                const float corr = m_o == -INFINITY ? 0.f : ex2(m_o - sc);
                l_o *= corr;
#pragma unroll
                for (int c = 0; c < 64; ++c) oacc[c] *= corr;
                m_o = sc;
            }
            const float pk = valid ? ex2(sc - m_o) : 0.f;
            l_o += pk;
            const uint32_t pb = pack_bf16x2(pk, 0.f);
            s = seq % kRing;
            mbar_wait(B_FULL(s), (seq / kRing) & 1, aborted, p.err);
            const uint8_t* vrow = smem + kOffRing + s * kTileBytes;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 w = *reinterpret_cast<const uint4*>(vrow + sw128_off(r, c));
                axpy2_bf16(pb, w.x, oacc[8 * c + 0], oacc[8 * c + 1]);
                axpy2_bf16(pb, w.y, oacc[8 * c + 2], oacc[8 * c + 3]);
                axpy2_bf16(pb, w.z, oacc[8 * c + 4], oacc[8 * c + 5]);
                axpy2_bf16(pb, w.w, oacc[8 * c + 6], oacc[8 * c + 7]);
            }
            mbar_arrive(B_EMPTY(s));
            ++seq;
        }

        // ---- epilogue: merge the band and offset softmax parts
        mbar_wait(B_O, (n_groups - 1) & 1, aborted, p.err);
        tc_fence_after();
        const float m = fmaxf(m_b, m_o);
        const float mu = m == -INFINITY ? 0.f : m;
        const float fb = m_b == -INFINITY ? 0.f : ex2(m_b - mu);
        const float fo = m_o == -INFINITY ? 0.f : ex2(m_o - mu);
        const float l = l_b * fb + l_o * fo;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        uint8_t* orow = smem + kOffQ;  // Q tile is free: stage O there for the TMA store
        for (int h = 0; h < 2; ++h) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + kTmemO + 32 * h, v);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint4 w;
                const int e = 8 * c;
                const int d = 32 * h + e;
                w.x = pack_bf16x2((__uint_as_float(v[e + 0]) * fb + oacc[d + 0] * fo) * inv,
                                  (__uint_as_float(v[e + 1]) * fb + oacc[d + 1] * fo) * inv);
                w.y = pack_bf16x2((__uint_as_float(v[e + 2]) * fb + oacc[d + 2] * fo) * inv,
                                  (__uint_as_float(v[e + 3]) * fb + oacc[d + 3] * fo) * inv);
                w.z = pack_bf16x2((__uint_as_float(v[e + 4]) * fb + oacc[d + 4] * fo) * inv,
                                  (__uint_as_float(v[e + 5]) * fb + oacc[d + 5] * fo) * inv);
                w.w = pack_bf16x2((__uint_as_float(v[e + 6]) * fb + oacc[d + 6] * fo) * inv,
                                  (__uint_as_float(v[e + 7]) * fb + oacc[d + 7] * fo) * inv);
                *reinterpret_cast<uint4*>(orow + sw128_off(r, 4 * h + c)) = w;
            }
        }
        if (i < T) p.lse[slice * T + i] = (m + lg2(l)) * 0.69314718055994531f;
        fence_proxy_async_smem();
        tc_fence_before();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (tid == 0 && !aborted) {
            tma_store_3d(&p.tm_o, sbase + kOffQ, 0, i0, z);
            if (i0 + kChunk < T) tma_store_3d(&p.tm_o, sbase + kOffQ + kChunkBytes, 0, i0 + kChunk, z);
            tma_store_commit();
            tma_store_wait_read0();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

fibattn_status launch_fwd_tc_bf16(const void* q, const void* k, const void* v, void* o, float* lse,
                                  const AttnShape& sh, const OffsetTables& t, cudaStream_t st) {
    const int64_t slices = sh.slices_per_layer * sh.n_layers;
    if (slices > 0x7fffffff) return FIBATTN_ERR_INVALID_ARG;
    const int32_t tiles = (sh.T + kRows - 1) / kRows;
    const int64_t gx = (int64_t)tiles * sh.slices_per_layer;
    if (gx > 0x7fffffff) return FIBATTN_ERR_INVALID_ARG;
    FwdParams P;
    // the error-word lookup is a runtime call: it binds the device's primary context to this
    // thread (a fresh thread may have none), which the tensor-map encoding below needs
    P.err = device_error_word();
    if (!P.err) return cuda_fail(-1, "cudaGetSymbolAddress (error word)");
    const void* bases[4] = {q, k, v, o};
    CUtensorMap* maps[4] = {&P.tm_q, &P.tm_k, &P.tm_v, &P.tm_o};
    for (int m = 0; m < 4; ++m) {
        const int r = make_bf16_rows_map(maps[m], bases[m], slices, sh.T);
        if (r != 0) return cuda_fail(r, "cuTensorMapEncodeTiled (fwd)");
    }
    P.lse = lse;
    P.slices_per_layer = sh.slices_per_layer;
    P.T = sh.T;
    P.W = sh.W;
    P.tiles_per_slice = tiles;
    P.scale_log2 = sh.scale * 1.4426950408889634f;
    P.tabs = t;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail((int32_t)e, "cudaGetDevice");
    static bool attr_set[64] = {};
    if (dev < 0 || dev >= 64) return FIBATTN_ERR_UNSUPPORTED;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemAlloc);
        if (e != cudaSuccess) return cuda_fail((int32_t)e, "cudaFuncSetAttribute (fwd)");
        attr_set[dev] = true;
    }
    dim3 grid((unsigned)gx, sh.n_layers);
    {
        KernelScope ks("fwd_tc_bf16", st);
        fwd_tc_kernel<<<grid, kThreads, kSmemAlloc, st>>>(P);
    }
    return launch_status("launch fwd_tc_bf16");
}

}  // namespace fibattn
