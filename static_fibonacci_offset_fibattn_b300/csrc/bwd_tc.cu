// bwd_tc.cu -- bf16 backward of Fibonacci-offset sparse attention on sm_103a tensor cores.
//
// Gradient of o_i = sum_{j in S_i} P_ij v_j, P_ij = exp(scale q_i.k_j - lse_i), over the
// attended set of "Depth-Staggered Fibonacci Spacing for Sparse Attention" (gist.science
// explainer, Metodologia / Arquitetura, "Conjunto Atendido": the window i-W+1..i plus the
// keys i-o of the layer's offsets):
//   D_i = dO_i . o_i,  dP_ij = dO_i . v_j,  dS_ij = P_ij (dP_ij - D_i),
//   dq_i = scale sum_j dS_ij k_j,  dk_j = scale sum_i dS_ij q_i,  dv_j = sum_i P_ij dO_i.
//
// Two kernels, each the only writer of its outputs (no atomics anywhere):
//
// bwd_dq_tc (query owner; one CTA = 128 queries [i0, i0+128) of a slice, 192 threads)
//   warps 0-3 : one thread per query row (TMEM lane = row).
//   warp 4    : TMEM allocation, TMA loads of Q, dO and the band K/V chunks, tcgen05.mma.
//   warp 5    : TMA loads of the shifted offset tiles K[i0-o ..], V[i0-o ..] into a ring.
//   Preamble: D_i from o_i and dO_i (written to the workspace for the second kernel).
//   Band, per 64-key chunk: S = Q K^T and dP = dO V^T (M=128, N=64) into TMEM; each row
//   thread forms dS = P (dP - D) in fp32 and writes it back as bf16 over S; then
//   dQ += dS K (A = dS from TMEM, B = K chunk MN-major) accumulates in TMEM.
//   Offsets (a diagonal per table entry): s = q.k_{i-o}, dp = dO.v_{i-o} by CUDA-core row
//   dot products, dq += ds k_{i-o} in registers; (P, dS) of each (row, offset) pair is
//   written to the workspace as a bf16 pair.
//   Epilogue: dq = scale (dQ_band + dq_off), bf16, TMA store.
//
// bwd_dkdv_tc (key owner; one CTA = 128 keys [j0, j0+128) of a slice, 320 threads)
//   warps 0-7 : two threads per key row: warps w and w+4 share TMEM lanes 32(w%4)..+31 and
//               split the 64 head dims (and the band columns) in halves.
//   warp 8    : TMEM allocation, TMA loads of K, V and the band Q/dO chunks (lane 0), the
//               band's lse/D values staged into shared memory (all lanes), tcgen05.mma.
//   warp 9    : TMA loads of the shifted offset tiles Q[j0+o ..], dO[j0+o ..].
//   Band, per 64-query chunk: S^T = K Q^T and dP^T = V dO^T into TMEM; row threads form
//   P^T and dS^T (bf16, over S^T and dP^T); dV += P^T dO and dK += dS^T Q in TMEM.
//   Offsets: key j receives dk_j += dS q_{j+o}, dv_j += P dO_{j+o} from the (P, dS) pairs
//   the first kernel stored, so no dot product is recomputed.
//   Epilogue: dk = scale (dK_band + dk_off), dv = dV_band + dv_off, bf16, TMA stores.
//
// Every mbarrier wait is bounded (tc::mbar_wait); a wait that runs out latches the device
// error word, later waits return at once, and the CTA still releases its TMEM.
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

constexpr int kRows = 128;                      // rows (queries or keys) per tile
constexpr int kChunk = kTmaBoxRows;             // band chunk (one TMA box)
constexpr uint32_t kTileBytes = kRows * 128;    // 16 KB
constexpr uint32_t kChunkBytes = kChunk * 128;  // 8 KB
constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_do;  // inputs, 3D {64, T, slices}, box {64, 64, 1}
    CUtensorMap tm_dq, tm_dk, tm_dv;      // outputs
    const __nv_bfloat16* o;               // forward output (for D)
    const float* lse;                     // [slices][T]
    float* delta;                         // workspace: D [slices][T]
    uint32_t* pds;                        // workspace: (P, dS) bf16 pairs [slices][n_max][T]
    int32_t* err;
    int64_t slices_per_layer;
    int32_t T, W;
    int32_t tiles_per_slice;
    int32_t n_max;                        // offsets per layer slot in pds
    float scale;
    float scale_log2;                     // scale * log2(e)
    OffsetTables tabs;
};

__device__ __forceinline__ uint32_t bar_at(uint32_t sbase, uint32_t off, int idx) {
    return sbase + off + 8u * idx;
}

__device__ __forceinline__ void load_row_sw(const uint8_t* tile, int r, uint32_t (&w)[32]) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 x = *reinterpret_cast<const uint4*>(tile + sw128_off(r, c));
        w[4 * c + 0] = x.x; w[4 * c + 1] = x.y; w[4 * c + 2] = x.z; w[4 * c + 3] = x.w;
    }
}

// ====================================================================== dQ (query owner)
namespace dq {

constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 64, kColP = 128;  // dQ accumulator in columns [0, 64)

constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffDO = kOffQ + kTileBytes;
constexpr uint32_t kOffK = kOffDO + kTileBytes;      // 2 stages x 8 KB
constexpr uint32_t kOffV = kOffK + 2 * kChunkBytes;  // 2 stages x 8 KB
constexpr uint32_t kOffRing = kOffV + 2 * kChunkBytes;
constexpr uint32_t kOffBar = kOffRing + 2 * kTileBytes;
// barriers: 0 q+dO, 1-2 band K/V full, 3 S/dP ready, 4 dS written (128), 5 dQ MMA done,
// 6-7 ring full, 8-9 ring empty (128)
constexpr int kNumBars = 10;
constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemAlloc = kOffTmemSlot + 16 + 1024;

__global__ void __launch_bounds__(kThreads, 2) kernel(const __grid_constant__ BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - smem_u32(smem_raw));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int layer = blockIdx.y;
    const int tile = blockIdx.x % p.tiles_per_slice;
    const int64_t zl = (int64_t)layer * p.slices_per_layer + blockIdx.x / p.tiles_per_slice;
    const int32_t z = (int32_t)zl;
    const int32_t T = p.T, W = p.W;
    const int32_t i0 = tile * kRows;

    const uint32_t B_QDO = bar_at(sbase, kOffBar, 0);
    auto B_KV = [&](int s) { return bar_at(sbase, kOffBar, 1 + s); };
    const uint32_t B_S = bar_at(sbase, kOffBar, 3), B_DS = bar_at(sbase, kOffBar, 4);
    const uint32_t B_DQ = bar_at(sbase, kOffBar, 5);
    auto B_FULL = [&](int s) { return bar_at(sbase, kOffBar, 6 + s); };
    auto B_EMPTY = [&](int s) { return bar_at(sbase, kOffBar, 8 + s); };

    const int32_t kstart = i0 - W + 1 > 0 ? i0 - W + 1 : 0;
    const int32_t klast = (i0 + kRows - 1 < T - 1) ? i0 + kRows - 1 : T - 1;
    const int32_t c_lo = kstart / kChunk;
    const int32_t n_chunks = klast / kChunk - c_lo + 1;
    const int32_t* offs = p.tabs.off[layer];
    int32_t n_act = 0;
    for (int e = 0; e < p.tabs.count[layer]; ++e)
        if (offs[e] <= klast) n_act = e + 1;

    if (tid == 0) {
        for (int b = 0; b < kNumBars; ++b)
            mbar_init(bar_at(sbase, kOffBar, b), (b == 4 || b >= 8) ? kRows : 1);
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
        if (lane == 0) {
            prefetch_tmap(&p.tm_q);
            prefetch_tmap(&p.tm_do);
            prefetch_tmap(&p.tm_k);
            prefetch_tmap(&p.tm_v);
            mbar_arrive_expect_tx(B_QDO, 2 * kTileBytes);
            tma_load_3d(sbase + kOffQ, &p.tm_q, B_QDO, 0, i0, z);
            tma_load_3d(sbase + kOffQ + kChunkBytes, &p.tm_q, B_QDO, 0, i0 + kChunk, z);
            tma_load_3d(sbase + kOffDO, &p.tm_do, B_QDO, 0, i0, z);
            tma_load_3d(sbase + kOffDO + kChunkBytes, &p.tm_do, B_QDO, 0, i0 + kChunk, z);
            auto load_chunk = [&](int c) {
                const int s = c & 1;
                const int32_t y = (c_lo + c) * kChunk;
                mbar_arrive_expect_tx(B_KV(s), 2 * kChunkBytes);
                tma_load_3d(sbase + kOffK + s * kChunkBytes, &p.tm_k, B_KV(s), 0, y, z);
                tma_load_3d(sbase + kOffV + s * kChunkBytes, &p.tm_v, B_KV(s), 0, y, z);
            };
            load_chunk(0);
            if (n_chunks > 1) load_chunk(1);
            mbar_wait(B_QDO, 0, aborted, p.err);
            const uint32_t idesc_s = idesc_bf16(128, 64, 0, 0);
            const uint32_t idesc_q = idesc_bf16(128, 64, 0, 1);
            for (int c = 0; c < n_chunks; ++c) {
                const int s = c & 1;
                mbar_wait(B_KV(s), (c >> 1) & 1, aborted, p.err);
                if (c > 0) mbar_wait(B_DQ, (c - 1) & 1, aborted, p.err);
                tc_fence_after();
                const uint32_t kaddr = sbase + kOffK + s * kChunkBytes;
                const uint32_t vaddr = sbase + kOffV + s * kChunkBytes;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tmem + kColS, sdesc_sw128(sbase + kOffQ + 32 * kk, 16, 1024),
                           sdesc_sw128(kaddr + 32 * kk, 16, 1024), idesc_s, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tmem + kColP, sdesc_sw128(sbase + kOffDO + 32 * kk, 16, 1024),
                           sdesc_sw128(vaddr + 32 * kk, 16, 1024), idesc_s, kk > 0);
                mma_commit(B_S);
                mbar_wait(B_DS, c & 1, aborted, p.err);
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ts(tmem, tmem + kColS + 8 * kk, sdesc_sw128(kaddr + 2048 * kk, 0, 1024),
                           idesc_q, (c > 0 || kk > 0) ? 1u : 0u);
                mma_commit(B_DQ);
                if (c + 2 < n_chunks) {
                    mbar_wait(B_DQ, c & 1, aborted, p.err);
                    load_chunk(c + 2);
                }
            }
            mbar_wait(B_DQ, (n_chunks - 1) & 1, aborted, p.err);
        }
    } else if (warp == 5) {
        if (lane == 0 && n_act > 0) {
            uint32_t seq = 0;
            for (int k = 0; k < n_act; ++k) {
                const int32_t y = i0 - offs[k];
                for (int h = 0; h < 2; ++h, ++seq) {
                    const CUtensorMap* map = h == 0 ? &p.tm_k : &p.tm_v;
                    const int s = seq & 1;
                    mbar_wait(B_EMPTY(s), ((seq >> 1) & 1) ^ 1, aborted, p.err);
                    mbar_arrive_expect_tx(B_FULL(s), kTileBytes);
                    tma_load_3d(sbase + kOffRing + s * kTileBytes, map, B_FULL(s), 0, y, z);
                    tma_load_3d(sbase + kOffRing + s * kTileBytes + kChunkBytes, map, B_FULL(s), 0,
                                y + kChunk, z);
                }
            }
            for (uint32_t q = seq > 2 ? seq - 2 : 0; q < seq; ++q)
                mbar_wait(B_FULL(q & 1), (q >> 1) & 1, aborted, p.err);
        }
    } else {
        // ------------------------------------------------ row threads
        const int r = tid;
        const int32_t i = i0 + r;
        const bool row_ok = i < T;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const float sl2 = p.scale_log2;
        const int64_t grow = zl * T + i;  // row index into lse / delta
        const float lse2 = row_ok ? p.lse[grow] * kLog2e : 0.f;

        // D_i = dO_i . o_i (o read straight from global memory, dO from the tile)
        uint4 orow[8];
        if (row_ok) {
            const uint4* op = reinterpret_cast<const uint4*>(p.o + grow * 64);
#pragma unroll
            for (int c = 0; c < 8; ++c) orow[c] = __ldg(op + c);
        } else {
#pragma unroll
            for (int c = 0; c < 8; ++c) orow[c] = make_uint4(0u, 0u, 0u, 0u);
        }
        mbar_wait(B_QDO, 0, aborted, p.err);
        uint32_t gw[32];  // dO row (bf16 pairs)
        load_row_sw(smem + kOffDO, r, gw);
        float D;
        {
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                fma2_bf16(gw[4 * c + 0], orow[c].x, a0, a1);
                fma2_bf16(gw[4 * c + 1], orow[c].y, a2, a3);
                fma2_bf16(gw[4 * c + 2], orow[c].z, a0, a1);
                fma2_bf16(gw[4 * c + 3], orow[c].w, a2, a3);
            }
            D = (a0 + a1) + (a2 + a3);
        }
        if (row_ok) p.delta[grow] = D;

        // ---- band: dS over the window, written back to TMEM as the dQ MMA's A operand
        for (int c = 0; c < n_chunks; ++c) {
            const int32_t kb = (c_lo + c) * kChunk;
            const int32_t d0 = i - kb;
            mbar_wait(B_S, c & 1, aborted, p.err);
            tc_fence_after();
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                // does any (row of this warp, key of this 32-column half) pair lie in the window?
                const int32_t rlo = i0 + warp * 32, klo = kb + 32 * hh;
                const bool need = (rlo + 31 - klo >= 0) && (rlo - (klo + 31) < W);
                uint32_t pk[16];
                if (need) {
                    uint32_t sv[32], dv[32];
                    tmem_ld32(tmem + lane_base + kColS + 32 * hh, sv);
                    tmem_ld32(tmem + lane_base + kColP + 32 * hh, dv);
                    tmem_ld_wait();
                    const int32_t dj = d0 - 32 * hh;
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const bool ok0 = row_ok && (uint32_t)(dj - e) < (uint32_t)W;
                        const bool ok1 = row_ok && (uint32_t)(dj - e - 1) < (uint32_t)W;
                        const float p0 = ok0 ? ex2(__uint_as_float(sv[e]) * sl2 - lse2) : 0.f;
                        const float p1 = ok1 ? ex2(__uint_as_float(sv[e + 1]) * sl2 - lse2) : 0.f;
                        pk[e >> 1] = pack_bf16x2(p0 * (__uint_as_float(dv[e]) - D),
                                                 p1 * (__uint_as_float(dv[e + 1]) - D));
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) pk[e] = 0u;
                }
                tmem_st16(tmem + lane_base + kColS + 16 * hh, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(B_DS);
        }

        // ---- offsets: one diagonal per table entry
        float dq[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) dq[c] = 0.f;
        uint32_t seq = 0;
        const int64_t pds_row = (int64_t)z * p.n_max * T + i;
#pragma unroll 1
        for (int k = 0; k < n_act; ++k) {
            const bool valid = row_ok && i - offs[k] >= 0;
            int s = seq & 1;
            mbar_wait(B_FULL(s), (seq >> 1) & 1, aborted, p.err);
            uint32_t kw[32];
            load_row_sw(smem + kOffRing + s * kTileBytes, r, kw);
            mbar_arrive(B_EMPTY(s));
            ++seq;
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
            {
                const uint8_t* qrow = smem + kOffQ;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 x = *reinterpret_cast<const uint4*>(qrow + sw128_off(r, c));
                    fma2_bf16(x.x, kw[4 * c + 0], a0, a1);
                    fma2_bf16(x.y, kw[4 * c + 1], a2, a3);
                    fma2_bf16(x.z, kw[4 * c + 2], a0, a1);
                    fma2_bf16(x.w, kw[4 * c + 3], a2, a3);
                }
            }
            const float sdot = (a0 + a1) + (a2 + a3);
            s = seq & 1;
            mbar_wait(B_FULL(s), (seq >> 1) & 1, aborted, p.err);
            float b0 = 0.f, b1 = 0.f, b2 = 0.f, b3 = 0.f;
            {
                const uint8_t* vrow = smem + kOffRing + s * kTileBytes;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 x = *reinterpret_cast<const uint4*>(vrow + sw128_off(r, c));
                    fma2_bf16(gw[4 * c + 0], x.x, b0, b1);
                    fma2_bf16(gw[4 * c + 1], x.y, b2, b3);
                    fma2_bf16(gw[4 * c + 2], x.z, b0, b1);
                    fma2_bf16(gw[4 * c + 3], x.w, b2, b3);
                }
            }
            mbar_arrive(B_EMPTY(s));
            ++seq;
            const float dpd = (b0 + b1) + (b2 + b3);
            const float pr = valid ? ex2(sdot * sl2 - lse2) : 0.f;
            const float ds = pr * (dpd - D);
            const uint32_t pair = pack_bf16x2(pr, ds);  // lo = P, hi = dS
            if (row_ok) p.pds[pds_row + (int64_t)k * T] = pair;
            const uint32_t dsb = pair >> 16;  // dS as bf16 in the low half
#pragma unroll
            for (int c = 0; c < 32; ++c) axpy2_bf16(dsb, kw[c], dq[2 * c], dq[2 * c + 1]);
        }

        // ---- epilogue: dq = scale (dQ_band + dq_off), staged in the Q tile, TMA store
        mbar_wait(B_DQ, (n_chunks - 1) & 1, aborted, p.err);
        tc_fence_after();
        uint8_t* stage = smem + kOffQ;
        for (int h = 0; h < 2; ++h) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + 32 * h, v);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int e = 8 * c, d = 32 * h + e;
                uint4 w;
                w.x = pack_bf16x2((__uint_as_float(v[e + 0]) + dq[d + 0]) * p.scale,
                                  (__uint_as_float(v[e + 1]) + dq[d + 1]) * p.scale);
                w.y = pack_bf16x2((__uint_as_float(v[e + 2]) + dq[d + 2]) * p.scale,
                                  (__uint_as_float(v[e + 3]) + dq[d + 3]) * p.scale);
                w.z = pack_bf16x2((__uint_as_float(v[e + 4]) + dq[d + 4]) * p.scale,
                                  (__uint_as_float(v[e + 5]) + dq[d + 5]) * p.scale);
                w.w = pack_bf16x2((__uint_as_float(v[e + 6]) + dq[d + 6]) * p.scale,
                                  (__uint_as_float(v[e + 7]) + dq[d + 7]) * p.scale);
                *reinterpret_cast<uint4*>(stage + sw128_off(r, 4 * h + c)) = w;
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (tid == 0 && !aborted) {
            tma_store_3d(&p.tm_dq, sbase + kOffQ, 0, i0, z);
            if (i0 + kChunk < T) tma_store_3d(&p.tm_dq, sbase + kOffQ + kChunkBytes, 0, i0 + kChunk, z);
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

}  // namespace dq

// ====================================================================== dK/dV (key owner)
namespace dkdv {

constexpr int kThreads = 320;
constexpr int kRowThreads = 256;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColDK = 0, kColDV = 64, kColS = 128, kColP = 192;

constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kOffK + kTileBytes;
constexpr uint32_t kOffBand = kOffV + kTileBytes;           // 2 stages x (Q 8 KB + dO 8 KB)
constexpr uint32_t kOffRing = kOffBand + 4 * kChunkBytes;   // 2 x 16 KB
constexpr uint32_t kOffLD = kOffRing + 2 * kTileBytes;      // 2 stages x (lse2[64], D[64])
constexpr uint32_t kOffBar = kOffLD + 2 * 2 * kChunk * 4;
// barriers: 0 K+V, 1-2 band full (32 arrivals + tx), 3 S^T/dP^T ready, 4 P^T/dS^T written
// (256), 5 dK/dV MMAs done, 6-7 ring full, 8-9 ring empty (256)
constexpr int kNumBars = 10;
constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemAlloc = kOffTmemSlot + 16 + 1024;

__global__ void __launch_bounds__(kThreads, 2) kernel(const __grid_constant__ BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - smem_u32(smem_raw));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int layer = blockIdx.y;
    const int tile = blockIdx.x % p.tiles_per_slice;
    const int64_t zl = (int64_t)layer * p.slices_per_layer + blockIdx.x / p.tiles_per_slice;
    const int32_t z = (int32_t)zl;
    const int32_t T = p.T, W = p.W;
    const int32_t j0 = tile * kRows;

    const uint32_t B_KV = bar_at(sbase, kOffBar, 0);
    auto B_BAND = [&](int s) { return bar_at(sbase, kOffBar, 1 + s); };
    const uint32_t B_S = bar_at(sbase, kOffBar, 3), B_PDS = bar_at(sbase, kOffBar, 4);
    const uint32_t B_MM = bar_at(sbase, kOffBar, 5);
    auto B_FULL = [&](int s) { return bar_at(sbase, kOffBar, 6 + s); };
    auto B_EMPTY = [&](int s) { return bar_at(sbase, kOffBar, 8 + s); };

    // band queries [j0, min(T-1, j0+127+W-1)] in 64-query chunks; active offsets o <= T-1-j0
    const int64_t qlast64 = (int64_t)j0 + kRows - 1 + W - 1;
    const int32_t qlast = qlast64 < T - 1 ? (int32_t)qlast64 : T - 1;
    const int32_t q_lo = j0 / kChunk;
    const int32_t n_chunks = qlast / kChunk - q_lo + 1;
    const int32_t* offs = p.tabs.off[layer];
    int32_t n_act = 0;
    for (int e = 0; e < p.tabs.count[layer]; ++e)
        if (offs[e] <= T - 1 - j0) n_act = e + 1;

    if (tid == 0) {
        for (int b = 0; b < kNumBars; ++b) {
            uint32_t cnt = 1;
            if (b == 1 || b == 2) cnt = 32;
            if (b == 4 || b >= 8) cnt = kRowThreads;
            mbar_init(bar_at(sbase, kOffBar, b), cnt);
        }
        fence_mbar_init();
    }
    if (warp == 8) {
        tmem_alloc(sbase + kOffTmemSlot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmemSlot);
    bool aborted = false;

    float* lds = reinterpret_cast<float*>(smem + kOffLD);  // [stage][lse2 64 | D 64]

    if (warp == 8) {
        // ------------------------------------------------ band loads + MMA issue (whole warp)
        auto load_band = [&](int c) {
            const int s = c & 1;
            const int32_t y = (q_lo + c) * kChunk;
            float* st = lds + s * 2 * kChunk;
            for (int t = lane; t < kChunk; t += 32) {
                const int32_t i = y + t;
                const bool ok = i < T;
                st[t] = ok ? p.lse[zl * T + i] * kLog2e : 0.f;
                st[kChunk + t] = ok ? p.delta[zl * T + i] : 0.f;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(B_BAND(s), 2 * kChunkBytes);
                const uint32_t dst = sbase + kOffBand + s * 2 * kChunkBytes;
                tma_load_3d(dst, &p.tm_q, B_BAND(s), 0, y, z);
                tma_load_3d(dst + kChunkBytes, &p.tm_do, B_BAND(s), 0, y, z);
            } else {
                mbar_arrive(B_BAND(s));
            }
        };
        if (lane == 0) {
            prefetch_tmap(&p.tm_q);
            prefetch_tmap(&p.tm_do);
            prefetch_tmap(&p.tm_k);
            prefetch_tmap(&p.tm_v);
            mbar_arrive_expect_tx(B_KV, 2 * kTileBytes);
            tma_load_3d(sbase + kOffK, &p.tm_k, B_KV, 0, j0, z);
            tma_load_3d(sbase + kOffK + kChunkBytes, &p.tm_k, B_KV, 0, j0 + kChunk, z);
            tma_load_3d(sbase + kOffV, &p.tm_v, B_KV, 0, j0, z);
            tma_load_3d(sbase + kOffV + kChunkBytes, &p.tm_v, B_KV, 0, j0 + kChunk, z);
        }
        load_band(0);
        if (n_chunks > 1) load_band(1);
        if (lane == 0) mbar_wait(B_KV, 0, aborted, p.err);
        const uint32_t idesc_s = idesc_bf16(128, 64, 0, 0);
        const uint32_t idesc_o = idesc_bf16(128, 64, 0, 1);
        for (int c = 0; c < n_chunks; ++c) {
            const int s = c & 1;
            if (lane == 0) {
                const uint32_t qaddr = sbase + kOffBand + s * 2 * kChunkBytes;
                const uint32_t gaddr = qaddr + kChunkBytes;
                mbar_wait(B_BAND(s), (c >> 1) & 1, aborted, p.err);
                if (c > 0) mbar_wait(B_MM, (c - 1) & 1, aborted, p.err);
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tmem + kColS, sdesc_sw128(sbase + kOffK + 32 * kk, 16, 1024),
                           sdesc_sw128(qaddr + 32 * kk, 16, 1024), idesc_s, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tmem + kColP, sdesc_sw128(sbase + kOffV + 32 * kk, 16, 1024),
                           sdesc_sw128(gaddr + 32 * kk, 16, 1024), idesc_s, kk > 0);
                mma_commit(B_S);
                mbar_wait(B_PDS, c & 1, aborted, p.err);
                tc_fence_after();
                // P^T / dS^T of queries 32h..32h+31 sit in columns [32h, 32h+16) of their block
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t acol = 32 * (kk >> 1) + 8 * (kk & 1);
                    const uint32_t acc = (c > 0 || kk > 0) ? 1u : 0u;
                    mma_ts(tmem + kColDV, tmem + kColS + acol,
                           sdesc_sw128(gaddr + 2048 * kk, 0, 1024), idesc_o, acc);
                    mma_ts(tmem + kColDK, tmem + kColP + acol,
                           sdesc_sw128(qaddr + 2048 * kk, 0, 1024), idesc_o, acc);
                }
                mma_commit(B_MM);
                if (c + 2 < n_chunks) mbar_wait(B_MM, c & 1, aborted, p.err);
            }
            __syncwarp();
            if (c + 2 < n_chunks) load_band(c + 2);
        }
        if (lane == 0) mbar_wait(B_MM, (n_chunks - 1) & 1, aborted, p.err);
    } else if (warp == 9) {
        if (lane == 0 && n_act > 0) {
            uint32_t seq = 0;
            for (int k = 0; k < n_act; ++k) {
                const int32_t y = j0 + offs[k];
                for (int h = 0; h < 2; ++h, ++seq) {
                    const CUtensorMap* map = h == 0 ? &p.tm_q : &p.tm_do;
                    const int s = seq & 1;
                    mbar_wait(B_EMPTY(s), ((seq >> 1) & 1) ^ 1, aborted, p.err);
                    mbar_arrive_expect_tx(B_FULL(s), kTileBytes);
                    tma_load_3d(sbase + kOffRing + s * kTileBytes, map, B_FULL(s), 0, y, z);
                    tma_load_3d(sbase + kOffRing + s * kTileBytes + kChunkBytes, map, B_FULL(s), 0,
                                y + kChunk, z);
                }
            }
            for (uint32_t q = seq > 2 ? seq - 2 : 0; q < seq; ++q)
                mbar_wait(B_FULL(q & 1), (q >> 1) & 1, aborted, p.err);
        }
    } else {
        // ------------------------------------------------ row threads: key row r, dim half h
        const int q4 = warp & 3, h = warp >> 2;
        const int r = 32 * q4 + lane;
        const int32_t j = j0 + r;
        const bool row_ok = j < T;
        const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
        const float sl2 = p.scale_log2;

        // ---- band: P^T and dS^T of this thread's 32 query columns
        for (int c = 0; c < n_chunks; ++c) {
            const int32_t qb = (q_lo + c) * kChunk + 32 * h;  // first query of my columns
            mbar_wait(B_S, c & 1, aborted, p.err);
            tc_fence_after();
            const int32_t klo = j0 + 32 * q4;
            const bool need = (qb + 31 - klo >= 0) && (qb - (klo + 31) < W) && qb < T;
            uint32_t pp[16], pd[16];
            if (need) {
                uint32_t sv[32], dv[32];
                tmem_ld32(tmem + lane_base + kColS + 32 * h, sv);
                tmem_ld32(tmem + lane_base + kColP + 32 * h, dv);
                tmem_ld_wait();
                const float* L = lds + (c & 1) * 2 * kChunk + 32 * h;
                const float* Dd = L + kChunk;
                const int32_t dist0 = qb - j;
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const bool ok0 = row_ok && (uint32_t)(dist0 + e) < (uint32_t)W && qb + e < T;
                    const bool ok1 = row_ok && (uint32_t)(dist0 + e + 1) < (uint32_t)W && qb + e + 1 < T;
                    const float p0 = ok0 ? ex2(__uint_as_float(sv[e]) * sl2 - L[e]) : 0.f;
                    const float p1 = ok1 ? ex2(__uint_as_float(sv[e + 1]) * sl2 - L[e + 1]) : 0.f;
                    pp[e >> 1] = pack_bf16x2(p0, p1);
                    pd[e >> 1] = pack_bf16x2(p0 * (__uint_as_float(dv[e]) - Dd[e]),
                                             p1 * (__uint_as_float(dv[e + 1]) - Dd[e + 1]));
                }
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) pp[e] = pd[e] = 0u;
            }
            tmem_st16(tmem + lane_base + kColS + 32 * h, pp);
            tmem_st16(tmem + lane_base + kColP + 32 * h, pd);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(B_PDS);
        }

        // ---- offsets: dk_j += dS q_{j+o}, dv_j += P dO_{j+o} over my 32 dims
        float dk[32], dv[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) dk[c] = dv[c] = 0.f;
        const uint32_t* pds = p.pds + (int64_t)z * p.n_max * T;
        uint32_t seq = 0;
        uint32_t nxt = 0;
        if (n_act > 0 && row_ok && j + offs[0] < T) nxt = pds[j + offs[0]];
#pragma unroll 1
        for (int k = 0; k < n_act; ++k) {
            const uint32_t pair = nxt;
            if (k + 1 < n_act) {
                const int32_t i1 = j + offs[k + 1];
                nxt = (row_ok && i1 < T) ? pds[(int64_t)(k + 1) * T + i1] : 0u;
            }
            const uint32_t pb = pair & 0xFFFFu, dsb = pair >> 16;
            int s = seq & 1;
            mbar_wait(B_FULL(s), (seq >> 1) & 1, aborted, p.err);
            {
                const uint8_t* row = smem + kOffRing + s * kTileBytes;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 x = *reinterpret_cast<const uint4*>(row + sw128_off(r, 4 * h + c));
                    axpy2_bf16(dsb, x.x, dk[8 * c + 0], dk[8 * c + 1]);
                    axpy2_bf16(dsb, x.y, dk[8 * c + 2], dk[8 * c + 3]);
                    axpy2_bf16(dsb, x.z, dk[8 * c + 4], dk[8 * c + 5]);
                    axpy2_bf16(dsb, x.w, dk[8 * c + 6], dk[8 * c + 7]);
                }
            }
            mbar_arrive(B_EMPTY(s));
            ++seq;
            s = seq & 1;
            mbar_wait(B_FULL(s), (seq >> 1) & 1, aborted, p.err);
            {
                const uint8_t* row = smem + kOffRing + s * kTileBytes;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 x = *reinterpret_cast<const uint4*>(row + sw128_off(r, 4 * h + c));
                    axpy2_bf16(pb, x.x, dv[8 * c + 0], dv[8 * c + 1]);
                    axpy2_bf16(pb, x.y, dv[8 * c + 2], dv[8 * c + 3]);
                    axpy2_bf16(pb, x.z, dv[8 * c + 4], dv[8 * c + 5]);
                    axpy2_bf16(pb, x.w, dv[8 * c + 6], dv[8 * c + 7]);
                }
            }
            mbar_arrive(B_EMPTY(s));
            ++seq;
        }

        // ---- epilogue: dk = scale (band + offsets) into the K tile, dv into the V tile
        mbar_wait(B_MM, (n_chunks - 1) & 1, aborted, p.err);
        tc_fence_after();
        {
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + kColDK + 32 * h, v);
            tmem_ld_wait();
            uint8_t* st = smem + kOffK;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int e = 8 * c;
                uint4 w;
                w.x = pack_bf16x2((__uint_as_float(v[e + 0]) + dk[e + 0]) * p.scale,
                                  (__uint_as_float(v[e + 1]) + dk[e + 1]) * p.scale);
                w.y = pack_bf16x2((__uint_as_float(v[e + 2]) + dk[e + 2]) * p.scale,
                                  (__uint_as_float(v[e + 3]) + dk[e + 3]) * p.scale);
                w.z = pack_bf16x2((__uint_as_float(v[e + 4]) + dk[e + 4]) * p.scale,
                                  (__uint_as_float(v[e + 5]) + dk[e + 5]) * p.scale);
                w.w = pack_bf16x2((__uint_as_float(v[e + 6]) + dk[e + 6]) * p.scale,
                                  (__uint_as_float(v[e + 7]) + dk[e + 7]) * p.scale);
                *reinterpret_cast<uint4*>(st + sw128_off(r, 4 * h + c)) = w;
            }
            tmem_ld32(tmem + lane_base + kColDV + 32 * h, v);
            tmem_ld_wait();
            st = smem + kOffV;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int e = 8 * c;
                uint4 w;
                w.x = pack_bf16x2(__uint_as_float(v[e + 0]) + dv[e + 0], __uint_as_float(v[e + 1]) + dv[e + 1]);
                w.y = pack_bf16x2(__uint_as_float(v[e + 2]) + dv[e + 2], __uint_as_float(v[e + 3]) + dv[e + 3]);
                w.z = pack_bf16x2(__uint_as_float(v[e + 4]) + dv[e + 4], __uint_as_float(v[e + 5]) + dv[e + 5]);
                w.w = pack_bf16x2(__uint_as_float(v[e + 6]) + dv[e + 6], __uint_as_float(v[e + 7]) + dv[e + 7]);
                *reinterpret_cast<uint4*>(st + sw128_off(r, 4 * h + c)) = w;
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (tid == 0 && !aborted) {
            tma_store_3d(&p.tm_dk, sbase + kOffK, 0, j0, z);
            tma_store_3d(&p.tm_dv, sbase + kOffV, 0, j0, z);
            if (j0 + kChunk < T) {
                tma_store_3d(&p.tm_dk, sbase + kOffK + kChunkBytes, 0, j0 + kChunk, z);
                tma_store_3d(&p.tm_dv, sbase + kOffV + kChunkBytes, 0, j0 + kChunk, z);
            }
            tma_store_commit();
            tma_store_wait_read0();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace dkdv

fibattn_status set_smem(const void* fn, uint32_t bytes, bool (&done)[64]) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail((int32_t)e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return FIBATTN_ERR_UNSUPPORTED;
    if (!done[dev]) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        if (e != cudaSuccess) return cuda_fail((int32_t)e, "cudaFuncSetAttribute (bwd)");
        done[dev] = true;
    }
    return FIBATTN_OK;
}

}  // namespace

int32_t bwd_tc_n_max(const OffsetTables& t, int32_t n_layers) {
    int32_t n = 0;
    for (int l = 0; l < n_layers; ++l) n = t.count[l] > n ? t.count[l] : n;
    return n;
}

fibattn_status launch_bwd_tc_bf16(const void* q, const void* k, const void* v, const void* o,
                                  const float* lse, const void* dO, void* dq, void* dk, void* dv,
                                  float* delta, uint32_t* pds, int32_t n_max, const AttnShape& sh,
                                  const OffsetTables& t, cudaStream_t st) {
    const int64_t slices = sh.slices_per_layer * sh.n_layers;
    if (slices > 0x7fffffff) return FIBATTN_ERR_INVALID_ARG;
    const int32_t tiles = (sh.T + kRows - 1) / kRows;
    const int64_t gx = (int64_t)tiles * sh.slices_per_layer;
    if (gx > 0x7fffffff) return FIBATTN_ERR_INVALID_ARG;
    BwdParams P;
    // the error-word lookup is a runtime call: it binds the device's primary context to this
    // thread (a fresh thread, e.g. autograd's, may have none), which the encoding needs
    P.err = device_error_word();
    if (!P.err) return cuda_fail(-1, "cudaGetSymbolAddress (error word)");
    const void* bases[7] = {q, k, v, dO, dq, dk, dv};
    CUtensorMap* maps[7] = {&P.tm_q, &P.tm_k, &P.tm_v, &P.tm_do, &P.tm_dq, &P.tm_dk, &P.tm_dv};
    for (int m = 0; m < 7; ++m) {
        const int r = make_bf16_rows_map(maps[m], bases[m], slices, sh.T);
        if (r != 0) return cuda_fail(r, "cuTensorMapEncodeTiled (bwd)");
    }
    P.o = static_cast<const __nv_bfloat16*>(o);
    P.lse = lse;
    P.delta = delta;
    P.pds = pds;
    P.slices_per_layer = sh.slices_per_layer;
    P.T = sh.T;
    P.W = sh.W;
    P.tiles_per_slice = tiles;
    P.n_max = n_max;
    P.scale = sh.scale;
    P.scale_log2 = sh.scale * kLog2e;
    P.tabs = t;
    static bool dq_set[64] = {}, dkdv_set[64] = {};
    fibattn_status s0 = set_smem((const void*)dq::kernel, dq::kSmemAlloc, dq_set);
    if (s0 != FIBATTN_OK) return s0;
    s0 = set_smem((const void*)dkdv::kernel, dkdv::kSmemAlloc, dkdv_set);
    if (s0 != FIBATTN_OK) return s0;
    dim3 grid((unsigned)gx, sh.n_layers);
    {
        KernelScope ks("bwd_dq_tc", st);
        dq::kernel<<<grid, dq::kThreads, dq::kSmemAlloc, st>>>(P);
    }
    s0 = launch_status("launch bwd_dq_tc");
    if (s0 != FIBATTN_OK) return s0;
    {
        KernelScope ks("bwd_dkdv_tc", st);
        dkdv::kernel<<<grid, dkdv::kThreads, dkdv::kSmemAlloc, st>>>(P);
    }
    return launch_status("launch bwd_dkdv_tc");
}

}  // namespace fibattn
