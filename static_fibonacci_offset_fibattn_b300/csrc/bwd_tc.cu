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
//   Preamble: D_i from o_i (the first item of the offset ring) and dO_i, written to the
//   workspace for the second kernel.
//   Band, per 64-key chunk: S = Q K^T and dP = dO V^T (M=128, N=64) into TMEM; each row
//   thread forms dS = P (dP - D) in fp32 and writes it as bf16 to TMEM columns of its own;
//   then dQ += dS K (A = dS from TMEM, B = K chunk MN-major) accumulates in TMEM. At head
//   size 64 the row threads signal once a chunk's S and dP are in their registers, and the
//   next chunk's S and dP form while they compute dS (chunks past the two K/V stages are
//   prefetched into L2 at the start).
//   Offsets (a diagonal per table entry): s = q.k_{i-o}, dp = dO.v_{i-o} by CUDA-core row
//   dot products, dq += ds k_{i-o} in registers; (P, dS) of each (row, offset) pair is
//   written to the workspace as a bf16 pair, indexed by the key row i-o; D and lse log2(e)
//   go to the workspace too (rows padded to a multiple of 4 so the second kernel can fetch
//   them with 16-byte-aligned bulk copies).
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
//   Offsets: key j receives dk_j += dS q_{j+o} (first pass over the Q tiles of all offsets)
//   and dv_j += P dO_{j+o} (second pass over the dO tiles) from the (P, dS) pairs the first
//   kernel stored, so no dot product is recomputed; each pass is added into TMEM.
//   Epilogue: dk = scale dK, dv = dV, bf16, TMA stores.
//
// Fractional offsets (the learned-alpha variant; Metodologia / Arquitetura, "Implementacao":
// keys and values linearly interpolated between rows so that the gradient reaches alpha),
// kFrac: a real distance d is held as c = ceil(d) and the weight w = c - d of the row after
// i - c. The query owner reads both rows of each shifted item (the item carries the 8 rows
// after its tile), forms s~ = lerp(q.k_lo, q.k_lo+1), dp~ likewise, dq += dS k~ with k~ the
// interpolated row, stores (P, dS) under the key row lo = i - c, and adds the query's share
// of dL/dalpha, g_i = sum_k f_k [dS scale q.(k_lo - k_lo+1) + P dO.(v_lo - v_lo+1)], to a
// per-row array that a reduction kernel sums per layer. The key owner takes, per distance,
// the pair of query j + c (key j as row lo, weight 1 - w) and that of query j + c - 1 (key j
// as row lo + 1, weight w); its shifted Q/dO items carry the 8 rows before their tile.
//
// Every mbarrier wait is bounded (tc::mbar_wait); a wait that runs out latches the device
// error word, later waits return at once, and the CTA still releases its TMEM, after a fixed
// wait that lets its own copies and MMAs in flight land (tc::settle_if_aborted).
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "internal.h"
#include "ring.cuh"
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
    CUtensorMap tm_dq, tm_dk, tm_dv;      // outputs (K, V, dK, dV over the kv slices)
    CUtensorMap tm_o;                     // forward output (for D)
    const float* lse;                     // [slices][T]
    float* delta;                         // workspace: D [slices][T_pad]
    float* lse2;                          // workspace: lse * log2(e) [slices][T_pad]
    uint32_t* pds;                        // workspace: (P, dS) bf16 pairs [slices][n_max][T_pad],
                                          // entry k of key row j = the pair (j + o_k, j)
    int32_t* err;
    int64_t slices_per_layer;             // query slices per layer (B * H)
    uint32_t group;                       // query heads per kv head
    uint32_t slices_per_layer_kv32;       // kv slices per layer (B * H / group), for the
                                          // key owner's persistent tile walk
    uint32_t total_tiles;                 // tiles of the launch (<= INT32_MAX)
    int32_t T, W;
    int32_t T_pad;                        // T rounded up to 4: rows of the workspace arrays
    int32_t tiles_per_slice;
    int32_t n_max;                        // offsets per layer slot in pds
    float scale;
    float scale_log2;                     // scale * log2(e)
    OffsetTables tabs;                    // fractional mode: ceil(d) of each real distance d
};

template <bool kFrac>
struct BwdArgs : BwdParams {};

template <>
struct BwdArgs<true> : BwdParams {
    CUtensorMap tm_k8, tm_v8;   // 8-row boxes: the rows after a shifted K/V tile (query owner)
    CUtensorMap tm_q8, tm_do8;  // 8-row boxes: the rows before a shifted Q/dO tile (key owner)
    float* galpha;              // [slices][tiles]: sum over the tile's queries of
                                // g_i = sum_k f_k dL/dd_k (fixed order)
    float w[kMaxLayersPerLaunch][kMaxOffsets];  // weight ceil(d) - d of the later row
    float f[kMaxLayersPerLaunch][kMaxOffsets];  // base value F of the distance (dd/dalpha)
};

__device__ __forceinline__ uint32_t bar_at(uint32_t sbase, uint32_t off, int idx) {
    return sbase + off + 8u * idx;
}

__device__ __forceinline__ void load_row_sw(const uint8_t* tile, int r, uint32_t* w) {
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
// dQ accumulator in columns [0, 64), S and dP of a 64-key chunk in [64, 128) and [128, 192),
// the chunk's dS (bf16 pairs, the dQ MMA's A operand) in [192, 224): the row threads free the
// S and dP columns as soon as they hold them in registers, so that the next chunk's S and dP
// form while they compute this chunk's dS (head size 64)
constexpr uint32_t kColS = 64, kColP = 128, kColDS = 192;

// barriers: 0 q+dO, 1-2 band K/V full, 3 S/dP ready, 4 dS written (128), 5 dQ MMA done,
// 6-7 ring full, 8-9 ring empty (128), 10 band done (every band MMA has completed),
// 11 S/dP read out (4 warps)
constexpr int kNumBars = 12;
// Shared memory: the Q and dO tiles, two stages of K and V chunks, the two ring slots (a
// tile, plus in the fractional mode the 8 rows after it). Head size 128 (kWide) doubles the
// tiles (two 64-column halves each) but keeps one stage of K and V chunks (both halves: 16 KB
// each), and that stage's memory is also the ring: slot 0 = the K stage, slot 1 = the V stage.
// The ring's O items (for D) use it before the band, its offset items after the band. So the
// CTA needs 97 KB and two fit on an SM.
template <bool kFrac, bool kWide = false>
struct Layout {
    static constexpr uint32_t kTileQ = kWide ? 2 * kTileBytes : kTileBytes;
    static constexpr uint32_t kStage = kWide ? 2 * kChunkBytes : kChunkBytes;
    static constexpr uint32_t kStages = kWide ? 1 : 2;
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffDO = kOffQ + kTileQ;
    static constexpr uint32_t kOffK = kOffDO + kTileQ;  // kStages stages
    static constexpr uint32_t kOffV = kOffK + kStages * kStage;  // kStages stages
    static constexpr uint32_t kOffRing = kWide ? kOffK : kOffV + kStages * kStage;
    static constexpr uint32_t kSlot = kTileBytes + (kFrac ? 1024u : 0u);
    static constexpr uint32_t kOffBar = kWide ? kOffV + kStage : kOffRing + 2 * kSlot;
    static constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
    static constexpr uint32_t kOffRed = kOffTmemSlot + 16;  // 4 floats: per-warp dalpha sums
    static constexpr uint32_t kSmemAlloc = kOffRed + 16 + 1024;
};

// Head size 128 (kWide): two CTAs per tile (blockIdx.x = 2 * tile index + half); both form
// the full S = Q K^T and dP = dO V^T (8 MMA k-steps over the two column halves) and the full
// offset dots, and each accumulates dq for its own 64 output columns (dS K_half); half 0
// alone writes D, lse log2(e) and the (P, dS) pairs.
template <bool kFrac, bool kWide>
__global__ void __launch_bounds__(kThreads, 2) bwd_dq_tc_kernel(const __grid_constant__ BwdArgs<kFrac> p) {
    static_assert(!(kFrac && kWide), "the fractional mode is for head size 64");
    using L = Layout<kFrac, kWide>;
    constexpr uint32_t kOffBar = L::kOffBar, kOffTmemSlot = L::kOffTmemSlot, kSlot = L::kSlot;
    constexpr uint32_t kOffQ = L::kOffQ, kOffDO = L::kOffDO, kOffK = L::kOffK, kOffV = L::kOffV,
                       kOffRing = L::kOffRing, kStage = L::kStage;
    constexpr int kHalves = kWide ? 2 : 1;  // 64-column halves of a row
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - smem_u32(smem_raw));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int layer = blockIdx.y;
    const int half = kWide ? (int)(blockIdx.x & 1u) : 0;
    const uint32_t bt = kWide ? blockIdx.x >> 1 : blockIdx.x;
    const int tile = bt % p.tiles_per_slice;
    const int64_t zl = (int64_t)layer * p.slices_per_layer + bt / p.tiles_per_slice;
    const int32_t z = (int32_t)zl;
    // the kv slice: query head h of batch b reads kv head h / group
    const int32_t zk = (int32_t)((int64_t)layer * p.slices_per_layer_kv32 +
                                 (uint32_t)(bt / p.tiles_per_slice) / p.group);
    const int32_t T = p.T, W = p.W;
    const int32_t i0 = tile * kRows;

    const uint32_t B_QDO = bar_at(sbase, kOffBar, 0);
    auto B_KV = [&](int s) { return bar_at(sbase, kOffBar, 1 + s); };
    const uint32_t B_S = bar_at(sbase, kOffBar, 3), B_DS = bar_at(sbase, kOffBar, 4);
    const uint32_t B_DQ = bar_at(sbase, kOffBar, 5);
    auto B_FULL = [&](int s) { return bar_at(sbase, kOffBar, 6 + s); };
    auto B_EMPTY = [&](int s) { return bar_at(sbase, kOffBar, 8 + s); };
    const uint32_t B_BD = bar_at(sbase, kOffBar, 10), B_F = bar_at(sbase, kOffBar, 11);
    static_assert(!kWide || (L::kOffRing == L::kOffK && L::kOffV == L::kOffK + kSlot && L::kStage == kSlot),
                  "head size 128: the ring slots are the K and V stages");

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
            mbar_init(bar_at(sbase, kOffBar, b), (b == 4 || b == 8 || b == 9) ? kRows : (b == 11 ? 4 : 1));
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
            mbar_arrive_expect_tx(B_QDO, 2 * L::kTileQ);
            for (int qh = 0; qh < kHalves; ++qh) {
                const uint32_t o = qh * kTileBytes;
                tma_load_3d(sbase + kOffQ + o, &p.tm_q, B_QDO, 64 * qh, i0, z);
                tma_load_3d(sbase + kOffQ + o + kChunkBytes, &p.tm_q, B_QDO, 64 * qh, i0 + kChunk, z);
                tma_load_3d(sbase + kOffDO + o, &p.tm_do, B_QDO, 64 * qh, i0, z);
                tma_load_3d(sbase + kOffDO + o + kChunkBytes, &p.tm_do, B_QDO, 64 * qh, i0 + kChunk, z);
            }
            auto load_chunk = [&](int c) {
                const int s = kWide ? 0 : (c & 1);
                const int32_t y = (c_lo + c) * kChunk;
                mbar_arrive_expect_tx(B_KV(s), 2 * kStage);
                for (int qh = 0; qh < kHalves; ++qh) {
                    tma_load_3d(sbase + kOffK + s * kStage + qh * kChunkBytes, &p.tm_k, B_KV(s), 64 * qh, y, zk);
                    tma_load_3d(sbase + kOffV + s * kStage + qh * kChunkBytes, &p.tm_v, B_KV(s), 64 * qh, y, zk);
                }
            };
            if constexpr (kWide) {
                // the stage memory holds the ring's O items until the row threads have formed D
                mbar_wait(B_EMPTY(0), 0, aborted, p.err);
                mbar_wait(B_EMPTY(1), 0, aborted, p.err);
                load_chunk(0);
            } else {
                load_chunk(0);
                if (n_chunks > 1) load_chunk(1);
                // the later chunks load only once a stage frees: bring them into L2 now
                for (int c = 2; c < n_chunks; ++c) {
                    const int32_t y = (c_lo + c) * kChunk;
                    tma_prefetch_l2_3d(&p.tm_k, 0, y, zk);
                    tma_prefetch_l2_3d(&p.tm_v, 0, y, zk);
                }
            }
            mbar_wait(B_QDO, 0, aborted, p.err);
            const uint32_t idesc_s = idesc_bf16(128, 64, 0, 0);
            const uint32_t idesc_q = idesc_bf16(128, 64, 0, 1);
            // S = Q K_c^T and dP = dO V_c^T of chunk c
            auto issue_sdp = [&](int c) {
                const int s = kWide ? 0 : (c & 1);
                mbar_wait(B_KV(s), (kWide ? c : c >> 1) & 1, aborted, p.err);
                tc_fence_after();
                const uint32_t kaddr = sbase + kOffK + s * kStage;
                const uint32_t vaddr = sbase + kOffV + s * kStage;
                // K-dim over the row halves: k-steps 4h .. 4h+3 read half h of Q/dO and of K/V
#pragma unroll
                for (int kk = 0; kk < 4 * kHalves; ++kk)
                    mma_ss(tmem + kColS,
                           sdesc_sw128(sbase + kOffQ + (kk >> 2) * kTileBytes + 32 * (kk & 3), 16, 1024),
                           sdesc_sw128(kaddr + (kk >> 2) * kChunkBytes + 32 * (kk & 3), 16, 1024),
                           idesc_s, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4 * kHalves; ++kk)
                    mma_ss(tmem + kColP,
                           sdesc_sw128(sbase + kOffDO + (kk >> 2) * kTileBytes + 32 * (kk & 3), 16, 1024),
                           sdesc_sw128(vaddr + (kk >> 2) * kChunkBytes + 32 * (kk & 3), 16, 1024),
                           idesc_s, kk > 0);
                mma_commit(B_S);
            };
            // dQ (own output half) += dS_c K_c_half, once the row threads have written dS_c;
            // then the chunk's stage takes the chunk after next
            auto issue_dq = [&](int c) {
                const int s = kWide ? 0 : (c & 1);
                const uint32_t kaddr = sbase + kOffK + s * kStage;
                mbar_wait(B_DS, c & 1, aborted, p.err);
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ts(tmem, tmem + kColDS + 8 * kk,
                           sdesc_sw128(kaddr + half * kChunkBytes + 2048 * kk, 0, 1024),
                           idesc_q, (c > 0 || kk > 0) ? 1u : 0u);
                mma_commit(B_DQ);
                const int next = c + (kWide ? 1 : 2);  // the chunk that reuses this stage
                if (next < n_chunks) {
                    mbar_wait(B_DQ, c & 1, aborted, p.err);
                    load_chunk(next);
                }
            };
            if constexpr (kWide) {
                // one stage: chunk c + 1 loads into it once dQ of chunk c is done
                for (int c = 0; c < n_chunks; ++c) {
                    issue_sdp(c);
                    issue_dq(c);
                }
            } else {
                // S/dP of chunk c as soon as the row threads hold chunk c - 1's, then dQ of c - 1
                issue_sdp(0);
                for (int c = 1; c < n_chunks; ++c) {
                    mbar_wait(B_F, (c - 1) & 1, aborted, p.err);
                    issue_sdp(c);
                    issue_dq(c - 1);
                }
                issue_dq(n_chunks - 1);
            }
            mma_commit(B_BD);  // the stage memory is free for the ring once every MMA completes
            mbar_wait(B_DQ, (n_chunks - 1) & 1, aborted, p.err);
        }
    } else if (warp == 5) {
        // ring items: the O tile (for D), then K_o and V_o per active offset
        if (lane == 0) {
            prefetch_tmap(&p.tm_o);
            if constexpr (kFrac) {
                prefetch_tmap(&p.tm_k8);
                prefetch_tmap(&p.tm_v8);
            }
            // items: the O tile (head size 128: its two halves), then per offset K_o and V_o
            // (each by halves at head size 128)
            uint32_t seq = 0;
            auto put = [&](const CUtensorMap* map, int32_t x, int32_t y, int32_t zz, bool side8) {
                const int s = seq & 1;
                const uint32_t dst = sbase + kOffRing + s * kSlot;
                mbar_wait(B_EMPTY(s), ((seq >> 1) & 1) ^ 1, aborted, p.err);
                mbar_arrive_expect_tx(B_FULL(s), side8 ? kSlot : kTileBytes);
                tma_load_3d(dst, map, B_FULL(s), x, y, zz);
                tma_load_3d(dst + kChunkBytes, map, B_FULL(s), x, y + kChunk, zz);
                return dst;
            };
            for (int qh = 0; qh < kHalves; ++qh, ++seq) put(&p.tm_o, 64 * qh, i0, z, false);
            if constexpr (kWide) {
                if (n_act > 0) mbar_wait(B_BD, 0, aborted, p.err);  // the band chunks are done with the memory
            }
            for (int k = 0; k < n_act; ++k) {
                const int32_t y = i0 - offs[k];
                for (int h = 0; h < 2; ++h)
                    for (int qh = 0; qh < kHalves; ++qh, ++seq) {
                        const CUtensorMap* map = h == 0 ? &p.tm_k : &p.tm_v;
                        // fractional mode: every item also carries the 8 rows after its tile
                        // (the derivative in d needs row lo + 1 even where w = 0)
                        const uint32_t dst = put(map, 64 * qh, y, zk, kFrac);
                        if constexpr (kFrac)
                            tma_load_3d(dst + kTileBytes, h == 0 ? &p.tm_k8 : &p.tm_v8,
                                        B_FULL(seq & 1), 0, y + kRows, zk);
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
        const int64_t grow = zl * T + i;  // row index into lse
        const int64_t wrow = zl * p.T_pad + i;  // row index into the workspace arrays
        const float lse2 = row_ok ? p.lse[grow] * kLog2e : 0.f;

        // D_i = dO_i . o_i (dO from its tile, o from the first ring item(s))
        mbar_wait(B_QDO, 0, aborted, p.err);
        uint32_t gw[32 * kHalves];  // dO row (bf16 pairs)
#pragma unroll
        for (int qh = 0; qh < kHalves; ++qh) load_row_sw(smem + kOffDO + qh * kTileBytes, r, gw + 32 * qh);
        float D;
        {
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int qh = 0; qh < kHalves; ++qh) {  // items 0 (and 1): slots 0 (and 1), phase 0
                mbar_wait(B_FULL(qh), 0, aborted, p.err);
                const uint8_t* orow = smem + kOffRing + qh * kSlot;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 x = *reinterpret_cast<const uint4*>(orow + sw128_off(r, c));
                    fma2_bf16(gw[32 * qh + 4 * c + 0], x.x, a0, a1);
                    fma2_bf16(gw[32 * qh + 4 * c + 1], x.y, a2, a3);
                    fma2_bf16(gw[32 * qh + 4 * c + 2], x.z, a0, a1);
                    fma2_bf16(gw[32 * qh + 4 * c + 3], x.w, a2, a3);
                }
                fence_proxy_async_smem();  // generic reads before the TMA refill
                mbar_arrive(B_EMPTY(qh));
            }
            D = (a0 + a1) + (a2 + a3);
        }
        if (row_ok && half == 0) {
            p.delta[wrow] = D;
            p.lse2[wrow] = lse2;
        }

        // ---- band: dS over the window, into TMEM as the dQ MMA's A operand
        for (int c = 0; c < n_chunks; ++c) {
            const int32_t kb = (c_lo + c) * kChunk;
            const int32_t d0 = i - kb;
            mbar_wait(B_S, c & 1, aborted, p.err);
            tc_fence_after();
            __syncwarp();  // converged for the warp-collective TMEM accesses below
            uint32_t pk[2][16];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                // does any (row of this warp, key of this 32-column half) pair lie in the window?
                const int32_t rlo = i0 + warp * 32, klo = kb + 32 * hh;
                const bool need = (rlo + 31 - klo >= 0) && (rlo - (klo + 31) < W);
                uint32_t sv[32], dv[32];
                if (need) {
                    tmem_ld32(tmem + lane_base + kColS + 32 * hh, sv);
                    tmem_ld32(tmem + lane_base + kColP + 32 * hh, dv);
                    tmem_ld_wait(sv, dv);
                }
                if (hh == 1) {
                    // both halves are in registers: the S and dP columns are free
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(B_F);
                }
                if (need) {
                    const int32_t dj = d0 - 32 * hh;
                    // bit e: key kb + 32 hh + e is in this query's window
                    const uint32_t okm = row_ok ? window_bits(dj, W) : 0u;
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const bool ok0 = (okm >> e) & 1u;
                        const bool ok1 = (okm >> (e + 1)) & 1u;
                        const float p0 = ok0 ? ex2(__uint_as_float(sv[e]) * sl2 - lse2) : 0.f;
                        const float p1 = ok1 ? ex2(__uint_as_float(sv[e + 1]) * sl2 - lse2) : 0.f;
                        pk[hh][e >> 1] = pack_bf16x2(p0 * (__uint_as_float(dv[e]) - D),
                                                     p1 * (__uint_as_float(dv[e + 1]) - D));
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) pk[hh][e] = 0u;
                }
            }
            // dQ of the chunk before has read the dS columns
            if (c > 0) {
                mbar_wait(B_DQ, (c - 1) & 1, aborted, p.err);
                tc_fence_after();
            }
            __syncwarp();  // converged for the warp-collective TMEM accesses below
            tmem_st16(tmem + lane_base + kColDS, pk[0]);
            tmem_st16(tmem + lane_base + kColDS + 16, pk[1]);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(B_DS);
        }

        // ---- offsets: one diagonal per table entry
        float dq[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) dq[c] = 0.f;
        uint32_t seq = kHalves;  // the first ring item(s) held the O tile
        const int64_t pds_row = (int64_t)z * p.n_max * p.T_pad + i;
        float ga = 0.f;  // fractional mode: this query's share of dL/dalpha
#pragma unroll 1
        for (int k = 0; k < n_act; ++k) {
            const bool valid = row_ok && i - offs[k] >= 0;
            if constexpr (kFrac) {
                // k~ = k_lo + w (k_lo+1 - k_lo) into registers (bf16), the two row dots exact
                const float wk = p.w[layer][k];
                int s = seq & 1;
                mbar_wait(B_FULL(s), (seq >> 1) & 1, aborted, p.err);
                const uint8_t* krow = smem + kOffRing + s * kSlot;
                const uint8_t* qrow = smem + kOffQ;
                uint32_t kt[32];
                float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f, b0 = 0.f, b1 = 0.f, b2 = 0.f, b3 = 0.f;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 x = *reinterpret_cast<const uint4*>(krow + sw128_off(r, c));
                    const uint4 y = *reinterpret_cast<const uint4*>(krow + sw128_off(r + 1, c));
                    const uint4 qq = *reinterpret_cast<const uint4*>(qrow + sw128_off(r, c));
                    fma2_bf16(qq.x, x.x, a0, a1);
                    fma2_bf16(qq.y, x.y, a2, a3);
                    fma2_bf16(qq.z, x.z, a0, a1);
                    fma2_bf16(qq.w, x.w, a2, a3);
                    fma2_bf16(qq.x, y.x, b0, b1);
                    fma2_bf16(qq.y, y.y, b2, b3);
                    fma2_bf16(qq.z, y.z, b0, b1);
                    fma2_bf16(qq.w, y.w, b2, b3);
                    kt[4 * c + 0] = lerp_bf16x2(x.x, y.x, wk);
                    kt[4 * c + 1] = lerp_bf16x2(x.y, y.y, wk);
                    kt[4 * c + 2] = lerp_bf16x2(x.z, y.z, wk);
                    kt[4 * c + 3] = lerp_bf16x2(x.w, y.w, wk);
                }
                fence_proxy_async_smem();  // generic reads before the TMA refill
                mbar_arrive(B_EMPTY(s));
                ++seq;
                const float slo = (a0 + a1) + (a2 + a3), shi = (b0 + b1) + (b2 + b3);
                s = seq & 1;
                mbar_wait(B_FULL(s), (seq >> 1) & 1, aborted, p.err);
                const uint8_t* vrow = smem + kOffRing + s * kSlot;
                a0 = a1 = a2 = a3 = b0 = b1 = b2 = b3 = 0.f;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 x = *reinterpret_cast<const uint4*>(vrow + sw128_off(r, c));
                    const uint4 y = *reinterpret_cast<const uint4*>(vrow + sw128_off(r + 1, c));
                    fma2_bf16(gw[4 * c + 0], x.x, a0, a1);
                    fma2_bf16(gw[4 * c + 1], x.y, a2, a3);
                    fma2_bf16(gw[4 * c + 2], x.z, a0, a1);
                    fma2_bf16(gw[4 * c + 3], x.w, a2, a3);
                    fma2_bf16(gw[4 * c + 0], y.x, b0, b1);
                    fma2_bf16(gw[4 * c + 1], y.y, b2, b3);
                    fma2_bf16(gw[4 * c + 2], y.z, b0, b1);
                    fma2_bf16(gw[4 * c + 3], y.w, b2, b3);
                }
                fence_proxy_async_smem();  // generic reads before the TMA refill
                mbar_arrive(B_EMPTY(s));
                ++seq;
                const float dlo = (a0 + a1) + (a2 + a3), dhi = (b0 + b1) + (b2 + b3);
                const float sdot = fmaf(wk, shi - slo, slo), dpd = fmaf(wk, dhi - dlo, dlo);
                const float pr = valid ? ex2(sdot * sl2 - lse2) : 0.f;
                const float ds = pr * (dpd - D);
                const uint32_t pair = pack_bf16x2(pr, ds);  // lo = P, hi = dS
                if (valid) p.pds[pds_row + (int64_t)k * p.T_pad - offs[k]] = pair;  // key row lo
                ga += p.f[layer][k] * (ds * p.scale * (slo - shi) + pr * (dlo - dhi));
                const uint32_t dsb = pair >> 16;
#pragma unroll
                for (int c = 0; c < 32; ++c) axpy2_bf16(dsb, kt[c], dq[2 * c], dq[2 * c + 1]);
                continue;
            }
            if constexpr (kWide) {
                // both halves of K_o for the score, the own half kept for dq; both halves of V_o
                uint32_t kw[32];
                float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
                for (int qh = 0; qh < 2; ++qh, ++seq) {
                    const int s = seq & 1;
                    mbar_wait(B_FULL(s), (seq >> 1) & 1, aborted, p.err);
                    const uint8_t* krow = smem + kOffRing + s * kSlot;
                    const uint8_t* qrow = smem + kOffQ + qh * kTileBytes;
                    if (qh == half) load_row_sw(krow, r, kw);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 x = *reinterpret_cast<const uint4*>(qrow + sw128_off(r, c));
                        const uint4 y = *reinterpret_cast<const uint4*>(krow + sw128_off(r, c));
                        fma2_bf16(x.x, y.x, a0, a1);
                        fma2_bf16(x.y, y.y, a2, a3);
                        fma2_bf16(x.z, y.z, a0, a1);
                        fma2_bf16(x.w, y.w, a2, a3);
                    }
                    fence_proxy_async_smem();  // generic reads before the TMA refill
                    mbar_arrive(B_EMPTY(s));
                }
                const float sdot = (a0 + a1) + (a2 + a3);
                float b0 = 0.f, b1 = 0.f, b2 = 0.f, b3 = 0.f;
#pragma unroll
                for (int qh = 0; qh < 2; ++qh, ++seq) {
                    const int s = seq & 1;
                    mbar_wait(B_FULL(s), (seq >> 1) & 1, aborted, p.err);
                    const uint8_t* vrow = smem + kOffRing + s * kSlot;
                    // the dO row half from its resident tile (not held in registers: that keeps
                    // the kernel within the registers of two CTAs per SM)
                    const uint8_t* grow = smem + kOffDO + qh * kTileBytes;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 x = *reinterpret_cast<const uint4*>(vrow + sw128_off(r, c));
                        const uint4 g = *reinterpret_cast<const uint4*>(grow + sw128_off(r, c));
                        fma2_bf16(g.x, x.x, b0, b1);
                        fma2_bf16(g.y, x.y, b2, b3);
                        fma2_bf16(g.z, x.z, b0, b1);
                        fma2_bf16(g.w, x.w, b2, b3);
                    }
                    fence_proxy_async_smem();  // generic reads before the TMA refill
                    mbar_arrive(B_EMPTY(s));
                }
                const float dpd = (b0 + b1) + (b2 + b3);
                const float pr = valid ? ex2(sdot * sl2 - lse2) : 0.f;
                const float ds = pr * (dpd - D);
                const uint32_t pair = pack_bf16x2(pr, ds);  // lo = P, hi = dS
                if (valid && half == 0) p.pds[pds_row + (int64_t)k * p.T_pad - offs[k]] = pair;
                const uint32_t dsb = pair >> 16;
#pragma unroll
                for (int c = 0; c < 32; ++c) axpy2_bf16(dsb, kw[c], dq[2 * c], dq[2 * c + 1]);
                continue;
            }
            int s = seq & 1;
            mbar_wait(B_FULL(s), (seq >> 1) & 1, aborted, p.err);
            uint32_t kw[32];
            load_row_sw(smem + kOffRing + s * kSlot, r, kw);
            fence_proxy_async_smem();  // generic reads before the TMA refill
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
                const uint8_t* vrow = smem + kOffRing + s * kSlot;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 x = *reinterpret_cast<const uint4*>(vrow + sw128_off(r, c));
                    fma2_bf16(gw[4 * c + 0], x.x, b0, b1);
                    fma2_bf16(gw[4 * c + 1], x.y, b2, b3);
                    fma2_bf16(gw[4 * c + 2], x.z, b0, b1);
                    fma2_bf16(gw[4 * c + 3], x.w, b2, b3);
                }
            }
            fence_proxy_async_smem();  // generic reads before the TMA refill
            mbar_arrive(B_EMPTY(s));
            ++seq;
            const float dpd = (b0 + b1) + (b2 + b3);
            const float pr = valid ? ex2(sdot * sl2 - lse2) : 0.f;
            const float ds = pr * (dpd - D);
            const uint32_t pair = pack_bf16x2(pr, ds);  // lo = P, hi = dS
            if (valid) p.pds[pds_row + (int64_t)k * p.T_pad - offs[k]] = pair;  // key row i - o
            const uint32_t dsb = pair >> 16;  // dS as bf16 in the low half
#pragma unroll
            for (int c = 0; c < 32; ++c) axpy2_bf16(dsb, kw[c], dq[2 * c], dq[2 * c + 1]);
        }

        if constexpr (kFrac) {
            // the tile's share of dL/dalpha: warp sums, then thread 0 adds the four in order
            // after the epilogue's barrier
            float g = ga;  // 0 on rows past T
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) g += __shfl_xor_sync(0xffffffffu, g, m);
            if (lane == 0) reinterpret_cast<float*>(smem + L::kOffRed)[warp] = g;
        }

        // ---- epilogue: dq = scale (dQ_band + dq_off), staged in the Q tile, TMA store
        mbar_wait(B_DQ, (n_chunks - 1) & 1, aborted, p.err);
        tc_fence_after();
        __syncwarp();  // converged for the warp-collective TMEM accesses below
        uint8_t* stage = smem + kOffQ;
        for (int h = 0; h < 2; ++h) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + 32 * h, v);
            tmem_ld_wait(v);
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
        if constexpr (kFrac) {
            if (tid == 0) {
                const float* red = reinterpret_cast<const float*>(smem + L::kOffRed);
                p.galpha[zl * p.tiles_per_slice + tile] = ((red[0] + red[1]) + red[2]) + red[3];
            }
        }
        if (tid == 0 && !aborted) {
            const int32_t xo = 64 * half;  // the CTA's output columns
            tma_store_3d(&p.tm_dq, sbase + kOffQ, xo, i0, z);
            if (i0 + kChunk < T) tma_store_3d(&p.tm_dq, sbase + kOffQ + kChunkBytes, xo, i0 + kChunk, z);
            tma_store_commit();
            tma_store_wait_read0();
        }
    }

    // after a timeout in this CTA, its own copies and MMAs in flight land before TMEM is released
    tc_fence_before();
    settle_if_aborted(__syncthreads_or(aborted ? 1 : 0));
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace dq

// ====================================================================== dK/dV (key owner)
namespace dkdv {

constexpr int kThreads = 320;
constexpr int kRowWarps = 8;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColDK = 0, kColDV = 64, kColS = 128, kColP = 192;
constexpr uint32_t kSlots = 6;
constexpr int kMaxGroupChunks = 4;    // band chunks per K/V copy: 2 + 4 ring items
constexpr uint32_t kFullArrivals = 1;  // the producer's arrival with the byte count

// barriers: FULL[kSlots], EMPTY[kSlots], S^T/dP^T ready, P^T/dS^T written (8 warps),
// dK/dV MMAs done, TMEM free (8 warps)
constexpr uint32_t kBarS = 2 * kSlots, kBarP = kBarS + 1, kBarM = kBarS + 2, kBarT = kBarS + 3;
constexpr uint32_t kNumBars = kBarT + 1;
// Shared memory: the ring slots, then per slot its side words, then the barriers. In the
// fractional mode a shifted Q/dO item puts the 8 rows before its tile at the slot's start
// and the tile 1 KB further (kPre), and its side data holds the pairs of key rows j0-4 ..
// j0+127 (132 words).
template <bool kFrac>
struct Layout {
    static constexpr uint32_t kPre = kFrac ? 1024u : 0u;
    static constexpr uint32_t kSlot = ring::kSlotBytes + kPre;
    static constexpr uint32_t kSide = kFrac ? 640u : 512u;  // bytes of side data per slot
    static constexpr uint32_t kOffSide = kSlots * kSlot;
    static constexpr uint32_t kOffBar = kOffSide + kSlots * kSide;
    static constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
    static constexpr uint32_t kSmemAlloc = kOffTmemSlot + 16 + 1024;
};

// Band queries [j0, min(T-1, j0+127+W-1)] in 64-query chunks, grouped by kMaxGroupChunks
// (each group re-reads the K and V tiles, so no ring item waits on a later one); active
// offsets o <= T-1-j0. Head size 128 (kWide): K and V take two items each (their column
// halves) and a chunk two (Q, dO: both halves each), so a group holds one chunk (6 items).
template <bool kWide>
struct Plan {
    static constexpr int kKV = kWide ? 2 : 1;        // items per K (and per V) tile
    static constexpr int kCI = kWide ? 2 : 1;        // items per band chunk
    static constexpr int kMaxGC = kWide ? 1 : kMaxGroupChunks;
    int32_t j0, q_lo, n_chunks, n_groups, n_act;
    __device__ __forceinline__ int nch(int g) const {
        return min(kMaxGC, n_chunks - g * kMaxGC);
    }
    __device__ __forceinline__ uint32_t group_items(int g) const { return 2 * kKV + kCI * nch(g); }
};

// Launch query slice of query head hq (of the `group` heads that read the tile's kv head).
__device__ __forceinline__ int64_t query_slice(const BwdParams& p, const ring::Tile& tl, int hq) {
    return (int64_t)tl.layer * p.slices_per_layer + (int64_t)tl.s * p.group + hq;
}

template <bool kWide>
__device__ __forceinline__ Plan<kWide> make_plan(const BwdParams& p, int layer, int32_t j0) {
    Plan<kWide> pl;
    pl.j0 = j0;
    const int64_t qlast64 = (int64_t)j0 + kRows - 1 + p.W - 1;
    const int32_t qlast = qlast64 < p.T - 1 ? (int32_t)qlast64 : p.T - 1;
    pl.q_lo = j0 / kChunk;
    pl.n_chunks = qlast / kChunk - pl.q_lo + 1;
    pl.n_groups = (pl.n_chunks + Plan<kWide>::kMaxGC - 1) / Plan<kWide>::kMaxGC;
    const int32_t* offs = p.tabs.off[layer];
    int32_t n = 0;
    for (int e = 0; e < p.tabs.count[layer]; ++e)
        if (offs[e] <= p.T - 1 - j0) n = e + 1;
    pl.n_act = n;
    return pl;
}

// Tile walk: at head size 128 each kv tile is taken twice, by output half (the fastest index).
template <bool kWide>
__device__ __forceinline__ ring::Tile tile_at(const BwdParams& p, uint32_t idx, int& half) {
    half = kWide ? (int)(idx & 1u) : 0;
    return ring::tile_of(kWide ? idx >> 1 : idx, p.tiles_per_slice, p.slices_per_layer_kv32);
}

// Head size 128 (kWide): two CTAs per kv tile, one per half of the dK/dV columns; both form
// the full S^T = K Q^T and dP^T = V dO^T (8 k-steps over the column halves), each takes
// dV_half += P^T dO_half and dK_half += dS^T Q_half and, in the offsets, the own half of
// the Q_o / dO_o rows.
template <bool kFrac, bool kWide>
__global__ void __launch_bounds__(kThreads, 2) bwd_dkdv_tc_kernel(const __grid_constant__ BwdArgs<kFrac> p) {
    static_assert(!(kFrac && kWide), "the fractional mode is for head size 64");
    using PL = Plan<kWide>;
    using L = Layout<kFrac>;
    constexpr uint32_t kOffBar = L::kOffBar, kOffTmemSlot = L::kOffTmemSlot, kPre = L::kPre;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - smem_u32(smem_raw));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t T = p.T, W = p.W;
    const ring::Ring rg{sbase, sbase + kOffBar, kSlots, kRowWarps, L::kSlot};
    auto bar = [&](uint32_t idx) { return sbase + kOffBar + 8u * idx; };
    const uint32_t B_S = bar(kBarS), B_P = bar(kBarP), B_M = bar(kBarM), B_T = bar(kBarT);
    auto side_addr = [&](uint32_t seq) { return sbase + L::kOffSide + rg.slot(seq) * L::kSide; };
    auto side_ptr = [&](uint32_t seq) {
        return reinterpret_cast<const float*>(smem + L::kOffSide + rg.slot(seq) * L::kSide);
    };
    auto slot_ptr = [&](uint32_t seq) { return smem + (rg.addr(seq) - sbase); };

    if (tid == 0) {
        ring::init_ring_barriers(rg, kFullArrivals);
        mbar_init(B_S, 1);
        mbar_init(B_P, kRowWarps);
        mbar_init(B_M, 1);
        mbar_init(B_T, kRowWarps);
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

    if (warp == 9) {
        // ------------------------------------------------ producer (lane 0)
        if (lane == 0) {
            prefetch_tmap(&p.tm_q);
            prefetch_tmap(&p.tm_do);
            prefetch_tmap(&p.tm_k);
            prefetch_tmap(&p.tm_v);
            prefetch_tmap(&p.tm_dk);
            prefetch_tmap(&p.tm_dv);
            if constexpr (kFrac) {
                prefetch_tmap(&p.tm_q8);
                prefetch_tmap(&p.tm_do8);
            }
            uint32_t seq = 0;
            const int32_t Tp = p.T_pad;
            for (uint32_t idx = blockIdx.x; idx < p.total_tiles; idx += gridDim.x) {
                int half;
                const ring::Tile tl = tile_at<kWide>(p, idx, half);
                const PL pl = make_plan<kWide>(p, tl.layer, tl.row0);
                const int32_t z = (int32_t)tl.zl;  // the kv slice of the tile
                for (int hq = 0; hq < (int)p.group; ++hq)
                for (int g = 0; g < pl.n_groups; ++g) {
                    // the query slice: head hq of the heads that read this kv head
                    const int64_t zq64 = query_slice(p, tl, hq);
                    const int32_t zq = (int32_t)zq64;
                    const float* l2_row = p.lse2 + zq64 * Tp;
                    const float* d_row = p.delta + zq64 * Tp;
                    // K and V tiles (head size 128: each by column halves)
                    for (int h = 0; h < 2; ++h)
                        for (int xh = 0; xh < PL::kKV; ++xh, ++seq) {
                            if (!rg.acquire(seq, aborted, p.err)) continue;
                            const CUtensorMap* map = h == 0 ? &p.tm_k : &p.tm_v;
                            mbar_arrive_expect_tx(rg.full(seq), ring::kSlotBytes);
                            tma_load_3d(rg.addr(seq), map, rg.full(seq), 64 * xh, pl.j0, z);
                            tma_load_3d(rg.addr(seq) + kChunkBytes, map, rg.full(seq), 64 * xh,
                                        pl.j0 + kChunk, z);
                        }
                    // band chunks: Q and dO rows qb.., with lse*log2(e) and D of those rows
                    // (head size 128: the Q chunk's two halves, then the dO chunk's)
                    for (int c = 0; c < pl.nch(g); ++c) {
                        const int32_t qb = (pl.q_lo + g * PL::kMaxGC + c) * kChunk;
                        const uint32_t side_bytes = 4u * (uint32_t)min(kChunk, Tp - qb);
                        if constexpr (kWide) {
                            for (int h = 0; h < 2; ++h, ++seq) {
                                if (!rg.acquire(seq, aborted, p.err)) continue;
                                const CUtensorMap* map = h == 0 ? &p.tm_q : &p.tm_do;
                                mbar_arrive_expect_tx(rg.full(seq), 2 * kChunkBytes + (h == 0 ? 2 * side_bytes : 0u));
                                tma_load_3d(rg.addr(seq), map, rg.full(seq), 0, qb, zq);
                                tma_load_3d(rg.addr(seq) + kChunkBytes, map, rg.full(seq), 64, qb, zq);
                                if (h == 0) {
                                    bulk_load(side_addr(seq), l2_row + qb, side_bytes, rg.full(seq));
                                    bulk_load(side_addr(seq) + 256, d_row + qb, side_bytes, rg.full(seq));
                                }
                            }
                            continue;
                        }
                        if (!rg.acquire(seq, aborted, p.err)) { ++seq; continue; }
                        mbar_arrive_expect_tx(rg.full(seq), 2 * kChunkBytes + 2 * side_bytes);
                        tma_load_3d(rg.addr(seq), &p.tm_q, rg.full(seq), 0, qb, zq);
                        tma_load_3d(rg.addr(seq) + kChunkBytes, &p.tm_do, rg.full(seq), 0, qb, zq);
                        bulk_load(side_addr(seq), l2_row + qb, side_bytes, rg.full(seq));
                        bulk_load(side_addr(seq) + 256, d_row + qb, side_bytes, rg.full(seq));
                        ++seq;
                    }
                }
                // Q_o of every offset, then dO_o of every offset; both carry the (P, dS) pairs of
                // the tile's key rows as side data. Fractional mode: pairs from key row j0 - 4
                // (from row 0 at j0 = 0, leaving words 0-3 unread) and, where w != 0, the 8 rows
                // before the tile.
                const int32_t* offs = p.tabs.off[tl.layer];
                const int32_t pfirst = kFrac ? max(pl.j0 - 4, 0) : pl.j0;
                const uint32_t pskip = kFrac ? 4u * (uint32_t)(pfirst - (pl.j0 - 4)) : 0u;
                const uint32_t pair_bytes =
                    4u * (uint32_t)min(kRows + (int32_t)(kFrac ? 4 : 0) - (int32_t)(pskip / 4u), Tp - pfirst);
                for (int h = 0; h < 2; ++h)
                for (int hq = 0; hq < (int)p.group; ++hq) {
                    const int32_t zq = (int32_t)query_slice(p, tl, hq);
                    for (int k = 0; k < pl.n_act; ++k, ++seq) {
                        if (!rg.acquire(seq, aborted, p.err)) continue;
                        const int32_t y = pl.j0 + offs[k];
                        const CUtensorMap* map = h == 0 ? &p.tm_q : &p.tm_do;
                        bool pre = false;
                        if constexpr (kFrac) pre = p.w[tl.layer][k] != 0.f;
                        mbar_arrive_expect_tx(rg.full(seq), ring::kSlotBytes + (pre ? 1024u : 0u) + pair_bytes);
                        const int32_t xo = 64 * half;  // the own half (head size 128)
                        tma_load_3d(rg.addr(seq) + kPre, map, rg.full(seq), xo, y, zq);
                        tma_load_3d(rg.addr(seq) + kPre + kChunkBytes, map, rg.full(seq), xo, y + kChunk, zq);
                        if constexpr (kFrac) {
                            if (pre)
                                tma_load_3d(rg.addr(seq), h == 0 ? &p.tm_q8 : &p.tm_do8, rg.full(seq), 0,
                                            y - 8, zq);
                        }
                        bulk_load(side_addr(seq) + pskip, p.pds + ((int64_t)zq * p.n_max + k) * Tp + pfirst,
                                  pair_bytes, rg.full(seq));
                    }
                }
                // staging slots of the dK and dV tiles
                for (int h = 0; h < 2; ++h, ++seq)
                    if (rg.acquire(seq, aborted, p.err)) rg.publish_empty(seq);
            }
            // teardown: the last fills have landed (no copy may still be writing this CTA's
            // shared memory when it exits) and every slot's last use has been released
            for (uint32_t q = seq > kSlots ? seq - kSlots : 0; q < seq; ++q)
                rg.wait_full(q, aborted, p.err);
            for (uint32_t q = seq > kSlots ? seq - kSlots : 0; q < seq; ++q)
                rg.acquire(q + kSlots, aborted, p.err);
        }
    } else if (warp == 8) {
        // ------------------------------------------------ MMA issue
        if (lane == 0) {
            uint32_t seq = 0, mcount = 0, tcount = 0;
            const uint32_t idesc_s = idesc_bf16(128, 64, 0, 0);
            const uint32_t idesc_o = idesc_bf16(128, 64, 0, 1);
            // descriptors of shared address sbase; an operand at sbase + x adds x >> 4
            const uint64_t dkm = sdesc_sw128(sbase, 16, 1024), dmn = sdesc_sw128(sbase, 0, 1024);
            for (uint32_t idx = blockIdx.x; idx < p.total_tiles; idx += gridDim.x, ++tcount) {
                int half;
                const ring::Tile tl = tile_at<kWide>(p, idx, half);
                const PL pl = make_plan<kWide>(p, tl.layer, tl.row0);
                if (tcount > 0) mbar_wait(B_T, (tcount - 1) & 1, aborted, p.err);
                int cg = 0;  // chunk index within the tile (over every query head)
                for (int hq = 0; hq < (int)p.group; ++hq)
                for (int g = 0; g < pl.n_groups; ++g) {
                    const int nch = pl.nch(g);
                    const uint32_t kseq = seq, vseq = seq + PL::kKV, bseq = seq + 2 * PL::kKV;
                    seq += pl.group_items(g);
                    for (int j = 0; j < PL::kKV; ++j) {
                        rg.wait_full(kseq + j, aborted, p.err);
                        rg.wait_full(vseq + j, aborted, p.err);
                    }
                    for (int c = 0; c < nch; ++c, ++cg, ++mcount) {
                        // the chunk's Q (and dO) operands; head size 128: two items, each the
                        // chunk's two column halves
                        const uint32_t qaddr = rg.addr(bseq + PL::kCI * c);
                        const uint32_t gaddr = kWide ? rg.addr(bseq + PL::kCI * c + 1) : qaddr + kChunkBytes;
                        for (int j = 0; j < PL::kCI; ++j) rg.wait_full(bseq + PL::kCI * c + j, aborted, p.err);
                        // S^T/dP^T columns hold the previous chunk's P^T/dS^T until its MMAs finish
                        if (cg > 0) mbar_wait(B_M, (mcount - 1) & 1, aborted, p.err);
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 4 * PL::kKV; ++kk) {
                            // k-steps 4h .. 4h+3: column half h of K (its item) and of the Q chunk
                            const uint64_t a = dkm + ((rg.addr(kseq + (kk >> 2)) - sbase) >> 4) + 2 * (kk & 3);
                            const uint64_t b = dkm + ((qaddr + (kk >> 2) * kChunkBytes - sbase) >> 4) + 2 * (kk & 3);
                            mma_ss(tmem + kColS, a, b, idesc_s, kk > 0);
                        }
#pragma unroll
                        for (int kk = 0; kk < 4 * PL::kKV; ++kk) {
                            const uint64_t a = dkm + ((rg.addr(vseq + (kk >> 2)) - sbase) >> 4) + 2 * (kk & 3);
                            const uint64_t b = dkm + ((gaddr + (kk >> 2) * kChunkBytes - sbase) >> 4) + 2 * (kk & 3);
                            mma_ss(tmem + kColP, a, b, idesc_s, kk > 0);
                        }
                        mma_commit(B_S);
                        if (c == nch - 1) {
                            for (int j = 0; j < PL::kKV; ++j) {
                                rg.release_mma(kseq + j);
                                rg.release_mma(vseq + j);
                            }
                        }
                        mbar_wait(B_P, mcount & 1, aborted, p.err);
                        tc_fence_after();
                        // P^T / dS^T of queries 32h..32h+31 sit in columns [32h, 32h+16) of their block
                        // dV (own half) += P^T dO_half, dK (own half) += dS^T Q_half
                        const uint32_t ho = kWide ? half * kChunkBytes : 0u;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t acol = 32 * (kk >> 1) + 8 * (kk & 1);
                            const uint32_t acc = (cg > 0 || kk > 0) ? 1u : 0u;
                            mma_ts(tmem + kColDV, tmem + kColS + acol,
                                   dmn + ((gaddr + ho - sbase) >> 4) + 128 * kk, idesc_o, acc);
                            mma_ts(tmem + kColDK, tmem + kColP + acol,
                                   dmn + ((qaddr + ho - sbase) >> 4) + 128 * kk, idesc_o, acc);
                        }
                        mma_commit(B_M);
                        for (int j = 0; j < PL::kCI; ++j) rg.release_mma(bseq + PL::kCI * c + j);
                    }
                }
                seq += 2 * p.group * pl.n_act + 2;
            }
            if (mcount > 0) mbar_wait(B_M, (mcount - 1) & 1, aborted, p.err);
        }
    } else {
        // ------------------------------------------------ row threads: key row r, dim half h
        const int q4 = warp & 3, h = warp >> 2;
        const int r = 32 * q4 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
        const float sl2 = p.scale_log2;
        uint32_t seq = 0, mcount = 0;
        for (uint32_t idx = blockIdx.x; idx < p.total_tiles; idx += gridDim.x) {
            int half;
            const ring::Tile tl = tile_at<kWide>(p, idx, half);
            const PL pl = make_plan<kWide>(p, tl.layer, tl.row0);
            const int32_t j0 = pl.j0;
            const int32_t j = j0 + r;
            const bool row_ok = j < T;
            const int32_t* offs = p.tabs.off[tl.layer];

            // ---- band: P^T and dS^T of this thread's 32 query columns, 16 at a time (for every
            // query head reading this kv head)
            for (int hq = 0; hq < (int)p.group; ++hq)
            for (int g = 0; g < pl.n_groups; ++g) {
                const int nch = pl.nch(g);
                const uint32_t bseq = seq + 2 * PL::kKV;
                seq += pl.group_items(g);
                for (int c = 0; c < nch; ++c, ++mcount) {
                    const int32_t qb = (pl.q_lo + g * PL::kMaxGC + c) * kChunk + 32 * h;
                    const uint32_t cseq = bseq + PL::kCI * c;  // the chunk's (first) item
                    mbar_wait(B_S, mcount & 1, aborted, p.err);
                    rg.wait_full(cseq, aborted, p.err);  // lse*log2(e) / D side data
                    tc_fence_after();
                    __syncwarp();  // converged for the warp-collective TMEM accesses below
                    const int32_t klo = j0 + 32 * q4;
                    const bool need = (qb + 31 - klo >= 0) && (qb - (klo + 31) < W) && qb < T;
                    const float* L = side_ptr(cseq) + 32 * h;
                    const float* Dd = L + kChunk;
                    const int32_t dist0 = qb - j;
                    // bit c: query qb + c is this key row's (0 <= qb + c - j < W, qb + c < T)
                    uint32_t okm = 0u;
                    if (row_ok) {
                        const int32_t lo = max(0, -dist0);
                        const int32_t hi = min(32, min(W - dist0, T - qb));
                        if (hi > lo)
                            okm = (hi == 32 ? 0xffffffffu : (1u << hi) - 1u) & ~((1u << lo) - 1u);
                    }
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const uint32_t col = 32 * h + 16 * half;
                        uint32_t pp[8], pd[8];
                        if (need) {
                            uint32_t sv[16], dv[16];
                            tmem_ld16(tmem + lane_base + kColS + col, sv);
                            tmem_ld16(tmem + lane_base + kColP + col, dv);
                            tmem_ld_wait(sv, dv);
#pragma unroll
                            for (int e = 0; e < 16; e += 4) {
                                const int ee = 16 * half + e;
                                const float4 l4 = *reinterpret_cast<const float4*>(L + ee);
                                const float4 d4 = *reinterpret_cast<const float4*>(Dd + ee);
                                const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
                                const float dd[4] = {d4.x, d4.y, d4.z, d4.w};
                                float pv[4], ds[4];
#pragma unroll
                                for (int u = 0; u < 4; ++u) {
                                    const bool ok = (okm >> (ee + u)) & 1u;
                                    pv[u] = ok ? ex2(__uint_as_float(sv[e + u]) * sl2 - lv[u]) : 0.f;
                                    // selects, not products with p = 0: for a query column at or
                                    // past T, Dd holds bytes this call never wrote (pad rows of
                                    // the workspace, or slot memory past the side copy), possibly
                                    // non-finite, and 0 * NaN would reach dK through the MMA
                                    ds[u] = ok ? pv[u] * (__uint_as_float(dv[e + u]) - dd[u]) : 0.f;
                                }
                                pp[e >> 1] = pack_bf16x2(pv[0], pv[1]);
                                pp[(e >> 1) + 1] = pack_bf16x2(pv[2], pv[3]);
                                pd[e >> 1] = pack_bf16x2(ds[0], ds[1]);
                                pd[(e >> 1) + 1] = pack_bf16x2(ds[2], ds[3]);
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) pp[e] = pd[e] = 0u;
                        }
                        // packed over the columns this thread already read (16*half .. +16)
                        tmem_st8(tmem + lane_base + kColS + 32 * h + 8 * half, pp);
                        tmem_st8(tmem + lane_base + kColP + 32 * h + 8 * half, pd);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    // the item's side data was read with generic loads; the MMA warp releases
                    // the slot to the next bulk copy after this arrival
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(B_P);
                }
            }

            // ---- offsets, first pass: dk_j += dS q_{j+o} over my 32 dims, then folded into the
            // dK accumulator in TMEM. The pass accumulates in registers, so it overlaps the band's
            // last dK/dV MMAs; their completion is awaited only before TMEM is touched (the fold,
            // or the epilogue when no offset is active). The ring's parity waits do not need it:
            // every band item was known to have landed before the B_S waits above returned.
            bool band_done = false;
            auto await_band = [&]() {
                if (band_done) return;
                mbar_wait(B_M, (mcount - 1) & 1, aborted, p.err);
                tc_fence_after();
                band_done = true;
            };
            float acc[32];
            for (int pass = 0; pass < 2; ++pass) {
#pragma unroll
                for (int c = 0; c < 32; ++c) acc[c] = 0.f;
#pragma unroll 1
                for (int e = 0; e < (int)p.group * pl.n_act; ++e) {
                    const int k = e % pl.n_act;  // the offset (the query head is e / n_act)
                    rg.wait_full(seq, aborted, p.err);
                    if constexpr (kFrac) {
                        // key j is row lo of query j + c (weight 1 - w: pair of key row j) and
                        // row lo + 1 of query j + c - 1 (weight w: pair of key row j - 1); the
                        // tile's row r is virtual row r + 8 of the slot, the row before it r + 7
                        const float wk = p.w[tl.layer][k];
                        const uint32_t* pw = reinterpret_cast<const uint32_t*>(side_ptr(seq));
                        const uint32_t plo = (row_ok && j + offs[k] < T) ? pw[r + 4] : 0u;
                        const uint32_t phi =
                            (wk != 0.f && row_ok && j >= 1 && j + offs[k] - 1 < T) ? pw[r + 3] : 0u;
                        const float xlo = pass == 0 ? bf16hi(plo) : bf16lo(plo);  // dS or P
                        const float xhi = pass == 0 ? bf16hi(phi) : bf16lo(phi);
                        const uint32_t clo = pack_bf16x2((1.f - wk) * xlo, 0.f);
                        const uint32_t chi = pack_bf16x2(wk * xhi, 0.f);
                        const uint8_t* row = slot_ptr(seq);
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint4 x = *reinterpret_cast<const uint4*>(row + sw128_off(r + 8, 4 * h + c));
                            axpy2_bf16(clo, x.x, acc[8 * c + 0], acc[8 * c + 1]);
                            axpy2_bf16(clo, x.y, acc[8 * c + 2], acc[8 * c + 3]);
                            axpy2_bf16(clo, x.z, acc[8 * c + 4], acc[8 * c + 5]);
                            axpy2_bf16(clo, x.w, acc[8 * c + 6], acc[8 * c + 7]);
                        }
                        if (wk != 0.f) {
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const uint4 x = *reinterpret_cast<const uint4*>(row + sw128_off(r + 7, 4 * h + c));
                                axpy2_bf16(chi, x.x, acc[8 * c + 0], acc[8 * c + 1]);
                                axpy2_bf16(chi, x.y, acc[8 * c + 2], acc[8 * c + 3]);
                                axpy2_bf16(chi, x.z, acc[8 * c + 4], acc[8 * c + 5]);
                                axpy2_bf16(chi, x.w, acc[8 * c + 6], acc[8 * c + 7]);
                            }
                        }
                        rg.release_warp(seq, lane);
                        ++seq;
                        continue;
                    }
                    const uint32_t pair = (row_ok && j + offs[k] < T)
                                              ? reinterpret_cast<const uint32_t*>(side_ptr(seq))[r] : 0u;
                    const uint32_t sc = pass == 0 ? pair >> 16 : pair & 0xFFFFu;  // dS or P (bf16)
                    const uint8_t* row = slot_ptr(seq);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 x = *reinterpret_cast<const uint4*>(row + sw128_off(r, 4 * h + c));
                        axpy2_bf16(sc, x.x, acc[8 * c + 0], acc[8 * c + 1]);
                        axpy2_bf16(sc, x.y, acc[8 * c + 2], acc[8 * c + 3]);
                        axpy2_bf16(sc, x.z, acc[8 * c + 4], acc[8 * c + 5]);
                        axpy2_bf16(sc, x.w, acc[8 * c + 6], acc[8 * c + 7]);
                    }
                    rg.release_warp(seq, lane);
                    ++seq;
                }
                // add into TMEM: dK columns [32h, +32) after the first pass, dV after the second
                if (pl.n_act > 0) {
                    await_band();
                    __syncwarp();  // converged for the warp-collective TMEM accesses below
                    const uint32_t col = (pass == 0 ? kColDK : kColDV) + 32 * h;
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        uint32_t v[16];
                        tmem_ld16(tmem + lane_base + col + 16 * q, v);
                        tmem_ld_wait(v);
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            v[c] = __float_as_uint(__uint_as_float(v[c]) + acc[16 * q + c]);
                        tmem_st16(tmem + lane_base + col + 16 * q, v);
                    }
                    tmem_st_wait();
                }
            }

            // ---- epilogue: dk = scale * dK, dv = dV (band + offsets), staged, TMA stores
            const uint32_t kst = seq, vst = seq + 1;
            seq += 2;
            await_band();
            rg.wait_full(kst, aborted, p.err);
            rg.wait_full(vst, aborted, p.err);
            __syncwarp();  // converged for the warp-collective TMEM accesses below
            {
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + kColDK + 32 * h, v);
                tmem_ld_wait(v);
                uint8_t* st = slot_ptr(kst);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int e = 8 * c;
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(v[e + 0]) * p.scale, __uint_as_float(v[e + 1]) * p.scale);
                    w.y = pack_bf16x2(__uint_as_float(v[e + 2]) * p.scale, __uint_as_float(v[e + 3]) * p.scale);
                    w.z = pack_bf16x2(__uint_as_float(v[e + 4]) * p.scale, __uint_as_float(v[e + 5]) * p.scale);
                    w.w = pack_bf16x2(__uint_as_float(v[e + 6]) * p.scale, __uint_as_float(v[e + 7]) * p.scale);
                    *reinterpret_cast<uint4*>(st + sw128_off(r, 4 * h + c)) = w;
                }
                tmem_ld32(tmem + lane_base + kColDV + 32 * h, v);
                tmem_ld_wait(v);
                st = slot_ptr(vst);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int e = 8 * c;
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(v[e + 0]), __uint_as_float(v[e + 1]));
                    w.y = pack_bf16x2(__uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
                    w.z = pack_bf16x2(__uint_as_float(v[e + 4]), __uint_as_float(v[e + 5]));
                    w.w = pack_bf16x2(__uint_as_float(v[e + 6]), __uint_as_float(v[e + 7]));
                    *reinterpret_cast<uint4*>(st + sw128_off(r, 4 * h + c)) = w;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B_T);  // TMEM free for the next tile's MMAs
            fence_proxy_async_smem();
            asm volatile("bar.sync 1, 256;" ::: "memory");
            if (tid == 0) {
                if (!aborted) {
                    const int32_t z = (int32_t)tl.zl;
                    const int32_t xo = 64 * half;  // the CTA's output columns
                    tma_store_3d(&p.tm_dk, rg.addr(kst), xo, j0, z);
                    tma_store_3d(&p.tm_dv, rg.addr(vst), xo, j0, z);
                    if (j0 + kChunk < T) {
                        tma_store_3d(&p.tm_dk, rg.addr(kst) + kChunkBytes, xo, j0 + kChunk, z);
                        tma_store_3d(&p.tm_dv, rg.addr(vst) + kChunkBytes, xo, j0 + kChunk, z);
                    }
                    tma_store_commit();
                    tma_store_wait_read0();
                }
                rg.release_stage(kst);
                rg.release_stage(vst);
            }
        }
    }

    // after a timeout in this CTA, its own copies and MMAs in flight land before TMEM is released
    tc_fence_before();
    settle_if_aborted(__syncthreads_or(aborted ? 1 : 0));
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

namespace {

template <bool kFrac, bool kWide>
fibattn_status launch_bwd(const void* q, const void* k, const void* v, const void* o,
                          const float* lse, const void* dO, void* dq, void* dk, void* dv,
                          float* delta, float* lse2, uint32_t* pds, int32_t n_max,
                          const AttnShape& sh, const OffsetTables& t, const FracTables* ft,
                          float* galpha, cudaStream_t st) {
    const int64_t slices = sh.slices_per_layer * sh.n_layers;
    if (slices > 0x7fffffff) return FIBATTN_ERR_INVALID_ARG;
    const int64_t slices_kv = slices / sh.group;
    const int32_t tiles = (sh.T + kRows - 1) / kRows;
    const int64_t halves = kWide ? 2 : 1;  // CTAs per tile (head size 128: one per column half)
    const int64_t gx = (int64_t)tiles * sh.slices_per_layer * halves;
    if (gx > 0x7fffffff || (int64_t)tiles * slices * halves > 0x7fffffff) return FIBATTN_ERR_INVALID_ARG;
    BwdArgs<kFrac> P;
    // the error-word lookup is a runtime call: it binds the device's primary context to this
    // thread (a fresh thread, e.g. autograd's, may have none), which the encoding needs
    P.err = device_error_word();
    if (!P.err) return cuda_fail(-1, "cudaGetSymbolAddress (error word)");
    const void* bases[8] = {q, k, v, dO, dq, dk, dv, o};
    CUtensorMap* maps[8] = {&P.tm_q, &P.tm_k, &P.tm_v, &P.tm_do, &P.tm_dq, &P.tm_dk, &P.tm_dv, &P.tm_o};
    for (int m = 0; m < 8; ++m) {
        // k, v, dk, dv (maps 1, 2, 5, 6) over the kv slices
        const bool kvmap = m == 1 || m == 2 || m == 5 || m == 6;
        const int64_t sl = kvmap ? slices_kv : slices;
        const int r = kWide ? make_bf16_rows_map_d(maps[m], bases[m], sl, sh.T, 128)
                            : make_bf16_rows_map(maps[m], bases[m], sl, sh.T);
        if (r != 0) return cuda_fail(r, "cuTensorMapEncodeTiled (bwd)");
    }
    if constexpr (kFrac) {
        const void* b8[4] = {k, v, q, dO};
        CUtensorMap* m8[4] = {&P.tm_k8, &P.tm_v8, &P.tm_q8, &P.tm_do8};
        for (int m = 0; m < 4; ++m) {
            const int r = make_bf16_rows8_map(m8[m], b8[m], m < 2 ? slices_kv : slices, sh.T);
            if (r != 0) return cuda_fail(r, "cuTensorMapEncodeTiled (bwd, 8-row box)");
        }
        P.galpha = galpha;
        for (int l = 0; l < kMaxLayersPerLaunch; ++l)
            for (int e = 0; e < kMaxOffsets; ++e) {
                P.w[l][e] = ft->w[l][e];
                P.f[l][e] = ft->f[l][e];
            }
    }
    P.lse = lse;
    P.delta = delta;
    P.lse2 = lse2;
    P.pds = pds;
    P.slices_per_layer = sh.slices_per_layer;
    P.group = (uint32_t)sh.group;
    P.slices_per_layer_kv32 = (uint32_t)(sh.slices_per_layer / sh.group);
    P.total_tiles = (uint32_t)((int64_t)tiles * slices_kv * halves);  // the key owner walks kv tiles
    P.T = sh.T;
    P.W = sh.W;
    P.T_pad = (sh.T + 3) & ~3;
    P.tiles_per_slice = tiles;
    P.n_max = n_max;
    P.scale = sh.scale;
    P.scale_log2 = sh.scale * kLog2e;
    P.tabs = t;
    static bool dq_set[64] = {}, dkdv_set[64] = {};
    static int n_sm[64] = {};
    fibattn_status s0 = set_smem((const void*)dq::bwd_dq_tc_kernel<kFrac, kWide>,
                                 dq::Layout<kFrac, kWide>::kSmemAlloc, dq_set);
    if (s0 != FIBATTN_OK) return s0;
    s0 = set_smem((const void*)dkdv::bwd_dkdv_tc_kernel<kFrac, kWide>,
                  dkdv::Layout<kFrac>::kSmemAlloc, dkdv_set);
    if (s0 != FIBATTN_OK) return s0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail((int32_t)e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return FIBATTN_ERR_UNSUPPORTED;
    if (n_sm[dev] == 0) {
        e = cudaDeviceGetAttribute(&n_sm[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail((int32_t)e, "cudaDeviceGetAttribute");
    }
    const int64_t pgrid = (int64_t)P.total_tiles < 2LL * n_sm[dev] ? (int64_t)P.total_tiles : 2LL * n_sm[dev];
    dim3 grid((unsigned)gx, sh.n_layers);
    const char* n_dq = kFrac ? "bwd_dq_frac_tc" : (kWide ? "bwd_dq_tc128" : "bwd_dq_tc");
    const char* n_kv = kFrac ? "bwd_dkdv_frac_tc" : (kWide ? "bwd_dkdv_tc128" : "bwd_dkdv_tc");
    {
        KernelScope ks(n_dq, st);
        dq::bwd_dq_tc_kernel<kFrac, kWide>
            <<<grid, dq::kThreads, dq::Layout<kFrac, kWide>::kSmemAlloc, st>>>(P);
    }
    s0 = launch_status(n_dq);
    if (s0 != FIBATTN_OK) return s0;
    {
        KernelScope ks(n_kv, st);
        dkdv::bwd_dkdv_tc_kernel<kFrac, kWide>
            <<<(unsigned)pgrid, dkdv::kThreads, dkdv::Layout<kFrac>::kSmemAlloc, st>>>(P);
    }
    return launch_status(n_kv);
}

}  // namespace

fibattn_status launch_bwd_tc_bf16(const void* q, const void* k, const void* v, const void* o,
                                  const float* lse, const void* dO, void* dq, void* dk, void* dv,
                                  float* delta, float* lse2, uint32_t* pds, int32_t n_max,
                                  const AttnShape& sh, const OffsetTables& t, cudaStream_t st) {
    if (sh.d == 128)
        return launch_bwd<false, true>(q, k, v, o, lse, dO, dq, dk, dv, delta, lse2, pds, n_max, sh,
                                       t, nullptr, nullptr, st);
    return launch_bwd<false, false>(q, k, v, o, lse, dO, dq, dk, dv, delta, lse2, pds, n_max, sh, t,
                                    nullptr, nullptr, st);
}

fibattn_status launch_bwd_frac_tc_bf16(const void* q, const void* k, const void* v, const void* o,
                                       const float* lse, const void* dO, void* dq, void* dk,
                                       void* dv, float* delta, float* lse2, uint32_t* pds,
                                       int32_t n_max, float* galpha, const AttnShape& sh,
                                       const FracTables& t, cudaStream_t st) {
    return launch_bwd<true, false>(q, k, v, o, lse, dO, dq, dk, dv, delta, lse2, pds, n_max, sh,
                                   t.c, &t, galpha, st);
}

}  // namespace fibattn
