// bwd_fused.cu -- the one-pass bf16 backward: one thread block per 128-row tile owns both dq
// of the tile's queries and dk, dv of the tile's keys (head size 64, one kv head per query
// head).
//
// The gradient is that of bwd_tc.cu (softmax attention over the attended set of
// "Depth-Staggered Fibonacci Spacing for Sparse Attention", gist.science explainer,
// Metodologia / Arquitetura, "Conjunto Atendido": the window i-W+1..i plus the keys i-o of the
// layer's offsets):
//   D_i = dO_i . o_i,  P_ij = exp(scale q_i.k_j - lse_i),  dS_ij = P_ij (dO_i . v_j - D_i),
//   dq_i = scale sum_j dS_ij k_j,  dk_j = scale sum_i dS_ij q_i,  dv_j = sum_i P_ij dO_i.
//
// Two launches:
//   bwd_prep    D = dO . o and lse log2(e) of every row into the workspace (a block's keys reach
//               the rows of other tiles, so these cannot come from the block that owns them).
//   bwd_fused   one block (320 threads) per tile [t0, t0+128) of a slice, two blocks per SM:
//     warps 0-7 : two threads per row: warps w and w+4 share TMEM lanes 32(w%4)..+31 and split
//                 the band columns and the 64 head dims of the outputs in halves.
//     warp 8    : TMEM allocation and tcgen05.mma.
//     warp 9    : TMA loads: the tile's Q, dO, K and V rows (resident for the whole block) and
//                 an in-order ring of two 16 KB slots for the rest.
//   dq phase (the block's 128 queries):
//     band, per 64-key chunk: S = Q K^T and dP = dO V^T into TMEM; the row threads form dS,
//     write it back as bf16; dQ += dS K in TMEM. The chunks below the tile come through the
//     ring, those of the tile itself are its resident K and V rows.
//     offsets: per table entry the shifted tiles K[t0-o ..], V[t0-o ..] (ring); each thread
//     forms q.k and dO.v over the 64 dims (both threads of a row alike), P and dS, and adds
//     dS k to its 32 dims of dq.
//     epilogue: dq = scale (dQ + dq_off), staged in a ring slot, TMA store.
//   dk/dv phase (the block's 128 keys):
//     band, per 64-query chunk: S^T = K Q^T, dP^T = V dO^T; P^T, dS^T written back as bf16;
//     dV += P^T dO, dK += dS^T Q in TMEM (the tile's own two chunks are the resident Q and dO
//     rows, later ones come through the ring with their lse log2(e) and D).
//     offsets: per table entry the shifted tiles Q[t0+o ..], dO[t0+o ..] (ring); the pair of
//     key j and query j+o is formed again here (q.k, dO.v), so the block needs no pairs from
//     other blocks; dk += dS q and dv += P dO in registers.
//     epilogue: dk = scale (dK + dk_off), dv = dV + dv_off, staged, TMA stores.
// No atomics: every output row has one writer. Each pair's P and dS are formed from the same
// operands in the same order as the two-kernel backward's query owner does, and every sum is
// taken in the same order, so the two backwards agree bit for bit.
//
// Every mbarrier wait is bounded (tc::mbar_wait); a wait that runs out latches the device
// error word, later waits return at once, and the block still releases its TMEM, after a
// fixed wait that lets its own copies and MMAs in flight land (tc::settle_if_aborted).
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

constexpr int kRows = 128;
constexpr int kChunk = kTmaBoxRows;
constexpr uint32_t kTileBytes = kRows * 128;    // 16 KB
constexpr uint32_t kChunkBytes = kChunk * 128;  // 8 KB
constexpr float kLog2e = 1.4426950408889634f;

constexpr int kThreads = 320;
constexpr int kRowWarps = 8;
constexpr uint32_t kTmemCols = 256;
// dq phase: dQ [0, 64); dk/dv phase: dK [0, 64), dV [64, 128); both: S [128, 192), dP [192, 256)
constexpr uint32_t kColDQ = 0, kColDK = 0, kColDV = 64, kColS = 128, kColP = 192;
constexpr uint32_t kSlots = 2;

// barriers: FULL[kSlots], EMPTY[kSlots], resident tiles loaded, S/dP ready, dS written
// (8 warps), dQ or dK/dV MMAs of a chunk done, dQ read out of TMEM (8 warps)
constexpr uint32_t kBarRes = 2 * kSlots, kBarS = kBarRes + 1, kBarP = kBarRes + 2,
                   kBarM = kBarRes + 3, kBarDQ = kBarRes + 4;
constexpr uint32_t kNumBars = kBarDQ + 1;

// Shared memory: the tile's Q, dO, K, V rows; the ring slots; per slot 512 bytes of side data
// (lse log2(e) and D of a 64-query band chunk); lse log2(e) and D of the tile's own rows.
constexpr uint32_t kOffQ = 0, kOffG = kTileBytes, kOffK = 2 * kTileBytes, kOffV = 3 * kTileBytes;
constexpr uint32_t kOffRing = 4 * kTileBytes;
constexpr uint32_t kSide = 512;
constexpr uint32_t kOffSide = kOffRing + kSlots * kTileBytes;
constexpr uint32_t kOffOwn = kOffSide + kSlots * kSide;  // lse2 [128] at +0, D [128] at +512
constexpr uint32_t kOffBar = kOffOwn + 1024;
constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemAlloc = kOffTmemSlot + 16 + 1024;  // + alignment slack

struct FusedParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_do;  // inputs, 3D {64, T, slices}, box {64, 64, 1}
    CUtensorMap tm_dq, tm_dk, tm_dv;      // outputs
    const float* delta;                   // workspace: D [slices][T_pad]
    const float* lse2;                    // workspace: lse * log2(e) [slices][T_pad]
    int32_t* err;
    int64_t slices_per_layer;
    int32_t T, W, T_pad, tiles_per_slice;
    float scale, scale_log2;
    OffsetTables tabs;
};

// The work of one tile.
struct Plan {
    int32_t qc_lo;    // first 64-key chunk of the dq phase's band
    int32_t n_qc;     // its chunks; the first n_qring lie below the tile (ring items)
    int32_t n_qring;
    int32_t n_qoff;   // active offsets of the dq phase (o <= the tile's last query)
    int32_t n_kc;     // 64-query chunks of the dk/dv phase's band, from the tile's first row;
                      // chunks 0 and 1 are the tile's own rows, the rest ring items
    int32_t n_koff;   // active offsets of the dk/dv phase (o <= T - 1 - t0)
};

__device__ __forceinline__ Plan make_plan(const FusedParams& p, int layer, int32_t t0) {
    Plan pl;
    const int32_t T = p.T, W = p.W;
    const int32_t kstart = t0 - W + 1 > 0 ? t0 - W + 1 : 0;
    const int32_t klast = t0 + kRows - 1 < T - 1 ? t0 + kRows - 1 : T - 1;
    pl.qc_lo = kstart / kChunk;
    pl.n_qc = klast / kChunk - pl.qc_lo + 1;
    pl.n_qring = t0 / kChunk - pl.qc_lo;
    const int64_t qlast64 = (int64_t)t0 + kRows - 1 + W - 1;
    const int32_t qlast = qlast64 < T - 1 ? (int32_t)qlast64 : T - 1;
    pl.n_kc = qlast / kChunk - t0 / kChunk + 1;
    const int32_t* offs = p.tabs.off[layer];
    int32_t nq = 0, nk = 0;
    for (int e = 0; e < p.tabs.count[layer]; ++e) {
        if (offs[e] <= klast) nq = e + 1;
        if (offs[e] <= T - 1 - t0) nk = e + 1;
    }
    pl.n_qoff = nq;
    pl.n_koff = nk;
    return pl;
}

// s += x . y over a 64-dim row pair (bf16 words of two swizzled rows), in the accumulation
// order of the two-kernel backward's offset dots.
__device__ __forceinline__ float row_dot(const uint8_t* xt, const uint8_t* yt, int r) {
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 x = *reinterpret_cast<const uint4*>(xt + sw128_off(r, c));
        const uint4 y = *reinterpret_cast<const uint4*>(yt + sw128_off(r, c));
        fma2_bf16(x.x, y.x, a0, a1);
        fma2_bf16(x.y, y.y, a2, a3);
        fma2_bf16(x.z, y.z, a0, a1);
        fma2_bf16(x.w, y.w, a2, a3);
    }
    return (a0 + a1) + (a2 + a3);
}

// The 16 bf16 words of dims [32h, 32h + 32) of row r.
__device__ __forceinline__ void load_half_sw(const uint8_t* tile, int r, int h, uint32_t (&w)[16]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint4 x = *reinterpret_cast<const uint4*>(tile + sw128_off(r, 4 * h + c));
        w[4 * c + 0] = x.x; w[4 * c + 1] = x.y; w[4 * c + 2] = x.z; w[4 * c + 3] = x.w;
    }
}

// D and lse log2(e) of every row, rows padded to T_pad (pad rows written as 0). Each warp takes
// 32 consecutive rows: the o and dO rows are copied through shared memory with coalesced
// 16-byte loads (a load instruction covers four whole rows), then lane l sums row l alone, in
// the order the tensor-core backward uses for its offset dots.
constexpr int kPrepWarps = 8;
constexpr int kPrepStride = 9;  // uint4 per staged row: 8 + 1 of padding (conflict-free reads)

__global__ void __launch_bounds__(32 * kPrepWarps) bwd_prep_kernel(const uint4* __restrict__ o,
                                                                   const uint4* __restrict__ dO,
                                                                   const float* __restrict__ lse,
                                                                   float* __restrict__ delta,
                                                                   float* __restrict__ lse2,
                                                                   int64_t slices, int32_t T,
                                                                   int32_t T_pad) {
    __shared__ uint4 stage[kPrepWarps][32 * kPrepStride];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint4* buf = stage[warp];
    const int64_t rows = slices * T;  // source rows, [slices][T][64] bf16 = 8 uint4 per row
    const int64_t step = (int64_t)gridDim.x * kPrepWarps * 32;
    for (int64_t base = ((int64_t)blockIdx.x * kPrepWarps + warp) * 32; base < rows; base += step) {
        const int nr = rows - base < 32 ? (int)(rows - base) : 32;
        uint4 x[8];
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            const uint4* src = pass == 0 ? o : dO;
            // lane l copies chunk l % 8 of rows l / 8, l / 8 + 4, ...
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int rr = 4 * k + (lane >> 3);
                if (rr < nr) buf[rr * kPrepStride + (lane & 7)] = src[(base + rr) * 8 + (lane & 7)];
            }
            __syncwarp();
            if (pass == 0) {
#pragma unroll
                for (int c = 0; c < 8; ++c) x[c] = buf[lane * kPrepStride + c];
                __syncwarp();  // every lane has its o row before the dO rows overwrite them
            }
        }
        if (lane < nr) {
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 g = buf[lane * kPrepStride + c];
                fma2_bf16(g.x, x[c].x, a0, a1);
                fma2_bf16(g.y, x[c].y, a2, a3);
                fma2_bf16(g.z, x[c].z, a0, a1);
                fma2_bf16(g.w, x[c].w, a2, a3);
            }
            const int64_t row = base + lane;
            const int64_t z = row / T;
            const int64_t w = z * T_pad + (row - z * T);
            delta[w] = (a0 + a1) + (a2 + a3);
            lse2[w] = lse[row] * kLog2e;
        }
        __syncwarp();  // the dO rows are read before the next rows' o overwrite them
    }
    // pad rows T .. T_pad - 1 of every slice
    const int32_t npad = T_pad - T;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < slices * npad;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t z = idx / npad;
        const int64_t w = z * T_pad + T + (idx - z * npad);
        delta[w] = 0.f;
        lse2[w] = 0.f;
    }
}

__global__ void __launch_bounds__(kThreads, 2) bwd_fused_kernel(const __grid_constant__ FusedParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - smem_u32(smem_raw));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int layer = blockIdx.y;
    const int tile = blockIdx.x % p.tiles_per_slice;
    const int64_t zl = (int64_t)layer * p.slices_per_layer + blockIdx.x / p.tiles_per_slice;
    const int32_t z = (int32_t)zl;
    const int32_t T = p.T, W = p.W, Tp = p.T_pad;
    const int32_t t0 = tile * kRows;
    const Plan pl = make_plan(p, layer, t0);
    const int32_t* offs = p.tabs.off[layer];
    const int n_kring = pl.n_kc > 2 ? pl.n_kc - 2 : 0;
    // ring item sequence: dq band chunks below the tile, K_o and V_o per dq offset, the dq
    // staging slot, dk/dv band chunks past the tile, Q_o and dO_o per dk/dv offset, the dk and
    // dv staging slots
    const uint32_t seq_qoff = (uint32_t)pl.n_qring;
    const uint32_t seq_dqst = seq_qoff + 2u * pl.n_qoff;
    const uint32_t seq_kring = seq_dqst + 1u;
    const uint32_t seq_koff = seq_kring + (uint32_t)n_kring;
    const uint32_t seq_kvst = seq_koff + 2u * pl.n_koff;
    const uint32_t n_items = seq_kvst + 2u;

    const ring::Ring rg{sbase + kOffRing, sbase + kOffBar, kSlots, kRowWarps, ring::kSlotBytes};
    auto bar = [&](uint32_t idx) { return sbase + kOffBar + 8u * idx; };
    const uint32_t B_RES = bar(kBarRes), B_S = bar(kBarS), B_P = bar(kBarP), B_M = bar(kBarM),
                   B_DQ = bar(kBarDQ);
    auto slot_ptr = [&](uint32_t seq) { return smem + (rg.addr(seq) - sbase); };
    auto side_off = [&](uint32_t seq) { return kOffSide + rg.slot(seq) * kSide; };

    if (tid == 0) {
        ring::init_ring_barriers(rg, 1);
        mbar_init(B_RES, 1);
        mbar_init(B_S, 1);
        mbar_init(B_P, kRowWarps);
        mbar_init(B_M, 1);
        mbar_init(B_DQ, kRowWarps);
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
            const int64_t wrow = zl * Tp;  // the slice's first workspace row
            const uint32_t own_bytes = 4u * (uint32_t)min(kRows, Tp - t0);
            mbar_arrive_expect_tx(B_RES, 4 * kTileBytes + 2 * own_bytes);
            const CUtensorMap* res_maps[4] = {&p.tm_q, &p.tm_do, &p.tm_k, &p.tm_v};
            for (int m = 0; m < 4; ++m) {
                tma_load_3d(sbase + m * kTileBytes, res_maps[m], B_RES, 0, t0, z);
                tma_load_3d(sbase + m * kTileBytes + kChunkBytes, res_maps[m], B_RES, 0, t0 + kChunk, z);
            }
            bulk_load(sbase + kOffOwn, p.lse2 + wrow + t0, own_bytes, B_RES);
            bulk_load(sbase + kOffOwn + 512, p.delta + wrow + t0, own_bytes, B_RES);
            // a 128-row tile from rows y.. of one tensor into the slot of item seq
            auto put_tile = [&](uint32_t seq, const CUtensorMap* map, int32_t y) {
                if (!rg.acquire(seq, aborted, p.err)) return;
                mbar_arrive_expect_tx(rg.full(seq), kTileBytes);
                tma_load_3d(rg.addr(seq), map, rg.full(seq), 0, y, z);
                tma_load_3d(rg.addr(seq) + kChunkBytes, map, rg.full(seq), 0, y + kChunk, z);
            };
            uint32_t seq = 0;
            for (int c = 0; c < pl.n_qring; ++c, ++seq) {
                // a K chunk and the V chunk of the same rows
                if (!rg.acquire(seq, aborted, p.err)) continue;
                const int32_t kb = (pl.qc_lo + c) * kChunk;
                mbar_arrive_expect_tx(rg.full(seq), 2 * kChunkBytes);
                tma_load_3d(rg.addr(seq), &p.tm_k, rg.full(seq), 0, kb, z);
                tma_load_3d(rg.addr(seq) + kChunkBytes, &p.tm_v, rg.full(seq), 0, kb, z);
            }
            for (int k = 0; k < pl.n_qoff; ++k) {
                put_tile(seq++, &p.tm_k, t0 - offs[k]);
                put_tile(seq++, &p.tm_v, t0 - offs[k]);
            }
            if (rg.acquire(seq, aborted, p.err)) rg.publish_empty(seq);  // dq staging
            ++seq;
            for (int c = 2; c < pl.n_kc; ++c, ++seq) {
                // a Q chunk, the dO chunk of the same rows, and their lse log2(e) and D
                if (!rg.acquire(seq, aborted, p.err)) continue;
                const int32_t qb = (t0 / kChunk + c) * kChunk;
                const uint32_t side_bytes = 4u * (uint32_t)min(kChunk, Tp - qb);
                mbar_arrive_expect_tx(rg.full(seq), 2 * kChunkBytes + 2 * side_bytes);
                tma_load_3d(rg.addr(seq), &p.tm_q, rg.full(seq), 0, qb, z);
                tma_load_3d(rg.addr(seq) + kChunkBytes, &p.tm_do, rg.full(seq), 0, qb, z);
                bulk_load(sbase + side_off(seq), p.lse2 + wrow + qb, side_bytes, rg.full(seq));
                bulk_load(sbase + side_off(seq) + 256, p.delta + wrow + qb, side_bytes, rg.full(seq));
            }
            for (int k = 0; k < pl.n_koff; ++k) {
                put_tile(seq++, &p.tm_q, t0 + offs[k]);
                put_tile(seq++, &p.tm_do, t0 + offs[k]);
            }
            for (int h = 0; h < 2; ++h, ++seq)  // dk and dv staging
                if (rg.acquire(seq, aborted, p.err)) rg.publish_empty(seq);
            // teardown: the last fills have landed and every slot's last use has been released
            for (uint32_t q = n_items > kSlots ? n_items - kSlots : 0; q < n_items; ++q)
                rg.wait_full(q, aborted, p.err);
            for (uint32_t q = n_items > kSlots ? n_items - kSlots : 0; q < n_items; ++q)
                rg.acquire(q + kSlots, aborted, p.err);
        }
    } else if (warp == 8) {
        // ------------------------------------------------ MMA issue (lane 0)
        if (lane == 0) {
            const uint32_t idesc_s = idesc_bf16(128, 64, 0, 0);
            const uint32_t idesc_o = idesc_bf16(128, 64, 0, 1);
            mbar_wait(B_RES, 0, aborted, p.err);
            uint32_t m = 0;  // band chunks issued (both phases)
            // dq phase: S = Q K^T, dP = dO V^T, then dQ += dS K
            for (int c = 0; c < pl.n_qc; ++c, ++m) {
                const bool ring = c < pl.n_qring;
                const uint32_t seq = (uint32_t)c;
                uint32_t kaddr, vaddr;
                if (ring) {
                    rg.wait_full(seq, aborted, p.err);
                    kaddr = rg.addr(seq);
                    vaddr = kaddr + kChunkBytes;
                } else {
                    const uint32_t rc = (uint32_t)(pl.qc_lo + c - t0 / kChunk);  // 0 or 1
                    kaddr = sbase + kOffK + rc * kChunkBytes;
                    vaddr = sbase + kOffV + rc * kChunkBytes;
                }
                if (m > 0) mbar_wait(B_M, (m - 1) & 1, aborted, p.err);  // S/dP columns free
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tmem + kColS, sdesc_sw128(sbase + kOffQ + 32 * kk, 16, 1024),
                           sdesc_sw128(kaddr + 32 * kk, 16, 1024), idesc_s, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tmem + kColP, sdesc_sw128(sbase + kOffG + 32 * kk, 16, 1024),
                           sdesc_sw128(vaddr + 32 * kk, 16, 1024), idesc_s, kk > 0);
                mma_commit(B_S);
                mbar_wait(B_P, m & 1, aborted, p.err);
                tc_fence_after();
                // dS of keys 16kk..16kk+15 sits in columns 32(kk/2) + 8(kk%2) of the S block
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ts(tmem + kColDQ, tmem + kColS + 32 * (kk >> 1) + 8 * (kk & 1),
                           sdesc_sw128(kaddr + 2048 * kk, 0, 1024), idesc_o, (c > 0 || kk > 0) ? 1u : 0u);
                mma_commit(B_M);
                if (ring) rg.release_mma(seq);
            }
            // dk/dv phase: S^T = K Q^T, dP^T = V dO^T, then dV += P^T dO, dK += dS^T Q
            for (int c = 0; c < pl.n_kc; ++c, ++m) {
                const bool ring = c >= 2;
                const uint32_t seq = seq_kring + (uint32_t)(c - 2);
                uint32_t qaddr, gaddr;
                if (ring) {
                    // the items before it have landed: the row threads consumed them before
                    // their B_DQ arrival, awaited at c = 0
                    rg.wait_full(seq, aborted, p.err);
                    qaddr = rg.addr(seq);
                    gaddr = qaddr + kChunkBytes;
                } else {
                    qaddr = sbase + kOffQ + (uint32_t)c * kChunkBytes;
                    gaddr = sbase + kOffG + (uint32_t)c * kChunkBytes;
                }
                mbar_wait(B_M, (m - 1) & 1, aborted, p.err);  // S/dP columns free
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
                mbar_wait(B_P, m & 1, aborted, p.err);
                if (c == 0) mbar_wait(B_DQ, 0, aborted, p.err);  // dQ left TMEM: dK may overwrite it
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t acol = 32 * (kk >> 1) + 8 * (kk & 1);
                    const uint32_t acc = (c > 0 || kk > 0) ? 1u : 0u;
                    mma_ts(tmem + kColDV, tmem + kColS + acol, sdesc_sw128(gaddr + 2048 * kk, 0, 1024),
                           idesc_o, acc);
                    mma_ts(tmem + kColDK, tmem + kColP + acol, sdesc_sw128(qaddr + 2048 * kk, 0, 1024),
                           idesc_o, acc);
                }
                mma_commit(B_M);
                if (ring) rg.release_mma(seq);
            }
            mbar_wait(B_M, (m - 1) & 1, aborted, p.err);
        }
    } else {
        // ------------------------------------------------ row threads: row r, half h
        const int q4 = warp & 3, h = warp >> 2;
        const int r = 32 * q4 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
        const float sl2 = p.scale_log2;
        const int32_t i = t0 + r;  // this thread's query (dq phase) and key (dk/dv phase)
        const bool row_ok = i < T;
        const float* own_l2 = reinterpret_cast<const float*>(smem + kOffOwn);
        const float* own_D = own_l2 + kRows;
        mbar_wait(B_RES, 0, aborted, p.err);
        const float lse2_i = row_ok ? own_l2[r] : 0.f;
        const float D_i = row_ok ? own_D[r] : 0.f;
        uint32_t m = 0;

        // ---- dq phase, band: dS of this thread's 32 key columns of each chunk
        for (int c = 0; c < pl.n_qc; ++c, ++m) {
            const int32_t kb = (pl.qc_lo + c) * kChunk + 32 * h;  // first key of my columns
            mbar_wait(B_S, m & 1, aborted, p.err);
            tc_fence_after();
            __syncwarp();  // converged for the warp-collective TMEM accesses below
            const int32_t rlo = t0 + 32 * q4;
            const bool need = (rlo + 31 - kb >= 0) && (rlo - (kb + 31) < W);
            const int32_t d0 = i - kb;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const uint32_t col = 32 * h + 16 * hf;
                uint32_t pk[8];
                if (need) {
                    uint32_t sv[16], dv[16];
                    tmem_ld16(tmem + lane_base + kColS + col, sv);
                    tmem_ld16(tmem + lane_base + kColP + col, dv);
                    tmem_ld_wait(sv, dv);
#pragma unroll
                    for (int e = 0; e < 16; e += 2) {
                        const int32_t dj = d0 - 16 * hf - e;
                        const bool ok0 = row_ok && (uint32_t)dj < (uint32_t)W;
                        const bool ok1 = row_ok && (uint32_t)(dj - 1) < (uint32_t)W;
                        const float p0 = ok0 ? ex2(__uint_as_float(sv[e]) * sl2 - lse2_i) : 0.f;
                        const float p1 = ok1 ? ex2(__uint_as_float(sv[e + 1]) * sl2 - lse2_i) : 0.f;
                        pk[e >> 1] = pack_bf16x2(p0 * (__uint_as_float(dv[e]) - D_i),
                                                 p1 * (__uint_as_float(dv[e + 1]) - D_i));
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) pk[e] = 0u;
                }
                tmem_st8(tmem + lane_base + kColS + 32 * h + 8 * hf, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B_P);
        }

        // ---- dq phase, offsets: q.k_{i-o} and dO.v_{i-o} over all 64 dims, dq of my 32 dims
        uint32_t seq = seq_qoff;
        {
            float dq[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) dq[c] = 0.f;
#pragma unroll 1
            for (int k = 0; k < pl.n_qoff; ++k) {
                const bool valid = row_ok && i - offs[k] >= 0;
                rg.wait_full(seq, aborted, p.err);
                const uint8_t* kt = slot_ptr(seq);
                const float sdot = row_dot(smem + kOffQ, kt, r);
                uint32_t kh[16];
                load_half_sw(kt, r, h, kh);
                rg.release_warp(seq, lane);
                ++seq;
                rg.wait_full(seq, aborted, p.err);
                const float dpd = row_dot(smem + kOffG, slot_ptr(seq), r);
                rg.release_warp(seq, lane);
                ++seq;
                const float pr = valid ? ex2(sdot * sl2 - lse2_i) : 0.f;
                const float ds = pr * (dpd - D_i);
                const uint32_t dsb = pack_bf16x2(pr, ds) >> 16;  // dS as bf16 in the low half
#pragma unroll
                for (int c = 0; c < 16; ++c) axpy2_bf16(dsb, kh[c], dq[2 * c], dq[2 * c + 1]);
            }

            // ---- dq epilogue: dq = scale (dQ + dq_off), staged in a ring slot, TMA store
            rg.wait_full(seq, aborted, p.err);
            mbar_wait(B_M, (uint32_t)(pl.n_qc - 1) & 1, aborted, p.err);
            tc_fence_after();
            __syncwarp();  // converged for the warp-collective TMEM accesses below
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + kColDQ + 32 * h, v);
            tmem_ld_wait(v);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B_DQ);  // the dK MMAs may take these columns
            uint8_t* st = slot_ptr(seq);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int e = 8 * c;
                uint4 w;
                w.x = pack_bf16x2((__uint_as_float(v[e + 0]) + dq[e + 0]) * p.scale,
                                  (__uint_as_float(v[e + 1]) + dq[e + 1]) * p.scale);
                w.y = pack_bf16x2((__uint_as_float(v[e + 2]) + dq[e + 2]) * p.scale,
                                  (__uint_as_float(v[e + 3]) + dq[e + 3]) * p.scale);
                w.z = pack_bf16x2((__uint_as_float(v[e + 4]) + dq[e + 4]) * p.scale,
                                  (__uint_as_float(v[e + 5]) + dq[e + 5]) * p.scale);
                w.w = pack_bf16x2((__uint_as_float(v[e + 6]) + dq[e + 6]) * p.scale,
                                  (__uint_as_float(v[e + 7]) + dq[e + 7]) * p.scale);
                *reinterpret_cast<uint4*>(st + sw128_off(r, 4 * h + c)) = w;
            }
            fence_proxy_async_smem();
            asm volatile("bar.sync 1, 256;" ::: "memory");
            if (tid == 0) {
                if (!aborted) {
                    tma_store_3d(&p.tm_dq, rg.addr(seq), 0, t0, z);
                    if (t0 + kChunk < T) tma_store_3d(&p.tm_dq, rg.addr(seq) + kChunkBytes, 0, t0 + kChunk, z);
                    tma_store_commit();
                    tma_store_wait_read0();
                }
                rg.release_stage(seq);
            }
            ++seq;
        }

        // ---- dk/dv phase, band: P^T and dS^T of this thread's 32 query columns of each chunk
        for (int c = 0; c < pl.n_kc; ++c, ++m) {
            const bool ring = c >= 2;
            const uint32_t cseq = seq_kring + (uint32_t)(c - 2);
            const int32_t qc0 = (t0 / kChunk + c) * kChunk;
            const int32_t qb = qc0 + 32 * h;  // first query of my columns
            mbar_wait(B_S, m & 1, aborted, p.err);
            if (ring) rg.wait_full(cseq, aborted, p.err);  // lse log2(e) / D side data
            tc_fence_after();
            __syncwarp();  // converged for the warp-collective TMEM accesses below
            const int32_t klo = t0 + 32 * q4;
            const bool need = (qb + 31 - klo >= 0) && (qb - (klo + 31) < W) && qb < T;
            const float* L = ring ? reinterpret_cast<const float*>(smem + side_off(cseq)) + 32 * h
                                  : own_l2 + (qc0 - t0) + 32 * h;
            const float* Dd = ring ? L + kChunk : L + kRows;
            const int32_t dist0 = qb - i;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const uint32_t col = 32 * h + 16 * hf;
                uint32_t pp[8], pd[8];
                if (need) {
                    uint32_t sv[16], dv[16];
                    tmem_ld16(tmem + lane_base + kColS + col, sv);
                    tmem_ld16(tmem + lane_base + kColP + col, dv);
                    tmem_ld_wait(sv, dv);
#pragma unroll
                    for (int e = 0; e < 16; e += 2) {
                        const int ee = 16 * hf + e;
                        const bool ok0 = row_ok && (uint32_t)(dist0 + ee) < (uint32_t)W && qb + ee < T;
                        const bool ok1 = row_ok && (uint32_t)(dist0 + ee + 1) < (uint32_t)W && qb + ee + 1 < T;
                        const float p0 = ok0 ? ex2(__uint_as_float(sv[e]) * sl2 - L[ee]) : 0.f;
                        const float p1 = ok1 ? ex2(__uint_as_float(sv[e + 1]) * sl2 - L[ee + 1]) : 0.f;
                        pp[e >> 1] = pack_bf16x2(p0, p1);
                        // selects: a query column at or past T reads lse/D bytes this call did
                        // not write (slot or pad memory), which must not reach dK through 0 * x
                        pd[e >> 1] = pack_bf16x2(ok0 ? p0 * (__uint_as_float(dv[e]) - Dd[ee]) : 0.f,
                                                 ok1 ? p1 * (__uint_as_float(dv[e + 1]) - Dd[ee + 1]) : 0.f);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) pp[e] = pd[e] = 0u;
                }
                tmem_st8(tmem + lane_base + kColS + 32 * h + 8 * hf, pp);
                tmem_st8(tmem + lane_base + kColP + 32 * h + 8 * hf, pd);
            }
            tmem_st_wait();
            tc_fence_before();
            // the side data was read with generic loads; the MMA warp releases the slot to the
            // next bulk copy after this arrival
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(B_P);
        }
        seq = seq_koff;

        // ---- dk/dv phase, offsets: the pair (key i, query i+o) formed again, dk and dv of my
        // 32 dims in registers
        float dka[32], dva[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) dka[c] = dva[c] = 0.f;
        const int64_t wrow = zl * Tp;
#pragma unroll 1
        for (int k = 0; k < pl.n_koff; ++k) {
            const int32_t jq = i + offs[k];
            const bool valid = row_ok && jq < T;
            const float l2q = valid ? p.lse2[wrow + jq] : 0.f;
            const float Dq = valid ? p.delta[wrow + jq] : 0.f;
            rg.wait_full(seq, aborted, p.err);
            const uint8_t* qt = slot_ptr(seq);
            const float sdot = row_dot(qt, smem + kOffK, r);
            uint32_t qh[16];
            load_half_sw(qt, r, h, qh);
            rg.release_warp(seq, lane);
            ++seq;
            const float pr = valid ? ex2(sdot * sl2 - l2q) : 0.f;
            rg.wait_full(seq, aborted, p.err);
            const uint8_t* gt = slot_ptr(seq);
            const float dpd = row_dot(gt, smem + kOffV, r);
            const float ds = pr * (dpd - Dq);
            const uint32_t pair = valid ? pack_bf16x2(pr, ds) : 0u;  // lo = P, hi = dS
            const uint32_t pb = pair & 0xFFFFu, dsb = pair >> 16;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint4 x = *reinterpret_cast<const uint4*>(gt + sw128_off(r, 4 * h + c));
                axpy2_bf16(pb, x.x, dva[8 * c + 0], dva[8 * c + 1]);
                axpy2_bf16(pb, x.y, dva[8 * c + 2], dva[8 * c + 3]);
                axpy2_bf16(pb, x.z, dva[8 * c + 4], dva[8 * c + 5]);
                axpy2_bf16(pb, x.w, dva[8 * c + 6], dva[8 * c + 7]);
            }
            rg.release_warp(seq, lane);
            ++seq;
#pragma unroll
            for (int c = 0; c < 16; ++c) axpy2_bf16(dsb, qh[c], dka[2 * c], dka[2 * c + 1]);
        }

        // ---- dk/dv epilogue: dk = scale (dK + dk_off), dv = dV + dv_off, staged, TMA stores
        const uint32_t kst = seq, vst = seq + 1;
        mbar_wait(B_M, (m - 1) & 1, aborted, p.err);
        tc_fence_after();
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
                w.x = pack_bf16x2((__uint_as_float(v[e + 0]) + dka[e + 0]) * p.scale,
                                  (__uint_as_float(v[e + 1]) + dka[e + 1]) * p.scale);
                w.y = pack_bf16x2((__uint_as_float(v[e + 2]) + dka[e + 2]) * p.scale,
                                  (__uint_as_float(v[e + 3]) + dka[e + 3]) * p.scale);
                w.z = pack_bf16x2((__uint_as_float(v[e + 4]) + dka[e + 4]) * p.scale,
                                  (__uint_as_float(v[e + 5]) + dka[e + 5]) * p.scale);
                w.w = pack_bf16x2((__uint_as_float(v[e + 6]) + dka[e + 6]) * p.scale,
                                  (__uint_as_float(v[e + 7]) + dka[e + 7]) * p.scale);
                *reinterpret_cast<uint4*>(st + sw128_off(r, 4 * h + c)) = w;
            }
            tmem_ld32(tmem + lane_base + kColDV + 32 * h, v);
            tmem_ld_wait(v);
            st = slot_ptr(vst);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int e = 8 * c;
                uint4 w;
                w.x = pack_bf16x2(__uint_as_float(v[e + 0]) + dva[e + 0], __uint_as_float(v[e + 1]) + dva[e + 1]);
                w.y = pack_bf16x2(__uint_as_float(v[e + 2]) + dva[e + 2], __uint_as_float(v[e + 3]) + dva[e + 3]);
                w.z = pack_bf16x2(__uint_as_float(v[e + 4]) + dva[e + 4], __uint_as_float(v[e + 5]) + dva[e + 5]);
                w.w = pack_bf16x2(__uint_as_float(v[e + 6]) + dva[e + 6], __uint_as_float(v[e + 7]) + dva[e + 7]);
                *reinterpret_cast<uint4*>(st + sw128_off(r, 4 * h + c)) = w;
            }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (tid == 0) {
            if (!aborted) {
                tma_store_3d(&p.tm_dk, rg.addr(kst), 0, t0, z);
                tma_store_3d(&p.tm_dv, rg.addr(vst), 0, t0, z);
                if (t0 + kChunk < T) {
                    tma_store_3d(&p.tm_dk, rg.addr(kst) + kChunkBytes, 0, t0 + kChunk, z);
                    tma_store_3d(&p.tm_dv, rg.addr(vst) + kChunkBytes, 0, t0 + kChunk, z);
                }
                tma_store_commit();
                tma_store_wait_read0();
            }
            rg.release_stage(kst);
            rg.release_stage(vst);
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

}  // namespace

fibattn_status launch_bwd_fused_tc_bf16(const void* q, const void* k, const void* v,
                                        const void* o, const float* lse, const void* dO, void* dq,
                                        void* dk, void* dv, float* delta, float* lse2,
                                        const AttnShape& sh, const OffsetTables& t, cudaStream_t st) {
    if (sh.group != 1 || sh.d != 64) return FIBATTN_ERR_UNSUPPORTED;
    const int64_t slices = sh.slices_per_layer * sh.n_layers;
    if (slices > 0x7fffffff) return FIBATTN_ERR_INVALID_ARG;
    const int32_t tiles = (sh.T + kRows - 1) / kRows;
    const int64_t gx = (int64_t)tiles * sh.slices_per_layer;
    if (gx > 0x7fffffff) return FIBATTN_ERR_INVALID_ARG;
    FusedParams P;
    // the error-word lookup is a runtime call: it binds the device's primary context to this
    // thread, which the tensor-map encoding needs
    P.err = device_error_word();
    if (!P.err) return cuda_fail(-1, "cudaGetSymbolAddress (error word)");
    const void* bases[7] = {q, k, v, dO, dq, dk, dv};
    CUtensorMap* maps[7] = {&P.tm_q, &P.tm_k, &P.tm_v, &P.tm_do, &P.tm_dq, &P.tm_dk, &P.tm_dv};
    for (int m = 0; m < 7; ++m) {
        const int r = make_bf16_rows_map(maps[m], bases[m], slices, sh.T);
        if (r != 0) return cuda_fail(r, "cuTensorMapEncodeTiled (fused bwd)");
    }
    P.delta = delta;
    P.lse2 = lse2;
    P.slices_per_layer = sh.slices_per_layer;
    P.T = sh.T;
    P.W = sh.W;
    P.T_pad = (sh.T + 3) & ~3;
    P.tiles_per_slice = tiles;
    P.scale = sh.scale;
    P.scale_log2 = sh.scale * kLog2e;
    P.tabs = t;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail((int32_t)e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return FIBATTN_ERR_UNSUPPORTED;
    static bool smem_set[64] = {};
    static int n_sm[64] = {};
    if (!smem_set[dev]) {
        e = cudaFuncSetAttribute((const void*)bwd_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemAlloc);
        if (e != cudaSuccess) return cuda_fail((int32_t)e, "cudaFuncSetAttribute (fused bwd)");
        smem_set[dev] = true;
    }
    if (n_sm[dev] == 0) {
        e = cudaDeviceGetAttribute(&n_sm[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail((int32_t)e, "cudaDeviceGetAttribute");
    }
    {
        // one warp per 32 rows; six blocks (37 KB of shared memory each) fit on an SM
        const int64_t rows = slices * sh.T;
        const int64_t want = (rows + 32 * kPrepWarps - 1) / (32 * kPrepWarps);
        const int64_t cap = 6LL * n_sm[dev];
        KernelScope ks("bwd_prep", st);
        bwd_prep_kernel<<<(unsigned)(want < cap ? want : cap), 32 * kPrepWarps, 0, st>>>(
            static_cast<const uint4*>(o), static_cast<const uint4*>(dO), lse, delta, lse2, slices,
            sh.T, P.T_pad);
    }
    fibattn_status s0 = launch_status("bwd_prep");
    if (s0 != FIBATTN_OK) return s0;
    {
        KernelScope ks("bwd_fused_tc", st);
        bwd_fused_kernel<<<dim3((unsigned)gx, (unsigned)sh.n_layers), kThreads, kSmemAlloc, st>>>(P);
    }
    return launch_status("bwd_fused_tc");
}

}  // namespace fibattn
