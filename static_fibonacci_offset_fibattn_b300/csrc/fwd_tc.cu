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
// Persistent kernel: 2 CTAs per SM, each walking tiles of 128 queries [i0, i0+128) of a
// (layer, batch, head) slice (ring.cuh). Per CTA:
//   warps 0-3 : one thread per query row (TMEM lane = row); softmax, offsets, epilogue.
//   warp 4    : TMEM allocation and tcgen05.mma issue (lane 0).
//   warp 5    : the producer (lane 0): TMA loads into the ring, running ahead across tiles.
// Ring items of one tile, in order: per band group a copy of Q, its K chunks, then its V
// chunks (two 64-key chunks per slot); per active offset o the shifted tiles K[i0-o ..] and
// V[i0-o ..] (negative rows zero-filled); a staging slot for the output tile. Every item is
// released without waiting on a later one, so the in-order ring cannot stall.
// Band: keys [max(0, i0-W+1), i0+127] in 64-key chunks, up to 3 chunks per group:
//   S = Q K^T (tcgen05, M=128, K=64) -> TMEM columns [0, 192): one N=192 MMA per k-step when
//   the three chunks sit in consecutive slots, else N=128 for the two chunks of a slot and
//   N=64 for a lone one (each tcgen05.mma costs the issuing thread about 100 cycles, and the
//   tile's S is on the row threads' path)
//   masked online softmax per row (fp32, log2 domain), P (bf16) written back over S
//   O_band += P V (tcgen05, A = P from TMEM, B = V MN-major in smem) -> TMEM [192, 256)
// Offsets: thread r takes row r of each shifted tile: s = q_r . k_{i-o}, then accumulates
//   exp(s - m) v_{i-o} in registers. The band and offset parts keep separate running
//   maxima and are merged once in the epilogue.
// Epilogue: O = (O_band 2^(m_b-m) + O_off 2^(m_o-m)) / l, staged in a ring slot,
//   TMA-stored; lse = (m + log2 l) ln 2.
//
// Fractional offsets (the learned-alpha variant; Metodologia / Arquitetura, "Implementacao":
// keys and values linearly interpolated between rows so that the gradient reaches alpha)
// reuse the same kernel (kFrac): a real distance d is held as c = ceil(d) and the weight
// w = c - d of the row after i - c, and query i >= c attends
//   k~ = (1 - w) k_{i-c} + w k_{i-c+1},  v~ likewise.
// Each shifted item then also carries the 8 rows after its 128-row tile (a 17 KB slot), so
// that row r finds both of its rows, r and r + 1, in the slot; the score is the lerp of the
// two row dot products and the value update two axpys with p (1 - w) and p w. A distance
// with w = 0 takes the static code path, so integer alphas give the static results.
//
// RoPE inside the kernel (kRope; Metodologia / Arquitetura, "Implementacao": RoPE applied
// before the gather, vanilla, no scaling): q and k arrive unrotated with the cos/sin table of
// every position. Before each band group's S MMAs the row threads rotate the group's Q copy
// and K chunks in their ring slots (row i by i theta_p, the unfused rotation's arithmetic and
// bf16 rounding), so the band is the attention of the rotated tensors. The offsets need no
// rotated copy: with R_a the rotation by the angles a theta_p,
//   (R_i q_i) . (R_(i-o) k_(i-o)) = (R_o q_i) . k_(i-o),
// one angle per offset for the whole tile, taken from table row o. Per pair p, with
// a = q_2p k_2p + q_2p+1 k_2p+1 and b = q_2p k_2p+1 - q_2p+1 k_2p, the score gains
// cos(o theta_p) a + sin(o theta_p) b. The row threads keep their unrotated q row in
// registers for this (read before the rotation), and v is never rotated.
//
// Head size 128 (kWide): rows are two 64-column halves (two 128-byte swizzle atoms). Each
// tile is taken by two CTAs, CTA half h writing output columns [64h, 64h+64): both compute
// the full scores (S over both halves of Q and K: 8 MMA k-steps; the offsets' row dots over
// 128 dims), and each accumulates P V and the offsets' p v over its own half of V, so TMEM
// (S 192 + O 64 columns), the ring and the row threads' O registers keep their 64-wide form.
// Ring items of a group: two Q items (the halves), one K chunk per slot (both halves), the
// own half of the V chunks two per slot; per offset the two K halves and the own V half.
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

constexpr int kRows = 128;          // queries per tile
constexpr int kChunk = kTmaBoxRows; // keys per band chunk (one TMA box)
constexpr int kMaxGroupChunks = 3;  // band chunks per S group (N <= 192)
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTmemO = 192;    // O accumulator columns [192, 256)
constexpr uint32_t kChunkBytes = kChunk * 128;  // 8 KB
constexpr uint32_t kSlots = 6;

// shared memory: the ring slots, then the barriers, then the TMEM address word
template <bool kFrac>
struct Layout {
    static constexpr uint32_t kSlot = ring::kSlotBytes + (kFrac ? 1024u : 0u);
    static constexpr uint32_t kOffBar = kSlots * kSlot;
};
// barriers: FULL[kSlots], EMPTY[kSlots], then S ready, P written (4 warps), PV done,
// TMEM free (4 warps), band items landed; then the TMEM address word. The Q slot is released
// by the row warps once they hold their q rows (the S MMAs reading it are complete by then).
// The row threads skip the MMA warp's ring items; before they wait on the offset slots
// (whose previous use may be a band slot) they wait for "band items landed", which the MMA
// warp signals once it has waited for every band item of the tile -- a parity wait is only
// exact when the slot's previous use is known to have landed.
constexpr uint32_t kBarS = 2 * kSlots, kBarP = kBarS + 1, kBarO = kBarS + 2, kBarT = kBarS + 3,
                   kBarL = kBarS + 4, kBarR = kBarS + 5;
constexpr uint32_t kNumBars = kBarR + 1;  // kBarR: a group's Q and K rotated (RoPE mode)
template <bool kFrac>
__host__ __device__ constexpr uint32_t tmem_slot_off() { return Layout<kFrac>::kOffBar + kNumBars * 8; }
template <bool kFrac>
__host__ __device__ constexpr uint32_t smem_alloc() { return tmem_slot_off<kFrac>() + 16 + 1024; }  // + alignment slack

struct FwdParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_o;  // 3D {64, T, slices}, box {64, 64, 1}, 128B swizzle
                                         // (tm_k, tm_v over the kv slices)
    float* lse;
    int32_t* err;
    uint32_t slices_per_layer;
    uint32_t group;             // query heads per kv head (1: one kv head per query head)
    uint32_t slices_per_layer_kv;  // slices_per_layer / group
    uint32_t total_tiles;       // <= INT32_MAX
    int32_t T, W;
    int32_t tiles_per_slice;
    float scale_log2;  // scale * log2(e)
    OffsetTables tabs;          // fractional mode: ceil(d) of each real distance d
    const float4* rope;         // RoPE mode: cos/sin table [rows][16] (pairs (cos, sin))
};

template <bool kFrac>
struct FwdArgs : FwdParams {};

template <>
struct FwdArgs<true> : FwdParams {
    CUtensorMap tm_k8, tm_v8;  // 8-row boxes: the rows just past a shifted tile
    float w[kMaxLayersPerLaunch][kMaxOffsets];  // weight ceil(d) - d of the later row
};

// The band and offset extents of one tile; every role derives the same item sequence.
template <bool kWide>
struct Plan {
    static constexpr int kQItems = kWide ? 2 : 1;   // Q copy items per group
    static constexpr int kKItems = kWide ? 2 : 1;   // K items per offset
    int32_t i0, klast, c_lo, n_chunks, n_groups, n_act;
    __device__ __forceinline__ int nch(int g) const {
        return min(kMaxGroupChunks, n_chunks - g * kMaxGroupChunks);
    }
    __device__ __forceinline__ int band_slots(int g) const { return (nch(g) + 1) / 2; }
    __device__ __forceinline__ int k_slots(int g) const { return kWide ? nch(g) : band_slots(g); }
    // ring items of group g: the Q copy, its K slots, its V slots (at most 5 before the V
    // slots, so a group never waits on a later item of the ring)
    __device__ __forceinline__ uint32_t group_items(int g) const {
        return kQItems + k_slots(g) + band_slots(g);
    }
    __device__ __forceinline__ uint32_t band_items() const {
        uint32_t n = 0;
        for (int g = 0; g < n_groups; ++g) n += group_items(g);
        return n;
    }
};

template <bool kWide>
__device__ __forceinline__ Plan<kWide> make_plan(const FwdParams& p, int layer, int32_t i0) {
    Plan<kWide> pl;
    pl.i0 = i0;
    const int32_t kstart = i0 - p.W + 1 > 0 ? i0 - p.W + 1 : 0;
    pl.klast = (i0 + kRows - 1 < p.T - 1) ? i0 + kRows - 1 : p.T - 1;
    pl.c_lo = kstart / kChunk;
    pl.n_chunks = pl.klast / kChunk - pl.c_lo + 1;
    pl.n_groups = (pl.n_chunks + kMaxGroupChunks - 1) / kMaxGroupChunks;
    const int32_t* offs = p.tabs.off[layer];
    int32_t n = 0;
    for (int e = 0; e < p.tabs.count[layer]; ++e)
        if (offs[e] <= pl.klast) n = e + 1;
    pl.n_act = n;
    return pl;
}

// Tile walk: at head size 128 each tile is taken twice, by output half (the fastest index).
template <bool kWide>
__device__ __forceinline__ ring::Tile tile_at(const FwdParams& p, uint32_t idx, int& half) {
    half = kWide ? (int)(idx & 1u) : 0;
    return ring::tile_of(kWide ? idx >> 1 : idx, p.tiles_per_slice, p.slices_per_layer);
}

// Rotation of one bf16 pair (x0, x1) by the angle with cosine c and sine s, rounded to bf16:
// (x0 c - x1 s, x0 s + x1 c), the arithmetic of the standalone rotation kernel.
__device__ __forceinline__ uint32_t rot_bf16x2(uint32_t w, float c, float s) {
    const float x0 = bf16lo(w), x1 = bf16hi(w);
    return pack_bf16x2(x0 * c - x1 * s, x0 * s + x1 * c);
}

// Rotates row `row` (0..127 of a 1024-byte aligned 128-byte-swizzled tile) by its position's
// angles, table row `pos` (16 float4: (cos, sin) of pairs 2m and 2m + 1).
__device__ __forceinline__ void rotate_row_sw(uint8_t* tile, int row, const float4* trow) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint4* ptr = reinterpret_cast<uint4*>(tile + sw128_off(row, c));
        uint4 w = *ptr;
        const float4 t0 = __ldg(trow + 2 * c), t1 = __ldg(trow + 2 * c + 1);
        w.x = rot_bf16x2(w.x, t0.x, t0.y);
        w.y = rot_bf16x2(w.y, t0.z, t0.w);
        w.z = rot_bf16x2(w.z, t1.x, t1.y);
        w.w = rot_bf16x2(w.w, t1.z, t1.w);
        *ptr = w;
    }
}

// acc += c (q0 k0 + q1 k1) + s (q0 k1 - q1 k0) for one bf16 pair of q and of k: the pair's
// share of (R q) . k with R the rotation by (c, s). Products of bf16 values are exact in fp32.
__device__ __forceinline__ void rope_dot_pair(uint32_t q, uint32_t k, float c, float s, float& acc) {
    asm("{\n\t.reg .b16 q0, q1, k0, k1;\n\t.reg .f32 a, b;\n\t"
        "mov.b32 {q0, q1}, %1;\n\tmov.b32 {k0, k1}, %2;\n\t"
        "fma.rn.f32.bf16 a, q1, k1, 0f00000000;\n\tfma.rn.f32.bf16 a, q0, k0, a;\n\t"
        "fma.rn.f32.bf16 b, q1, k0, 0f00000000;\n\tneg.f32 b, b;\n\t"
        "fma.rn.f32.bf16 b, q0, k1, b;\n\t"
        "fma.rn.f32 %0, %3, a, %0;\n\tfma.rn.f32 %0, %4, b, %0;\n\t}"
        : "+f"(acc)
        : "r"(q), "r"(k), "f"(c), "f"(s));
}

template <bool kFrac, bool kWide, bool kRope = false>
__global__ void __launch_bounds__(kThreads, 2)
fwd_tc_kernel(const __grid_constant__ FwdArgs<kFrac> p) {
    static_assert(!(kFrac && kWide), "the fractional mode is for head size 64");
    static_assert(!kRope || (!kFrac && !kWide), "the RoPE mode is the static head-size-64 path");
    using PL = Plan<kWide>;
    using L = Layout<kFrac>;
    constexpr uint32_t kOffTmemSlot = tmem_slot_off<kFrac>();
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - smem_u32(smem_raw));

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int32_t T = p.T, W = p.W;

    const ring::Ring rg{sbase, sbase + L::kOffBar, kSlots, 4, L::kSlot};  // 4 row warps
    auto bar = [&](uint32_t idx) { return sbase + L::kOffBar + 8u * idx; };
    const uint32_t B_S = bar(kBarS), B_P = bar(kBarP), B_O = bar(kBarO), B_T = bar(kBarT),
                   B_L = bar(kBarL), B_R = bar(kBarR);
    auto slot_ptr = [&](uint32_t seq) { return smem + (rg.addr(seq) - sbase); };

    if (tid == 0) {
        ring::init_ring_barriers(rg, 1);
        mbar_init(B_S, 1);
        mbar_init(B_P, 4);
        mbar_init(B_O, 1);
        mbar_init(B_T, 4);
        mbar_init(B_L, 1);
        mbar_init(B_R, 4);
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

    if (warp == 5) {
        // ------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&p.tm_q);
            prefetch_tmap(&p.tm_k);
            prefetch_tmap(&p.tm_v);
            prefetch_tmap(&p.tm_o);
            if constexpr (kFrac) {
                prefetch_tmap(&p.tm_k8);
                prefetch_tmap(&p.tm_v8);
            }
            uint32_t seq = 0;
            for (uint32_t idx = blockIdx.x; idx < p.total_tiles; idx += gridDim.x) {
                int half;
                const ring::Tile tl = tile_at<kWide>(p, idx, half);
                const PL pl = make_plan<kWide>(p, tl.layer, tl.row0);
                const int32_t z = (int32_t)tl.zl;
                const int32_t xv = 64 * half;  // the own half of V
                // the kv slice: query head h of batch b reads kv head h / group
                const int32_t zk = (int32_t)((int64_t)tl.layer * p.slices_per_layer_kv +
                                             (uint32_t)tl.s / p.group);
                // band: per group a copy of Q, its K chunks, then its V chunks (two per slot)
                for (int g = 0; g < pl.n_groups; ++g) {
                    for (int qh = 0; qh < PL::kQItems; ++qh, ++seq) {  // Q (head size 128: by halves)
                        if (!rg.acquire(seq, aborted, p.err)) continue;
                        mbar_arrive_expect_tx(rg.full(seq), ring::kSlotBytes);
                        tma_load_3d(rg.addr(seq), &p.tm_q, rg.full(seq), 64 * qh, pl.i0, z);
                        tma_load_3d(rg.addr(seq) + kChunkBytes, &p.tm_q, rg.full(seq), 64 * qh,
                                    pl.i0 + kChunk, z);
                    }
                    const int nch = pl.nch(g);
                    for (int h = 0; h < 2; ++h) {
                        const CUtensorMap* map = h == 0 ? &p.tm_k : &p.tm_v;
                        if (kWide && h == 0) {
                            // one K chunk per slot: its two column halves
                            for (int c = 0; c < nch; ++c, ++seq) {
                                const int32_t y = (pl.c_lo + g * kMaxGroupChunks + c) * kChunk;
                                if (!rg.acquire(seq, aborted, p.err)) continue;
                                mbar_arrive_expect_tx(rg.full(seq), 2 * kChunkBytes);
                                tma_load_3d(rg.addr(seq), map, rg.full(seq), 0, y, zk);
                                tma_load_3d(rg.addr(seq) + kChunkBytes, map, rg.full(seq), 64, y, zk);
                            }
                            continue;
                        }
                        const int32_t x = h == 0 ? 0 : xv;
                        for (int c = 0; c < nch; c += 2, ++seq) {
                            const int n2 = min(2, nch - c);
                            const int32_t y = (pl.c_lo + g * kMaxGroupChunks + c) * kChunk;
                            if (!rg.acquire(seq, aborted, p.err)) continue;
                            mbar_arrive_expect_tx(rg.full(seq), n2 * kChunkBytes);
                            tma_load_3d(rg.addr(seq), map, rg.full(seq), x, y, zk);
                            if (n2 == 2)
                                tma_load_3d(rg.addr(seq) + kChunkBytes, map, rg.full(seq), x, y + kChunk, zk);
                        }
                    }
                }
                // offsets: K_o then V_o (fractional w != 0: plus the 8 rows after the tile)
                const int32_t* offs = p.tabs.off[tl.layer];
                for (int k = 0; k < pl.n_act; ++k) {
                    const int32_t y = pl.i0 - offs[k];
                    bool side = false;
                    if constexpr (kFrac) side = p.w[tl.layer][k] != 0.f;
                    // K_o (head size 128: its two halves), then the own half of V_o
                    for (int h = 0; h < PL::kKItems + 1; ++h, ++seq) {
                        const bool is_k = h < PL::kKItems;
                        const CUtensorMap* map = is_k ? &p.tm_k : &p.tm_v;
                        const int32_t x = is_k ? 64 * h : xv;
                        if (!rg.acquire(seq, aborted, p.err)) continue;
                        mbar_arrive_expect_tx(rg.full(seq), ring::kSlotBytes + (side ? 1024u : 0u));
                        tma_load_3d(rg.addr(seq), map, rg.full(seq), x, y, zk);
                        tma_load_3d(rg.addr(seq) + kChunkBytes, map, rg.full(seq), x, y + kChunk, zk);
                        if constexpr (kFrac) {
                            if (side)
                                tma_load_3d(rg.addr(seq) + ring::kSlotBytes, h == 0 ? &p.tm_k8 : &p.tm_v8,
                                            rg.full(seq), 0, y + kRows, zk);
                        }
                    }
                }
                // output staging slot
                if (rg.acquire(seq, aborted, p.err)) rg.publish_empty(seq);
                ++seq;
            }
            // teardown: the last fills have landed (no copy may still be writing this CTA's
            // shared memory when it exits) and every slot's last use has been released
            for (uint32_t q = seq > kSlots ? seq - kSlots : 0; q < seq; ++q)
                rg.wait_full(q, aborted, p.err);
            for (uint32_t q = seq > kSlots ? seq - kSlots : 0; q < seq; ++q)
                rg.acquire(q + kSlots, aborted, p.err);
        }
    } else if (warp == 4) {
        // ------------------------------------------------ MMA issue
        if (lane == 0) {
            uint32_t seq = 0, gcount = 0, tcount = 0;
            const uint32_t idesc_o = idesc_bf16(128, 64, 0, 1);
            const uint32_t idesc_s = idesc_bf16(128, 64, 0, 0);
            const uint32_t idesc_s2 = idesc_bf16(128, 128, 0, 0);
            const uint32_t idesc_s3 = idesc_bf16(128, 192, 0, 0);
            for (uint32_t idx = blockIdx.x; idx < p.total_tiles; idx += gridDim.x, ++tcount) {
                int half;
                const ring::Tile tl = tile_at<kWide>(p, idx, half);
                const PL pl = make_plan<kWide>(p, tl.layer, tl.row0);
                // TMEM of the previous tile read out (and its PV finished) before S is rewritten
                if (tcount > 0) mbar_wait(B_T, (tcount - 1) & 1, aborted, p.err);
                for (int g = 0; g < pl.n_groups; ++g, ++gcount) {
                    const int nch = pl.nch(g);
                    const int ns = pl.band_slots(g);
                    const int nk = pl.k_slots(g);
                    const uint32_t qseq = seq, kseq = seq + PL::kQItems, vseq = kseq + nk;
                    seq += pl.group_items(g);
                    if (g > 0) mbar_wait(B_O, (gcount - 1) & 1, aborted, p.err);  // P of g-1 consumed
                    for (int j = 0; j < PL::kQItems; ++j) rg.wait_full(qseq + j, aborted, p.err);
                    for (int j = 0; j < nk; ++j) rg.wait_full(kseq + j, aborted, p.err);
                    if constexpr (kRope) mbar_wait(B_R, gcount & 1, aborted, p.err);  // rotated in place
                    tc_fence_after();
                    // head size 64, three chunks in two consecutive slots that do not wrap
                    // around the ring: 192 key rows at one stride, one N = 192 MMA per k-step
                    // (the fractional mode's 17 KB slots break the stride)
                    const bool one_n192 = !kWide && !kFrac && nch == 3 && rg.slot(kseq) + 1 < kSlots;
                    if (one_n192) {
                        const uint32_t qaddr = rg.addr(qseq), kaddr = rg.addr(kseq);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_ss(tmem, sdesc_sw128(qaddr + 32 * kk, 16, 1024),
                                   sdesc_sw128(kaddr + 32 * kk, 16, 1024), idesc_s3, kk > 0);
                    }
                    for (int c = 0; c < (one_n192 ? 0 : nch); ++c) {
                        if (!kWide && (c & 1) == 0 && c + 1 < nch) {
                            // two chunks of one slot (128 contiguous key rows): one N = 128 MMA
                            // per k-step into columns [64c, 64c + 128)
                            const uint32_t qaddr = rg.addr(qseq);
                            const uint32_t kaddr = rg.addr(kseq + c / 2);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_ss(tmem + 64 * c, sdesc_sw128(qaddr + 32 * kk, 16, 1024),
                                       sdesc_sw128(kaddr + 32 * kk, 16, 1024), idesc_s2, kk > 0);
                            ++c;
                            continue;
                        }
                        if constexpr (kWide) {
                            // K-dim 128: Q half 0 against the chunk's columns 0-63, then half 1
                            const uint32_t kaddr = rg.addr(kseq + c);
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk)
                                mma_ss(tmem + 64 * c,
                                       sdesc_sw128(rg.addr(qseq + (kk >> 2)) + 32 * (kk & 3), 16, 1024),
                                       sdesc_sw128(kaddr + (kk >> 2) * kChunkBytes + 32 * (kk & 3), 16, 1024),
                                       idesc_s, kk > 0);
                        } else {
                            const uint32_t qaddr = rg.addr(qseq);
                            const uint32_t kaddr = rg.addr(kseq + c / 2) + (c & 1) * kChunkBytes;
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_ss(tmem + 64 * c, sdesc_sw128(qaddr + 32 * kk, 16, 1024),
                                       sdesc_sw128(kaddr + 32 * kk, 16, 1024), idesc_s, kk > 0);
                        }
                    }
                    mma_commit(B_S);
                    for (int j = 0; j < nk; ++j) rg.release_mma(kseq + j);
                    // the last group's Q copy is released by the row warps once they hold q
                    if (g < pl.n_groups - 1)
                        for (int j = 0; j < PL::kQItems; ++j) rg.release_mma(qseq + j);
                    mbar_wait(B_P, gcount & 1, aborted, p.err);
                    tc_fence_after();
                    for (int j = 0; j < ns; ++j) rg.wait_full(vseq + j, aborted, p.err);
                    if (g == pl.n_groups - 1) mbar_arrive(B_L);  // every band item has landed
                    tc_fence_after();
                    for (int kk = 0; kk < nch * (kChunk / 16); ++kk) {
                        const int c = kk >> 2;
                        const uint32_t vaddr = rg.addr(vseq + c / 2) + (c & 1) * kChunkBytes + 2048 * (kk & 3);
                        mma_ts(tmem + kTmemO, tmem + 8 * kk, sdesc_sw128(vaddr, 0, 1024), idesc_o,
                               (g > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(B_O);
                    for (int j = 0; j < ns; ++j) rg.release_mma(vseq + j);
                }
                seq += (PL::kKItems + 1) * pl.n_act + 1;  // offset and staging slots are the row threads'
            }
            // teardown: the last commit must have landed before TMEM is released
            if (gcount > 0) mbar_wait(B_O, (gcount - 1) & 1, aborted, p.err);
        }
    } else {
        // ------------------------------------------------ row threads
        const int r = tid;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const float sl2 = p.scale_log2;
        uint32_t seq = 0, gbase = 0, tcount = 0;
        for (uint32_t idx = blockIdx.x; idx < p.total_tiles; idx += gridDim.x, ++tcount) {
            int half;
            const ring::Tile tl = tile_at<kWide>(p, idx, half);
            const PL pl = make_plan<kWide>(p, tl.layer, tl.row0);
            const int32_t i0 = pl.i0, c_lo = pl.c_lo, n_chunks = pl.n_chunks, n_groups = pl.n_groups;
            const int32_t i = i0 + r;
            const int32_t z = (int32_t)tl.zl;
            const int32_t* offs = p.tabs.off[tl.layer];

            uint32_t qseq = seq;  // the last group's Q copy
            for (int g = 0; g + 1 < n_groups; ++g) qseq += pl.group_items(g);
            uint32_t gseq = seq;  // the current group's first item (RoPE mode)
            seq += pl.band_items();
            uint32_t qw[32 * PL::kQItems];  // the q row (head size 128: both halves)

            // ---- band: masked online softmax over the S groups. Only the 32-column chunks
            // that some row of this warp can reach are read (3 of 6 at W = 64).
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
                if constexpr (kRope) {
                    // rotate the group's Q copy and K chunks in their slots before its S MMAs
                    // (every row a thread touches is its own: no barrier among the row threads)
                    rg.wait_full(gseq, aborted, p.err);
                    for (int j = 0; j < pl.k_slots(g); ++j) rg.wait_full(gseq + 1 + j, aborted, p.err);
                    uint8_t* qt = slot_ptr(gseq);
                    if (g == n_groups - 1) {  // the unrotated q row, for the offsets
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const uint4 w = *reinterpret_cast<const uint4*>(qt + sw128_off(r, c));
                            qw[4 * c + 0] = w.x; qw[4 * c + 1] = w.y; qw[4 * c + 2] = w.z; qw[4 * c + 3] = w.w;
                        }
                    }
                    if (i < T) rotate_row_sw(qt, r, p.rope + (int64_t)i * 16);
                    for (int rr = r; rr < nch * kChunk; rr += kRows) {
                        const int32_t j = kbase + rr;  // the key's position
                        if (j < T) {
                            const int c = rr / kChunk;
                            uint8_t* kt = slot_ptr(gseq + 1 + c / 2) + (c & 1) * kChunkBytes;
                            rotate_row_sw(kt, rr % kChunk, p.rope + (int64_t)j * 16);
                        }
                    }
                    fence_proxy_async_smem();  // generic writes before the MMAs' reads
                    __syncwarp();
                    if (lane == 0) mbar_arrive(B_R);
                    gseq += pl.group_items(g);
                }
                mbar_wait(B_S, (gbase + g) & 1, aborted, p.err);
                tc_fence_after();
                __syncwarp();  // converged for the warp-collective TMEM accesses below
                float mn = m_b;
                {
                    // two passes over the reachable 32-column chunks: the row max, then the
                    // exponentials (one chunk of registers at a time)
                    uint32_t v[32];
                    float mx = -INFINITY;
                    for (int j = 0; j < n_need; ++j) {
                        tmem_ld32(tmem + lane_base + 32 * (ccA + j), v);
                        tmem_ld_wait(v);
                        const int32_t dj = d0 - 32 * (ccA + j);
    #pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if ((uint32_t)(dj - e) < (uint32_t)W) mx = fmaxf(mx, __uint_as_float(v[e]) * sl2);
                    }
                    mn = fmaxf(m_b, mx);
                    if (g > 0) {
                        mbar_wait(B_O, (gbase + g - 1) & 1, aborted, p.err);
                        tc_fence_after();
                        const float corr = (m_b == -INFINITY) ? 0.f : ex2(m_b - mn);
                        if (__any_sync(0xffffffffu, mn != m_b)) {
                            for (int h = 0; h < 2; ++h) {
                                tmem_ld32(tmem + lane_base + kTmemO + 32 * h, v);
                                tmem_ld_wait(v);
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
                            tmem_ld_wait(v);
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
                __syncwarp();
                if (lane == 0) mbar_arrive(B_P);
            }

            // ---- offsets: one pass per offset; the running max starts at the band's max and
            // is only raised when a score exceeds it by more than 2^8 (rare rescale)
            // q row into registers, then the Q slot goes back to the producer (every S MMA
            // reading it has completed: B_S was waited for each group). Holding the slot through
            // the offsets would stall the in-order ring.
#pragma unroll
            for (int qh = 0; qh < PL::kQItems; ++qh) {
                if constexpr (!kRope) {  // (RoPE mode: read before the rotation)
                    rg.wait_full(qseq + qh, aborted, p.err);
                    const uint8_t* qrow = slot_ptr(qseq + qh);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 w = *reinterpret_cast<const uint4*>(qrow + sw128_off(r, c));
                        qw[32 * qh + 4 * c + 0] = w.x; qw[32 * qh + 4 * c + 1] = w.y;
                        qw[32 * qh + 4 * c + 2] = w.z; qw[32 * qh + 4 * c + 3] = w.w;
                    }
                }
                rg.release_warp(qseq + qh, lane);
            }
            mbar_wait(B_L, tcount & 1, aborted, p.err);
            float m_o = m_b, l_o = 0.f;
            float oacc[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) oacc[c] = 0.f;
#pragma unroll 1
            for (int k = 0; k < pl.n_act; ++k) {
                const bool valid = i - offs[k] >= 0;
                float wk = 0.f;  // weight of row r + 1 (fractional mode); uniform over the CTA
                if constexpr (kFrac) wk = p.w[tl.layer][k];
                const bool lerp = kFrac && wk != 0.f;
                float s = 0.f;
                if constexpr (kRope) {
                    // (R_o q) . k_(i-o) from the unrotated rows: one angle per offset
                    const float4* trow = p.rope + (int64_t)offs[k] * 16;
                    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
                    rg.wait_full(seq, aborted, p.err);
                    const uint8_t* krow = slot_ptr(seq);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 w = *reinterpret_cast<const uint4*>(krow + sw128_off(r, c));
                        const float4 t0 = __ldg(trow + 2 * c), t1 = __ldg(trow + 2 * c + 1);
                        rope_dot_pair(qw[4 * c + 0], w.x, t0.x, t0.y, a0);
                        rope_dot_pair(qw[4 * c + 1], w.y, t0.z, t0.w, a1);
                        rope_dot_pair(qw[4 * c + 2], w.z, t1.x, t1.y, a2);
                        rope_dot_pair(qw[4 * c + 3], w.w, t1.z, t1.w, a3);
                    }
                    s = (a0 + a1) + (a2 + a3);
                    rg.release_warp(seq, lane);
                    ++seq;
                } else {
                    // the row dot over the K item(s): head size 128 takes its two halves
                    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
                    for (int kh = 0; kh < PL::kKItems; ++kh) {
                        rg.wait_full(seq, aborted, p.err);
                        const uint8_t* krow = slot_ptr(seq);
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const uint4 w = *reinterpret_cast<const uint4*>(krow + sw128_off(r, c));
                            fma2_bf16(qw[32 * kh + 4 * c + 0], w.x, a0, a1);
                            fma2_bf16(qw[32 * kh + 4 * c + 1], w.y, a2, a3);
                            fma2_bf16(qw[32 * kh + 4 * c + 2], w.z, a0, a1);
                            fma2_bf16(qw[32 * kh + 4 * c + 3], w.w, a2, a3);
                        }
                        if (kh == PL::kKItems - 1) {
                            s = (a0 + a1) + (a2 + a3);
                            if (lerp) {
                                // row r + 1 of the item (row 128 is the first of the 8 extra rows)
                                float b0 = 0.f, b1 = 0.f, b2 = 0.f, b3 = 0.f;
#pragma unroll
                                for (int c = 0; c < 8; ++c) {
                                    const uint4 w = *reinterpret_cast<const uint4*>(krow + sw128_off(r + 1, c));
                                    fma2_bf16(qw[4 * c + 0], w.x, b0, b1);
                                    fma2_bf16(qw[4 * c + 1], w.y, b2, b3);
                                    fma2_bf16(qw[4 * c + 2], w.z, b0, b1);
                                    fma2_bf16(qw[4 * c + 3], w.w, b2, b3);
                                }
                                s = fmaf(wk, ((b0 + b1) + (b2 + b3)) - s, s);
                            }
                        }
                        rg.release_warp(seq, lane);
                        ++seq;
                    }
                }
                const float sc = valid ? s * sl2 : -INFINITY;
                if (sc > m_o + 8.f) {
                    const float corr = m_o == -INFINITY ? 0.f : ex2(m_o - sc);
                    l_o *= corr;
#pragma unroll
                    for (int c = 0; c < 64; ++c) oacc[c] *= corr;
                    m_o = sc;
                }
                const float pk = valid ? ex2(sc - m_o) : 0.f;
                l_o += pk;
                const float phi = pk * wk;  // fractional mode: the later row's share
                const uint32_t pb = pack_bf16x2(lerp ? pk - phi : pk, 0.f);
                rg.wait_full(seq, aborted, p.err);
                const uint8_t* vrow = slot_ptr(seq);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 w = *reinterpret_cast<const uint4*>(vrow + sw128_off(r, c));
                    axpy2_bf16(pb, w.x, oacc[8 * c + 0], oacc[8 * c + 1]);
                    axpy2_bf16(pb, w.y, oacc[8 * c + 2], oacc[8 * c + 3]);
                    axpy2_bf16(pb, w.z, oacc[8 * c + 4], oacc[8 * c + 5]);
                    axpy2_bf16(pb, w.w, oacc[8 * c + 6], oacc[8 * c + 7]);
                }
                if (lerp) {
                    const uint32_t ph = pack_bf16x2(phi, 0.f);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 w = *reinterpret_cast<const uint4*>(vrow + sw128_off(r + 1, c));
                        axpy2_bf16(ph, w.x, oacc[8 * c + 0], oacc[8 * c + 1]);
                        axpy2_bf16(ph, w.y, oacc[8 * c + 2], oacc[8 * c + 3]);
                        axpy2_bf16(ph, w.z, oacc[8 * c + 4], oacc[8 * c + 5]);
                        axpy2_bf16(ph, w.w, oacc[8 * c + 6], oacc[8 * c + 7]);
                    }
                }
                rg.release_warp(seq, lane);
                ++seq;
            }

            // ---- epilogue: merge the band and offset softmax parts
            mbar_wait(B_O, (gbase + n_groups - 1) & 1, aborted, p.err);
            tc_fence_after();
            const float m = fmaxf(m_b, m_o);
            const float mu = m == -INFINITY ? 0.f : m;
            const float fb = m_b == -INFINITY ? 0.f : ex2(m_b - mu);
            const float fo = m_o == -INFINITY ? 0.f : ex2(m_o - mu);
            const float l = l_b * fb + l_o * fo;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const uint32_t oseq = seq++;
            rg.wait_full(oseq, aborted, p.err);
            uint8_t* orow = slot_ptr(oseq);
            __syncwarp();  // converged for the warp-collective TMEM accesses below
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + kTmemO + 32 * h, v);
                tmem_ld_wait(v);
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
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B_T);  // TMEM free for the next tile's MMAs
            gbase += n_groups;
            if (i < T && half == 0) p.lse[tl.zl * T + i] = (m + lg2(l)) * 0.69314718055994531f;
            fence_proxy_async_smem();
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (tid == 0) {
                if (!aborted) {
                    const int32_t xo = 64 * half;  // the CTA's output columns
                    tma_store_3d(&p.tm_o, rg.addr(oseq), xo, i0, z);
                    if (i0 + kChunk < T) tma_store_3d(&p.tm_o, rg.addr(oseq) + kChunkBytes, xo, i0 + kChunk, z);
                    tma_store_commit();
                    tma_store_wait_read0();
                }
                rg.release_stage(oseq);
            }
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

}  // namespace

namespace {

template <bool kFrac, bool kWide, bool kRope = false>
fibattn_status launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                          const AttnShape& sh, const OffsetTables& t,
                          const float (*w)[kMaxOffsets], const char* name, cudaStream_t st,
                          const float* rope = nullptr) {
    const int64_t slices = sh.slices_per_layer * sh.n_layers;
    const int32_t tiles = (sh.T + kRows - 1) / kRows;
    const int64_t halves = kWide ? 2 : 1;  // CTAs per tile
    if (slices > 0x7fffffff || (int64_t)tiles * slices * halves > 0x7fffffff)
        return FIBATTN_ERR_INVALID_ARG;
    FwdArgs<kFrac> P;
    // the error-word lookup is a runtime call: it binds the device's primary context to this
    // thread (a fresh thread may have none), which the tensor-map encoding below needs
    P.err = device_error_word();
    if (!P.err) return cuda_fail(-1, "cudaGetSymbolAddress (error word)");
    const int64_t slices_kv = slices / sh.group;
    const void* bases[4] = {q, k, v, o};
    CUtensorMap* maps[4] = {&P.tm_q, &P.tm_k, &P.tm_v, &P.tm_o};
    for (int m = 0; m < 4; ++m) {
        const int64_t sl = (m == 1 || m == 2) ? slices_kv : slices;
        const int r = kWide ? make_bf16_rows_map_d(maps[m], bases[m], sl, sh.T, 128)
                            : make_bf16_rows_map(maps[m], bases[m], sl, sh.T);
        if (r != 0) return cuda_fail(r, "cuTensorMapEncodeTiled (fwd)");
    }
    if constexpr (kFrac) {
        int r = make_bf16_rows8_map(&P.tm_k8, k, slices_kv, sh.T);
        if (r == 0) r = make_bf16_rows8_map(&P.tm_v8, v, slices_kv, sh.T);
        if (r != 0) return cuda_fail(r, "cuTensorMapEncodeTiled (fwd, 8-row box)");
        for (int l = 0; l < kMaxLayersPerLaunch; ++l)
            for (int e = 0; e < kMaxOffsets; ++e) P.w[l][e] = w[l][e];
    }
    P.lse = lse;
    P.rope = reinterpret_cast<const float4*>(rope);
    P.slices_per_layer = (uint32_t)sh.slices_per_layer;
    P.group = (uint32_t)sh.group;
    P.slices_per_layer_kv = (uint32_t)(sh.slices_per_layer / sh.group);
    P.total_tiles = (uint32_t)((int64_t)tiles * slices * halves);
    P.T = sh.T;
    P.W = sh.W;
    P.tiles_per_slice = tiles;
    P.scale_log2 = sh.scale * 1.4426950408889634f;
    P.tabs = t;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail((int32_t)e, "cudaGetDevice");
    static bool attr_set[64] = {};
    static int n_sm[64] = {};
    if (dev < 0 || dev >= 64) return FIBATTN_ERR_UNSUPPORTED;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(fwd_tc_kernel<kFrac, kWide, kRope>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem_alloc<kFrac>());
        if (e != cudaSuccess) return cuda_fail((int32_t)e, "cudaFuncSetAttribute (fwd)");
        e = cudaDeviceGetAttribute(&n_sm[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail((int32_t)e, "cudaDeviceGetAttribute");
        attr_set[dev] = true;
    }
    const int64_t grid = (int64_t)P.total_tiles < 2LL * n_sm[dev] ? (int64_t)P.total_tiles : 2LL * n_sm[dev];
    {
        KernelScope ks(name, st);
        fwd_tc_kernel<kFrac, kWide, kRope><<<(unsigned)grid, kThreads, smem_alloc<kFrac>(), st>>>(P);
    }
    return launch_status(name);
}

}  // namespace

fibattn_status launch_fwd_tc_bf16(const void* q, const void* k, const void* v, void* o, float* lse,
                                  const AttnShape& sh, const OffsetTables& t, cudaStream_t st) {
    return launch_fwd<false, false>(q, k, v, o, lse, sh, t, nullptr, "fwd_tc_bf16", st);
}

fibattn_status launch_fwd_rope_tc_bf16(const void* q, const void* k, const void* v, void* o,
                                       float* lse, const AttnShape& sh, const OffsetTables& t,
                                       const float* rope_table, cudaStream_t st) {
    return launch_fwd<false, false, true>(q, k, v, o, lse, sh, t, nullptr, "fwd_rope_tc_bf16", st,
                                          rope_table);
}

fibattn_status launch_fwd_tc128_bf16(const void* q, const void* k, const void* v, void* o,
                                     float* lse, const AttnShape& sh, const OffsetTables& t,
                                     cudaStream_t st) {
    return launch_fwd<false, true>(q, k, v, o, lse, sh, t, nullptr, "fwd_tc128_bf16", st);
}

fibattn_status launch_fwd_frac_tc_bf16(const void* q, const void* k, const void* v, void* o,
                                       float* lse, const AttnShape& sh, const FracTables& t,
                                       cudaStream_t st) {
    return launch_fwd<true, false>(q, k, v, o, lse, sh, t.c, t.w, "fwd_frac_tc_bf16", st);
}

}  // namespace fibattn
