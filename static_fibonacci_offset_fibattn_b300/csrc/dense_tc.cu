// dense_tc.cu -- dense causal attention forward (bf16, head size 64) on sm_103a tensor cores.
//
// When the window covers every earlier key (W >= T) no offset survives the table rule and the
// attended set of "Depth-Staggered Fibonacci Spacing for Sparse Attention" (gist.science
// explainer, Metodologia / Arquitetura e Mecanismo de Atencao, "Conjunto Atendido") is the
// causal prefix: o_i = softmax_j<=i(scale q_i . k_j) . v_j. That is the dense baseline the pages
// compare against (Metodologia / Controles; Principais Contribuicoes 3), so it gets a kernel
// laid out for it instead of the sparse kernel's 64-key window chunks.
//
// One CTA (192 threads) per 128-query tile [t0, t0+128) of a (layer, batch, head) slice, two
// CTAs per SM, the tiles with the most key blocks launched first:
//   warps 0-3 : one thread per query row (TMEM lane = row): softmax and epilogue.
//   warp 4    : TMEM allocation and tcgen05.mma issue (lane 0).
//   warp 5    : TMA loads (lane 0): the tile's Q rows, then K_j and V_j of every key block
//               j = 0 .. t0/128 through a five-slot ring.
// Per key block j (keys [128j, 128j+128)):
//   S = Q K_j^T (M=128, N=128, K=64) into TMEM columns [0, 128);
//   each row thread reads its score row into registers (the columns are then free, and the
//   tensor core forms S_{j+1} while the row threads work on block j), takes the row max over
//   its allowed keys (all of them, or k <= i in the diagonal block) and raises its running
//   max m only when the block's max exceeds it by more than 2^8 (then O and the sum l are
//   rescaled, once PV_{j-1} has completed); the exponentials 2^(s - m) <= 2^8 are formed in
//   registers as bf16 pairs and go to TMEM columns [192, 256) once PV_{j-1}, which reads
//   those columns, has completed (so its latency is not on the row threads' path);
//   O += P V_j (A = P from TMEM, B = V_j MN-major) into TMEM columns [128, 192).
// Epilogue: O / l staged in the Q buffer (every S MMA that read it has completed), TMA store;
// lse = (m + log2 l) ln 2.
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

constexpr int kRows = 128;                       // queries per tile, keys per block
constexpr int kBox = kTmaBoxRows;                // rows of one TMA box
constexpr int kThreads = 192;
constexpr uint32_t kTileBytes = kRows * 128;     // 16 KB
constexpr uint32_t kBoxBytes = kBox * 128;       // 8 KB
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0, kColO = 128, kColP = 192;  // S [0, 128), O [128, 192), P [192, 256)
constexpr uint32_t kSlots = 5;
constexpr float kRescale = 8.f;                  // log2 of the largest unnormalised P

// barriers: FULL[kSlots], EMPTY[kSlots], Q loaded, S ready, S read out (4 warps), P written
// (4 warps), PV done
constexpr uint32_t kBarQ = 2 * kSlots, kBarS = kBarQ + 1, kBarF = kBarQ + 2, kBarP = kBarQ + 3,
                   kBarO = kBarQ + 4;
constexpr uint32_t kNumBars = kBarO + 1;
// shared memory: Q (later the output staging), the ring, the barriers, the TMEM address word
constexpr uint32_t kOffQ = 0, kOffRing = kTileBytes, kOffBar = kOffRing + kSlots * kTileBytes;
constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemAlloc = kOffTmemSlot + 16 + 1024;  // + alignment slack

struct DenseParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_o;  // 3D {64, T, slices}, box {64, 64, 1} (k, v over kv slices)
    float* lse;
    int32_t* err;
    uint32_t slices_per_layer;
    uint32_t group;                // query heads per kv head
    uint32_t slices_per_layer_kv;
    int32_t T;
    int32_t tiles_per_slice;
    float scale_log2;              // scale * log2(e)
};

// The largest raw score of a row: every column, or columns c <= r (the diagonal block). Four
// partial maxima keep the dependency chains short.
template <bool kDiag>
__device__ __forceinline__ float row_max(const uint32_t (&v)[4][32], int r) {
    float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc)
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
            const int c = 32 * cc + e;
            a0 = fmaxf(a0, (!kDiag || c + 0 <= r) ? __uint_as_float(v[cc][e + 0]) : -INFINITY);
            a1 = fmaxf(a1, (!kDiag || c + 1 <= r) ? __uint_as_float(v[cc][e + 1]) : -INFINITY);
            a2 = fmaxf(a2, (!kDiag || c + 2 <= r) ? __uint_as_float(v[cc][e + 2]) : -INFINITY);
            a3 = fmaxf(a3, (!kDiag || c + 3 <= r) ? __uint_as_float(v[cc][e + 3]) : -INFINITY);
        }
    return fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
}

// p = 2^(s sl2 - m) of a row (0 for masked columns) as bf16 pairs, 32-column chunk cc in
// pk[cc] (for TMEM columns 16cc ..); returns the sum of the p (four partial sums). The pairs
// stay in registers so that the exponentials need not wait for the previous block's P V.
template <bool kDiag>
__device__ __forceinline__ float row_exp(const uint32_t (&v)[4][32], int r, float sl2, float m,
                                         uint32_t (&pk)[4][16]) {
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
            const int c = 32 * cc + e;
            const float p0 = (!kDiag || c + 0 <= r) ? ex2(fmaf(__uint_as_float(v[cc][e + 0]), sl2, -m)) : 0.f;
            const float p1 = (!kDiag || c + 1 <= r) ? ex2(fmaf(__uint_as_float(v[cc][e + 1]), sl2, -m)) : 0.f;
            const float p2 = (!kDiag || c + 2 <= r) ? ex2(fmaf(__uint_as_float(v[cc][e + 2]), sl2, -m)) : 0.f;
            const float p3 = (!kDiag || c + 3 <= r) ? ex2(fmaf(__uint_as_float(v[cc][e + 3]), sl2, -m)) : 0.f;
            a0 += p0;
            a1 += p1;
            a2 += p2;
            a3 += p3;
            pk[cc][e >> 1] = pack_bf16x2(p0, p1);
            pk[cc][(e >> 1) + 1] = pack_bf16x2(p2, p3);
        }
    }
    return (a0 + a1) + (a2 + a3);
}

__global__ void __launch_bounds__(kThreads, 2) fwd_dense_tc_kernel(const __grid_constant__ DenseParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - smem_u32(smem_raw));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t T = p.T;
    const int layer = blockIdx.y;
    // the tiles with the most key blocks first, over every slice of the layer
    const int32_t tile = p.tiles_per_slice - 1 - (int32_t)(blockIdx.x / p.slices_per_layer);
    const uint32_t s = blockIdx.x % p.slices_per_layer;
    const int64_t zl = (int64_t)layer * p.slices_per_layer + s;
    const int32_t z = (int32_t)zl;
    const int32_t zk = (int32_t)((int64_t)layer * p.slices_per_layer_kv + s / p.group);
    const int32_t t0 = tile * kRows;
    const int nb = tile + 1;  // key blocks 0 .. tile

    const ring::Ring rg{sbase + kOffRing, sbase + kOffBar, kSlots, 1, ring::kSlotBytes};
    auto bar = [&](uint32_t idx) { return sbase + kOffBar + 8u * idx; };
    const uint32_t B_Q = bar(kBarQ), B_S = bar(kBarS), B_F = bar(kBarF), B_P = bar(kBarP),
                   B_O = bar(kBarO);

    if (tid == 0) {
        ring::init_ring_barriers(rg, 1);
        mbar_init(B_Q, 1);
        mbar_init(B_S, 1);
        mbar_init(B_F, 4);
        mbar_init(B_P, 4);
        mbar_init(B_O, 1);
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
        // ------------------------------------------------ producer (lane 0)
        if (lane == 0) {
            prefetch_tmap(&p.tm_q);
            prefetch_tmap(&p.tm_k);
            prefetch_tmap(&p.tm_v);
            prefetch_tmap(&p.tm_o);
            mbar_arrive_expect_tx(B_Q, kTileBytes);
            tma_load_3d(sbase + kOffQ, &p.tm_q, B_Q, 0, t0, z);
            tma_load_3d(sbase + kOffQ + kBoxBytes, &p.tm_q, B_Q, 0, t0 + kBox, z);
            uint32_t seq = 0;
            for (int j = 0; j < nb; ++j)
                for (int h = 0; h < 2; ++h, ++seq) {  // K_j, then V_j
                    if (!rg.acquire(seq, aborted, p.err)) continue;
                    const CUtensorMap* map = h == 0 ? &p.tm_k : &p.tm_v;
                    mbar_arrive_expect_tx(rg.full(seq), kTileBytes);
                    tma_load_3d(rg.addr(seq), map, rg.full(seq), 0, kRows * j, zk);
                    tma_load_3d(rg.addr(seq) + kBoxBytes, map, rg.full(seq), 0, kRows * j + kBox, zk);
                }
            // teardown: the last fills have landed and every slot's last use has been released
            for (uint32_t q = seq > kSlots ? seq - kSlots : 0; q < seq; ++q)
                rg.wait_full(q, aborted, p.err);
            for (uint32_t q = seq > kSlots ? seq - kSlots : 0; q < seq; ++q)
                rg.acquire(q + kSlots, aborted, p.err);
        }
    } else if (warp == 4) {
        // ------------------------------------------------ MMA issue (lane 0)
        if (lane == 0) {
            const uint32_t idesc_s = idesc_bf16(128, 128, 0, 0);
            const uint32_t idesc_o = idesc_bf16(128, 64, 0, 1);
            mbar_wait(B_Q, 0, aborted, p.err);
            // S_j as soon as the row threads hold S_{j-1} in registers, then PV_{j-1} once they
            // have written P_{j-1}: the tensor core forms S_j while they exponentiate S_{j-1}
            auto issue_pv = [&](int j) {
                const uint32_t vseq = 2u * j + 1u;
                mbar_wait(B_P, j & 1, aborted, p.err);
                rg.wait_full(vseq, aborted, p.err);
                tc_fence_after();
                // keys 16kk .. 16kk+15: P packed in columns 8kk .. 8kk+7, V rows 16kk ..
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(tmem + kColO, tmem + kColP + 8 * kk,
                           sdesc_sw128(rg.addr(vseq) + 2048 * kk, 0, 1024), idesc_o,
                           (j > 0 || kk > 0) ? 1u : 0u);
                mma_commit(B_O);
                rg.release_mma(vseq);
            };
            for (int j = 0; j < nb; ++j) {
                const uint32_t kseq = 2u * j;
                rg.wait_full(kseq, aborted, p.err);
                if (j > 0) mbar_wait(B_F, (j - 1) & 1, aborted, p.err);  // S_{j-1} read out
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tmem + kColS, sdesc_sw128(sbase + kOffQ + 32 * kk, 16, 1024),
                           sdesc_sw128(rg.addr(kseq) + 32 * kk, 16, 1024), idesc_s, kk > 0);
                mma_commit(B_S);
                rg.release_mma(kseq);
                if (j > 0) issue_pv(j - 1);
            }
            issue_pv(nb - 1);
            mbar_wait(B_O, (nb - 1) & 1, aborted, p.err);
        }
    } else {
        // ------------------------------------------------ row threads
        const int r = tid;
        const int32_t i = t0 + r;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const float sl2 = p.scale_log2;
        float m = -INFINITY, l = 0.f;
        for (int j = 0; j < nb; ++j) {
            const bool diag = j == nb - 1;  // keys t0 + c, allowed for c <= r
            mbar_wait(B_S, j & 1, aborted, p.err);
            tc_fence_after();
            __syncwarp();  // converged for the warp-collective TMEM accesses below
            // the whole score row (128 columns) in one round trip
            uint32_t v[4][32];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) tmem_ld32(tmem + lane_base + kColS + 32 * cc, v[cc]);
            tmem_ld_wait();
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                for (int e = 0; e < 32; ++e) asm volatile("" : "+r"(v[cc][e]));  // after the wait
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B_F);  // the S columns are free for S_{j+1}
            const float mx = (diag ? row_max<true>(v, r) : row_max<false>(v, r)) * sl2;
            // raise the running max only past 2^8: then l and (once PV_{j-1} is done) O are
            // rescaled
            const bool raise = mx > m + kRescale;
            const float corr = raise ? (m == -INFINITY ? 0.f : ex2(m - mx)) : 1.f;
            if (raise) {
                l *= corr;
                m = mx;
            }
            // the exponentials into registers, as bf16 pairs: they need only the scores
            uint32_t pk[4][16];
            l += diag ? row_exp<true>(v, r, sl2, m, pk) : row_exp<false>(v, r, sl2, m, pk);
            // PV_{j-1} must be done before the P columns are overwritten and before O is
            // rescaled: it reads the P columns and accumulates into O
            if (j > 0) {
                mbar_wait(B_O, (j - 1) & 1, aborted, p.err);
                tc_fence_after();
            }
            __syncwarp();  // converged for the warp-collective TMEM accesses below
            if (j > 0 && __any_sync(0xffffffffu, raise)) {
                // a warp rescales O together, rows whose max stays by a factor of 1;
                // 16 columns at a time: the P pairs stay in registers meanwhile
                for (int h = 0; h < 4; ++h) {
                    uint32_t w[16];
                    tmem_ld16(tmem + lane_base + kColO + 16 * h, w);
                    tmem_ld_wait(w);
#pragma unroll
                    for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(__uint_as_float(w[e]) * corr);
                    tmem_st16(tmem + lane_base + kColO + 16 * h, w);
                }
            }
            // P into its columns (chunk cc -> columns 16cc ..)
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) tmem_st16(tmem + lane_base + kColP + 16 * cc, pk[cc]);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B_P);
        }

        // ---- epilogue: O / l staged in the Q buffer, TMA store; lse
        mbar_wait(B_O, (nb - 1) & 1, aborted, p.err);
        tc_fence_after();
        __syncwarp();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        uint8_t* orow = smem + kOffQ;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t w[32];
            tmem_ld32(tmem + lane_base + kColO + 32 * h, w);
            tmem_ld_wait(w);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int e = 8 * c;
                uint4 x;
                x.x = pack_bf16x2(__uint_as_float(w[e + 0]) * inv, __uint_as_float(w[e + 1]) * inv);
                x.y = pack_bf16x2(__uint_as_float(w[e + 2]) * inv, __uint_as_float(w[e + 3]) * inv);
                x.z = pack_bf16x2(__uint_as_float(w[e + 4]) * inv, __uint_as_float(w[e + 5]) * inv);
                x.w = pack_bf16x2(__uint_as_float(w[e + 6]) * inv, __uint_as_float(w[e + 7]) * inv);
                *reinterpret_cast<uint4*>(orow + sw128_off(r, 4 * h + c)) = x;
            }
        }
        if (i < T) p.lse[zl * T + i] = (m + lg2(l)) * 0.69314718055994531f;
        tc_fence_before();
        fence_proxy_async_smem();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (tid == 0 && !aborted) {
            tma_store_3d(&p.tm_o, sbase + kOffQ, 0, t0, z);
            if (t0 + kBox < T) tma_store_3d(&p.tm_o, sbase + kOffQ + kBoxBytes, 0, t0 + kBox, z);
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

}  // namespace

fibattn_status launch_fwd_dense_tc_bf16(const void* q, const void* k, const void* v, void* o,
                                        float* lse, const AttnShape& sh, cudaStream_t st) {
    if (sh.d != 64) return FIBATTN_ERR_UNSUPPORTED;
    const int64_t slices = sh.slices_per_layer * sh.n_layers;
    const int32_t tiles = (sh.T + kRows - 1) / kRows;
    const int64_t gx = (int64_t)tiles * sh.slices_per_layer;
    if (slices > 0x7fffffff || gx > 0x7fffffff) return FIBATTN_ERR_INVALID_ARG;
    DenseParams P;
    // the error-word lookup is a runtime call: it binds the device's primary context to this
    // thread, which the tensor-map encoding below needs
    P.err = device_error_word();
    if (!P.err) return cuda_fail(-1, "cudaGetSymbolAddress (error word)");
    const int64_t slices_kv = slices / sh.group;
    const void* bases[4] = {q, k, v, o};
    CUtensorMap* maps[4] = {&P.tm_q, &P.tm_k, &P.tm_v, &P.tm_o};
    for (int m = 0; m < 4; ++m) {
        const int r = make_bf16_rows_map(maps[m], bases[m], (m == 1 || m == 2) ? slices_kv : slices, sh.T);
        if (r != 0) return cuda_fail(r, "cuTensorMapEncodeTiled (dense fwd)");
    }
    P.lse = lse;
    P.slices_per_layer = (uint32_t)sh.slices_per_layer;
    P.group = (uint32_t)sh.group;
    P.slices_per_layer_kv = (uint32_t)(sh.slices_per_layer / sh.group);
    P.T = sh.T;
    P.tiles_per_slice = tiles;
    P.scale_log2 = sh.scale * 1.4426950408889634f;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail((int32_t)e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return FIBATTN_ERR_UNSUPPORTED;
    static bool attr_set[64] = {};
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(fwd_dense_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemAlloc);
        if (e != cudaSuccess) return cuda_fail((int32_t)e, "cudaFuncSetAttribute (dense fwd)");
        attr_set[dev] = true;
    }
    {
        KernelScope ks("fwd_dense_tc_bf16", st);
        fwd_dense_tc_kernel<<<dim3((unsigned)gx, (unsigned)sh.n_layers), kThreads, kSmemAlloc, st>>>(P);
    }
    return launch_status("fwd_dense_tc_bf16");
}

}  // namespace fibattn
