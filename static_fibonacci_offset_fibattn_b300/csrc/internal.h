// internal.h -- types shared by the library's host code and its kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fibattn.h"

namespace fibattn {

// Layers handled by one kernel launch; longer calls are split into several launches.
constexpr int kMaxLayersPerLaunch = 16;
constexpr int kMaxOffsets = FIBATTN_MAX_OFFSETS;

// Per-launch offset tables, passed by value (__grid_constant__) so that they live in
// the kernel's constant bank: every launch carries its own copy, so concurrent calls
// on different streams cannot see each other's tables.
struct OffsetTables {
    int32_t count[kMaxLayersPerLaunch];
    int32_t off[kMaxLayersPerLaunch][kMaxOffsets];  // ascending, each in [W, T-1]
};

// Fractional-offset tables of one launch (the learned-alpha variant): for every real distance
// d = alpha * F kept by the table rule, `c.off` holds ceil(d) (ascending, possibly repeated),
// `w` the interpolation weight ceil(d) - d in [0, 1) of the row after i - ceil(d), and `f`
// the base value F (dd/dalpha, for the gradient of alpha).
struct FracTables {
    OffsetTables c;
    float w[kMaxLayersPerLaunch][kMaxOffsets];
    float f[kMaxLayersPerLaunch][kMaxOffsets];
};

// An exact alpha = num / den of one layer (num, den > 0, already reduced).
struct Alpha {
    int64_t num, den;
};

// Validates a schedule and a layer index; writes the layer's exact alpha.
fibattn_status layer_alpha(const fibattn_schedule* s, int32_t layer, Alpha* out);

// Host offset table of one layer under an exact alpha (see fibattn_offsets).
fibattn_status build_table(const fibattn_schedule* s, Alpha a, int32_t W, int32_t T, int32_t* out,
                           int32_t cap, int32_t* n_out);

// Fractional-offset table of one real alpha (see fibattn_frac_offsets).
fibattn_status build_frac_table(int32_t base, int64_t base_max, float alpha, int32_t W, int32_t T,
                                int32_t* c_out, float* w_out, float* f_out, int32_t cap,
                                int32_t* n_out);

// Builds FracTables for n launch layers with alphas[0..n).
fibattn_status build_frac_launch_tables(int32_t base, int64_t base_max, const float* alphas,
                                        int32_t n, int32_t W, int32_t T, FracTables* t);

// Builds OffsetTables for launch layers [layer0, layer0 + n).
fibattn_status build_launch_tables(const fibattn_schedule* s, int32_t layer0, int32_t n, int32_t W,
                                   int32_t T, OffsetTables* t);

// Brackets one kernel launch: counts it and, while profiling is enabled
// (fibattn_profile_enable), records a start/stop event pair on its stream.
class KernelScope {
  public:
    KernelScope(const char* name, cudaStream_t st);
    ~KernelScope();
    KernelScope(const KernelScope&) = delete;
    KernelScope& operator=(const KernelScope&) = delete;

  private:
    cudaStream_t st_;
    int rec_;
};

// Records a failed CUDA call (error code and a static description of the call) for
// fibattn_last_cuda_error and returns FIBATTN_ERR_CUDA.
fibattn_status cuda_fail(int32_t code, const char* where);
// Status of the kernel launch just issued on this thread: OK, or a recorded CUDA failure.
fibattn_status launch_status(const char* where);

// Device error word protocol (see fibattn_poll_device_error).
enum DeviceError : int32_t { kDevErrNone = 0, kDevErrTimeout = 1 };
int32_t* device_error_word();  // device address of the error word (current device)

// Launchers (defined in the .cu files).
fibattn_status launch_offsets_device(const fibattn_schedule* s, int32_t layer0, int32_t n,
                                     int32_t W, int32_t T, int32_t* d_tables, int32_t* d_counts,
                                     cudaStream_t st);
fibattn_status launch_keyset(const OffsetTables& t, int32_t W, int32_t T, uint32_t* d_mask,
                             cudaStream_t st);

struct AttnShape {
    int64_t slices_per_layer;  // B * H (query heads)
    int32_t T;
    int32_t W;                 // the window, clamped to T by every caller: a window of T keys
                               // already holds every causal key, and W + j or d - W in the
                               // kernels' 32-bit row arithmetic cannot overflow
    float scale;
    int32_t n_layers;          // layers in this launch
    int32_t group = 1;         // query heads per kv head: K/V (and dK/dV) have
                               // slices_per_layer / group slices per layer, query head h of
                               // batch b reading kv head h / group of batch b
    int32_t d = 64;            // head size: 64 or 128
};

fibattn_status launch_fwd_simt_f32(const float* q, const float* k, const float* v, float* o,
                                   float* lse, const AttnShape& sh, const OffsetTables& t,
                                   cudaStream_t st);
fibattn_status launch_fwd_tc_bf16(const void* q, const void* k, const void* v, void* o, float* lse,
                                  const AttnShape& sh, const OffsetTables& t, cudaStream_t st);
// Dense causal forward (bf16, head size 64): the W >= T case, where no offset survives and
// every earlier key is attended; 128 x 128 score blocks on the tensor cores.
fibattn_status launch_fwd_dense_tc_bf16(const void* q, const void* k, const void* v, void* o,
                                        float* lse, const AttnShape& sh, cudaStream_t st);
// The same forward at head size 128 (two CTAs per tile, one per half of the output columns).
fibattn_status launch_fwd_rope_tc_bf16(const void* q, const void* k, const void* v, void* o,
                                       float* lse, const AttnShape& sh, const OffsetTables& t,
                                       const float* rope_table, cudaStream_t st);
fibattn_status launch_fwd_tc128_bf16(const void* q, const void* k, const void* v, void* o,
                                     float* lse, const AttnShape& sh, const OffsetTables& t,
                                     cudaStream_t st);
// Fractional-offset forwards (the learned-alpha variant): fp32 SIMT and bf16 tensor cores.
fibattn_status launch_fwd_frac_simt_f32(const float* q, const float* k, const float* v, float* o,
                                        float* lse, const AttnShape& sh, const FracTables& t,
                                        cudaStream_t st);
fibattn_status launch_fwd_frac_tc_bf16(const void* q, const void* k, const void* v, void* o,
                                       float* lse, const AttnShape& sh, const FracTables& t,
                                       cudaStream_t st);
// SIMT backward (fp32 path, d = 64 or 128): D into `delta`, then dQ, then dK/dV.
fibattn_status launch_bwd_simt_f32(const float* q, const float* k, const float* v, const float* o,
                                   const float* lse, const float* dO, float* dq, float* dk,
                                   float* dv, float* delta, const AttnShape& sh,
                                   const OffsetTables& t, cudaStream_t st);

// Fractional-offset backwards: dq/dk/dv as the static ones with interpolated rows, plus the
// partials of dL/dalpha (g_i = sum_k f_k dL/dd_k of query i) into galpha: per query,
// [slices][T], on the SIMT path; per 128-query tile, [slices][tiles], on the tensor-core
// path (reduced per layer by launch_dalpha_reduce). Workspace as the static bf16 backward
// (n_max from the frac tables).
fibattn_status launch_bwd_frac_simt_f32(const float* q, const float* k, const float* v,
                                        const float* o, const float* lse, const float* dO,
                                        float* dq, float* dk, float* dv, float* delta,
                                        float* galpha, const AttnShape& sh, const FracTables& t,
                                        cudaStream_t st);
fibattn_status launch_bwd_frac_tc_bf16(const void* q, const void* k, const void* v, const void* o,
                                       const float* lse, const void* dO, void* dq, void* dk,
                                       void* dv, float* delta, float* lse2, uint32_t* pds,
                                       int32_t n_max, float* galpha, const AttnShape& sh,
                                       const FracTables& t, cudaStream_t st);
// dalpha[l] = sum of galpha over the rows_per_layer rows of launch layer l, for n layers
// (fixed summation order, fp64 accumulation: deterministic).
fibattn_status launch_dalpha_reduce(const float* galpha, float* dalpha, int32_t n,
                                    int64_t rows_per_layer, cudaStream_t st);

// Rotary position embedding (rope.cu): the cos/sin table [T][32] (float2, fp64-computed) and
// the rotation of rows [rows][64] (row r at position r % T), y = R x or R^T x.
fibattn_status launch_rope_table(float* table, int32_t T, double base, cudaStream_t st);
fibattn_status launch_rope(const void* x, void* y, int64_t rows, int32_t T, int32_t dtype,
                           const float* table, bool inverse, cudaStream_t st);

// Tensor-core backward (bf16 path). Workspace rows are padded to T_pad = T rounded up to 4:
// delta and lse2 [slices][T_pad] fp32, pds [slices][n_max][T_pad] (P, dS) bf16 pairs indexed
// by key row, n_max >= every launch layer's table size.
fibattn_status launch_bwd_tc_bf16(const void* q, const void* k, const void* v, const void* o,
                                  const float* lse, const void* dO, void* dq, void* dk, void* dv,
                                  float* delta, float* lse2, uint32_t* pds, int32_t n_max,
                                  const AttnShape& sh, const OffsetTables& t, cudaStream_t st);

// One-pass backward (bf16, head size 64, one kv head per query head): a pre-pass writes D and
// lse log2(e) into delta / lse2 ([slices][T_pad], T_pad = T rounded up to 4), then one tensor-core
// kernel whose thread block per 128-row tile writes dq of the tile's queries and dk, dv of its
// keys. UNSUPPORTED for other head sizes or grouped kv heads.
fibattn_status launch_bwd_fused_tc_bf16(const void* q, const void* k, const void* v,
                                        const void* o, const float* lse, const void* dO, void* dq,
                                        void* dk, void* dv, float* delta, float* lse2,
                                        const AttnShape& sh, const OffsetTables& t, cudaStream_t st);

}  // namespace fibattn
