/*
 * fibattn.h -- C ABI of the B300 (sm_103a) Fibonacci-offset sparse attention library.
 *
 * The operation ("Depth-Staggered Fibonacci Spacing for Sparse Attention: Static
 * Schedules Beat Learned Dilation and Extrapolate Where Dense Attention Fails",
 * gist.science explainer, Metodologia / Arquitetura e Mecanismo de Atencao):
 * causal softmax attention in which query i of layer l attends
 *     S_i = { j : 0 <= i - j < W }  U  { i - o : o in O_l, i - o >= 0 }
 * where O_l is the layer's offset table: the base offsets F (Fibonacci
 * 1, 2, 3, 5, ..., 987, or the power-of-two control 2^k) scaled by the layer's
 * alpha_l and rounded, alpha_l coming from a static per-layer schedule
 * (Metodologia / Variaveis Experimentais and Controles).
 *
 * Conventions shared by every entry point:
 *   - All tensors are dense, contiguous, row-major [Lc][B][H][T][d] (Lc = layers in
 *     the call); lse is [Lc][B][H][T] float32, natural log. Call-layer c
 *     uses schedule layer (layer0 + c).
 *   - The caller owns every buffer; the library allocates no device memory apart
 *     from a 4-byte device error word and the fixed scratch array of
 *     fibattn_bwd_noalloc (both static). Device pointers must be 16-byte aligned.
 *   - No output (o, lse, dq, dk, dv, dalpha, the workspace) may share a byte with another
 *     output or an input of the same attention call; inputs may share memory (k == v). The
 *     extents are compared on the host and an overlap returns FIBATTN_ERR_INVALID_ARG
 *     (fibattn_fwd_bwd compares them within each layer group's forward and backward).
 *     fibattn_rope alone allows x == y (in place).
 *   - Work is enqueued on `cuda_stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns once launched; results are ready when the stream is.
 *     (fibattn_fwd_bwd forks its work to internal streams and joins it back into
 *     cuda_stream, so the same holds for it.)
 *   - Nothing is printed. Errors are returned as fibattn_status; kernel-side
 *     failures (a bounded wait that ran out) are latched in the device error word
 *     and reported by fibattn_poll_device_error().
 *   - d (head size) is 64, or 128 for the static and grouped-query forward and backward
 *     (the fractional-offset and RoPE calls take 64); dtype FIBATTN_F32 or FIBATTN_BF16, the
 *     same for every q/k/v/o/dO/dq/dk/dv tensor of a call.
 *   - T (sequence length) is in [1, FIBATTN_T_MAX] for every call that launches work, so
 *     that tile counts, padded row counts and row coordinates stay in 32 bits; a larger T
 *     returns FIBATTN_ERR_INVALID_ARG. The host table calls (fibattn_offsets,
 *     fibattn_frac_offsets) take any T >= 1.
 */
#ifndef FIBATTN_H
#define FIBATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported symbols (the library is built with hidden visibility by default). */
#if defined(FIBATTN_BUILD) && defined(__GNUC__)
#define FIBATTN_API __attribute__((visibility("default")))
#else
#define FIBATTN_API
#endif

typedef enum {
    FIBATTN_OK = 0,
    FIBATTN_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer, bad schedule */
    FIBATTN_ERR_UNSUPPORTED = 2, /* valid but not implemented (a head size or dtype) */
    FIBATTN_ERR_CAPACITY = 3,    /* an offset table does not fit the given capacity */
    FIBATTN_ERR_CUDA = 4,        /* a CUDA runtime call or a launch failed */
    FIBATTN_ERR_TIMEOUT = 5,     /* a kernel's bounded wait ran out (device error word) */
    FIBATTN_ERR_SCRATCH_LIMIT = 6 /* fibattn_bwd_noalloc: workspace larger than its fixed array */
} fibattn_status;

typedef enum { FIBATTN_BASE_FIB = 0, FIBATTN_BASE_POW2 = 1 } fibattn_base;
typedef enum { FIBATTN_SCHED_FIXED = 0, FIBATTN_SCHED_LINEAR = 1, FIBATTN_SCHED_COPRIME = 2 } fibattn_sched;
typedef enum { FIBATTN_F32 = 0, FIBATTN_BF16 = 1 } fibattn_dtype;

/* An exact rational alpha = num / den; 1 <= num, den <= FIBATTN_RATIO_MAX. */
typedef struct { int32_t num, den; } fibattn_ratio;
#define FIBATTN_RATIO_MAX (1 << 20)
#define FIBATTN_LAYERS_MAX (1 << 20)
#define FIBATTN_T_MAX (1 << 30)

/*
 * A per-layer alpha schedule (Metodologia / Variaveis Experimentais):
 *   FIXED   : alpha_l = alpha for every layer.
 *   LINEAR  : alpha_l = alpha_min + (alpha_max - alpha_min) * l / (n_layers - 1)
 *             (n_layers = 1 gives alpha_min), the static linear stagger.
 *   COPRIME : alpha_l = LINEAR alpha of layer (coprime_c * l mod n_layers); requires
 *             gcd(coprime_c, n_layers) = 1, coprime_c >= 1 (the coprime reassignment).
 * base      : FIBATTN_BASE_FIB (1, 2, 3, 5, ..., 987) or FIBATTN_BASE_POW2 (1, 2, 4, ...:
 *             the power-of-two control of Metodologia / Controles).
 * base_max  : 0 = default (Fibonacci stops at 987; powers of two run while the scaled
 *             offset is <= T - 1); > 0 = largest base value used, for either base.
 * n_layers  : L >= 1; every layer index passed to the library must be in [0, L).
 * Offsets of layer l: o = floor(alpha_l * F + 1/2) (exact, round half up) for each base
 * value F, kept when W <= o <= T - 1, ascending and without duplicates.
 */
typedef struct {
    int32_t base;                  /* fibattn_base */
    int32_t kind;                  /* fibattn_sched */
    fibattn_ratio alpha;           /* FIXED */
    fibattn_ratio alpha_min;       /* LINEAR, COPRIME */
    fibattn_ratio alpha_max;       /* LINEAR, COPRIME */
    int32_t n_layers;              /* L */
    int32_t coprime_c;             /* COPRIME */
    int64_t base_max;              /* 0 = default */
} fibattn_schedule;

/* Most offsets one layer's table may hold inside the kernels. */
#define FIBATTN_MAX_OFFSETS 64

/*
 * Offset table of one layer, on the host (Metodologia / Arquitetura, "Escalonamento":
 * target distance d_k = alpha * f_k). Writes *n_out entries to out[0..cap).
 * Errors: INVALID_ARG (null, W < 1, T < 1, bad schedule or layer), CAPACITY (more than
 * `cap` entries; *n_out then holds the needed count).
 */
FIBATTN_API fibattn_status fibattn_offsets(const fibattn_schedule* sched, int32_t layer, int32_t W, int32_t T,
                               int32_t* out, int32_t cap, int32_t* n_out);

/*
 * The same tables built by a device kernel, for n_layers_call layers starting at layer0:
 * d_tables is a device int32 [n_layers_call][FIBATTN_MAX_OFFSETS] (unused entries -1),
 * d_counts a device int32 [n_layers_call]. Used to cross-check the device integer
 * arithmetic bit-exactly against the host. Errors as fibattn_offsets (checked on the
 * host first), plus CUDA.
 */
FIBATTN_API fibattn_status fibattn_offsets_device(const fibattn_schedule* sched, int32_t layer0,
                                      int32_t n_layers_call, int32_t W, int32_t T,
                                      int32_t* d_tables, int32_t* d_counts, void* cuda_stream);

/*
 * Forward (the attended set of Metodologia / Arquitetura; scores scale * q.k, softmax
 * over S_i, output sum_j p_ij v_j):
 *   q, k, v : [Lc][B][H][T][d] device, dtype `dtype` (RoPE, if any, already applied:
 *             the pages apply it before the gather).
 *   o       : [Lc][B][H][T][d] device, written, same dtype.
 *   lse     : [Lc][B][H][T] float32 device, written: log sum_j exp(scale * q_i.k_j).
 *   scale   : <= 0 or NaN selects 1/sqrt(d); +inf returns FIBATTN_ERR_INVALID_ARG.
 *   W >= 1 (W >= T gives dense causal attention). bf16 runs on the tcgen05 tensor-core
 *   kernel (d = 128: two CTAs per 128-query tile, one per half of the output columns; d = 64
 *   with W >= T: a dense causal kernel over 128 x 128 score blocks); f32 on the SIMT fp32
 *   kernel.
 * Errors: INVALID_ARG, UNSUPPORTED, CAPACITY (a layer table above FIBATTN_MAX_OFFSETS),
 * CUDA (launch failure).
 */
FIBATTN_API fibattn_status fibattn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                           int32_t B, int32_t H, int32_t T, int32_t d, int32_t dtype, int32_t W,
                           float scale, const fibattn_schedule* sched, int32_t layer0,
                           int32_t n_layers_call, void* cuda_stream);

/*
 * Grouped-query forms of fibattn_fwd / fibattn_bwd (GQA; MQA at H_kv = 1): H query heads
 * share H_kv key/value heads, H a multiple of H_kv, query head h of batch b reading kv head
 * h / (H / H_kv) of batch b. q, o, dO, dq, lse are [Lc][B][H][T](d) as above; k, v, dk, dv
 * are [Lc][B][H_kv][T][d]. dk, dv of a kv row sum the contributions of every query head that
 * reads it (computed by the one thread block that owns the row: no atomics). The workspace is
 * fibattn_bwd_workspace_size(B, H, ...) (it is indexed by query rows). H_kv = H is exactly
 * fibattn_fwd / fibattn_bwd. Errors as those, plus INVALID_ARG when H_kv < 1 or H % H_kv != 0.
 * (This shape is not on the pages, which study 8 heads of 64; it is the head sharing of larger
 * models.)
 */
FIBATTN_API fibattn_status fibattn_fwd_gqa(const void* q, const void* k, const void* v, void* o,
                                           float* lse, int32_t B, int32_t H, int32_t H_kv,
                                           int32_t T, int32_t d, int32_t dtype, int32_t W,
                                           float scale, const fibattn_schedule* sched,
                                           int32_t layer0, int32_t n_layers_call,
                                           void* cuda_stream);
FIBATTN_API fibattn_status fibattn_bwd_gqa(const void* q, const void* k, const void* v,
                                           const void* o, const float* lse, const void* dO,
                                           void* dq, void* dk, void* dv, void* workspace,
                                           uint64_t workspace_bytes, int32_t B, int32_t H,
                                           int32_t H_kv, int32_t T, int32_t d, int32_t dtype,
                                           int32_t W, float scale, const fibattn_schedule* sched,
                                           int32_t layer0, int32_t n_layers_call,
                                           void* cuda_stream);

/*
 * Forward and backward of a layer stack in one call (a training step of the attention):
 * the call's Lc layers are split into min(n_streams, Lc) contiguous groups of sizes
 * differing by at most one, and group g runs fibattn_fwd_gqa then fibattn_bwd_gqa on its
 * layers on an internal stream of the library. The internal streams (non-blocking, created
 * once per device) are forked from cuda_stream by an event and joined back into it by
 * another, so the work is ordered after what cuda_stream holds and everything queued on
 * cuda_stream later waits for it; the pattern is also valid inside CUDA-graph capture.
 * Layers are independent problems, so the groups' kernels overlap on the GPU while every
 * output equals the sequential fibattn_fwd_gqa + fibattn_bwd_gqa calls bit for bit.
 *   q, k, v, dO : inputs as fibattn_bwd_gqa; o, lse : written (the forward's outputs);
 *   dq, dk, dv  : written. n_streams in [1, FIBATTN_STEP_STREAMS_MAX]; 1 runs both calls on
 *   cuda_stream itself.
 *   workspace   : 256-byte aligned, at least fibattn_fwd_bwd_workspace_size() bytes: each
 *                 group's backward workspace, 256-aligned, one after the other.
 * The first call with n_streams > 1 on a device creates that device's internal streams: make
 * it before any stream capture (creating a stream is not allowed while one is captured).
 * Calls on different host threads share the internal streams of a device (their work is
 * ordered, not raced). Errors: those of fibattn_fwd_gqa / fibattn_bwd_gqa, checked for every
 * group before anything is enqueued; INVALID_ARG for n_streams out of range or a short
 * workspace; CUDA for a failed stream or event call.
 */
#define FIBATTN_STEP_STREAMS_MAX 8
FIBATTN_API fibattn_status fibattn_fwd_bwd_workspace_size(int32_t B, int32_t H, int32_t T,
                                                          int32_t d, int32_t dtype, int32_t W,
                                                          const fibattn_schedule* sched,
                                                          int32_t layer0, int32_t n_layers_call,
                                                          int32_t n_streams, uint64_t* bytes);
FIBATTN_API fibattn_status fibattn_fwd_bwd(const void* q, const void* k, const void* v,
                                           const void* dO, void* o, float* lse, void* dq,
                                           void* dk, void* dv, void* workspace,
                                           uint64_t workspace_bytes, int32_t B, int32_t H,
                                           int32_t H_kv, int32_t T, int32_t d, int32_t dtype,
                                           int32_t W, float scale, const fibattn_schedule* sched,
                                           int32_t layer0, int32_t n_layers_call,
                                           int32_t n_streams, void* cuda_stream);

/*
 * Fractional-offset table of one real alpha: the learned-alpha variant of the pages
 * (Metodologia / Arquitetura, "Implementacao": keys and values are linearly interpolated
 * between rows so that the gradient reaches alpha when alpha * F is not an integer).
 * Real distances d = (double)alpha * F for the base values F of `base` / `base_max` (as in
 * fibattn_schedule), kept when W <= d <= T - 1, ascending. Entry n: ceil_out[n] = ceil(d),
 * w_out[n] = (float)(ceil(d) - d), the weight of the row after i - ceil(d) (0 for an
 * integer d). alpha: finite, 0 < alpha <= FIBATTN_RATIO_MAX.
 * Errors: INVALID_ARG (null with cap > 0, W < 1, T < 1, bad base, bad alpha), CAPACITY (more
 * than `cap` entries; *n_out then holds the needed count).
 */
FIBATTN_API fibattn_status fibattn_frac_offsets(float alpha, int32_t base, int64_t base_max,
                                                int32_t W, int32_t T, int32_t* ceil_out,
                                                float* w_out, int32_t cap, int32_t* n_out);

/*
 * Forward with fractional offsets (same page and passage): query i of call-layer c attends
 * its window i-W+1..i and, for every distance d of alphas[c]'s table (fibattn_frac_offsets)
 * with i >= d, the key and value interpolated at the real position i - d:
 *     x~ = (1 - w) x[i - ceil(d)] + w x[i - ceil(d) + 1],  w = ceil(d) - d,
 * with softmax over all of them. An integer alpha gives exactly the static forward's
 * attended set (fibattn_fwd with alpha num/1).
 *   alphas : host float [n_layers_call], read during the call.
 *   base, base_max : as in fibattn_schedule. Other arguments as fibattn_fwd.
 * bf16 runs on the tcgen05 forward kernel in its fractional mode; f32 on a SIMT kernel.
 * Errors: INVALID_ARG (also a bad alpha or base), UNSUPPORTED, CAPACITY (a table above
 * FIBATTN_MAX_OFFSETS), CUDA.
 */
FIBATTN_API fibattn_status fibattn_fwd_frac(const void* q, const void* k, const void* v, void* o,
                                            float* lse, int32_t B, int32_t H, int32_t T,
                                            int32_t d, int32_t dtype, int32_t W, float scale,
                                            int32_t base, int64_t base_max, const float* alphas,
                                            int32_t n_layers_call, void* cuda_stream);

/*
 * Workspace of fibattn_bwd_frac for one call, in bytes: the static backward's layout
 * (fibattn_bwd_workspace_size, with n_max = the largest fractional table of the call's
 * layers) followed, 256-byte aligned, by the per-query dalpha partials [Lc][B][H][T] float32.
 * Errors as fibattn_fwd_frac.
 */
FIBATTN_API fibattn_status fibattn_bwd_frac_workspace_size(int32_t B, int32_t H, int32_t T,
                                                           int32_t d, int32_t dtype, int32_t W,
                                                           int32_t base, int64_t base_max,
                                                           const float* alphas,
                                                           int32_t n_layers_call, uint64_t* bytes);

/*
 * Backward of fibattn_fwd_frac (same passage): the gradient reaches alpha through the
 * interpolation weights. With k~ = (1 - w) k[lo] + w k[lo + 1] (lo = i - ceil(d)), v~ likewise:
 *   P = exp(scale q_i.k~ - lse_i),  dS = P (dO_i.v~ - D_i),
 *   dq_i += scale dS k~,  dk[lo] += (1 - w) scale dS q_i,  dk[lo + 1] += w scale dS q_i,
 *   dv[lo] += (1 - w) P dO_i,  dv[lo + 1] += w P dO_i,
 *   dL/dd = sum_i dS scale q_i.(k[lo] - k[lo + 1]) + P dO_i.(v[lo] - v[lo + 1])
 *   (the derivative on the segment [lo, lo + 1]: for an integer d, that for d decreasing),
 *   dalpha[c] = sum_k F_k dL/dd_k over the distances of call-layer c, for the loss whose
 *   gradient with respect to o is dO.
 *   dq, dk, dv : written as in fibattn_bwd.
 *   dalpha     : float32 device [n_layers_call], written (4-byte aligned).
 *   workspace  : 256-byte aligned, at least fibattn_bwd_frac_workspace_size() bytes.
 *   Other arguments as fibattn_fwd_frac / fibattn_bwd. The per-layer sums run in a fixed
 *   order (deterministic). bf16 runs the tcgen05 backward kernels in their fractional mode;
 *   f32 runs SIMT kernels.
 * Errors as fibattn_fwd_frac, plus INVALID_ARG when workspace_bytes is too small.
 */
FIBATTN_API fibattn_status fibattn_bwd_frac(const void* q, const void* k, const void* v,
                                            const void* o, const float* lse, const void* dO,
                                            void* dq, void* dk, void* dv, float* dalpha,
                                            void* workspace, uint64_t workspace_bytes, int32_t B,
                                            int32_t H, int32_t T, int32_t d, int32_t dtype,
                                            int32_t W, float scale, int32_t base,
                                            int64_t base_max, const float* alphas,
                                            int32_t n_layers_call, void* cuda_stream);

/*
 * Workspace the backward needs for one call, in bytes (write it to *bytes). f32 calls:
 *   D [Lc][B][H][T] float32 (D_i = dO_i . o_i). bf16 calls, with rows padded to
 *   T_pad = T rounded up to a multiple of 4: D and lse * log2(e), each [Lc][B][H][T_pad]
 *   float32 and 256-byte aligned, then the (P, dS) pair (two bf16) of every (query, offset)
 *   diagonal entry, [Lc][B][H][n_max][T_pad] indexed by the key row, n_max = the largest
 *   table size among the call's layers at this (W, T).
 * Errors: INVALID_ARG, UNSUPPORTED and CAPACITY as fibattn_bwd (same checks).
 */
FIBATTN_API fibattn_status fibattn_bwd_workspace_size(int32_t B, int32_t H, int32_t T, int32_t d,
                                                      int32_t dtype, int32_t W,
                                                      const fibattn_schedule* sched,
                                                      int32_t layer0, int32_t n_layers_call,
                                                      uint64_t* bytes);

/*
 * Backward from the saved forward (the analytic gradient of softmax attention over S_i):
 *   D_i = dO_i . o_i,  P_ij = exp(scale q_i.k_j - lse_i),  dS_ij = P_ij (dO_i . v_j - D_i),
 *   dq_i = scale sum_j dS_ij k_j,  dk_j = scale sum_i dS_ij q_i,  dv_j = sum_i P_ij dO_i.
 *   q, k, v, o, dO : inputs as in fibattn_fwd; lse : the forward's lse.
 *   dq, dk, dv     : written (every element; no accumulation into old contents).
 *   workspace      : device scratch owned by the caller, 256-byte aligned, at least
 *                    fibattn_bwd_workspace_size() bytes (workspace_bytes says how many);
 *                    its contents on entry do not matter: the backward writes every value
 *                    it uses, and the few bytes it reads without writing (the pad rows of
 *                    D and lse * log2(e) past T, pairs of queries past T) are discarded by
 *                    selects, so stale or non-finite contents cannot reach the outputs.
 * bf16 runs two tcgen05 tensor-core kernels (query owner: D and dq; key owner: dk, dv);
 * f32 runs SIMT kernels. No atomics: each dq/dk/dv row is summed by the one thread block
 * that owns it.
 * Errors as fibattn_fwd, plus INVALID_ARG when workspace_bytes is too small.
 */
FIBATTN_API fibattn_status fibattn_bwd(const void* q, const void* k, const void* v, const void* o,
                           const float* lse, const void* dO, void* dq, void* dk, void* dv,
                           void* workspace, uint64_t workspace_bytes, int32_t B, int32_t H,
                           int32_t T, int32_t d, int32_t dtype, int32_t W, float scale,
                           const fibattn_schedule* sched, int32_t layer0, int32_t n_layers_call,
                           void* cuda_stream);

/*
 * The same backward in one pass over the tiles: a thread block per 128-row tile of a
 * (layer, batch, head) slice writes both dq of the tile's queries and dk, dv of its keys.
 * The key side forms each diagonal pair (key j, query j + o) again instead of reading it
 * from a workspace, so the only workspace is D and lse * log2(e) (written by a pre-pass).
 *   Arguments, layouts and results as fibattn_bwd; the outputs equal fibattn_bwd's bit
 *   for bit (each P and dS is formed from the same operands in the same order, and every
 *   sum is taken in the same order). No atomics.
 *   workspace : 256-byte aligned, at least 2 x 256-aligned [Lc][B][H][T_pad] float32
 *               (D, then lse * log2(e); T_pad = T rounded up to 4);
 *               fibattn_bwd_workspace_size() bytes always suffice. Contents on entry do
 *               not matter (the pre-pass writes every row, pad rows as 0).
 * Errors as fibattn_bwd; UNSUPPORTED unless dtype is FIBATTN_BF16 and d is 64.
 */
FIBATTN_API fibattn_status fibattn_bwd_fused(const void* q, const void* k, const void* v,
                                             const void* o, const float* lse, const void* dO,
                                             void* dq, void* dk, void* dv, void* workspace,
                                             uint64_t workspace_bytes, int32_t B, int32_t H,
                                             int32_t T, int32_t d, int32_t dtype, int32_t W,
                                             float scale, const fibattn_schedule* sched,
                                             int32_t layer0, int32_t n_layers_call,
                                             void* cuda_stream);

/*
 * fibattn_bwd for callers that cannot allocate device memory. The paper has no
 * counterpart: this is a deployment variant of the backward above, identical in
 * arguments, results and errors except that no workspace is passed.
 * Some callers cannot call cudaMalloc: an operator hosted by a framework that owns the
 * device allocator and hands it no workspace, or a latency-critical loop where
 * cudaMalloc/cudaFree would synchronise the device. This entry point takes the backward's
 * workspace from a fixed file-scope __device__ array of FIBATTN_NOALLOC_SCRATCH_BYTES
 * (40 MiB, held on every GPU that loads the library until the process exits) and
 * allocates nothing.
 *   - Calls whose fibattn_bwd_workspace_size() exceeds FIBATTN_NOALLOC_SCRATCH_BYTES
 *     return FIBATTN_ERR_SCRATCH_LIMIT without launching anything. The 16-layer
 *     B=8, H=8, T=1024, W=64 bf16 training step (32 MiB) fits.
 *   - The first call on a device (that device current) looks up the array's device
 *     address with cudaGetSymbolAddress; make that first call before any stream capture.
 *   - All calls on a device share the array and it keeps the last call's contents. Nothing
 *     needs clearing: the backward writes every value it uses, and what it reads without
 *     writing (pad rows past T, pairs of queries past T) is discarded by selects, so an
 *     earlier call's contents, even non-finite ones, cannot reach the outputs. Calls whose
 *     kernels can overlap on the GPU (unordered streams) race on it.
 */
#define FIBATTN_NOALLOC_SCRATCH_BYTES (40ull << 20)
FIBATTN_API fibattn_status fibattn_bwd_noalloc(const void* q, const void* k, const void* v,
                                               const void* o, const float* lse, const void* dO,
                                               void* dq, void* dk, void* dv, int32_t B, int32_t H,
                                               int32_t T, int32_t d, int32_t dtype, int32_t W,
                                               float scale, const fibattn_schedule* sched,
                                               int32_t layer0, int32_t n_layers_call,
                                               void* cuda_stream);

/*
 * The attended key sets of one layer, materialised by a device kernel from the same
 * table and predicate the attention kernels use: d_mask is a device uint32
 * [T][ceil(T/32)] bitmask, bit (j % 32) of word [i][j / 32] set iff j is in S_i.
 * For testing only (O(T^2) memory). Errors as fibattn_offsets, plus CUDA.
 */
FIBATTN_API fibattn_status fibattn_keyset_debug(const fibattn_schedule* sched, int32_t layer, int32_t W,
                                    int32_t T, uint32_t* d_mask, void* cuda_stream);

/*
 * Rotary position embedding, applied to q and k before the attention (Metodologia /
 * Arquitetura, "Implementacao": RoPE is applied before the gather; Significancia: vanilla
 * RoPE without scaling). Row i, pair (2p, 2p+1) is rotated by the angle i * theta_p,
 * theta_p = base^(-2p/d).
 * fibattn_rope_table: writes table, float32 device [T][d/2][2] (cos, sin of i * theta_p,
 *   computed in fp64 and rounded once), 16-byte aligned, caller-owned; build it once per
 *   (T, base) and pass it to every fibattn_rope call. base > 1 (10000 is the usual value).
 * fibattn_rope: y = x rotated, x and y [slices][T][d] of dtype `dtype` (row r of a slice at
 *   position r); inverse != 0 rotates by the opposite angles (R^T: it carries dq and dk back
 *   through the rotation, and undoes it). x == y (in place) is allowed; a partial overlap is
 *   INVALID_ARG. table_rows (>= T) is the number of rows the table was built with.
 * fibattn_fwd_rope: the forward with RoPE before the gather, in one call: q and k rotated into
 *   the caller's q_rot ([Lc][B][H][T][d]) and k_rot ([Lc][B][H_kv][T][d]) by fibattn_rope,
 *   then fibattn_fwd_gqa on them. Keep q_rot and k_rot for the backward.
 * fibattn_bwd_rope: the backward through RoPE from the forward's q_rot and k_rot: the
 *   attention backward of fibattn_bwd_gqa, then dq and dk rotated back in place (R^T,
 *   fibattn_rope), so they are the gradients of the unrotated q and k. Workspace as
 *   fibattn_bwd_workspace_size.
 * Errors: INVALID_ARG (null or misaligned pointers, sizes, base, a table shorter than T),
 * UNSUPPORTED (d != 64, dtype), and those of the attention calls; CUDA.
 */
FIBATTN_API fibattn_status fibattn_rope_table(float* table, int32_t T, int32_t d, double base,
                                              void* cuda_stream);
FIBATTN_API fibattn_status fibattn_rope(const void* x, void* y, int64_t slices, int32_t T,
                                        int32_t d, int32_t dtype, const float* table,
                                        int32_t table_rows, int32_t inverse, void* cuda_stream);
FIBATTN_API fibattn_status fibattn_fwd_rope(const void* q, const void* k, const void* v,
                                            void* q_rot, void* k_rot, void* o, float* lse,
                                            int32_t B, int32_t H, int32_t H_kv, int32_t T,
                                            int32_t d, int32_t dtype, int32_t W, float scale,
                                            const fibattn_schedule* sched, int32_t layer0,
                                            int32_t n_layers_call, const float* rope_table,
                                            int32_t table_rows, void* cuda_stream);
/*
 * The forward with RoPE applied inside the attention kernel (same passages as
 * fibattn_fwd_rope): q and k are read unrotated and no rotated copy is written. The band's
 * Q and K tiles are rotated in shared memory (the standalone rotation's arithmetic and bf16
 * rounding). Each offset's score is taken as (R_o q_i) . k_(i-o), equal to the rotated
 * tensors' score since rotations compose, with the angle o theta_p of table row o. Results
 * agree with fibattn_fwd_rope to rounding; o and lse as fibattn_fwd.
 * For callers without room or use for the rotated copies: a forward-only (inference) pass
 * that keeps no q_rot/k_rot buffers, 2 x [Lc][B][H(_kv)][T][d] bf16 less memory. Training keeps
 * fibattn_fwd_rope, whose rotated tensors the backward needs.
 * bf16, d = 64 (others: UNSUPPORTED). Other arguments and errors as fibattn_fwd_rope.
 */
FIBATTN_API fibattn_status fibattn_fwd_rope_fused(const void* q, const void* k, const void* v,
                                                  void* o, float* lse, int32_t B, int32_t H,
                                                  int32_t H_kv, int32_t T, int32_t d,
                                                  int32_t dtype, int32_t W, float scale,
                                                  const fibattn_schedule* sched, int32_t layer0,
                                                  int32_t n_layers_call, const float* rope_table,
                                                  int32_t table_rows, void* cuda_stream);
FIBATTN_API fibattn_status fibattn_bwd_rope(const void* q_rot, const void* k_rot, const void* v,
                                            const void* o, const float* lse, const void* dO,
                                            void* dq, void* dk, void* dv, void* workspace,
                                            uint64_t workspace_bytes, int32_t B, int32_t H,
                                            int32_t H_kv, int32_t T, int32_t d, int32_t dtype,
                                            int32_t W, float scale, const fibattn_schedule* sched,
                                            int32_t layer0, int32_t n_layers_call,
                                            const float* rope_table, int32_t table_rows,
                                            void* cuda_stream);

/*
 * Synchronises `cuda_stream`, then reads and clears the device error word.
 * Returns OK, TIMEOUT (a kernel gave up a bounded wait and returned early; its
 * outputs are undefined) or CUDA (a CUDA error is pending on the context).
 */
FIBATTN_API fibattn_status fibattn_poll_device_error(void* cuda_stream);

/*
 * A check of the failure path, for tests: launches one small kernel whose thread waits, with
 * the bounded wait every attention kernel uses (limit_ms, 1..10000), on an mbarrier that
 * nothing arrives on. The wait runs out, the kernel latches the device error word and
 * returns; fibattn_poll_device_error then reports TIMEOUT once (and clears it), and the
 * context stays usable. No fault, trap or hang is involved. Errors: INVALID_ARG, CUDA.
 */
FIBATTN_API fibattn_status fibattn_debug_wait_timeout(int32_t limit_ms, void* cuda_stream);

/* Static English text for a status value (never NULL). */
FIBATTN_API const char* fibattn_status_string(fibattn_status status);

/*
 * Kernel timing without a profiler. While enabled (on != 0), every kernel the library
 * launches is bracketed by a pair of CUDA events recorded on the launch stream (the
 * events are created and pooled by the library; no device memory is allocated).
 * fibattn_profile_read synchronises the recorded events and, per kernel name, writes
 * the summed device milliseconds and the number of launches since the previous read,
 * then resets them. names is a char [cap][name_len] buffer (NUL-terminated names).
 * Returns the number of kernel names known (may exceed cap).
 */
FIBATTN_API fibattn_status fibattn_profile_enable(int32_t on);
FIBATTN_API int32_t fibattn_profile_read(char* names, int32_t name_len, double* total_ms,
                                         int64_t* launches, int32_t cap);

/*
 * The cudaError_t value behind the most recent FIBATTN_ERR_CUDA returned by any call in
 * the process (0 if none yet), and in *where (if not NULL) a static text naming the
 * CUDA call that failed (-1 for a tensor-map encoding the driver rejected).
 */
FIBATTN_API int32_t fibattn_last_cuda_error(const char** where);

/* Kernels launched by the library since it was loaded (always counted). */
FIBATTN_API int64_t fibattn_launch_count(void);

/* Library version, major * 10000 + minor * 100 + patch. */
FIBATTN_API int32_t fibattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FIBATTN_H */
