// api.cu -- the extern "C" entry points declared in include/fibattn.h: argument
// validation, offset-table construction, and dispatch to the kernels.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <initializer_list>

#include "internal.h"

using namespace fibattn;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A buffer of a call: its first byte and its length in bytes.
struct Span {
    const void* p;
    uint64_t n;
};

bool spans_overlap(Span a, Span b) {
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a.p), pb = reinterpret_cast<uintptr_t>(b.p);
    return a.n > 0 && b.n > 0 && pa < pb + b.n && pb < pa + a.n;
}

// True when an output overlaps another output or an input. Inputs may share memory (k == v):
// they are only read.
bool outputs_overlap(std::initializer_list<Span> outs, std::initializer_list<Span> ins) {
    for (const Span* a = outs.begin(); a != outs.end(); ++a) {
        for (const Span* b = a + 1; b != outs.end(); ++b)
            if (spans_overlap(*a, *b)) return true;
        for (const Span& b : ins)
            if (spans_overlap(*a, b)) return true;
    }
    return false;
}

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Shared checks of fibattn_fwd / fibattn_bwd.
fibattn_status check_common(int32_t B, int32_t H, int32_t T, int32_t d, int32_t dtype, int32_t W,
                            const fibattn_schedule* sched, int32_t layer0, int32_t n_layers_call) {
    if (!sched) return FIBATTN_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || T < 1 || T > FIBATTN_T_MAX || W < 1 || n_layers_call < 1 || layer0 < 0)
        return FIBATTN_ERR_INVALID_ARG;
    if (sched->n_layers < 1 || (int64_t)layer0 + n_layers_call > sched->n_layers)
        return FIBATTN_ERR_INVALID_ARG;
    if (dtype != FIBATTN_F32 && dtype != FIBATTN_BF16) return FIBATTN_ERR_UNSUPPORTED;
    if (d != 64 && d != 128) return FIBATTN_ERR_UNSUPPORTED;
    // rows of one launch layer must index within int32 grids and int64 offsets
    const int64_t rows = (int64_t)B * H * T;
    if (rows > ((int64_t)1 << 34)) return FIBATTN_ERR_INVALID_ARG;
    if (rows * (int64_t)n_layers_call > ((int64_t)1 << 40)) return FIBATTN_ERR_INVALID_ARG;
    // validate every layer's schedule and table size before launching anything
    for (int32_t c = 0; c < n_layers_call; c += kMaxLayersPerLaunch) {
        int32_t n = n_layers_call - c < kMaxLayersPerLaunch ? n_layers_call - c : kMaxLayersPerLaunch;
        OffsetTables t;
        fibattn_status st = build_launch_tables(sched, layer0 + c, n, W, T, &t);
        if (st != FIBATTN_OK) return st;
    }
    return FIBATTN_OK;
}

size_t elt_size(int32_t dtype) { return dtype == FIBATTN_F32 ? 4 : 2; }

// The softmax scale: <= 0 or NaN selects 1/sqrt(d); +inf is refused (every score would be
// infinite).
bool resolve_scale(float& scale, int32_t d) {
    if (scale == INFINITY) return false;
    if (!(scale > 0.f)) scale = 1.0f / sqrtf((float)d);
    return true;
}

// Layout of the backward workspace. f32 path: D [rows] (rows of T). bf16 path: rows padded to
// T_pad = T rounded up to 4 (16-byte rows for bulk copies): D [rows_pad], lse*log2(e)
// [rows_pad], then the (P, dS) pairs [slices][n_max][T_pad]; each array starts 256-aligned.
struct BwdWorkspace {
    uint64_t lse2_offset;    // bytes
    uint64_t pds_offset;     // bytes
    uint64_t galpha_offset;  // bytes (fractional backward only)
    uint64_t total;          // bytes
    int32_t n_max;           // table entries per layer slot of the pairs array
    int32_t T_pad;
};

uint64_t align256(uint64_t x) { return (x + 255) & ~(uint64_t)255; }

// The layout for a given n_max; `frac` appends the per-query dalpha partials [rows].
BwdWorkspace workspace_layout(int32_t B, int32_t H, int32_t T, int32_t dtype, int32_t n_layers_call,
                              int32_t n_max, bool frac) {
    BwdWorkspace ws;
    const uint64_t rows = (uint64_t)n_layers_call * B * H * T;
    if (dtype != FIBATTN_BF16) {
        ws.lse2_offset = ws.pds_offset = 0;
        ws.galpha_offset = align256(rows * 4);
        ws.total = frac ? ws.galpha_offset + rows * 4 : rows * 4;
        ws.n_max = 0;
        ws.T_pad = T;
        return ws;
    }
    ws.T_pad = (T + 3) & ~3;
    const uint64_t rows_pad = (uint64_t)n_layers_call * B * H * ws.T_pad;
    ws.n_max = n_max;
    ws.lse2_offset = align256(rows_pad * 4);
    ws.pds_offset = ws.lse2_offset + align256(rows_pad * 4);
    ws.galpha_offset = align256(ws.pds_offset + rows_pad * (uint64_t)n_max * 4);
    ws.total = frac ? ws.galpha_offset + rows * 4 : ws.pds_offset + rows_pad * (uint64_t)n_max * 4;
    return ws;
}

// Callers have validated the arguments (check_common), so every table builds. The tensor-core
// layout is bf16 (d = 64 or 128); fp32 runs the SIMT backward (D only).
BwdWorkspace bwd_workspace(int32_t B, int32_t H, int32_t T, int32_t d, int32_t dtype, int32_t W,
                           const fibattn_schedule* sched, int32_t layer0, int32_t n_layers_call) {
    (void)d;
    if (dtype != FIBATTN_BF16)
        return workspace_layout(B, H, T, FIBATTN_F32, n_layers_call, 0, false);
    int32_t n_max = 0;
    for (int32_t c = 0; c < n_layers_call; ++c) {
        Alpha a;
        int32_t n = 0;
        if (layer_alpha(sched, layer0 + c, &a) == FIBATTN_OK &&
            build_table(sched, a, W, T, nullptr, 0, &n) != FIBATTN_ERR_INVALID_ARG)
            n_max = n > n_max ? n : n_max;
    }
    return workspace_layout(B, H, T, dtype, n_layers_call, n_max, false);
}

// Checks shared by the fractional-offset entry points (every layer's table validated).
fibattn_status check_frac(int32_t B, int32_t H, int32_t T, int32_t d, int32_t dtype, int32_t W,
                          int32_t base, int64_t base_max, const float* alphas,
                          int32_t n_layers_call, int32_t* n_max) {
    if (!alphas) return FIBATTN_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || T < 1 || T > FIBATTN_T_MAX || W < 1 || n_layers_call < 1 ||
        n_layers_call > FIBATTN_LAYERS_MAX)
        return FIBATTN_ERR_INVALID_ARG;
    if (dtype != FIBATTN_F32 && dtype != FIBATTN_BF16) return FIBATTN_ERR_UNSUPPORTED;
    if (d != 64) return FIBATTN_ERR_UNSUPPORTED;
    const int64_t per_layer = (int64_t)B * H * T;
    if (per_layer > ((int64_t)1 << 34) || per_layer * n_layers_call > ((int64_t)1 << 40))
        return FIBATTN_ERR_INVALID_ARG;
    int32_t m = 0;
    for (int32_t c = 0; c < n_layers_call; ++c) {
        int32_t n = 0;
        fibattn_status st =
            build_frac_table(base, base_max, alphas[c], W, T, nullptr, nullptr, nullptr, 0, &n);
        if (st == FIBATTN_ERR_INVALID_ARG) return st;
        if (n > kMaxOffsets) return FIBATTN_ERR_CAPACITY;
        m = n > m ? n : m;
    }
    if (n_max) *n_max = m;
    return FIBATTN_OK;
}

}  // namespace

extern "C" {

int32_t fibattn_version(void) { return 100; }

const char* fibattn_status_string(fibattn_status s) {
    switch (s) {
        case FIBATTN_OK: return "ok";
        case FIBATTN_ERR_INVALID_ARG: return "invalid argument";
        case FIBATTN_ERR_UNSUPPORTED: return "unsupported configuration";
        case FIBATTN_ERR_CAPACITY: return "offset table exceeds capacity";
        case FIBATTN_ERR_CUDA: return "CUDA error";
        case FIBATTN_ERR_TIMEOUT: return "kernel wait timed out";
        case FIBATTN_ERR_SCRATCH_LIMIT: return "call exceeds the fixed no-allocation scratch size";
    }
    return "unknown status";
}

fibattn_status fibattn_offsets(const fibattn_schedule* sched, int32_t layer, int32_t W, int32_t T,
                               int32_t* out, int32_t cap, int32_t* n_out) {
    if (!sched || !n_out || (cap > 0 && !out) || cap < 0) return FIBATTN_ERR_INVALID_ARG;
    if (W < 1 || T < 1) return FIBATTN_ERR_INVALID_ARG;
    Alpha a;
    fibattn_status st = layer_alpha(sched, layer, &a);
    if (st != FIBATTN_OK) return st;
    return build_table(sched, a, W, T, out, cap, n_out);
}

fibattn_status fibattn_offsets_device(const fibattn_schedule* sched, int32_t layer0,
                                      int32_t n_layers_call, int32_t W, int32_t T,
                                      int32_t* d_tables, int32_t* d_counts, void* cuda_stream) {
    if (!sched || !d_tables || !d_counts || n_layers_call < 1 || layer0 < 0)
        return FIBATTN_ERR_INVALID_ARG;
    if (W < 1 || T < 1 || T > FIBATTN_T_MAX) return FIBATTN_ERR_INVALID_ARG;
    if ((int64_t)layer0 + n_layers_call > sched->n_layers) return FIBATTN_ERR_INVALID_ARG;
    for (int32_t c = 0; c < n_layers_call; ++c) {  // same validation and capacity as the host
        Alpha a;
        fibattn_status st = layer_alpha(sched, layer0 + c, &a);
        if (st != FIBATTN_OK) return st;
        int32_t tmp[kMaxOffsets], n = 0;
        st = build_table(sched, a, W, T, tmp, kMaxOffsets, &n);
        if (st != FIBATTN_OK) return st;
    }
    return launch_offsets_device(sched, layer0, n_layers_call, W, T, d_tables, d_counts,
                                 as_stream(cuda_stream));
}

fibattn_status fibattn_keyset_debug(const fibattn_schedule* sched, int32_t layer, int32_t W,
                                    int32_t T, uint32_t* d_mask, void* cuda_stream) {
    if (!sched || !d_mask) return FIBATTN_ERR_INVALID_ARG;
    if (W < 1 || T < 1 || T > FIBATTN_T_MAX) return FIBATTN_ERR_INVALID_ARG;
    OffsetTables t;
    fibattn_status st = build_launch_tables(sched, layer, 1, W, T, &t);
    if (st != FIBATTN_OK) return st;
    return launch_keyset(t, W, T, d_mask, as_stream(cuda_stream));
}

fibattn_status fibattn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                               int32_t B, int32_t H, int32_t H_kv, int32_t T, int32_t d,
                               int32_t dtype, int32_t W, float scale, const fibattn_schedule* sched,
                               int32_t layer0, int32_t n_layers_call, void* cuda_stream) {
    if (!q || !k || !v || !o || !lse) return FIBATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FIBATTN_ERR_INVALID_ARG;
    if (H_kv < 1 || H < 1 || H % H_kv != 0) return FIBATTN_ERR_INVALID_ARG;
    fibattn_status st = check_common(B, H, T, d, dtype, W, sched, layer0, n_layers_call);
    if (st != FIBATTN_OK) return st;
    if (!resolve_scale(scale, d)) return FIBATTN_ERR_INVALID_ARG;
    const int64_t per_layer = (int64_t)B * H * T;
    const int64_t per_layer_kv = (int64_t)B * H_kv * T;
    const size_t es = elt_size(dtype);
    const uint64_t qb = (uint64_t)n_layers_call * per_layer * d * es;
    const uint64_t kb = (uint64_t)n_layers_call * per_layer_kv * d * es;
    const uint64_t lb = (uint64_t)n_layers_call * per_layer * 4;
    if (outputs_overlap({{o, qb}, {lse, lb}}, {{q, qb}, {k, kb}, {v, kb}}))
        return FIBATTN_ERR_INVALID_ARG;
    for (int32_t c = 0; c < n_layers_call; c += kMaxLayersPerLaunch) {
        const int32_t n = n_layers_call - c < kMaxLayersPerLaunch ? n_layers_call - c : kMaxLayersPerLaunch;
        OffsetTables t;
        st = build_launch_tables(sched, layer0 + c, n, W, T, &t);
        if (st != FIBATTN_OK) return st;
        AttnShape sh{(int64_t)B * H, T, W < T ? W : T, scale, n, H / H_kv, d};
        const size_t off = (size_t)c * per_layer * d * es;
        const size_t koff = (size_t)c * per_layer_kv * d * es;
        const char* qc = (const char*)q + off;
        const char* kc = (const char*)k + koff;
        const char* vc = (const char*)v + koff;
        char* oc = (char*)o + off;
        float* lc = lse + (size_t)c * per_layer;
        if (dtype == FIBATTN_F32)
            st = launch_fwd_simt_f32((const float*)qc, (const float*)kc, (const float*)vc,
                                     (float*)oc, lc, sh, t, as_stream(cuda_stream));
        else if (d == 64 && W >= T)  // every earlier key: dense causal attention
            st = launch_fwd_dense_tc_bf16(qc, kc, vc, oc, lc, sh, as_stream(cuda_stream));
        else if (d == 64)
            st = launch_fwd_tc_bf16(qc, kc, vc, oc, lc, sh, t, as_stream(cuda_stream));
        else
            st = launch_fwd_tc128_bf16(qc, kc, vc, oc, lc, sh, t, as_stream(cuda_stream));
        if (st != FIBATTN_OK) return st;
    }
    return FIBATTN_OK;
}

fibattn_status fibattn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                           int32_t B, int32_t H, int32_t T, int32_t d, int32_t dtype, int32_t W,
                           float scale, const fibattn_schedule* sched, int32_t layer0,
                           int32_t n_layers_call, void* cuda_stream) {
    return fibattn_fwd_gqa(q, k, v, o, lse, B, H, H, T, d, dtype, W, scale, sched, layer0,
                           n_layers_call, cuda_stream);
}

fibattn_status fibattn_frac_offsets(float alpha, int32_t base, int64_t base_max, int32_t W,
                                    int32_t T, int32_t* ceil_out, float* w_out, int32_t cap,
                                    int32_t* n_out) {
    if (!n_out || cap < 0 || (cap > 0 && (!ceil_out || !w_out))) return FIBATTN_ERR_INVALID_ARG;
    return build_frac_table(base, base_max, alpha, W, T, ceil_out, w_out, nullptr, cap, n_out);
}

fibattn_status fibattn_fwd_frac(const void* q, const void* k, const void* v, void* o, float* lse,
                                int32_t B, int32_t H, int32_t T, int32_t d, int32_t dtype,
                                int32_t W, float scale, int32_t base, int64_t base_max,
                                const float* alphas, int32_t n_layers_call, void* cuda_stream) {
    if (!q || !k || !v || !o || !lse || !alphas) return FIBATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FIBATTN_ERR_INVALID_ARG;
    // every layer's table is validated before anything is launched
    fibattn_status st0 = check_frac(B, H, T, d, dtype, W, base, base_max, alphas, n_layers_call, nullptr);
    if (st0 != FIBATTN_OK) return st0;
    const int64_t per_layer = (int64_t)B * H * T;
    if (!resolve_scale(scale, d)) return FIBATTN_ERR_INVALID_ARG;
    const size_t es = elt_size(dtype);
    const uint64_t qb = (uint64_t)n_layers_call * per_layer * d * es;
    if (outputs_overlap({{o, qb}, {lse, (uint64_t)n_layers_call * per_layer * 4}},
                        {{q, qb}, {k, qb}, {v, qb}}))
        return FIBATTN_ERR_INVALID_ARG;
    for (int32_t c = 0; c < n_layers_call; c += kMaxLayersPerLaunch) {
        const int32_t n = n_layers_call - c < kMaxLayersPerLaunch ? n_layers_call - c : kMaxLayersPerLaunch;
        FracTables t;
        fibattn_status st = build_frac_launch_tables(base, base_max, alphas + c, n, W, T, &t);
        if (st != FIBATTN_OK) return st;
        AttnShape sh{(int64_t)B * H, T, W < T ? W : T, scale, n};
        const size_t off = (size_t)c * per_layer * d * es;
        const char* qc = (const char*)q + off;
        const char* kc = (const char*)k + off;
        const char* vc = (const char*)v + off;
        char* oc = (char*)o + off;
        float* lc = lse + (size_t)c * per_layer;
        if (dtype == FIBATTN_F32)
            st = launch_fwd_frac_simt_f32((const float*)qc, (const float*)kc, (const float*)vc,
                                          (float*)oc, lc, sh, t, as_stream(cuda_stream));
        else
            st = launch_fwd_frac_tc_bf16(qc, kc, vc, oc, lc, sh, t, as_stream(cuda_stream));
        if (st != FIBATTN_OK) return st;
    }
    return FIBATTN_OK;
}

fibattn_status fibattn_bwd_workspace_size(int32_t B, int32_t H, int32_t T, int32_t d,
                                          int32_t dtype, int32_t W, const fibattn_schedule* sched,
                                          int32_t layer0, int32_t n_layers_call, uint64_t* bytes) {
    if (!bytes) return FIBATTN_ERR_INVALID_ARG;
    fibattn_status st = check_common(B, H, T, d, dtype, W, sched, layer0, n_layers_call);
    if (st != FIBATTN_OK) return st;
    const BwdWorkspace ws = bwd_workspace(B, H, T, d, dtype, W, sched, layer0, n_layers_call);
    *bytes = ws.total;
    return FIBATTN_OK;
}

namespace {

// The backward of fibattn_bwd_gqa / fibattn_bwd_rope (rope: the RoPE table or null).
fibattn_status bwd_common(const void* q, const void* k, const void* v, const void* o,
                          const float* lse, const void* dO, void* dq, void* dk, void* dv,
                          void* workspace, uint64_t workspace_bytes, int32_t B, int32_t H,
                          int32_t H_kv, int32_t T, int32_t d, int32_t dtype, int32_t W,
                          float scale, const fibattn_schedule* sched, int32_t layer0,
                          int32_t n_layers_call, void* cuda_stream) {
    const void* ptrs[] = {q, k, v, o, lse, dO, dq, dk, dv};
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return FIBATTN_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return FIBATTN_ERR_INVALID_ARG;
    if (H_kv < 1 || H < 1 || H % H_kv != 0) return FIBATTN_ERR_INVALID_ARG;
    fibattn_status st = check_common(B, H, T, d, dtype, W, sched, layer0, n_layers_call);
    if (st != FIBATTN_OK) return st;
    const BwdWorkspace ws = bwd_workspace(B, H, T, d, dtype, W, sched, layer0, n_layers_call);
    if (workspace_bytes < ws.total) return FIBATTN_ERR_INVALID_ARG;
    float* delta = static_cast<float*>(workspace);
    float* lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + ws.lse2_offset);
    uint32_t* pds = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + ws.pds_offset);
    const int64_t per_layer_pad = (int64_t)B * H * ws.T_pad;
    if (!resolve_scale(scale, d)) return FIBATTN_ERR_INVALID_ARG;
    const int64_t per_layer = (int64_t)B * H * T;
    const int64_t per_layer_kv = (int64_t)B * H_kv * T;
    const size_t es = elt_size(dtype);
    {
        const uint64_t qb = (uint64_t)n_layers_call * per_layer * d * es;
        const uint64_t kb = (uint64_t)n_layers_call * per_layer_kv * d * es;
        const uint64_t lb = (uint64_t)n_layers_call * per_layer * 4;
        if (outputs_overlap({{dq, qb}, {dk, kb}, {dv, kb}, {workspace, ws.total}},
                            {{q, qb}, {k, kb}, {v, kb}, {o, qb}, {lse, lb}, {dO, qb}}))
            return FIBATTN_ERR_INVALID_ARG;
    }
    for (int32_t c = 0; c < n_layers_call; c += kMaxLayersPerLaunch) {
        const int32_t n = n_layers_call - c < kMaxLayersPerLaunch ? n_layers_call - c : kMaxLayersPerLaunch;
        OffsetTables t;
        st = build_launch_tables(sched, layer0 + c, n, W, T, &t);
        if (st != FIBATTN_OK) return st;
        AttnShape sh{(int64_t)B * H, T, W < T ? W : T, scale, n, H / H_kv, d};
        const size_t off = (size_t)c * per_layer * d * es;
        const size_t koff = (size_t)c * per_layer_kv * d * es;
        const size_t loff = (size_t)c * per_layer;
        if (dtype == FIBATTN_F32) {
            st = launch_bwd_simt_f32((const float*)((const char*)q + off),
                                     (const float*)((const char*)k + koff),
                                     (const float*)((const char*)v + koff),
                                     (const float*)((const char*)o + off), lse + loff,
                                     (const float*)((const char*)dO + off),
                                     (float*)((char*)dq + off), (float*)((char*)dk + koff),
                                     (float*)((char*)dv + koff), delta + loff, sh, t,
                                     as_stream(cuda_stream));
        } else {
            const size_t poff = (size_t)c * per_layer_pad;
            st = launch_bwd_tc_bf16((const char*)q + off, (const char*)k + koff,
                                    (const char*)v + koff, (const char*)o + off, lse + loff,
                                    (const char*)dO + off, (char*)dq + off, (char*)dk + koff,
                                    (char*)dv + koff, delta + poff, lse2 + poff,
                                    pds + poff * ws.n_max, ws.n_max, sh, t,
                                    as_stream(cuda_stream));
        }
        if (st != FIBATTN_OK) return st;
    }
    return FIBATTN_OK;
}

}  // namespace

fibattn_status fibattn_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                               const float* lse, const void* dO, void* dq, void* dk, void* dv,
                               void* workspace, uint64_t workspace_bytes, int32_t B, int32_t H,
                               int32_t H_kv, int32_t T, int32_t d, int32_t dtype, int32_t W,
                               float scale, const fibattn_schedule* sched, int32_t layer0,
                               int32_t n_layers_call, void* cuda_stream) {
    return bwd_common(q, k, v, o, lse, dO, dq, dk, dv, workspace, workspace_bytes, B, H, H_kv, T,
                      d, dtype, W, scale, sched, layer0, n_layers_call, cuda_stream);
}

fibattn_status fibattn_bwd_rope(const void* q_rot, const void* k_rot, const void* v,
                                const void* o, const float* lse, const void* dO, void* dq,
                                void* dk, void* dv, void* workspace, uint64_t workspace_bytes,
                                int32_t B, int32_t H, int32_t H_kv, int32_t T, int32_t d,
                                int32_t dtype, int32_t W, float scale,
                                const fibattn_schedule* sched, int32_t layer0,
                                int32_t n_layers_call, const float* rope_table,
                                int32_t table_rows, void* cuda_stream) {
    if (!rope_table || !aligned16(rope_table) || table_rows < T) return FIBATTN_ERR_INVALID_ARG;
    if (d != 64) return FIBATTN_ERR_UNSUPPORTED;  // the rotation kernel's rows are 64 wide
    fibattn_status st = bwd_common(q_rot, k_rot, v, o, lse, dO, dq, dk, dv, workspace,
                                   workspace_bytes, B, H, H_kv, T, d, dtype, W, scale, sched,
                                   layer0, n_layers_call, cuda_stream);
    if (st != FIBATTN_OK) return st;
    // dq and dk of the rotated q and k, rotated back in place: the gradients of q and k
    st = fibattn_rope(dq, dq, (int64_t)n_layers_call * B * H, T, d, dtype, rope_table, table_rows,
                      1, cuda_stream);
    if (st != FIBATTN_OK) return st;
    return fibattn_rope(dk, dk, (int64_t)n_layers_call * B * H_kv, T, d, dtype, rope_table,
                        table_rows, 1, cuda_stream);
}

fibattn_status fibattn_fwd_rope_fused(const void* q, const void* k, const void* v, void* o,
                                      float* lse, int32_t B, int32_t H, int32_t H_kv, int32_t T,
                                      int32_t d, int32_t dtype, int32_t W, float scale,
                                      const fibattn_schedule* sched, int32_t layer0,
                                      int32_t n_layers_call, const float* rope_table,
                                      int32_t table_rows, void* cuda_stream) {
    if (!rope_table || !aligned16(rope_table) || table_rows < T) return FIBATTN_ERR_INVALID_ARG;
    if (!q || !k || !v || !o || !lse) return FIBATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FIBATTN_ERR_INVALID_ARG;
    if (H_kv < 1 || H < 1 || H % H_kv != 0) return FIBATTN_ERR_INVALID_ARG;
    fibattn_status st = check_common(B, H, T, d, dtype, W, sched, layer0, n_layers_call);
    if (st != FIBATTN_OK) return st;
    if (dtype != FIBATTN_BF16 || d != 64) return FIBATTN_ERR_UNSUPPORTED;
    if (!resolve_scale(scale, d)) return FIBATTN_ERR_INVALID_ARG;
    const int64_t per_layer = (int64_t)B * H * T;
    const int64_t per_layer_kv = (int64_t)B * H_kv * T;
    const size_t es = elt_size(dtype);
    {
        const uint64_t qb = (uint64_t)n_layers_call * per_layer * d * es;
        const uint64_t kb = (uint64_t)n_layers_call * per_layer_kv * d * es;
        if (outputs_overlap({{o, qb}, {lse, (uint64_t)n_layers_call * per_layer * 4}},
                            {{q, qb}, {k, kb}, {v, kb}, {rope_table, (uint64_t)table_rows * 256}}))
            return FIBATTN_ERR_INVALID_ARG;
    }
    for (int32_t c = 0; c < n_layers_call; c += kMaxLayersPerLaunch) {
        const int32_t n = n_layers_call - c < kMaxLayersPerLaunch ? n_layers_call - c : kMaxLayersPerLaunch;
        OffsetTables t;
        st = build_launch_tables(sched, layer0 + c, n, W, T, &t);
        if (st != FIBATTN_OK) return st;
        AttnShape sh{(int64_t)B * H, T, W < T ? W : T, scale, n, H / H_kv, d};
        const size_t off = (size_t)c * per_layer * d * es;
        const size_t koff = (size_t)c * per_layer_kv * d * es;
        st = launch_fwd_rope_tc_bf16((const char*)q + off, (const char*)k + koff,
                                     (const char*)v + koff, (char*)o + off,
                                     lse + (size_t)c * per_layer, sh, t, rope_table,
                                     as_stream(cuda_stream));
        if (st != FIBATTN_OK) return st;
    }
    return FIBATTN_OK;
}

fibattn_status fibattn_fwd_rope(const void* q, const void* k, const void* v, void* q_rot,
                                void* k_rot, void* o, float* lse, int32_t B, int32_t H,
                                int32_t H_kv, int32_t T, int32_t d, int32_t dtype, int32_t W,
                                float scale, const fibattn_schedule* sched, int32_t layer0,
                                int32_t n_layers_call, const float* rope_table,
                                int32_t table_rows, void* cuda_stream) {
    if (!rope_table || !aligned16(rope_table) || table_rows < T) return FIBATTN_ERR_INVALID_ARG;
    if (d != 64) return FIBATTN_ERR_UNSUPPORTED;  // the rotation kernel's rows are 64 wide
    if (!q || !k || !q_rot || !k_rot || !aligned16(q) || !aligned16(k) || !aligned16(q_rot) ||
        !aligned16(k_rot))
        return FIBATTN_ERR_INVALID_ARG;
    if (H_kv < 1 || H < 1 || H % H_kv != 0) return FIBATTN_ERR_INVALID_ARG;
    // every argument of the attention is checked before the first rotation is launched
    fibattn_status st = check_common(B, H, T, d, dtype, W, sched, layer0, n_layers_call);
    if (st != FIBATTN_OK) return st;
    if (!v || !o || !lse || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FIBATTN_ERR_INVALID_ARG;
    st = fibattn_rope(q, q_rot, (int64_t)n_layers_call * B * H, T, d, dtype, rope_table,
                      table_rows, 0, cuda_stream);
    if (st != FIBATTN_OK) return st;
    st = fibattn_rope(k, k_rot, (int64_t)n_layers_call * B * H_kv, T, d, dtype, rope_table,
                      table_rows, 0, cuda_stream);
    if (st != FIBATTN_OK) return st;
    return fibattn_fwd_gqa(q_rot, k_rot, v, o, lse, B, H, H_kv, T, d, dtype, W, scale, sched,
                           layer0, n_layers_call, cuda_stream);
}

fibattn_status fibattn_bwd(const void* q, const void* k, const void* v, const void* o,
                           const float* lse, const void* dO, void* dq, void* dk, void* dv,
                           void* workspace, uint64_t workspace_bytes, int32_t B, int32_t H,
                           int32_t T, int32_t d, int32_t dtype, int32_t W, float scale,
                           const fibattn_schedule* sched, int32_t layer0, int32_t n_layers_call,
                           void* cuda_stream) {
    return fibattn_bwd_gqa(q, k, v, o, lse, dO, dq, dk, dv, workspace, workspace_bytes, B, H, H,
                           T, d, dtype, W, scale, sched, layer0, n_layers_call, cuda_stream);
}
fibattn_status fibattn_bwd_fused(const void* q, const void* k, const void* v, const void* o,
                                 const float* lse, const void* dO, void* dq, void* dk, void* dv,
                                 void* workspace, uint64_t workspace_bytes, int32_t B, int32_t H,
                                 int32_t T, int32_t d, int32_t dtype, int32_t W, float scale,
                                 const fibattn_schedule* sched, int32_t layer0,
                                 int32_t n_layers_call, void* cuda_stream) {
    const void* ptrs[] = {q, k, v, o, lse, dO, dq, dk, dv};
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return FIBATTN_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return FIBATTN_ERR_INVALID_ARG;
    fibattn_status st = check_common(B, H, T, d, dtype, W, sched, layer0, n_layers_call);
    if (st != FIBATTN_OK) return st;
    if (dtype != FIBATTN_BF16 || d != 64) return FIBATTN_ERR_UNSUPPORTED;
    // D and lse * log2(e) only: the layout of the two-kernel backward without its pairs
    const BwdWorkspace ws = workspace_layout(B, H, T, dtype, n_layers_call, 0, false);
    if (workspace_bytes < ws.total) return FIBATTN_ERR_INVALID_ARG;
    float* delta = static_cast<float*>(workspace);
    float* lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + ws.lse2_offset);
    const int64_t per_layer_pad = (int64_t)B * H * ws.T_pad;
    if (!resolve_scale(scale, d)) return FIBATTN_ERR_INVALID_ARG;
    const int64_t per_layer = (int64_t)B * H * T;
    const size_t es = elt_size(dtype);
    {
        const uint64_t qb = (uint64_t)n_layers_call * per_layer * d * es;
        const uint64_t lb = (uint64_t)n_layers_call * per_layer * 4;
        if (outputs_overlap({{dq, qb}, {dk, qb}, {dv, qb}, {workspace, ws.total}},
                            {{q, qb}, {k, qb}, {v, qb}, {o, qb}, {lse, lb}, {dO, qb}}))
            return FIBATTN_ERR_INVALID_ARG;
    }
    for (int32_t c = 0; c < n_layers_call; c += kMaxLayersPerLaunch) {
        const int32_t n = n_layers_call - c < kMaxLayersPerLaunch ? n_layers_call - c : kMaxLayersPerLaunch;
        OffsetTables t;
        st = build_launch_tables(sched, layer0 + c, n, W, T, &t);
        if (st != FIBATTN_OK) return st;
        AttnShape sh{(int64_t)B * H, T, W < T ? W : T, scale, n, 1, d};
        const size_t off = (size_t)c * per_layer * d * es;
        const size_t poff = (size_t)c * per_layer_pad;
        st = launch_bwd_fused_tc_bf16((const char*)q + off, (const char*)k + off,
                                      (const char*)v + off, (const char*)o + off,
                                      lse + (size_t)c * per_layer, (const char*)dO + off,
                                      (char*)dq + off, (char*)dk + off, (char*)dv + off,
                                      delta + poff, lse2 + poff, sh, t, as_stream(cuda_stream));
        if (st != FIBATTN_OK) return st;
    }
    return FIBATTN_OK;
}

fibattn_status fibattn_bwd_frac_workspace_size(int32_t B, int32_t H, int32_t T, int32_t d,
                                               int32_t dtype, int32_t W, int32_t base,
                                               int64_t base_max, const float* alphas,
                                               int32_t n_layers_call, uint64_t* bytes) {
    if (!bytes) return FIBATTN_ERR_INVALID_ARG;
    int32_t n_max = 0;
    fibattn_status st = check_frac(B, H, T, d, dtype, W, base, base_max, alphas, n_layers_call, &n_max);
    if (st != FIBATTN_OK) return st;
    *bytes = workspace_layout(B, H, T, dtype, n_layers_call, n_max, true).total;
    return FIBATTN_OK;
}

fibattn_status fibattn_bwd_frac(const void* q, const void* k, const void* v, const void* o,
                                const float* lse, const void* dO, void* dq, void* dk, void* dv,
                                float* dalpha, void* workspace, uint64_t workspace_bytes,
                                int32_t B, int32_t H, int32_t T, int32_t d, int32_t dtype,
                                int32_t W, float scale, int32_t base, int64_t base_max,
                                const float* alphas, int32_t n_layers_call, void* cuda_stream) {
    const void* ptrs[] = {q, k, v, o, lse, dO, dq, dk, dv};
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return FIBATTN_ERR_INVALID_ARG;
    if (!dalpha || (reinterpret_cast<uintptr_t>(dalpha) & 3u) != 0) return FIBATTN_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return FIBATTN_ERR_INVALID_ARG;
    int32_t n_max = 0;
    fibattn_status st = check_frac(B, H, T, d, dtype, W, base, base_max, alphas, n_layers_call, &n_max);
    if (st != FIBATTN_OK) return st;
    const BwdWorkspace ws = workspace_layout(B, H, T, dtype, n_layers_call, n_max, true);
    if (workspace_bytes < ws.total) return FIBATTN_ERR_INVALID_ARG;
    char* wsb = static_cast<char*>(workspace);
    float* delta = reinterpret_cast<float*>(wsb);
    float* lse2 = reinterpret_cast<float*>(wsb + ws.lse2_offset);
    uint32_t* pds = reinterpret_cast<uint32_t*>(wsb + ws.pds_offset);
    float* galpha = reinterpret_cast<float*>(wsb + ws.galpha_offset);
    if (!resolve_scale(scale, d)) return FIBATTN_ERR_INVALID_ARG;
    const int64_t per_layer = (int64_t)B * H * T;
    const int64_t per_layer_pad = (int64_t)B * H * ws.T_pad;
    // dalpha partials per layer: one per query (f32) or one per 128-query tile (bf16)
    const int64_t parts = dtype == FIBATTN_F32 ? per_layer : (int64_t)B * H * ((T + 127) / 128);
    const size_t es = elt_size(dtype);
    {
        const uint64_t qb = (uint64_t)n_layers_call * per_layer * d * es;
        const uint64_t lb = (uint64_t)n_layers_call * per_layer * 4;
        if (outputs_overlap({{dq, qb}, {dk, qb}, {dv, qb}, {dalpha, (uint64_t)n_layers_call * 4},
                             {workspace, ws.total}},
                            {{q, qb}, {k, qb}, {v, qb}, {o, qb}, {lse, lb}, {dO, qb}}))
            return FIBATTN_ERR_INVALID_ARG;
    }
    cudaStream_t s = as_stream(cuda_stream);
    for (int32_t c = 0; c < n_layers_call; c += kMaxLayersPerLaunch) {
        const int32_t n = n_layers_call - c < kMaxLayersPerLaunch ? n_layers_call - c : kMaxLayersPerLaunch;
        FracTables t;
        st = build_frac_launch_tables(base, base_max, alphas + c, n, W, T, &t);
        if (st != FIBATTN_OK) return st;
        AttnShape sh{(int64_t)B * H, T, W < T ? W : T, scale, n};
        const size_t off = (size_t)c * per_layer * d * es;
        const size_t loff = (size_t)c * per_layer;
        if (dtype == FIBATTN_F32) {
            st = launch_bwd_frac_simt_f32((const float*)((const char*)q + off),
                                          (const float*)((const char*)k + off),
                                          (const float*)((const char*)v + off),
                                          (const float*)((const char*)o + off), lse + loff,
                                          (const float*)((const char*)dO + off),
                                          (float*)((char*)dq + off), (float*)((char*)dk + off),
                                          (float*)((char*)dv + off), delta + loff,
                                          galpha + (size_t)c * parts, sh, t, s);
        } else {
            const size_t poff = (size_t)c * per_layer_pad;
            st = launch_bwd_frac_tc_bf16((const char*)q + off, (const char*)k + off,
                                         (const char*)v + off, (const char*)o + off, lse + loff,
                                         (const char*)dO + off, (char*)dq + off, (char*)dk + off,
                                         (char*)dv + off, delta + poff, lse2 + poff,
                                         pds + poff * ws.n_max, ws.n_max, galpha + (size_t)c * parts,
                                         sh, t, s);
        }
        if (st != FIBATTN_OK) return st;
        st = launch_dalpha_reduce(galpha + (size_t)c * parts, dalpha + c, n, parts, s);
        if (st != FIBATTN_OK) return st;
    }
    return FIBATTN_OK;
}

fibattn_status fibattn_rope_table(float* table, int32_t T, int32_t d, double base,
                                  void* cuda_stream) {
    if (!table || (reinterpret_cast<uintptr_t>(table) & 15u) != 0 || T < 1 || T > FIBATTN_T_MAX)
        return FIBATTN_ERR_INVALID_ARG;
    if (!(base > 1.0) || !(base < 1e300)) return FIBATTN_ERR_INVALID_ARG;
    if (d != 64) return FIBATTN_ERR_UNSUPPORTED;
    return launch_rope_table(table, T, base, as_stream(cuda_stream));
}

fibattn_status fibattn_rope(const void* x, void* y, int64_t slices, int32_t T, int32_t d,
                            int32_t dtype, const float* table, int32_t table_rows,
                            int32_t inverse, void* cuda_stream) {
    if (!x || !y || !table || !aligned16(x) || !aligned16(y) || !aligned16(table))
        return FIBATTN_ERR_INVALID_ARG;
    if (table_rows < T) return FIBATTN_ERR_INVALID_ARG;
    // slices * T <= 2^40, tested without forming a product that could overflow
    if (slices < 1 || T < 1 || T > FIBATTN_T_MAX || slices > (((int64_t)1 << 40) / T))
        return FIBATTN_ERR_INVALID_ARG;
    if (dtype != FIBATTN_F32 && dtype != FIBATTN_BF16) return FIBATTN_ERR_UNSUPPORTED;
    if (d != 64) return FIBATTN_ERR_UNSUPPORTED;
    const int64_t bytes = slices * (int64_t)T * d * (int64_t)elt_size(dtype);
    const char* xb = static_cast<const char*>(x);
    const char* yb = static_cast<const char*>(y);
    if (xb != yb && xb < yb + bytes && yb < xb + bytes) return FIBATTN_ERR_INVALID_ARG;  // partial overlap
    return launch_rope(x, y, slices * (int64_t)T, T, dtype, table, inverse != 0,
                       as_stream(cuda_stream));
}

fibattn_status fibattn_poll_device_error(void* cuda_stream) {
    cudaError_t e = cudaStreamSynchronize(as_stream(cuda_stream));
    if (e != cudaSuccess) return cuda_fail((int32_t)e, "cudaStreamSynchronize");
    e = cudaPeekAtLastError();
    if (e != cudaSuccess) return cuda_fail((int32_t)e, "cudaPeekAtLastError");
    int32_t* w = device_error_word();
    if (!w) return cuda_fail(-1, "cudaGetSymbolAddress (error word)");
    int32_t h = 0;
    e = cudaMemcpy(&h, w, sizeof(h), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail((int32_t)e, "cudaMemcpy (error word)");
    if (h != kDevErrNone) {
        e = cudaMemset(w, 0, sizeof(int32_t));
        if (e != cudaSuccess) return cuda_fail((int32_t)e, "cudaMemset (error word)");
        return FIBATTN_ERR_TIMEOUT;
    }
    return FIBATTN_OK;
}

}  // extern "C"
