// schedule.cpp -- host side of the per-layer alpha schedules and offset tables.
//
// "Depth-Staggered Fibonacci Spacing for Sparse Attention" (gist.science explainer):
//   Metodologia / Arquitetura, "Escalonamento": offset f_k scaled to d_k = alpha * f_k;
//   Metodologia / Variaveis Experimentais: fixed alpha, linear stagger across depth,
//   coprime reassignment l -> (c * l mod L) of the same alphas;
//   Metodologia / Controles: the power-of-two base.
// Alphas are exact rationals; offsets are alpha * F rounded half up with integer
// arithmetic only, so host and device agree bit for bit.
// The learned-alpha variant (Metodologia / Arquitetura, "Implementacao": linear
// interpolation between key/value rows so that the gradient reaches alpha) takes a real
// float alpha instead: d = alpha * F in double (exact for F < 2^29), kept when
// W <= d <= T - 1, stored as ceil(d) and the weight ceil(d) - d of the following row.
#include <math.h>
#include <stdint.h>

#include "internal.h"

namespace fibattn {
namespace {

typedef __int128 i128;

int64_t gcd64(int64_t a, int64_t b) {
    if (a < 0) a = -a;
    if (b < 0) b = -b;
    while (b) {
        int64_t t = a % b;
        a = b;
        b = t;
    }
    return a;
}

bool ratio_ok(fibattn_ratio r) {
    return r.num >= 1 && r.den >= 1 && r.num <= FIBATTN_RATIO_MAX && r.den <= FIBATTN_RATIO_MAX;
}

// alpha_min + (alpha_max - alpha_min) * l / (L - 1), exact.
Alpha linear_alpha(fibattn_ratio lo, fibattn_ratio hi, int64_t l, int64_t L) {
    if (L == 1) return Alpha{lo.num, lo.den};
    // lo.n/lo.d + (hi.n/hi.d - lo.n/lo.d) * l/(L-1)
    //   = [lo.n*hi.d*(L-1) + (hi.n*lo.d - lo.n*hi.d)*l] / [lo.d*hi.d*(L-1)]
    i128 a = (i128)lo.num * hi.den;
    i128 b = (i128)hi.num * lo.den;
    i128 num = a * (L - 1) + (b - a) * l;
    i128 den = (i128)lo.den * hi.den * (L - 1);
    // |num|, den < 2^61 for ratios <= 2^20 and L <= 2^20; reduce to lowest terms
    int64_t n64 = (int64_t)num, d64 = (int64_t)den;
    int64_t g = gcd64(n64, d64);
    return Alpha{n64 / g, d64 / g};
}

}  // namespace

fibattn_status layer_alpha(const fibattn_schedule* s, int32_t layer, Alpha* out) {
    if (!s || !out) return FIBATTN_ERR_INVALID_ARG;
    if (s->n_layers < 1 || s->n_layers > FIBATTN_LAYERS_MAX) return FIBATTN_ERR_INVALID_ARG;
    if (layer < 0 || layer >= s->n_layers) return FIBATTN_ERR_INVALID_ARG;
    if (s->base != FIBATTN_BASE_FIB && s->base != FIBATTN_BASE_POW2) return FIBATTN_ERR_INVALID_ARG;
    if (s->base_max < 0) return FIBATTN_ERR_INVALID_ARG;
    switch (s->kind) {
        case FIBATTN_SCHED_FIXED: {
            if (!ratio_ok(s->alpha)) return FIBATTN_ERR_INVALID_ARG;
            int64_t g = gcd64(s->alpha.num, s->alpha.den);
            *out = Alpha{s->alpha.num / g, s->alpha.den / g};
            return FIBATTN_OK;
        }
        case FIBATTN_SCHED_LINEAR:
        case FIBATTN_SCHED_COPRIME: {
            if (!ratio_ok(s->alpha_min) || !ratio_ok(s->alpha_max)) return FIBATTN_ERR_INVALID_ARG;
            int64_t L = s->n_layers, l = layer;
            if (s->kind == FIBATTN_SCHED_COPRIME) {
                if (s->coprime_c < 1 || gcd64(s->coprime_c, L) != 1) return FIBATTN_ERR_INVALID_ARG;
                l = ((int64_t)s->coprime_c * l) % L;
            }
            *out = linear_alpha(s->alpha_min, s->alpha_max, l, L);
            return FIBATTN_OK;
        }
        default:
            return FIBATTN_ERR_INVALID_ARG;
    }
}

fibattn_status build_table(const fibattn_schedule* s, Alpha a, int32_t W, int32_t T, int32_t* out,
                           int32_t cap, int32_t* n_out) {
    if (W < 1 || T < 1 || cap < 0) return FIBATTN_ERR_INVALID_ARG;
    const bool fib = s->base == FIBATTN_BASE_FIB;
    const int64_t fmax = s->base_max > 0 ? s->base_max : (fib ? 987 : INT64_MAX);
    int32_t n = 0;
    int64_t last = -1;
    int64_t f = 1, g = 2;  // Fibonacci pair (f, next) or the power of two f
    while (f <= fmax) {
        // o = floor(alpha * f + 1/2) = floor((2 * num * f + den) / (2 * den))
        i128 o = ((i128)2 * a.num * f + a.den) / ((i128)2 * a.den);
        if (o > (i128)T - 1) break;  // o grows with f: nothing further fits
        if (o >= W && o != last) {
            if (n < cap) out[n] = (int32_t)o;
            ++n;
            last = (int64_t)o;
        }
        if (fib) {
            int64_t h = f + g;
            f = g;
            g = h;
        } else {
            if (f > INT64_MAX / 2) break;
            f *= 2;
        }
    }
    *n_out = n;
    return n > cap ? FIBATTN_ERR_CAPACITY : FIBATTN_OK;
}

fibattn_status build_frac_table(int32_t base, int64_t base_max, float alpha, int32_t W, int32_t T,
                                int32_t* c_out, float* w_out, float* f_out, int32_t cap,
                                int32_t* n_out) {
    if (W < 1 || T < 1 || cap < 0 || base_max < 0) return FIBATTN_ERR_INVALID_ARG;
    if (base != FIBATTN_BASE_FIB && base != FIBATTN_BASE_POW2) return FIBATTN_ERR_INVALID_ARG;
    if (!(alpha > 0.f) || !(alpha <= (float)FIBATTN_RATIO_MAX)) return FIBATTN_ERR_INVALID_ARG;
    const bool fib = base == FIBATTN_BASE_FIB;
    const double a = (double)alpha;
    int32_t n = 0;
    auto keep = [&](double d, int64_t f) {
        if (d < (double)W || d > (double)T - 1) return;
        if (n < cap) {
            const double c = ceil(d);
            c_out[n] = (int32_t)c;
            w_out[n] = (float)(c - d);
            if (f_out) f_out[n] = (float)f;
        }
        ++n;
    };
    if (fib) {
        const int64_t fmax = base_max > 0 ? base_max : 987;
        // The pair is carried in 128 bits: a tiny alpha keeps alpha * F below T - 1 for every
        // F up to fmax (at most 2^63 - 1), and the next term must not overflow on the way.
        for (i128 f = 1, g = 2; f <= (i128)fmax;) {
            const int64_t f64 = (int64_t)f;  // f <= fmax fits
            if (a * (double)f64 > (double)T - 1) break;  // d grows with F: nothing further fits
            keep(a * (double)f64, f64);
            const i128 h = f + g;
            f = g;
            g = h;
        }
    } else {
        for (int64_t f = 1; a * (double)f <= (double)T - 1 && (base_max <= 0 || f <= base_max);) {
            keep(a * (double)f, f);
            if (f > INT64_MAX / 2) break;
            f *= 2;
        }
    }
    *n_out = n;
    return n > cap ? FIBATTN_ERR_CAPACITY : FIBATTN_OK;
}

fibattn_status build_frac_launch_tables(int32_t base, int64_t base_max, const float* alphas,
                                        int32_t n, int32_t W, int32_t T, FracTables* t) {
    if (!alphas || n < 1 || n > kMaxLayersPerLaunch) return FIBATTN_ERR_INVALID_ARG;
    for (int c = 0; c < kMaxLayersPerLaunch; ++c) {
        t->c.count[c] = 0;
        for (int e = 0; e < kMaxOffsets; ++e) {
            t->c.off[c][e] = -1;
            t->w[c][e] = 0.f;
            t->f[c][e] = 0.f;
        }
    }
    for (int c = 0; c < n; ++c) {
        int32_t cnt = 0;
        fibattn_status st = build_frac_table(base, base_max, alphas[c], W, T, t->c.off[c], t->w[c],
                                             t->f[c], kMaxOffsets, &cnt);
        if (st != FIBATTN_OK) return st;
        t->c.count[c] = cnt;
    }
    return FIBATTN_OK;
}

fibattn_status build_launch_tables(const fibattn_schedule* s, int32_t layer0, int32_t n, int32_t W,
                                   int32_t T, OffsetTables* t) {
    if (n < 1 || n > kMaxLayersPerLaunch) return FIBATTN_ERR_INVALID_ARG;
    for (int c = 0; c < kMaxLayersPerLaunch; ++c) {
        t->count[c] = 0;
        for (int e = 0; e < kMaxOffsets; ++e) t->off[c][e] = -1;
    }
    for (int c = 0; c < n; ++c) {
        Alpha a;
        fibattn_status st = layer_alpha(s, layer0 + c, &a);
        if (st != FIBATTN_OK) return st;
        int32_t cnt = 0;
        st = build_table(s, a, W, T, t->off[c], kMaxOffsets, &cnt);
        if (st != FIBATTN_OK) return st;
        t->count[c] = cnt;
    }
    return FIBATTN_OK;
}

}  // namespace fibattn
