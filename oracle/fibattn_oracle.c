/*
 * fibattn_oracle.c -- the oracle: plain fp64 CPU sparse attention, forward and
 * backward, by the definition.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this library. It shares no source, header or helper with
 * the CUDA library and includes nothing from it.
 *
 * What it computes ("Depth-Staggered Fibonacci Spacing for Sparse Attention",
 * gist.science explainer, Metodologia / Arquitetura e Mecanismo de Atencao,
 * "Conjunto Atendido"): query i attends the dense local window of W keys
 * ending at i plus the keys i - o for every offset o of the layer's table.
 * For each (layer, batch, head) slice and each query i:
 *   1. materialise S_i = {j : 0 <= i-j < W, j >= 0} U {i-o : o in table, i-o >= 0},
 *      sorted and without duplicates;
 *   2. s_j = scale * sum_c q[i][c] * k[j][c] for j in S_i;
 *   3. m = max_j s_j, p_j = exp(s_j - m), l = sum_j p_j,
 *      out[i] = sum_j p_j v[j] / l, lse[i] = m + log(l).
 * Backward (the analytic gradient of softmax attention restricted to S_i):
 *   P_ij = exp(s_ij - lse_i), D_i = sum_c dO[i][c] * out[i][c],
 *   dS_ij = P_ij * (dO_i . v_j - D_i),
 *   dQ_i = scale * sum_j dS_ij k_j,  dK_j += scale * dS_ij q_i,  dV_j += P_ij dO_i.
 * RoPE is applied before the gather on the pages; here Q and K arrive rotated.
 *
 * Fractional ("learned") offsets (same page, "Implementacao" under Arquitetura: to let the
 * gradient reach alpha when offsets are not integers, keys and values are linearly
 * interpolated between rows): with real distances d_k = alpha * f_k, query i attends its
 * window plus, for every d_k <= i, one interpolated key/value at position p = i - d_k:
 *   lo = floor(p), w = p - lo,  k~ = (1 - w) k[lo] + w k[lo + 1],  v~ likewise
 * (lo + 1 <= i - W + 1 <= i because d_k >= W). Softmax over the window keys and the
 * interpolated keys together, as above.
 * Its backward is the same softmax gradient with the interpolated rows in place of k_j and
 * v_j, the interpolation weights carried to the two rows (dk[lo] += (1 - w) g, dk[lo+1] +=
 * w g, likewise dv), and the derivative with respect to each distance d: p = i - d, so
 * dk~/dd = k[lo] - k[lo+1] and dv~/dd = v[lo] - v[lo+1] on the segment holding p (at an
 * integer p that is the segment [p, p+1], the derivative for d decreasing), giving
 *   dL/dd = sum_i [ dS_i scale q_i.(k[lo] - k[lo+1]) + P_i dO_i.(v[lo] - v[lo+1]) ],
 * and dL/dalpha = sum_k f_k dL/dd_k (chain rule through d_k = alpha f_k).
 *
 * Layout: every tensor is [n_slices][T][d] row-major float64; lse is [n_slices][T].
 * Slices are independent; OpenMP runs them in parallel when built with -fopenmp.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int cmp_i64(const void* a, const void* b) {
    int64_t x = *(const int64_t*)a, y = *(const int64_t*)b;
    return (x > y) - (x < y);
}

/* Step 1: the attended key set of query i, sorted ascending, unique. Returns its size. */
static int64_t key_set(int64_t i, int64_t W, const int32_t* table, int n_table, int64_t* out) {
    int64_t n = 0;
    int64_t lo = i - W + 1;
    if (lo < 0) lo = 0;
    for (int64_t j = lo; j <= i; ++j) out[n++] = j;
    for (int t = 0; t < n_table; ++t) {
        int64_t j = i - (int64_t)table[t];
        if (j >= 0) out[n++] = j;
    }
    qsort(out, (size_t)n, sizeof(int64_t), cmp_i64);
    int64_t m = 0;
    for (int64_t a = 0; a < n; ++a)
        if (m == 0 || out[a] != out[m - 1]) out[m++] = out[a];
    return m;
}

/* Public: key set of query i (for the tests' cross-checks). */
int64_t oracle_key_set(int64_t i, int64_t W, const int32_t* table, int n_table, int64_t* out) {
    return key_set(i, W, table, n_table, out);
}

/* Forward of one slice: q, k, v [T][d]; writes out [T][d] and lse [T]. */
static void fwd_slice(const double* q, const double* k, const double* v, double* out, double* lse,
                      int64_t T, int64_t d, int64_t W, double scale, const int32_t* table,
                      int n_table, int64_t* keys, double* s) {
    for (int64_t i = 0; i < T; ++i) {
        int64_t n = key_set(i, W, table, n_table, keys);
        double m = -INFINITY;
        for (int64_t a = 0; a < n; ++a) {
            const double* kr = k + keys[a] * d;
            double acc = 0.0;
            for (int64_t c = 0; c < d; ++c) acc += q[i * d + c] * kr[c];
            s[a] = scale * acc;
            if (s[a] > m) m = s[a];
        }
        double l = 0.0;
        for (int64_t a = 0; a < n; ++a) {
            s[a] = exp(s[a] - m);
            l += s[a];
        }
        for (int64_t c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int64_t a = 0; a < n; ++a) acc += s[a] * v[keys[a] * d + c];
            out[i * d + c] = acc / l;
        }
        lse[i] = m + log(l);
    }
}

/* Backward of one slice. Needs the forward's out and lse (computed here, fp64). */
static void bwd_slice(const double* q, const double* k, const double* v, const double* dout,
                      const double* out, const double* lse, double* dq, double* dk, double* dv,
                      int64_t T, int64_t d, int64_t W, double scale, const int32_t* table,
                      int n_table, int64_t* keys) {
    memset(dk, 0, sizeof(double) * (size_t)(T * d));
    memset(dv, 0, sizeof(double) * (size_t)(T * d));
    for (int64_t i = 0; i < T; ++i) {
        const double* qi = q + i * d;
        const double* gi = dout + i * d;
        double Di = 0.0;
        for (int64_t c = 0; c < d; ++c) Di += gi[c] * out[i * d + c];
        for (int64_t c = 0; c < d; ++c) dq[i * d + c] = 0.0;
        int64_t n = key_set(i, W, table, n_table, keys);
        for (int64_t a = 0; a < n; ++a) {
            int64_t j = keys[a];
            const double* kj = k + j * d;
            const double* vj = v + j * d;
            double sij = 0.0, dpij = 0.0;
            for (int64_t c = 0; c < d; ++c) {
                sij += qi[c] * kj[c];
                dpij += gi[c] * vj[c];
            }
            double pij = exp(scale * sij - lse[i]);
            double dsij = pij * (dpij - Di);
            for (int64_t c = 0; c < d; ++c) {
                dq[i * d + c] += scale * dsij * kj[c];
                dk[j * d + c] += scale * dsij * qi[c];
                dv[j * d + c] += pij * gi[c];
            }
        }
    }
}

/* Forward of one slice with fractional offsets (dists: n_dist real distances, ascending). */
static void fwd_frac_slice(const double* q, const double* k, const double* v, double* out,
                           double* lse, int64_t T, int64_t d, int64_t W, double scale,
                           const double* dists, int n_dist, double* s, double* keyv, double* valv) {
    for (int64_t i = 0; i < T; ++i) {
        /* materialise the attended keys and values of query i */
        int64_t n = 0;
        int64_t lo_w = i - W + 1;
        if (lo_w < 0) lo_w = 0;
        for (int64_t j = lo_w; j <= i; ++j, ++n) {
            memcpy(keyv + n * d, k + j * d, sizeof(double) * (size_t)d);
            memcpy(valv + n * d, v + j * d, sizeof(double) * (size_t)d);
        }
        for (int t = 0; t < n_dist; ++t) {
            double pos = (double)i - dists[t];
            if (pos < 0.0) continue;
            int64_t lo = (int64_t)floor(pos);
            double w = pos - (double)lo;
            for (int64_t c = 0; c < d; ++c) {
                double khi = w != 0.0 ? k[(lo + 1) * d + c] : 0.0;
                double vhi = w != 0.0 ? v[(lo + 1) * d + c] : 0.0;
                keyv[n * d + c] = (1.0 - w) * k[lo * d + c] + w * khi;
                valv[n * d + c] = (1.0 - w) * v[lo * d + c] + w * vhi;
            }
            ++n;
        }
        /* softmax attention over them */
        double m = -INFINITY;
        for (int64_t a = 0; a < n; ++a) {
            double acc = 0.0;
            for (int64_t c = 0; c < d; ++c) acc += q[i * d + c] * keyv[a * d + c];
            s[a] = scale * acc;
            if (s[a] > m) m = s[a];
        }
        double l = 0.0;
        for (int64_t a = 0; a < n; ++a) {
            s[a] = exp(s[a] - m);
            l += s[a];
        }
        for (int64_t c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int64_t a = 0; a < n; ++a) acc += s[a] * valv[a * d + c];
            out[i * d + c] = acc / l;
        }
        lse[i] = m + log(l);
    }
}

/* Backward of one slice with fractional offsets: dq, dk, dv and dd[n_dist] = dL/dd per
 * distance, from the forward's out and lse (computed by fwd_frac_slice, fp64). */
static void bwd_frac_slice(const double* q, const double* k, const double* v, const double* dout,
                           const double* out, const double* lse, double* dq, double* dk,
                           double* dv, double* dd, int64_t T, int64_t d, int64_t W, double scale,
                           const double* dists, int n_dist, double* kt, double* vt) {
    memset(dk, 0, sizeof(double) * (size_t)(T * d));
    memset(dv, 0, sizeof(double) * (size_t)(T * d));
    for (int t = 0; t < n_dist; ++t) dd[t] = 0.0;
    for (int64_t i = 0; i < T; ++i) {
        const double* qi = q + i * d;
        const double* gi = dout + i * d;
        double Di = 0.0;
        for (int64_t c = 0; c < d; ++c) Di += gi[c] * out[i * d + c];
        for (int64_t c = 0; c < d; ++c) dq[i * d + c] = 0.0;
        /* window keys: the plain softmax gradient */
        int64_t lo_w = i - W + 1;
        if (lo_w < 0) lo_w = 0;
        for (int64_t j = lo_w; j <= i; ++j) {
            double sij = 0.0, dpij = 0.0;
            for (int64_t c = 0; c < d; ++c) {
                sij += qi[c] * k[j * d + c];
                dpij += gi[c] * v[j * d + c];
            }
            double pij = exp(scale * sij - lse[i]);
            double dsij = pij * (dpij - Di);
            for (int64_t c = 0; c < d; ++c) {
                dq[i * d + c] += scale * dsij * k[j * d + c];
                dk[j * d + c] += scale * dsij * qi[c];
                dv[j * d + c] += pij * gi[c];
            }
        }
        /* interpolated keys */
        for (int t = 0; t < n_dist; ++t) {
            double pos = (double)i - dists[t];
            if (pos < 0.0) continue;
            int64_t lo = (int64_t)floor(pos);
            double w = pos - (double)lo;
            int64_t hi = lo + 1; /* <= i - W + 1 <= i */
            for (int64_t c = 0; c < d; ++c) {
                kt[c] = (1.0 - w) * k[lo * d + c] + w * k[hi * d + c];
                vt[c] = (1.0 - w) * v[lo * d + c] + w * v[hi * d + c];
            }
            double s = 0.0, dp = 0.0, sdiff = 0.0, vdiff = 0.0;
            for (int64_t c = 0; c < d; ++c) {
                s += qi[c] * kt[c];
                dp += gi[c] * vt[c];
                sdiff += qi[c] * (k[lo * d + c] - k[hi * d + c]);
                vdiff += gi[c] * (v[lo * d + c] - v[hi * d + c]);
            }
            double P = exp(scale * s - lse[i]);
            double dS = P * (dp - Di);
            for (int64_t c = 0; c < d; ++c) {
                dq[i * d + c] += scale * dS * kt[c];
                dk[lo * d + c] += (1.0 - w) * scale * dS * qi[c];
                dk[hi * d + c] += w * scale * dS * qi[c];
                dv[lo * d + c] += (1.0 - w) * P * gi[c];
                dv[hi * d + c] += w * P * gi[c];
            }
            dd[t] += dS * scale * sdiff + P * vdiff;
        }
    }
}

static int set_threads(int n_threads) {
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
    return omp_get_max_threads();
#else
    (void)n_threads;
    return 1;
#endif
}

/* Number of threads the next parallel region will use. */
int oracle_threads(int n_threads) { return set_threads(n_threads); }

/*
 * Forward over n_slices slices. table_of_slice[s] indexes into `tables`
 * (row-major [n_tables][cap]) and `counts`.
 */
int oracle_fwd(const double* q, const double* k, const double* v, double* out, double* lse,
               int64_t n_slices, int64_t T, int64_t d, int64_t W, double scale,
               const int32_t* tables, const int32_t* counts, int64_t cap,
               const int32_t* table_of_slice, int n_threads) {
    set_threads(n_threads);
    int err = 0;
#pragma omp parallel
    {
        int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)(T + cap + 1));
        double* s = (double*)malloc(sizeof(double) * (size_t)(T + cap + 1));
        if (!keys || !s) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic)
            for (int64_t sl = 0; sl < n_slices; ++sl) {
                int32_t t = table_of_slice[sl];
                fwd_slice(q + sl * T * d, k + sl * T * d, v + sl * T * d, out + sl * T * d,
                          lse + sl * T, T, d, W, scale, tables + (int64_t)t * cap, counts[t],
                          keys, s);
            }
        }
        free(keys);
        free(s);
    }
    return err;
}

/* Backward over n_slices slices; also returns the fp64 forward (out, lse) it used. */
int oracle_bwd(const double* q, const double* k, const double* v, const double* dout,
               double* out, double* lse, double* dq, double* dk, double* dv,
               int64_t n_slices, int64_t T, int64_t d, int64_t W, double scale,
               const int32_t* tables, const int32_t* counts, int64_t cap,
               const int32_t* table_of_slice, int n_threads) {
    set_threads(n_threads);
    int err = 0;
#pragma omp parallel
    {
        int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)(T + cap + 1));
        double* s = (double*)malloc(sizeof(double) * (size_t)(T + cap + 1));
        if (!keys || !s) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic)
            for (int64_t sl = 0; sl < n_slices; ++sl) {
                int32_t t = table_of_slice[sl];
                const int32_t* tab = tables + (int64_t)t * cap;
                int64_t off = sl * T * d;
                fwd_slice(q + off, k + off, v + off, out + off, lse + sl * T, T, d, W, scale, tab,
                          counts[t], keys, s);
                bwd_slice(q + off, k + off, v + off, dout + off, out + off, lse + sl * T, dq + off,
                          dk + off, dv + off, T, d, W, scale, tab, counts[t], keys);
            }
        }
        free(keys);
        free(s);
    }
    return err;
}

/* Forward with fractional offsets over n_slices slices; dists is [n_tables][cap] doubles. */
int oracle_fwd_frac(const double* q, const double* k, const double* v, double* out, double* lse,
                    int64_t n_slices, int64_t T, int64_t d, int64_t W, double scale,
                    const double* dists, const int32_t* counts, int64_t cap,
                    const int32_t* table_of_slice, int n_threads) {
    set_threads(n_threads);
    int err = 0;
#pragma omp parallel
    {
        int64_t nk = T + cap + 1;
        double* s = (double*)malloc(sizeof(double) * (size_t)nk);
        double* keyv = (double*)malloc(sizeof(double) * (size_t)(nk * d));
        double* valv = (double*)malloc(sizeof(double) * (size_t)(nk * d));
        if (!s || !keyv || !valv) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic)
            for (int64_t sl = 0; sl < n_slices; ++sl) {
                int32_t t = table_of_slice[sl];
                fwd_frac_slice(q + sl * T * d, k + sl * T * d, v + sl * T * d, out + sl * T * d,
                               lse + sl * T, T, d, W, scale, dists + (int64_t)t * cap, counts[t],
                               s, keyv, valv);
            }
        }
        free(s);
        free(keyv);
        free(valv);
    }
    return err;
}

/* Backward with fractional offsets. out/lse are written (the forward, fp64); dd is
 * [n_slices][cap]: dL/dd of each slice's distances. */
int oracle_bwd_frac(const double* q, const double* k, const double* v, const double* dout,
                    double* dq, double* dk, double* dv, double* out, double* lse, double* dd,
                    int64_t n_slices, int64_t T, int64_t d, int64_t W, double scale,
                    const double* dists, const int32_t* counts, int64_t cap,
                    const int32_t* table_of_slice, int n_threads) {
    set_threads(n_threads);
    int err = 0;
#pragma omp parallel
    {
        int64_t nk = T + cap + 1;
        double* s = (double*)malloc(sizeof(double) * (size_t)nk);
        double* keyv = (double*)malloc(sizeof(double) * (size_t)(nk * d));
        double* valv = (double*)malloc(sizeof(double) * (size_t)(nk * d));
        if (!s || !keyv || !valv) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic)
            for (int64_t sl = 0; sl < n_slices; ++sl) {
                int32_t t = table_of_slice[sl];
                const double* ds = dists + (int64_t)t * cap;
                const int64_t o3 = sl * T * d;
                fwd_frac_slice(q + o3, k + o3, v + o3, out + o3, lse + sl * T, T, d, W, scale, ds,
                               counts[t], s, keyv, valv);
                bwd_frac_slice(q + o3, k + o3, v + o3, dout + o3, out + o3, lse + sl * T, dq + o3,
                               dk + o3, dv + o3, dd + sl * cap, T, d, W, scale, ds, counts[t],
                               keyv, valv);
            }
        }
        free(s);
        free(keyv);
        free(valv);
    }
    return err;
}
