/*
 * mk_oracle.c -- plain CPU oracle (TEST INFRASTRUCTURE ONLY; see mk_oracle.h).
 *
 * Written to be read against the definition, not to be fast: every loop
 * follows one step of the definition in mk_oracle.h, with fp64 arithmetic
 * and no blocking or reordering of a sum.  OpenMP only splits independent
 * tokens or rows across threads.
 */
#include "mk_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int mko_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* A logit is inside the contract when it is finite or -inf. */
static int logit_ok(float v) { return !(isnan(v) || (isinf(v) && v > 0)); }

/* Key order of step 1: expert a comes before expert b when its logit is
 * larger, or when the logits are equal and its id is smaller. */
static int precedes(const float* l, int a, int b) {
    if (l[a] > l[b]) return 1;
    if (l[a] == l[b] && a < b) return 1;
    return 0;
}

static double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int mko_route(const float* logits, int64_t T, int E, int k,
              int32_t* topk_idx, float* topk_gate) {
    if (T < 0 || E < 1 || k < 1 || k > E) return MKO_EARG;
    if (T > 0 && (!logits || !topk_idx || !topk_gate)) return MKO_EARG;
    for (int64_t i = 0; i < T * (int64_t)E; ++i)
        if (!logit_ok(logits[i])) return MKO_EBADVAL;

    int bad = 0;
#pragma omp parallel for schedule(static) reduction(|: bad)
    for (int64_t t = 0; t < T; ++t) {
        const float* l = logits + t * (int64_t)E;
        int* taken = (int*)calloc((size_t)E, sizeof(int));
        if (!taken) { bad = 1; continue; }
        /* Step 1: the first k positions of the key order, found one at a
         * time (a selection sort stopped after k picks). */
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || precedes(l, e, best)) best = e;
            }
            taken[best] = 1;
            topk_idx[t * k + j] = best;
        }
        free(taken);
        /* Step 2: softmax over the chosen logits, relative to slot 0. */
        double l0 = (double)l[topk_idx[t * k]];
        if (isinf(l0)) {
            for (int j = 0; j < k; ++j) topk_gate[t * k + j] = 0.0f;
        } else {
            double s = 0.0;
            for (int j = 0; j < k; ++j) s += exp((double)l[topk_idx[t * k + j]] - l0);
            for (int j = 0; j < k; ++j)
                topk_gate[t * k + j] = (float)(exp((double)l[topk_idx[t * k + j]] - l0) / s);
        }
    }
    return bad ? MKO_EARG : MKO_OK;
}

int mko_dispatch(const int32_t* topk_idx, const float* topk_gate,
                 int64_t T, int E, int k,
                 int32_t* expert_offsets, int32_t* src_index, float* gate_w) {
    if (T < 0 || E < 1 || k < 1 || k > E || !expert_offsets) return MKO_EARG;
    if (T > 0 && (!topk_idx || !topk_gate || !src_index || !gate_w)) return MKO_EARG;
    const int64_t n = T * (int64_t)k;
    for (int64_t i = 0; i < n; ++i)
        if (topk_idx[i] < 0 || topk_idx[i] >= E) return MKO_EARG;

    /* Step 3: histogram. */
    int64_t* count = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    if (!count) return MKO_EARG;
    for (int64_t i = 0; i < n; ++i) count[topk_idx[i]] += 1;

    /* Step 4: exclusive scan. */
    int64_t run = 0;
    for (int e = 0; e < E; ++e) {
        expert_offsets[e] = (int32_t)run;
        run += count[e];
    }
    expert_offsets[E] = (int32_t)run;
    free(count);

    /* Steps 5-6: rows ordered by (e, t, j). */
    int64_t r = 0;
    for (int e = 0; e < E; ++e)
        for (int64_t t = 0; t < T; ++t)
            for (int j = 0; j < k; ++j)
                if (topk_idx[t * k + j] == e) {
                    src_index[r] = (int32_t)(t * k + j);
                    gate_w[r] = topk_gate[t * k + j];
                    ++r;
                }
    return MKO_OK;
}

int mko_gated_rows(const uint16_t* x, const uint16_t* W1, const uint16_t* W3,
                   int64_t T, int H, int F, int E, int k,
                   const int32_t* expert_offsets, const int32_t* src_index,
                   const int64_t* rows, int64_t n, double* y) {
    if (T < 0 || H < 1 || F < 1 || E < 1 || k < 1 || n < 0) return MKO_EARG;
    if (n > 0 && (!x || !W1 || !W3 || !expert_offsets || !src_index || !rows || !y)) return MKO_EARG;
    const int64_t nrows = T * (int64_t)k;
    for (int64_t i = 0; i < n; ++i)
        if (rows[i] < 0 || rows[i] >= nrows) return MKO_EARG;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(|: bad)
    for (int64_t i = 0; i < n; ++i) {
        const int64_t r = rows[i];
        int e = 0;
        while (!(expert_offsets[e] <= r && r < expert_offsets[e + 1])) ++e;
        const int64_t t = src_index[r] / k;
        const uint16_t* xt = x + t * (int64_t)H;
        const uint16_t* W1e = W1 + (int64_t)e * H * F;
        const uint16_t* W3e = W3 + (int64_t)e * H * F;
        double* a = (double*)calloc((size_t)F, sizeof(double));
        double* b = (double*)calloc((size_t)F, sizeof(double));
        if (!a || !b) {
            free(a);
            free(b);
            bad = 1;
            continue;
        }
        for (int h = 0; h < H; ++h) {
            const double xv = bf16_to_double(xt[h]);
            for (int f = 0; f < F; ++f) {
                a[f] += xv * bf16_to_double(W1e[(int64_t)h * F + f]);
                b[f] += xv * bf16_to_double(W3e[(int64_t)h * F + f]);
            }
        }
        double* yr = y + i * (int64_t)F;
        for (int f = 0; f < F; ++f) yr[f] = a[f] / (1.0 + exp(-a[f])) * b[f];
        free(a);
        free(b);
    }
    return bad ? MKO_EARG : MKO_OK;
}

int mko_combine(const double* y, const int32_t* src_index, const float* gate_w,
                int64_t T, int k, int F, double* out) {
    if (T < 0 || k < 1 || F < 1) return MKO_EARG;
    if (T > 0 && (!y || !src_index || !gate_w || !out)) return MKO_EARG;
    const int64_t n = T * (int64_t)k;
    for (int64_t r = 0; r < n; ++r)
        if (src_index[r] < 0 || src_index[r] >= n) return MKO_EARG;
    for (int64_t i = 0; i < T * (int64_t)F; ++i) out[i] = 0.0;
    /* every sorted row adds its gated product to its token's row */
    for (int64_t r = 0; r < n; ++r) {
        const int64_t t = src_index[r] / k;
        const double g = (double)gate_w[r];
        for (int f = 0; f < F; ++f) out[t * F + f] += g * y[r * F + f];
    }
    return MKO_OK;
}

int mko_expert_rows(const uint16_t* x, const uint16_t* W,
                    int64_t T, int H, int F, int E, int k,
                    const int32_t* expert_offsets, const int32_t* src_index,
                    const int64_t* rows, int64_t n, double* y) {
    if (T < 0 || H < 1 || F < 1 || E < 1 || k < 1 || n < 0) return MKO_EARG;
    if (n > 0 && (!x || !W || !expert_offsets || !src_index || !rows || !y)) return MKO_EARG;
    const int64_t nrows = T * (int64_t)k;
    for (int64_t i = 0; i < n; ++i)
        if (rows[i] < 0 || rows[i] >= nrows) return MKO_EARG;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n; ++i) {
        const int64_t r = rows[i];
        /* The expert that owns sorted row r. */
        int e = 0;
        while (!(expert_offsets[e] <= r && r < expert_offsets[e + 1])) ++e;
        const int64_t t = src_index[r] / k;
        const uint16_t* xt = x + t * (int64_t)H;
        const uint16_t* We = W + (int64_t)e * H * F;
        double* yr = y + i * (int64_t)F;
        for (int f = 0; f < F; ++f) yr[f] = 0.0;
        /* Step 7: ascending h for every output column. */
        for (int h = 0; h < H; ++h) {
            const double xv = bf16_to_double(xt[h]);
            const uint16_t* wrow = We + (int64_t)h * F;
            for (int f = 0; f < F; ++f) yr[f] += xv * bf16_to_double(wrow[f]);
        }
    }
    return MKO_OK;
}

/* First token of rank r: floor(r*T/R). */
static int64_t ep_token0(int64_t T, int R, int r) { return (T * (int64_t)r) / R; }

int mko_ep_layout(const int32_t* topk_idx, int64_t T, int E, int k, int R,
                  int32_t* cnt, int32_t* recv_offsets, int32_t* recv_src) {
    if (T < 0 || E < 1 || k < 1 || k > E || R < 1 || E % R != 0) return MKO_EARG;
    if (!cnt || !recv_offsets || (T > 0 && (!topk_idx || !recv_src))) return MKO_EARG;
    const int epr = E / R;
    for (int64_t i = 0; i < T * (int64_t)k; ++i)
        if (topk_idx[i] < 0 || topk_idx[i] >= E) return MKO_EARG;

    /* Step 1: every source rank counts its own entries per expert.
     * Step 2: the all-gather leaves the whole table on every rank (one
     * table here stands for the R identical copies). */
    memset(cnt, 0, sizeof(int32_t) * (size_t)R * (size_t)E);
    for (int r = 0; r < R; ++r)
        for (int64_t t = ep_token0(T, R, r); t < ep_token0(T, R, r + 1); ++t)
            for (int j = 0; j < k; ++j) cnt[(int64_t)r * E + topk_idx[t * k + j]] += 1;

    /* Step 3: receive offsets of the ranks, then the start of every block
     * (e, r) inside its destination's buffer. */
    int64_t* block = (int64_t*)malloc(sizeof(int64_t) * (size_t)R * (size_t)E);
    if (!block) return MKO_EARG;
    int64_t run = 0;
    for (int q = 0; q < R; ++q) {
        recv_offsets[q] = (int32_t)run;
        for (int e = q * epr; e < (q + 1) * epr; ++e)
            for (int r = 0; r < R; ++r) {
                block[(int64_t)r * E + e] = run;
                run += cnt[(int64_t)r * E + e];
            }
    }
    recv_offsets[R] = (int32_t)run;

    /* Step 4: each source sends its entries in (t, j) order; a block fills
     * in arrival order. */
    int bad = 0;
    for (int r = 0; r < R; ++r)
        for (int64_t t = ep_token0(T, R, r); t < ep_token0(T, R, r + 1); ++t)
            for (int j = 0; j < k; ++j) {
                const int e = topk_idx[t * k + j];
                const int64_t at = block[(int64_t)r * E + e]++;
                if (at < 0 || at >= T * (int64_t)k) bad = 1;  /* a block outside the buffers */
                else recv_src[at] = (int32_t)(t * k + j);
            }
    free(block);
    return bad ? MKO_EARG : MKO_OK;
}
