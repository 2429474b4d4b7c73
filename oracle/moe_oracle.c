/*
 * moe_oracle.c -- plain, slow, fp64 CPU oracle for the forward pass of one
 * Mixture-of-Experts FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file: only the tests, __graft_entry__.smoke() and bench.py's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library; the only thing both sides see is the seeded input data.
 *
 * What is computed, and where the pages define it:
 *   - The MoE layer replaces the FFN with a router plus E small experts; the
 *     router picks experts per token (HARMOEny write-up, part 1 "What is MoE").
 *   - Each expert is a two-layer MLP x.W1.W2 with W1 of shape m x p and W2 of
 *     shape p x m (HARMOEny write-up, part 3.2 "expert prefetch").  The pages
 *     do not name the activation: the two-matrix form uses ReLU between the
 *     layers; the three-matrix (Mixtral / Phi-3.5-MoE) form uses
 *     SiLU(x.W1) * (x.W3) before W2.
 *   - The tokens are dispatched to their experts and the finished tokens are
 *     gathered back in token order (HARMOEny write-up, part 2, the two
 *     exchanges around expert compute; part 3.3 steps 4 and 6).  On one device
 *     the dispatch is a stable counting sort by expert.
 *
 * Readings chosen where the pages are silent:
 *   - top-k is taken on the raw logits, larger logit first, ties to the lower
 *     expert id; the k weights are the softmax renormalised over the k chosen,
 *     exp(l_j - l_0) / sum_j' exp(l_j' - l_0).
 *   - Inside one expert's segment, tokens keep flat-index order i = t*k + j.
 *   - The combine sums the k weighted expert outputs in ascending j.
 *   - int8 weights are per-output-column symmetric: scale = max|W[:,c]| / 127
 *     and code = round-half-even(W / scale) clamped to [-127, 127], both in
 *     fp32 (the precision the device uses for the same decision); an all-zero
 *     column gets scale 1 and codes 0.  The oracle then computes with
 *     code * scale in fp64.
 *
 * Every dot product runs in fp64 in ascending reduction index, starting from
 * its first product.  The optional operation counter counts exactly the
 * multiplies and adds these loops execute, so that the count can be checked
 * against the closed form |O| = q p (2m - 1) + q m (2p - 1) of the HARMOEny
 * write-up, part 3.2.
 *
 * Element types: 0 = fp32, 1 = bf16 (raw 16-bit patterns), 2 = int8 codes
 * (with a per-column fp32 scale), 3 = fp64.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_BF16 = 1, OR_I8 = 2, OR_F64 = 3 };
enum { OR_RELU2 = 0, OR_SWIGLU = 1 };

enum {
    OR_OK = 0,
    OR_BAD_ARG = 1,
    OR_NONFINITE = 2,
    OR_NOMEM = 3,
};

/* bf16 is the top half of an fp32 bit pattern; widening is exact. */
static double bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Element i of an array of the given type.  For int8 the caller applies the
 * column scale. */
static double elem(const void *base, int dtype, size_t i) {
    switch (dtype) {
    case OR_F32: return (double)((const float *)base)[i];
    case OR_BF16: return bf16_to_double(((const uint16_t *)base)[i]);
    case OR_I8: return (double)((const int8_t *)base)[i];
    default: return ((const double *)base)[i];
    }
}

/* Weight element W[r][c] of a row-major rows x cols matrix; int8 codes are
 * multiplied by the per-column scale. */
static double welem(const void *w, int dtype, const float *scale, size_t cols,
                    size_t r, size_t c) {
    double v = elem(w, dtype, r * cols + c);
    if (dtype == OR_I8) v *= (double)scale[c];
    return v;
}

/* ------------------------------------------------------------------------ */
/* Router GEMM: logits[t][e] = sum_c x[t][c] * Wr[c][e] (+ bias[e]).
 * abssum[t][e] = sum_c |x[t][c] * Wr[c][e]| bounds the rounding error of any
 * finite-precision evaluation of the same sum; it may be NULL.
 * Router: HARMOEny write-up part 1 and part 3.3 step 1; the gating network
 * runs on the GPU in the expert-cache article, section 3.1. */
int moe_oracle_router_logits(const void *x, int x_dtype, const void *wr,
                             int wr_dtype, const double *bias, int T, int m,
                             int E, double *logits, double *abssum) {
    if (!x || !wr || !logits || T < 0 || m <= 0 || E <= 0) return OR_BAD_ARG;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            double acc = 0.0, mag = 0.0;
            for (int c = 0; c < m; ++c) {
                double xv = elem(x, x_dtype, (size_t)t * m + c);
                double wv = elem(wr, wr_dtype, (size_t)c * E + e);
                double prod = xv * wv;
                if (!isfinite(xv) || !isfinite(wv)) bad = 1;
                acc = (c == 0) ? prod : acc + prod;
                mag += fabs(prod);
            }
            if (bias) acc += bias[e];
            logits[(size_t)t * E + e] = acc;
            if (abssum) abssum[(size_t)t * E + e] = mag;
        }
    }
    return bad ? OR_NONFINITE : OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Softmax + top-k + renormalisation.  For each token: order the experts by
 * (logit descending, expert id ascending), keep the first k, and give slot j
 * the weight exp(l_j - l_0) / sum_{j'<k} exp(l_j' - l_0).  This equals a full
 * softmax over E followed by renormalisation over the k chosen.
 * Selection is a pure comparison of the given values, so feeding fp32 logits
 * (widened exactly to fp64) reproduces an fp32 selection. */
int moe_oracle_topk(const double *logits, int T, int E, int k, int32_t *ids,
                    double *weights) {
    if (!logits || !ids || !weights || T < 0 || E <= 0 || k <= 0 || k > E)
        return OR_BAD_ARG;
    for (int t = 0; t < T; ++t) {
        const double *l = logits + (size_t)t * E;
        for (int e = 0; e < E; ++e)
            if (!isfinite(l[e])) return OR_NONFINITE;
        /* Selection sort on (value desc, id asc): slot j takes the best
         * expert not yet taken. */
        int32_t *out = ids + (size_t)t * k;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                int taken = 0;
                for (int jj = 0; jj < j; ++jj)
                    if (out[jj] == e) taken = 1;
                if (taken) continue;
                if (best < 0 || l[e] > l[best]) best = e; /* ties keep lower id */
            }
            out[j] = best;
        }
        double denom = 0.0;
        for (int j = 0; j < k; ++j) denom += exp(l[out[j]] - l[out[0]]);
        for (int j = 0; j < k; ++j)
            weights[(size_t)t * k + j] = exp(l[out[j]] - l[out[0]]) / denom;
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Histogram, exclusive scan and stable scatter of the n = T*k flat indices
 * i = t*k + j by expert id (the single-device form of the dispatch step,
 * HARMOEny write-up part 2 and part 3.3 step 4):
 *   counts[e]   = #{i : ids[i] == e}
 *   offsets[0]  = 0, offsets[e+1] = offsets[e] + counts[e]
 *   pos(i)      = offsets[ids[i]] + #{i' < i : ids[i'] == ids[i]}
 *   gather[pos(i)] = i,  scatter[i] = pos(i)
 * Returns OR_BAD_ARG if an id is out of range. */
int moe_oracle_permute(const int32_t *ids, int T, int k, int E, int32_t *counts,
                       int32_t *offsets, int32_t *gather, int32_t *scatter) {
    if (!ids || !counts || !offsets || !gather || !scatter || T < 0 || k <= 0 ||
        E <= 0)
        return OR_BAD_ARG;
    const int n = T * k;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= E) return OR_BAD_ARG;
        counts[ids[i]] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    for (int i = 0; i < n; ++i) {
        int e = ids[i];
        int before = 0;
        for (int i2 = 0; i2 < i; ++i2)
            if (ids[i2] == e) before += 1;
        int pos = offsets[e] + before;
        gather[pos] = i;
        scatter[i] = pos;
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Per-column symmetric int8 quantisation of a row-major rows x cols matrix
 * (DeepSpeed-Inference article, part 4: INT8 GEMM with quantise before and
 * dequantise after the product; the scheme itself is this build's reading).
 * The decisions are taken in fp32:
 *   scale[c] = fp32(max_r |W[r][c]|) / 127   (fp32 division)
 *   q[r][c]  = clamp(rint(fp32(W[r][c] / scale[c])), -127, 127)
 * with an all-zero column given scale 1 and codes 0.  fp32 division is
 * computed as an fp64 division rounded once to fp32, which equals the
 * correctly rounded fp32 quotient of two fp32 operands. */
int moe_oracle_quantize_cols(const void *w, int w_dtype, int rows, int cols,
                             int8_t *q, float *scale) {
    if (!w || !q || !scale || rows <= 0 || cols <= 0 || w_dtype == OR_I8)
        return OR_BAD_ARG;
    /* column maxima, scanning the matrix row by row */
    for (int c = 0; c < cols; ++c) scale[c] = 0.0f;
    for (int r = 0; r < rows; ++r) {
        for (int c = 0; c < cols; ++c) {
            float v = (float)elem(w, w_dtype, (size_t)r * cols + c);
            if (!isfinite(v)) return OR_NONFINITE;
            if (fabsf(v) > scale[c]) scale[c] = fabsf(v);
        }
    }
    for (int c = 0; c < cols; ++c)
        scale[c] = (scale[c] == 0.0f) ? 1.0f : (float)((double)scale[c] / 127.0);
    for (int r = 0; r < rows; ++r) {
        for (int c = 0; c < cols; ++c) {
            float v = (float)elem(w, w_dtype, (size_t)r * cols + c);
            float ratio = (float)((double)v / (double)scale[c]);
            double code = rint((double)ratio); /* default mode: half to even */
            if (code > 127.0) code = 127.0;
            if (code < -127.0) code = -127.0;
            q[(size_t)r * cols + c] = (int8_t)code;
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* One expert applied to one token row x (length m):
 *   two-matrix form : h = max(0, x.W1)                  (W1: m x p)
 *   three-matrix form: h = silu(x.W1) * (x.W3), silu(z) = z / (1 + e^-z)
 *   out = h.W2                                            (W2: p x m)
 * Expert shape and |E|, |O|: HARMOEny write-up part 3.2.
 * ops (may be NULL) accumulates [multiplies, adds, activations, gate
 * multiplies] actually executed; each dot product starts from its first
 * product, so a length-L dot costs L multiplies and L-1 adds. */
static int expert_row(const void *xrow, int x_dtype, size_t x_off,
                      const void *w1, const void *w2, const void *w3,
                      int w_dtype, const float *s1, const float *s2,
                      const float *s3, int m, int p, int kind, double *h,
                      double *u, double *out, long long *ops) {
    /* up projection(s): h[n] = sum_c x[c] W1[c][n], ascending c */
    for (int c = 0; c < m; ++c) {
        double xv = elem(xrow, x_dtype, x_off + (size_t)c);
        if (!isfinite(xv)) return OR_NONFINITE;
        for (int n = 0; n < p; ++n) {
            double prod = xv * welem(w1, w_dtype, s1, (size_t)p, (size_t)c, (size_t)n);
            h[n] = (c == 0) ? prod : h[n] + prod;
            if (kind == OR_SWIGLU) {
                double prod3 = xv * welem(w3, w_dtype, s3, (size_t)p, (size_t)c, (size_t)n);
                u[n] = (c == 0) ? prod3 : u[n] + prod3;
            }
        }
    }
    if (ops) {
        long long dots = (kind == OR_SWIGLU) ? 2LL * p : (long long)p;
        ops[0] += dots * m;
        ops[1] += dots * (m - 1);
    }
    for (int n = 0; n < p; ++n) {
        if (kind == OR_SWIGLU) {
            double g = h[n];
            h[n] = (g / (1.0 + exp(-g))) * u[n];
        } else {
            h[n] = h[n] > 0.0 ? h[n] : 0.0;
        }
    }
    if (ops) {
        ops[2] += p;
        if (kind == OR_SWIGLU) ops[3] += p;
    }
    /* down projection: out[r] = sum_n h[n] W2[n][r], ascending n */
    for (int n = 0; n < p; ++n) {
        for (int r = 0; r < m; ++r) {
            double prod = h[n] * welem(w2, w_dtype, s2, (size_t)m, (size_t)n, (size_t)r);
            out[r] = (n == 0) ? prod : out[r] + prod;
        }
    }
    if (ops) {
        ops[0] += (long long)m * p;
        ops[1] += (long long)m * (p - 1);
    }
    return OR_OK;
}

/* One expert on one token, exposed for the tests.  h_out (length p) receives
 * the activation, out (length m) the down projection; ops as above. */
int moe_oracle_expert(const void *x, int x_dtype, const void *w1, const void *w2,
                      const void *w3, int w_dtype, const float *s1,
                      const float *s2, const float *s3, int m, int p, int kind,
                      double *h_out, double *out, long long *ops) {
    if (!x || !w1 || !w2 || !h_out || !out || m <= 0 || p <= 0) return OR_BAD_ARG;
    if (kind == OR_SWIGLU && !w3) return OR_BAD_ARG;
    if (w_dtype == OR_I8 && (!s1 || !s2 || (kind == OR_SWIGLU && !s3)))
        return OR_BAD_ARG;
    double *u = (double *)malloc(sizeof(double) * (size_t)p);
    if (!u) return OR_NOMEM;
    int rc = expert_row(x, x_dtype, 0, w1, w2, w3, w_dtype, s1, s2, s3, m, p,
                        kind, h_out, u, out, ops);
    free(u);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Whole layer for a chosen list of tokens, given the routing:
 *   y[t] = sum_{j=0..k-1} w[t][j] * expert_{ids[t][j]}(x[t]),  ascending j.
 * w1/w2/w3/s1/s2/s3 are arrays of E per-expert pointers (row-major, as the
 * user hands them over); tokens lists the token indices to evaluate (NULL:
 * all T); y receives n_tokens x m values.  ops, if non-NULL, is an E x 4
 * array of per-expert operation counts and forces one thread. */
int moe_oracle_layer(const void *x, int x_dtype, int T, int m, int p, int E,
                     int k, const void *const *w1, const void *const *w2,
                     const void *const *w3, int w_dtype,
                     const float *const *s1, const float *const *s2,
                     const float *const *s3, int kind, const int32_t *ids,
                     const double *weights, const int32_t *tokens, int n_tokens,
                     double *y, long long *ops, int nthreads) {
    if (!x || !w1 || !w2 || !ids || !weights || !y || T < 0 || m <= 0 || p <= 0 ||
        E <= 0 || k <= 0)
        return OR_BAD_ARG;
    if (kind == OR_SWIGLU && !w3) return OR_BAD_ARG;
    if (!tokens) n_tokens = T;
    int rc_all = OR_OK;
#ifdef _OPENMP
    if (ops) nthreads = 1;
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#endif
#pragma omp parallel num_threads(nthreads) reduction(max : rc_all)
    {
        double *h = (double *)malloc(sizeof(double) * (size_t)p);
        double *u = (double *)malloc(sizeof(double) * (size_t)p);
        double *o = (double *)malloc(sizeof(double) * (size_t)m);
        if (!h || !u || !o) {
            rc_all = OR_NOMEM;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int s = 0; s < n_tokens; ++s) {
                int t = tokens ? tokens[s] : s;
                double *yt = y + (size_t)s * m;
                if (t < 0 || t >= T) {
                    rc_all = OR_BAD_ARG;
                    continue;
                }
                for (int j = 0; j < k; ++j) {
                    int e = ids[(size_t)t * k + j];
                    if (e < 0 || e >= E) {
                        rc_all = OR_BAD_ARG;
                        break;
                    }
                    int rc = expert_row(
                        x, x_dtype, (size_t)t * m, w1[e], w2[e],
                        w3 ? w3[e] : NULL, w_dtype, s1 ? s1[e] : NULL,
                        s2 ? s2[e] : NULL, s3 ? s3[e] : NULL, m, p, kind, h, u, o,
                        ops ? ops + 4 * (size_t)e : NULL);
                    if (rc != OR_OK) {
                        rc_all = rc;
                        break;
                    }
                    double wj = weights[(size_t)t * k + j];
                    for (int r = 0; r < m; ++r)
                        yt[r] = (j == 0) ? wj * o[r] : yt[r] + wj * o[r];
                }
            }
        }
        free(h);
        free(u);
        free(o);
    }
    return rc_all;
}

/* ------------------------------------------------------------------------ */
/* N-index x M-way set-associative expert cache with LRU replacement inside a
 * set, set = layer_id mod N (expert-cache article, section 2.2).  Replays a
 * sequence of (layer, expert) queries and writes 1 for a hit, 0 for a miss.
 * A miss inserts the expert, evicting the least recently used way of the set
 * when all M ways are full.  The slot number (set * M + way) that serves each
 * query is written to slot_out (may be NULL). */
int moe_oracle_cache_replay(int n_index, int n_way, int n_queries,
                            const int32_t *layer, const int32_t *expert,
                            int32_t *hit_out, int32_t *slot_out) {
    if (n_index <= 0 || n_way <= 0 || n_queries < 0 || !layer || !expert || !hit_out)
        return OR_BAD_ARG;
    size_t n_slots = (size_t)n_index * n_way;
    long long *tag_layer = (long long *)malloc(sizeof(long long) * n_slots);
    long long *tag_expert = (long long *)malloc(sizeof(long long) * n_slots);
    long long *last_use = (long long *)malloc(sizeof(long long) * n_slots);
    if (!tag_layer || !tag_expert || !last_use) {
        free(tag_layer);
        free(tag_expert);
        free(last_use);
        return OR_NOMEM;
    }
    for (size_t s = 0; s < n_slots; ++s) {
        tag_layer[s] = -1;
        tag_expert[s] = -1;
        last_use[s] = -1;
    }
    for (int qi = 0; qi < n_queries; ++qi) {
        int set = layer[qi] % n_index;
        size_t base = (size_t)set * n_way;
        int found = -1;
        for (int w = 0; w < n_way; ++w)
            if (tag_layer[base + w] == layer[qi] && tag_expert[base + w] == expert[qi])
                found = w;
        if (found < 0) {
            /* an empty way first (lowest index), else the least recently used */
            int victim = -1;
            for (int w = 0; w < n_way && victim < 0; ++w)
                if (tag_layer[base + w] < 0) victim = w;
            if (victim < 0) {
                victim = 0;
                for (int w = 1; w < n_way; ++w)
                    if (last_use[base + w] < last_use[base + victim]) victim = w;
            }
            tag_layer[base + victim] = layer[qi];
            tag_expert[base + victim] = expert[qi];
            found = victim;
            hit_out[qi] = 0;
        } else {
            hit_out[qi] = 1;
        }
        last_use[base + found] = qi;
        if (slot_out) slot_out[qi] = (int32_t)(base + found);
    }
    free(tag_layer);
    free(tag_expert);
    free(last_use);
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* The same cache driven by whole layer calls, with optional cross-layer
 * prefetch: experts chosen in layer l are fetched for layer l + 1 ahead of
 * its call (HARMOEny write-up, part 3.2: prefetch the next layer's experts
 * during the current layer's compute; expert-cache article, section 2.1:
 * consecutive layers often pick the same experts).
 *
 * Call c is layer call_layer[c] with per-expert token counts
 * counts[c * E .. c * E + E - 1].  For each call:
 *   1. demand: every expert with tokens, in ascending id, is looked up in set
 *      layer mod N; a miss takes an empty way (lowest index) or the least
 *      recently used way; every lookup makes the way most recently used;
 *   2. prefetch (n_prefetch > 0, layer + 1 < n_layers, and layer + 1 maps to a
 *      different set): the n_prefetch experts of this call with the most
 *      tokens (ties to the lower id) are looked up for layer + 1; one that is
 *      not resident is inserted as in a miss and becomes most recently used;
 *      one that is resident is left untouched.
 * Log entry i: layer_out, expert_out, kind_out (0 demand miss, 1 demand hit,
 * 2 prefetch insert, 3 demand hit on a prefetched entry not used before) and
 * slot_out (set * M + way).  Writes at most max_out entries; *n_out receives
 * the number of entries the replay produced. */
int moe_oracle_cache_replay_calls(int n_index, int n_way, int n_calls, const int32_t *call_layer,
                                  int E, const int32_t *counts, int n_layers, int n_prefetch,
                                  int32_t *layer_out, int32_t *expert_out, int32_t *kind_out,
                                  int32_t *slot_out, int max_out, int *n_out) {
    if (n_index <= 0 || n_way <= 0 || n_calls < 0 || E <= 0 || n_prefetch < 0 || !n_out ||
        (n_calls > 0 && (!call_layer || !counts)) || max_out < 0)
        return OR_BAD_ARG;
    size_t n_slots = (size_t)n_index * n_way;
    long long *tag_layer = (long long *)malloc(sizeof(long long) * n_slots);
    long long *tag_expert = (long long *)malloc(sizeof(long long) * n_slots);
    long long *last_use = (long long *)malloc(sizeof(long long) * n_slots);
    int *fetched = (int *)malloc(sizeof(int) * n_slots); /* inserted by prefetch, unused */
    int *order = (int *)malloc(sizeof(int) * (size_t)E);
    if (!tag_layer || !tag_expert || !last_use || !fetched || !order) {
        free(tag_layer);
        free(tag_expert);
        free(last_use);
        free(fetched);
        free(order);
        return OR_NOMEM;
    }
    for (size_t s = 0; s < n_slots; ++s) {
        tag_layer[s] = -1;
        tag_expert[s] = -1;
        last_use[s] = -1;
        fetched[s] = 0;
    }
    long long clock = 0;
    int n = 0;
#define OR_LOG(L_, E_, K_, S_)                              \
    do {                                                    \
        if (n < max_out) {                                  \
            if (layer_out) layer_out[n] = (int32_t)(L_);    \
            if (expert_out) expert_out[n] = (int32_t)(E_);  \
            if (kind_out) kind_out[n] = (int32_t)(K_);      \
            if (slot_out) slot_out[n] = (int32_t)(S_);      \
        }                                                   \
        ++n;                                                \
    } while (0)
    for (int c = 0; c < n_calls; ++c) {
        const int l = call_layer[c];
        const int32_t *cnt = counts + (size_t)c * E;
        /* 1. demand lookups */
        for (int e = 0; e < E; ++e) {
            if (cnt[e] <= 0) continue;
            size_t base = (size_t)(l % n_index) * n_way;
            int found = -1;
            for (int w = 0; w < n_way; ++w)
                if (tag_layer[base + w] == l && tag_expert[base + w] == e) found = w;
            int kind;
            if (found < 0) {
                int victim = -1;
                for (int w = 0; w < n_way && victim < 0; ++w)
                    if (tag_layer[base + w] < 0) victim = w;
                if (victim < 0) {
                    victim = 0;
                    for (int w = 1; w < n_way; ++w)
                        if (last_use[base + w] < last_use[base + victim]) victim = w;
                }
                tag_layer[base + victim] = l;
                tag_expert[base + victim] = e;
                fetched[base + victim] = 0;
                found = victim;
                kind = 0;
            } else {
                kind = fetched[base + found] ? 3 : 1;
                fetched[base + found] = 0;
            }
            last_use[base + found] = clock++;
            OR_LOG(l, e, kind, base + found);
        }
        /* 2. prefetch for the next layer */
        const int nl = l + 1;
        if (n_prefetch == 0 || nl >= n_layers || (nl % n_index) == (l % n_index)) continue;
        int n_cand = 0;
        for (int e = 0; e < E; ++e)
            if (cnt[e] > 0) order[n_cand++] = e;
        /* by count descending, ties to the lower id (insertion sort: stable) */
        for (int i = 1; i < n_cand; ++i) {
            int v = order[i], j = i - 1;
            while (j >= 0 && cnt[order[j]] < cnt[v]) {
                order[j + 1] = order[j];
                --j;
            }
            order[j + 1] = v;
        }
        if (n_cand > n_prefetch) n_cand = n_prefetch;
        size_t base = (size_t)(nl % n_index) * n_way;
        for (int i = 0; i < n_cand; ++i) {
            const int e = order[i];
            int found = -1;
            for (int w = 0; w < n_way; ++w)
                if (tag_layer[base + w] == nl && tag_expert[base + w] == e) found = w;
            if (found >= 0) continue;
            int victim = -1;
            for (int w = 0; w < n_way && victim < 0; ++w)
                if (tag_layer[base + w] < 0) victim = w;
            if (victim < 0) {
                victim = 0;
                for (int w = 1; w < n_way; ++w)
                    if (last_use[base + w] < last_use[base + victim]) victim = w;
            }
            tag_layer[base + victim] = nl;
            tag_expert[base + victim] = e;
            fetched[base + victim] = 1;
            last_use[base + victim] = clock++;
            OR_LOG(nl, e, 2, base + victim);
        }
    }
#undef OR_LOG
    *n_out = n;
    free(tag_layer);
    free(tag_expert);
    free(last_use);
    free(fetched);
    free(order);
    return OR_OK;
}
