/*
 * moe_oracle.c -- the CPU oracle for the Qwen3.6-35B-A3B mixture-of-experts layer
 * over MLX affine 4-bit (group-64) expert weights.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark load this file.  The CUDA library never calls it and shares
 * no code, header or constant with it.
 *
 * It is deliberately plain: one token at a time, one output at a time, inputs in
 * ascending order, every value held in double precision.  Tokens are independent,
 * so an OpenMP loop over tokens is the only parallelism.
 *
 * What the layer computes (sources are the three news pages about Perplexity's
 * Lily engine; "p1" is aimanavo.com "Why is Perplexity's local AI Lily faster than
 * MLX", "p3" is news.mantis.guru "Perplexity opened Lily -- a specialised inference
 * engine for Apple silicon"):
 *   - every token scores all 256 experts, keeps 8 and adds one shared expert
 *     (p1, section "Qwen3.6's 256 experts and two layer kinds make the MLX/Lily gap");
 *   - expert weights are MLX affine 4-bit with group size 64
 *     (p1, "Only one 4-bit checkpoint of a pinned revision runs"; p3, "Rust drives
 *     the model, Metal computes").
 * The pages give no formulas.  The plain reading used here, stated once:
 *   unpack   q[o][i] = (Wq[o][i/8] >> 4*(i%8)) & 15            (low nibble first)
 *   dequant  w[o][i] = scale[o][i/g] * q[o][i] + bias[o][i/g]
 *   router   l_e = fp32( sum_i x_i * Wr[e][i] ) (+ fp32 bias_e, an fp32 add)
 *            p = softmax(l); top-k by (p descending, expert ascending);
 *            w_k = p_k / sum of the k chosen p
 *   expert   g = Wg x, u = Wu x, h = silu(g) * u, y = Wd h;  silu(z) = z / (1 + e^-z)
 *   shared   s = sigmoid(g_s . x) multiplies the shared expert's y
 *   output   o = sum_k w_k y_k + s * y_shared (+ x when the residual is asked for),
 *            rounded once to bf16 (nearest, ties to even).
 *   norm     (stacked layers only) the layer's input is first RMS-normalised,
 *            x_n = bf16( x / sqrt(mean(x^2) + 1e-6) * norm_w ), and the residual adds
 *            the un-normalised x.  Without it a stack of these layers diverges: the
 *            SwiGLU output grows with the square of its input, so the residual stream
 *            grows doubly exponentially (it reaches inf within about 7 layers).  A norm
 *            before the mixture-of-experts block is how the real model keeps the scale;
 *            the pages name the 40-layer hybrid stack (p1, section "Qwen3.6's 256
 *            experts and two layer kinds make the MLX/Lily gap") but print no formula.
 * Router logits are fp32 values (the one place where the precision decides an
 * integer result, the chosen experts); they are the exact dot product rounded
 * once to fp32.  Everything else is double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#include "moe_oracle.h"

/* Planted mistakes, for the test that checks the pins catch them.  0 = none. */
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* ---------------------------------------------------------------- bf16 */

double oracle_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bfloat16 (ties to even) in one step: keep eight
 * significant bits (seven stored plus the hidden one), with the subnormal quantum
 * 2^-133 as the floor and overflow to infinity. */
uint16_t oracle_double_to_bf16(double v) {
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (isnan(v)) return 0x7FC0u;
    if (isinf(v)) return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                  /* a = m * 2^e, m in [0.5, 1) */
    int qexp = e - 8;              /* quantum of an 8-significant-bit value */
    if (qexp < -133) qexp = -133;  /* bf16 subnormals */
    double r = nearbyint(ldexp(a, -qexp)) ; /* default rounding mode: ties to even */
    double rv = ldexp(r, qexp);
    if (rv >= 0x1p128) return (uint16_t)(sign | 0x7F80u);
    float f = (float)rv;           /* exact: rv has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

/* ---------------------------------------------------------------- 4-bit */

void oracle_unpack4(uint32_t word, int q[8]) {
    for (int i = 0; i < 8; ++i) {
#if ORACLE_MUTANT == 1
        q[i] = (int)((word >> (4 * (7 - i))) & 0xFu);   /* planted: high nibble first */
#else
        q[i] = (int)((word >> (4 * i)) & 0xFu);
#endif
    }
}

void oracle_dequant_row(const uint32_t* q_row, const uint16_t* s_row, const uint16_t* b_row,
                        int in_dim, int group, double* w) {
    int q[8];
    for (int i = 0; i < in_dim; i += 8) {
        oracle_unpack4(q_row[i / 8], q);
        for (int j = 0; j < 8; ++j) {
            int col = i + j;
#if ORACLE_MUTANT == 5
            int g = (col / group + 1) % (in_dim / group);  /* planted: wrong group index */
#else
            int g = col / group;
#endif
            double s = oracle_bf16_to_double(s_row[g]);
            double b = oracle_bf16_to_double(b_row[g]);
#if ORACLE_MUTANT == 2
            w[col] = s * q[j];                             /* planted: bias dropped */
#else
            w[col] = s * q[j] + b;
#endif
        }
    }
}

/* y = W x for matrix number `mat` of a stack of [out_dim][in_dim] 4-bit matrices. */
void oracle_qmatvec(const oracle_qmat_t* m, long mat, int out_dim, int in_dim, int group,
                    const double* x, double* y) {
    double* w = (double*)malloc(sizeof(double) * (size_t)in_dim);
    const size_t qstride = (size_t)in_dim / 8, gstride = (size_t)in_dim / (size_t)group;
    const size_t qbase = (size_t)mat * out_dim * qstride, gbase = (size_t)mat * out_dim * gstride;
    for (int o = 0; o < out_dim; ++o) {
#if ORACLE_MUTANT == 7
        /* planted: operand transposed -- reads row (o + 1) */
        int ro = (o + 1) % out_dim;
#else
        int ro = o;
#endif
        oracle_dequant_row(m->q + qbase + (size_t)ro * qstride, m->scales + gbase + (size_t)ro * gstride,
                           m->biases + gbase + (size_t)ro * gstride, in_dim, group, w);
        double acc = 0.0;
        for (int i = 0; i < in_dim; ++i) acc += w[i] * x[i];
        y[o] = acc;
    }
    free(w);
}

/* ---------------------------------------------------------------- router */

void oracle_router_logits(const oracle_dims_t* d, const uint16_t* router_w, const float* router_bias,
                          const uint16_t* x_row, float* logits) {
    for (int e = 0; e < d->n_experts; ++e) {
        double acc = 0.0;
        for (int i = 0; i < d->hidden; ++i)
            acc += oracle_bf16_to_double(x_row[i]) * oracle_bf16_to_double(router_w[(size_t)e * d->hidden + i]);
        float l = (float)acc;
        if (router_bias) l = (float)((double)l + (double)router_bias[e]);
        logits[e] = l;
    }
}

/* Softmax over all experts, then the top-k by (p desc, index asc), renormalised.
 * p_sorted (optional, n_experts entries) receives the probabilities in that order and
 * order (optional) the expert ids in that order. */
void oracle_route_logits(const oracle_dims_t* d, const float* logits, int32_t* idx, double* w,
                         double* gap, double* p_sorted, int32_t* order) {
    const int E = d->n_experts, K = d->top_k;
    double* p = (double*)malloc(sizeof(double) * (size_t)E);
    char* taken = (char*)calloc((size_t)E, 1);
    double mx = -INFINITY;
    for (int e = 0; e < E; ++e) if ((double)logits[e] > mx) mx = logits[e];
    double z = 0.0;
    for (int e = 0; e < E; ++e) { p[e] = exp((double)logits[e] - mx); z += p[e]; }
    for (int e = 0; e < E; ++e) p[e] /= z;
    /* selection sort by (p desc, e asc): strictly-greater keeps the lowest index on ties */
    int n_order = (p_sorted || order || gap) ? E : K;
    if (n_order > E) n_order = E;
    double sel_sum = 0.0;
    double pk = 0.0, pk1 = 0.0;
    for (int r = 0; r < n_order; ++r) {
        int best = -1;
        for (int e = 0; e < E; ++e)
            if (!taken[e] && (best < 0 || p[e] > p[best])) best = e;
        taken[best] = 1;
        if (p_sorted) p_sorted[r] = p[best];
        if (order) order[r] = best;
        if (r < K) {
            idx[r] = best;
            w[r] = p[best];
            sel_sum += p[best];
        }
        if (r == K - 1) pk = p[best];
        if (r == K) pk1 = p[best];
    }
    for (int k = 0; k < K; ++k) {
#if ORACLE_MUTANT == 4
        (void)sel_sum;                           /* planted: no renormalisation */
#else
        w[k] = w[k] / sel_sum;
#endif
    }
    if (gap) *gap = (K < E) ? (pk - pk1) / sel_sum : INFINITY;
    free(p);
    free(taken);
}

/* ---------------------------------------------------------------- input norm */

void oracle_rmsnorm(int hidden, const uint16_t* x_row, const uint16_t* norm_w, uint16_t* out) {
    double ss = 0.0;
    for (int i = 0; i < hidden; ++i) {
        const double v = oracle_bf16_to_double(x_row[i]);
        ss += v * v;
    }
#if ORACLE_MUTANT == 9
    const double r = 1.0 / sqrt(ss / hidden);                  /* planted: epsilon dropped */
#else
    const double r = 1.0 / sqrt(ss / hidden + ORACLE_RMS_EPS);
#endif
    for (int i = 0; i < hidden; ++i)
        out[i] = oracle_double_to_bf16(oracle_bf16_to_double(x_row[i]) * r * oracle_bf16_to_double(norm_w[i]));
}

/* ---------------------------------------------------------------- experts */

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* y (hidden) = Wd silu(Wg x) * (Wu x) for expert `e` of a stack (e = 0 for an unstacked matrix). */
void oracle_expert(const oracle_dims_t* d, const oracle_qmat_t* gate, const oracle_qmat_t* up,
                   const oracle_qmat_t* down, long e, int inter, const double* x, double* y) {
    double* g = (double*)malloc(sizeof(double) * (size_t)inter);
    double* u = (double*)malloc(sizeof(double) * (size_t)inter);
    oracle_qmatvec(gate, e, inter, d->hidden, d->group, x, g);
    oracle_qmatvec(up, e, inter, d->hidden, d->group, x, u);
    for (int j = 0; j < inter; ++j) {
#if ORACLE_MUTANT == 6
        g[j] = silu(u[j]) * g[j];                /* planted: gate and up swapped */
#else
        g[j] = silu(g[j]) * u[j];
#endif
    }
    oracle_qmatvec(down, e, d->hidden, inter, d->group, g, y);
    free(g);
    free(u);
}

double oracle_shared_gate(const oracle_dims_t* d, const uint16_t* shared_gate_w, const uint16_t* x_row) {
    double acc = 0.0;
    for (int i = 0; i < d->hidden; ++i)
        acc += oracle_bf16_to_double(shared_gate_w[i]) * oracle_bf16_to_double(x_row[i]);
#if ORACLE_MUTANT == 3
    return 1.0 / (1.0 + exp(acc));               /* planted: sign of the sigmoid */
#else
    return 1.0 / (1.0 + exp(-acc));
#endif
}

/* One token through the layer with a given expert choice and weights (no routing). */
void oracle_token_forward(const oracle_dims_t* d, const oracle_weights_t* W, const uint16_t* x_row,
                          const int32_t* experts, const double* wts, int residual, double* out) {
    const int H = d->hidden;
    double* x = (double*)malloc(sizeof(double) * (size_t)H);
    double* y = (double*)malloc(sizeof(double) * (size_t)H);
    uint16_t* xn_row = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)H);
    if (W->norm_w) oracle_rmsnorm(H, x_row, W->norm_w, xn_row);
    else memcpy(xn_row, x_row, sizeof(uint16_t) * (size_t)H);
    for (int i = 0; i < H; ++i) { x[i] = oracle_bf16_to_double(xn_row[i]); out[i] = 0.0; }
    for (int k = 0; k < d->top_k; ++k) {
        oracle_expert(d, &W->gate, &W->up, &W->down, experts[k], d->inter, x, y);
        for (int i = 0; i < H; ++i) out[i] += wts[k] * y[i];
    }
    double s = oracle_shared_gate(d, W->shared_gate_w, xn_row);
    oracle_expert(d, &W->sh_gate, &W->sh_up, &W->sh_down, 0, d->shared_inter, x, y);
#if ORACLE_MUTANT != 8
    for (int i = 0; i < H; ++i) out[i] += s * y[i];   /* (mutant 8 drops the shared expert) */
#else
    (void)s;
#endif
    if (residual)
#if ORACLE_MUTANT == 10
        for (int i = 0; i < H; ++i) out[i] += x[i];                              /* planted: normalised input */
#else
        for (int i = 0; i < H; ++i) out[i] += oracle_bf16_to_double(x_row[i]);   /* the un-normalised input */
#endif
    free(x);
    free(y);
    free(xn_row);
}

/* ---------------------------------------------------------------- whole layer */

/* The layer's router logits for one token: on the normalised input when the layer has a norm. */
void oracle_layer_logits(const oracle_dims_t* d, const oracle_weights_t* W, const uint16_t* x_row, float* l) {
    if (W->norm_w) {
        uint16_t* xn = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)d->hidden);
        oracle_rmsnorm(d->hidden, x_row, W->norm_w, xn);
        oracle_router_logits(d, W->router_w, W->router_bias, xn, l);
        free(xn);
    } else {
        oracle_router_logits(d, W->router_w, W->router_bias, x_row, l);
    }
}

void oracle_route(const oracle_dims_t* d, const oracle_weights_t* W, const uint16_t* x, int T, int nthreads,
                  int32_t* idx, double* wts, double* gap, int32_t* counts, int32_t* offsets, int32_t* perm) {
    const int E = d->n_experts, K = d->top_k;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int t = 0; t < T; ++t) {
        float* l = (float*)malloc(sizeof(float) * (size_t)E);
        oracle_layer_logits(d, W, x + (size_t)t * d->hidden, l);
        oracle_route_logits(d, l, idx + (size_t)t * K, wts + (size_t)t * K, gap ? gap + t : NULL, NULL, NULL);
        free(l);
    }
    (void)nthreads;
    if (counts || offsets || perm) {
        int32_t* c = (int32_t*)calloc((size_t)E, sizeof(int32_t));
        for (long s = 0; s < (long)T * K; ++s) c[idx[s]]++;
        int32_t* off = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 1));
        off[0] = 0;
        for (int e = 0; e < E; ++e) off[e + 1] = off[e] + c[e];
        if (counts) memcpy(counts, c, sizeof(int32_t) * (size_t)E);
        if (offsets) memcpy(offsets, off, sizeof(int32_t) * (size_t)(E + 1));
        if (perm) {
            /* stable: slots of one expert in ascending slot id t*K + k */
            int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
            for (long s = 0; s < (long)T * K; ++s) {
                int e = idx[s];
                perm[off[e] + fill[e]++] = (int32_t)s;
            }
            free(fill);
        }
        free(c);
        free(off);
    }
}

void oracle_layer_forward(const oracle_dims_t* d, const oracle_weights_t* W, const uint16_t* x, int T,
                          int residual, int nthreads, uint16_t* out, int32_t* idx, double* wts, double* gap) {
    const int E = d->n_experts, K = d->top_k, H = d->hidden;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int t = 0; t < T; ++t) {
        float* l = (float*)malloc(sizeof(float) * (size_t)E);
        int32_t* ti = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
        double* tw = (double*)malloc(sizeof(double) * (size_t)K);
        double* o = (double*)malloc(sizeof(double) * (size_t)H);
        double tg;
        oracle_layer_logits(d, W, x + (size_t)t * H, l);
        oracle_route_logits(d, l, ti, tw, &tg, NULL, NULL);
        oracle_token_forward(d, W, x + (size_t)t * H, ti, tw, residual, o);
        for (int i = 0; i < H; ++i) out[(size_t)t * H + i] = oracle_double_to_bf16(o[i]);
        if (idx) memcpy(idx + (size_t)t * K, ti, sizeof(int32_t) * (size_t)K);
        if (wts) memcpy(wts + (size_t)t * K, tw, sizeof(double) * (size_t)K);
        if (gap) gap[t] = tg;
        free(l); free(ti); free(tw); free(o);
    }
    (void)nthreads;
}

/* One token forward with a caller-given expert list; weights are recomputed from the
 * token's own router probabilities renormalised over that list.  Used to evaluate the
 * other valid choices of a near-tie token (the list comes from oracle_route_logits'
 * full order, never from the GPU). */
void oracle_token_forward_choice(const oracle_dims_t* d, const oracle_weights_t* W, const uint16_t* x_row,
                                 const int32_t* experts, int residual, uint16_t* out, double* wts_out) {
    const int E = d->n_experts, K = d->top_k, H = d->hidden;
    float* l = (float*)malloc(sizeof(float) * (size_t)E);
    double* p = (double*)malloc(sizeof(double) * (size_t)E);
    double* w = (double*)malloc(sizeof(double) * (size_t)K);
    double* o = (double*)malloc(sizeof(double) * (size_t)H);
    oracle_layer_logits(d, W, x_row, l);
    double mx = -INFINITY, z = 0.0, sel = 0.0;
    for (int e = 0; e < E; ++e) if ((double)l[e] > mx) mx = l[e];
    for (int e = 0; e < E; ++e) { p[e] = exp((double)l[e] - mx); z += p[e]; }
    for (int k = 0; k < K; ++k) { w[k] = p[experts[k]] / z; sel += w[k]; }
    for (int k = 0; k < K; ++k) w[k] /= sel;
    oracle_token_forward(d, W, x_row, experts, w, residual, o);
    for (int i = 0; i < H; ++i) out[i] = oracle_double_to_bf16(o[i]);
    if (wts_out) memcpy(wts_out, w, sizeof(double) * (size_t)K);
    free(l); free(p); free(w); free(o);
}

int oracle_mutant(void) { return ORACLE_MUTANT; }
