/*
 * gqa_oracle.c -- the CPU oracle for grouped-query decode attention, the second decode
 * workload of the model's 10 full-attention layers.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark load this file.  The CUDA library never calls it and shares no code,
 * header or constant with it.
 *
 * What the pages say (aimanavo.com, "Why is Perplexity's local AI Lily faster than MLX"):
 *   - the full-attention layers have 16 query heads and only 2 key/value heads, an 8-to-1
 *     compression of the KV cache (section "Qwen3.6's 256 experts and two layer kinds
 *     make the MLX/Lily gap");
 *   - decode reads the KV cache at every step and is bound by memory bandwidth, and Lily
 *     packs the query heads of a group so that every KV row is read once (section
 *     "Prefill and decode are not treated as the same job"; dzen.guru, "Perplexity opened
 *     the Lily engine", section "Where the speed-up comes from").
 * The pages give no formula and no head size.  The plain reading used here: standard
 * scaled dot-product attention of one new query token per sequence over that sequence's
 * cached keys and values, query head h reading KV head h / (Hq / Hkv):
 *   s_i   = scale * sum_d q[h][d] * k[g][i][d]           i < len   (scale = 1/sqrt(D))
 *   p_i   = exp(s_i - max_j s_j) / sum_j exp(s_j - max_j s_j)
 *   o[d]  = sum_i p_i * v[g][i][d]
 * Every value is held in double precision; q, k and v are bf16 inputs.  Alongside o the
 * oracle returns a[d] = sum_i p_i * |v[g][i][d]|, the size that bounds the rounding error
 * of any implementation that rounds the p_i (the parity tolerance is derived from it).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#include "moe_oracle.h"

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

static double gqa_bf16(uint16_t b) {
    union {
        uint32_t u;
        float f;
    } c;
    c.u = (uint32_t)b << 16;
    return (double)c.f;
}

/* Layouts: q [B][Hq][D], k and v [B][Hkv][S_max][D] (bf16 bits), lens [B] (1..S_max),
 * out and abs_out [B][Hq][D] (double). */
void oracle_gqa_decode(int B, int Hq, int Hkv, int D, int S_max, const int32_t* lens, const uint16_t* q,
                       const uint16_t* k, const uint16_t* v, double scale, int nthreads, double* out,
                       double* abs_out) {
#if ORACLE_MUTANT == 11
    scale = 1.0 / (double)D; /* planted: scale 1/D instead of 1/sqrt(D) */
#endif
#ifdef _OPENMP
    omp_set_num_threads(nthreads > 0 ? nthreads : 1);
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
#endif
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < Hq; ++h) {
#if ORACLE_MUTANT == 12
            const int g = h % Hkv; /* planted: heads interleaved across groups */
#else
            const int g = h / (Hq / Hkv);
#endif
            int n = lens[b];
#if ORACLE_MUTANT == 13
            n = n - 1; /* planted: the last key dropped */
#endif
            const uint16_t* qh = q + ((size_t)b * Hq + h) * D;
            const uint16_t* kg = k + ((size_t)b * Hkv + g) * S_max * D;
#if ORACLE_MUTANT == 14
            const uint16_t* vg = kg; /* planted: values read from the keys */
#else
            const uint16_t* vg = v + ((size_t)b * Hkv + g) * S_max * D;
#endif
            double* o = out + ((size_t)b * Hq + h) * D;
            double* a = abs_out + ((size_t)b * Hq + h) * D;
            /* scores and their maximum */
            double m = -INFINITY;
            for (int i = 0; i < n; ++i) {
                double s = 0.0;
                for (int d = 0; d < D; ++d) s += gqa_bf16(qh[d]) * gqa_bf16(kg[(size_t)i * D + d]);
                s *= scale;
                if (s > m) m = s;
            }
            /* normaliser */
            double l = 0.0;
            for (int i = 0; i < n; ++i) {
                double s = 0.0;
                for (int d = 0; d < D; ++d) s += gqa_bf16(qh[d]) * gqa_bf16(kg[(size_t)i * D + d]);
                l += exp(s * scale - m);
            }
            /* weighted values, one output element at a time */
            for (int d = 0; d < D; ++d) {
                o[d] = 0.0;
                a[d] = 0.0;
            }
            for (int i = 0; i < n; ++i) {
                double s = 0.0;
                for (int e = 0; e < D; ++e) s += gqa_bf16(qh[e]) * gqa_bf16(kg[(size_t)i * D + e]);
                const double p = exp(s * scale - m) / l;
                for (int d = 0; d < D; ++d) {
                    const double vv = gqa_bf16(vg[(size_t)i * D + d]);
                    o[d] += p * vv;
                    a[d] += p * fabs(vv);
                }
            }
        }
    }
}
