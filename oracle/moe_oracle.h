/*
 * moe_oracle.h -- declarations of the CPU oracle (test infrastructure only; see
 * moe_oracle.c for what each function computes and where it comes from).
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int hidden, n_experts, top_k, inter, shared_inter, group;
} oracle_dims_t;

/* One 4-bit matrix or a stack of them: q uint32 [.., out, in/8] (low nibble first),
 * scales / biases bf16 bits [.., out, in/group]. */
typedef struct {
    const uint32_t* q;
    const uint16_t* scales;
    const uint16_t* biases;
} oracle_qmat_t;

typedef struct {
    oracle_qmat_t gate, up, down;          /* routed experts, stacked [E][..] */
    oracle_qmat_t sh_gate, sh_up, sh_down; /* the shared expert */
    const uint16_t* router_w;              /* bf16 [E][hidden] */
    const float* router_bias;              /* fp32 [E] or NULL */
    const uint16_t* shared_gate_w;         /* bf16 [hidden] */
    const uint16_t* norm_w;                /* bf16 [hidden]: RMSNorm of the layer input, or NULL */
} oracle_weights_t;

#define ORACLE_RMS_EPS 1e-6

double oracle_bf16_to_double(uint16_t b);
uint16_t oracle_double_to_bf16(double v);
void oracle_unpack4(uint32_t word, int q[8]);
void oracle_dequant_row(const uint32_t* q_row, const uint16_t* s_row, const uint16_t* b_row,
                        int in_dim, int group, double* w);
void oracle_qmatvec(const oracle_qmat_t* m, long mat, int out_dim, int in_dim, int group,
                    const double* x, double* y);
void oracle_router_logits(const oracle_dims_t* d, const uint16_t* router_w, const float* router_bias,
                          const uint16_t* x_row, float* logits);
void oracle_route_logits(const oracle_dims_t* d, const float* logits, int32_t* idx, double* w,
                         double* gap, double* p_sorted, int32_t* order);
void oracle_expert(const oracle_dims_t* d, const oracle_qmat_t* gate, const oracle_qmat_t* up,
                   const oracle_qmat_t* down, long e, int inter, const double* x, double* y);
void oracle_layer_logits(const oracle_dims_t* d, const oracle_weights_t* W, const uint16_t* x_row, float* l);
void oracle_rmsnorm(int hidden, const uint16_t* x_row, const uint16_t* norm_w, uint16_t* out);
double oracle_shared_gate(const oracle_dims_t* d, const uint16_t* shared_gate_w, const uint16_t* x_row);
void oracle_token_forward(const oracle_dims_t* d, const oracle_weights_t* W, const uint16_t* x_row,
                          const int32_t* experts, const double* wts, int residual, double* out);
void oracle_route(const oracle_dims_t* d, const oracle_weights_t* W, const uint16_t* x, int T, int nthreads,
                  int32_t* idx, double* wts, double* gap, int32_t* counts, int32_t* offsets, int32_t* perm);
void oracle_layer_forward(const oracle_dims_t* d, const oracle_weights_t* W, const uint16_t* x, int T,
                          int residual, int nthreads, uint16_t* out, int32_t* idx, double* wts, double* gap);
void oracle_token_forward_choice(const oracle_dims_t* d, const oracle_weights_t* W, const uint16_t* x_row,
                                 const int32_t* experts, int residual, uint16_t* out, double* wts_out);
int oracle_mutant(void);

/* Grouped-query decode attention (gqa_oracle.c): q [B][Hq][D], k and v [B][Hkv][S_max][D]
 * (bf16 bits), lens [B]; out and abs_out [B][Hq][D] (double). */
void oracle_gqa_decode(int B, int Hq, int Hkv, int D, int S_max, const int32_t* lens, const uint16_t* q,
                       const uint16_t* k, const uint16_t* v, double scale, int nthreads, double* out,
                       double* abs_out);

#ifdef __cplusplus
}
#endif

#endif
