/*
 * moe_layer.h -- C ABI of a GB300 (sm_103a) library for the mixture-of-experts
 * layer of Qwen3.6-35B-A3B over MLX affine 4-bit expert weights.
 *
 * What the layer is.  Lily, Perplexity's engine for this one model, scores all 256
 * experts for every token, keeps 8 and adds one shared expert (aimanavo.com, "Why is
 * Perplexity's local AI Lily faster than MLX", section "Qwen3.6's 256 experts and two
 * layer kinds make the MLX/Lily gap").  Its weights are MLX affine 4-bit with group
 * size 64, and anything else is refused when the model loads (same page, section
 * "Only one 4-bit checkpoint of a pinned revision runs"; news.mantis.guru, "Perplexity
 * opened Lily", section "Rust drives the model, Metal computes").  Prefill dequantises
 * the 4-bit weights inside grouped GEMMs and keeps routing on the GPU with no host
 * synchronisation; decode is bound by memory reads of the weights (aimanavo.com,
 * section "Prefill and decode are not treated as the same job"; dzen.guru,
 * "Perplexity opened the Lily engine", section "Where the speed-up comes from").
 *
 * The maths, per token x (bf16, hidden 2048):
 *   w[o][i]  = scale[o][i/64] * q[o][i] + bias[o][i/64]   q = nibble i%8 of word i/8,
 *                                                         low nibble first
 *   l_e      = fp32 dot(x, W_r[e]) (+ router_bias[e])     e = 0..255
 *   top-8 of softmax(l) (ties: lowest expert index), weights renormalised to sum 1
 *   y_e      = W_down,e ( silu(W_gate,e x) * (W_up,e x) )
 *   out      = sum_k w_k y_{e_k} + sigmoid(g_s . x) * y_shared   (+ x for *_residual)
 *   rounded once to bf16.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller, except the *_host
 *     entry, whose x/out are host pointers.  bf16 tensors are passed as void*.
 *   - Nothing throws.  A status code is returned; host-side argument checks return
 *     before any work is enqueued.
 *   - Calls are asynchronous on `stream` and never synchronise the host (except
 *     moe_layer_create, moe_layer_get_error and the *_host entry's copies as noted).
 *   - The library never allocates device memory: all scratch lives in the caller's
 *     workspace.  One workspace may back several layers that run one after another
 *     on one stream; two calls that overlap in time need two workspaces.
 *   - Device-side failures (a bounded wait that gave up, an index out of range) never
 *     trap: they set a word in the workspace that moe_layer_get_error reads.
 */
#ifndef MOE_LAYER_H
#define MOE_LAYER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_layer moe_layer_t;        /* opaque; owned by the library */
typedef struct CUstream_st* moe_stream_t;    /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,    /* NULL pointer, T out of range, aliasing not allowed */
    MOE_ERR_UNSUPPORTED = 2,    /* shapes or quantisation other than the one layer supported */
    MOE_ERR_ALIGNMENT = 3,      /* a pointer not 16-byte aligned (workspace: 256-byte) */
    MOE_ERR_CUDA = 4,           /* a CUDA runtime or driver call failed */
    MOE_ERR_TIMEOUT = 5,        /* a device-side bounded wait gave up */
    MOE_ERR_DEVICE_BOUNDS = 6,  /* a device-side index check failed */
    MOE_ERR_WORKSPACE = 7       /* workspace smaller than moe_workspace_bytes() */
} moe_status_t;

/* The layer's shape.  Only hidden 2048, 256 experts, top-8, intermediate 512, shared
 * intermediate 512, group 64, 4 bits is accepted (Lily's own load-time refusal of every
 * other checkpoint, cited above); max_tokens (1..65536) sizes the workspace. */
typedef struct {
    int hidden, n_experts, top_k, inter, shared_inter, group_size, bits, max_tokens;
} moe_config_t;

/* One MLX affine 4-bit matrix [out][in]: q uint32 [out][in/8] (eight codes per word,
 * low nibble first), scales and biases bf16 [out][in/64].  Routed experts are stacked
 * along a leading expert axis: q [256][out][in/8], scales/biases [256][out][in/64]. */
typedef struct {
    const void* q;
    const void* scales;
    const void* biases;
} moe_qmat_t;

typedef struct {
    moe_qmat_t gate, up, down;          /* routed: gate/up [256][512][2048], down [256][2048][512] */
    moe_qmat_t sh_gate, sh_up, sh_down; /* shared: gate/up [512][2048], down [2048][512] */
    const void* router_w;               /* bf16 [256][2048] */
    const float* router_bias;           /* fp32 [256] added to the logits before softmax, or NULL */
    const void* shared_gate_w;          /* bf16 [2048] */
    const void* norm_w;                 /* bf16 [2048]: the layer's input RMSNorm weight, or NULL.
                                         * With it the layer computes MoE(x_n), x_n = bf16(x /
                                         * sqrt(mean(x^2) + 1e-6) * norm_w), and the residual forms
                                         * add the un-normalised x (the form stacked layers need). */
} moe_weights_t;

/* Bytes of device workspace a layer with this config needs (0 if the config is refused).
 * The workspace holds the routing tables and the intermediates of the path the pages
 * describe for prefill: the on-GPU routing state, the permuted rows and the per-expert
 * activations between the grouped GEMMs (aimanavo.com, section "Prefill and decode are not
 * treated as the same job").  No allocation happens inside the library. */
size_t moe_workspace_bytes(const moe_config_t* cfg);

/* Validate the config and weights and bind them to `workspace` (device, 256-byte
 * aligned, at least moe_workspace_bytes bytes, owned by the caller and kept alive as
 * long as the layer).  Weights are borrowed for the layer's lifetime.  Like Lily, which
 * checks the checkpoint's layout at load time and refuses anything else (aimanavo.com,
 * section "Only one 4-bit checkpoint of a pinned revision runs"; news.mantis.guru,
 * section "Rust drives the model, Metal computes"), every shape, quantisation and
 * alignment check happens here, before any kernel runs.  Synchronises the current device
 * once (it zeroes the workspace words that must start at zero: the error word and the
 * decode hand-off tables).  On success *out receives a layer to free with
 * moe_layer_destroy.
 * Errors: INVALID_ARG (NULL), UNSUPPORTED (shape), ALIGNMENT, WORKSPACE, CUDA. */
moe_status_t moe_layer_create(const moe_config_t* cfg, const moe_weights_t* weights,
                              void* workspace, size_t workspace_bytes, moe_layer_t** out);

/* Routing only (router logits, softmax, top-8, renormalisation, expert histogram,
 * exclusive-scan offsets and the stable token permutation), all on the device with no
 * host synchronisation: the 256 experts scored and 8 kept per token (aimanavo.com,
 * section "Qwen3.6's 256 experts and two layer kinds make the MLX/Lily gap"), and the
 * routing kept on the GPU without a per-layer CPU sync (aimanavo.com, section "Prefill
 * and decode are not treated as the same job"; dzen.guru, section "Where the speed-up
 * comes from").
 *   x        bf16 [T][2048]
 *   topk_idx int32 [T][8]   experts in rank order
 *   topk_w   fp32  [T][8]   renormalised weights
 *   counts   int32 [256]    slots per expert
 *   offsets  int32 [257]    exclusive scan of counts
 *   perm     int32 [T*8]    slot ids t*8+k grouped by expert, ascending within one
 * Any output pointer may be NULL.  1 <= T <= max_tokens. */
moe_status_t moe_route(moe_layer_t* layer, const void* x, int T, int32_t* topk_idx, float* topk_w,
                       int32_t* counts, int32_t* offsets, int32_t* perm, moe_stream_t stream);

/* out[T][2048] (bf16) = the layer applied to x[T][2048] (bf16).  T <= 8 takes the
 * decode path (a memory-bound dequant-GEMV kernel), larger T the prefill path (grouped
 * tcgen05 GEMMs with the 4-bit weights dequantised inside the kernel): the two modes the
 * pages keep apart (aimanavo.com, section "Prefill and decode are not treated as the same
 * job"; news.mantis.guru, section "Prefill and decode are optimised as different modes").
 * out must not overlap x.  1 <= T <= max_tokens.
 * Errors: INVALID_ARG (NULL, T out of range, overlap), ALIGNMENT, CUDA (a launch failed;
 * moe_last_error_detail says which). */
moe_status_t moe_forward(moe_layer_t* layer, const void* x, int T, void* out, moe_stream_t stream);

/* out = x + layer(x), the residual form used between stacked layers of the model's
 * 40-layer stack (aimanavo.com, section "Qwen3.6's 256 experts and two layer kinds make
 * the MLX/Lily gap").  With norm_w set the layer computes x + MoE(RMSNorm(x)).  out == x
 * (in place) is allowed; a partial overlap is not.  Errors as moe_forward. */
moe_status_t moe_forward_residual(moe_layer_t* layer, const void* x, int T, void* out, moe_stream_t stream);

/* x_io <- layer[n-1]( ... layer[0](x_io) ... ) with the residual add after every layer,
 * in place on the device.  All layers must share one workspace.  For T <= 8 the whole
 * stack is one persistent decode launch per 48 layers: the counterpart of Lily's
 * overlapped decode kernels (aimanavo.com, section "Prefill and decode are not treated as
 * the same job").  Errors as moe_forward. */
moe_status_t moe_stack_forward(moe_layer_t* const* layers, int n_layers, void* x_io, int T, moe_stream_t stream);

/* The same stack from HOST memory: copies x_host (bf16 [T][2048]) into the shared
 * workspace's I/O buffer, runs the stack and copies the result to out_host, all
 * enqueued on `stream`.  With pinned host buffers the copies are asynchronous and the
 * caller must synchronise the stream before reading out_host.  (The pages' engine runs
 * on unified memory, where this step does not exist; it is the end-to-end entry of this
 * library.)  Errors as moe_forward. */
moe_status_t moe_stack_forward_host(moe_layer_t* const* layers, int n_layers, const void* x_host, int T,
                                    void* out_host, moe_stream_t stream);

/* The decode forward (1 <= T <= 8) for callers that cannot allocate device memory:
 * a plug-in whose host application owns all device memory and offers no allocator or
 * workspace, or a latency-critical decode loop that must never reach cudaMalloc (which
 * can synchronise the device).  No layer object and no workspace: the scratch of the
 * decode kernel lives in a fixed 3 MiB array of device memory inside the library,
 * held by every device that loads it until the process exits.  Nothing is allocated
 * (no cudaMalloc, no cudaFree, no allocating library routine).  The pages describe no
 * such entry point; it has no counterpart there.
 *   weights  as for moe_layer_create (device pointers, borrowed for the call)
 *   x, out   bf16 [T][2048] device pointers; out == x is allowed only with residual
 *   residual 0: out = layer(x); 1: out = x + layer(x) (with norm_w: x + MoE(norm(x)))
 * T above 8 (the array's limit) or below 1 returns MOE_ERR_INVALID_ARG and says why in
 * moe_last_error_detail.  The first call on a device looks up the array's device address
 * there (make that first call before any stream capture).  Every call on a device shares
 * the one array and leaves its contents behind; the parts that must start at zero start
 * at zero when the library is loaded and the kernel keeps them valid.  Calls that overlap
 * on the GPU (other streams, other threads) race on the array and corrupt each other:
 * serialise them.  Device-side errors of these calls (a bounded wait that gave up, an
 * index out of range) collect in the array's error word until
 * moe_decode_static_get_error reads it. */
moe_status_t moe_decode_forward_static(const moe_weights_t* weights, const void* x, int T, void* out,
                                       int residual, moe_stream_t stream);

/* Synchronise the current device, then read and clear the error word of
 * moe_decode_forward_static's array on that device: MOE_OK if none of its calls since the
 * last read recorded a device-side error, else MOE_ERR_TIMEOUT or MOE_ERR_DEVICE_BOUNDS
 * (MOE_ERR_CUDA if the synchronisation or the copy failed). */
moe_status_t moe_decode_static_get_error(void);

/* Number of kernel launches one moe_forward of T tokens on this layer enqueues
 * (for accounting); 0 for a NULL layer or T out of range. */
int moe_forward_launches(const moe_layer_t* layer, int T);

/* Number of kernel launches one moe_stack_forward of T tokens over these layers
 * enqueues (for T <= 8 the whole stack runs in one launch per 48 layers); 0 for a NULL
 * array or layer, n_layers < 1 or T out of range. */
int moe_stack_forward_launches(const moe_layer_t* const* layers, int n_layers, int T);

/* Synchronise the device, read and clear the layer's device error word.
 * MOE_OK if nothing was recorded. */
moe_status_t moe_layer_get_error(moe_layer_t* layer);

/* Free the layer object (not the workspace or the weights, which the caller owns). */
void moe_layer_destroy(moe_layer_t* layer);

/* Time limit, in nanoseconds, of every bounded device-side wait in the launches that
 * follow (process-wide; 0 restores the default of 2 s; below 1000, the device timer's
 * resolution, a wait gives up as soon as it finds its data not ready).  A wait that runs out sets
 * MOE_ERR_TIMEOUT in the error word and ends its launch early without trapping (the
 * copies and MMAs already in flight still land before a CTA exits), so a very short
 * limit is how the failure path is exercised on purpose.  The pages have no counterpart:
 * Lily's Metal kernels are not described at this level. */
void moe_set_wait_limit_ns(unsigned long long ns);

/* A static string naming a status code. */
const char* moe_status_string(moe_status_t status);

/* The calling thread's description of the last CUDA/driver failure behind an
 * MOE_ERR_CUDA status (empty if none).  Valid until the thread's next call. */
const char* moe_last_error_detail(void);

/* Pipeline tracing of the grouped GEMMs (only when the environment variable
 * MOE_PIPE_PROF=1 is set before the first forward): clock cycles that each warp role
 * spent waiting on its barriers, summed over all CTAs and launches since the last read.
 * out receives 32 counters, 16 for the gate/up kernel then 16 for the down kernel, each:
 * [0] MMA issuer waiting for the accumulator to drain, [1] for dequantised tiles, [2] for
 * TMA data, [3] MMA issuer total; [4] TMA producer waiting for a free stage, [5] its
 * total; [6] one dequant thread waiting for TMA data, [7] its total; [8] one epilogue
 * thread waiting for the accumulator, [9] its total; [10] tiles processed.
 * Synchronises the device, then zeroes the counters. */
moe_status_t moe_pipeline_counters(moe_layer_t* layer, unsigned long long* out);

/* Phase timestamps of the fused decode kernel (tracing; only when the environment
 * variable MOE_DECODE_TRACE=1 is set before the first forward).  For layer l of the most
 * recent decode launch on the workspace bound to `layer` and CTA c < 256, word
 * (l * 256 + c) * 16 + k holds the device's global timer (ns) when CTA c passed phase
 * boundary k: 0 layer start, 1 layer input received, 2 router rows staged, 3 router
 * logits published, 4 all logits received, 5 expert tables built, 6 weight copies
 * issued, 7 first gate/up batch landed, 8 gate/up done, 9 down rows staged, 10 first
 * batch of h' received, 11 layer output published, 12 first gate/up batch computed, 13
 * its h' published, 14 down products computed, 15 down sums reduced (phases A-C of the
 * kernel, described in its source).  Synchronises the device and copies
 * the first n_words words (at most 48 * 256 * 16) to out. */
moe_status_t moe_decode_trace(moe_layer_t* layer, unsigned long long* out, size_t n_words);

/* Kernel timing (tracing for benchmarks).  While enabled, every kernel this library
 * launches is bracketed by two CUDA events recorded on the launch's own stream. */
void moe_profiler_enable(int on);

/* Resolve the recorded events (waits for each one), add up the duration per kernel
 * kind and clear the record.  Fills up to `max` entries of names (static strings),
 * total_ms and launches (any may be NULL); returns the number of kernel kinds. */
int moe_profiler_read(const char** names, double* total_ms, long long* launches, int max);

#ifdef __cplusplus
}
#endif

#endif /* MOE_LAYER_H */
