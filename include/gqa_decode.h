/*
 * gqa_decode.h -- C ABI of the grouped-query decode attention of the same GB300 (sm_103a)
 * library: the full-attention layers of Qwen3.6-35B-A3B, whose 16 query heads share 2
 * key/value heads (aimanavo.com, "Why is Perplexity's local AI Lily faster than MLX",
 * section "Qwen3.6's 256 experts and two layer kinds make the MLX/Lily gap").  Decode reads
 * the whole KV cache at every step and is bound by memory bandwidth; Lily packs the query
 * heads of a group so that each KV row is read once for all of them (same page, section
 * "Prefill and decode are not treated as the same job"; dzen.guru, "Perplexity opened the
 * Lily engine", section "Where the speed-up comes from").  This entry does the same: each
 * key and value row crosses HBM once and serves the 8 query heads of its group.
 *
 * The maths, per sequence b and query head h (KV head g = h / 8), for its one new query
 * token over the len[b] cached positions:
 *   s_i  = (q[b][h] . k[b][g][i]) / sqrt(128)
 *   o    = sum_i softmax(s)_i v[b][g][i]
 * computed with fp32 scores, the softmax in fp32 with the probabilities rounded to bf16
 * for the value product (fp32 accumulation), and o rounded once to bf16.
 *
 * Conventions as in moe_layer.h: device pointers owned by the caller, status codes, no
 * host synchronisation, no allocation inside the library.
 */
#ifndef GQA_DECODE_H
#define GQA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#include "moe_layer.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of device workspace one call with B sequences needs (0 unless 1 <= B <= 64).  The
 * workspace holds the per-split partial results, the split tickets and an error word; it
 * must be zero-filled (cudaMemset) before its first use, after which every call leaves it
 * ready for the next. */
size_t gqa_decode_workspace_bytes(int B);

/* One decode step of grouped-query attention.
 *   q        bf16 [B][16][128]   the new query token of each sequence (device)
 *   k, v     bf16 [B][2][S_max][128]  the KV cache, position-major per KV head (device);
 *            rows at or past a sequence's length are never read into the result
 *   lens     int32 [B] HOST array, 1 <= lens[b] <= S_max
 *   out      bf16 [B][16][128] (device)
 *   workspace  >= gqa_decode_workspace_bytes(B) bytes, 256-byte aligned, zero-filled
 *            before first use; two calls that overlap in time need two workspaces
 * Errors: INVALID_ARG (NULL, B or S_max or a length out of range), ALIGNMENT (a tensor not
 * 16-byte aligned, the workspace not 256-byte aligned), WORKSPACE, CUDA (a launch or a
 * tensor-map encoding failed; moe_last_error_detail says which). */
moe_status_t gqa_decode_attention(const void* q, const void* k, const void* v, const int32_t* lens, int B,
                                  int S_max, void* out, void* workspace, size_t workspace_bytes,
                                  moe_stream_t stream);

/* Synchronise the current device, then read and clear the workspace's error word: MOE_OK,
 * MOE_ERR_TIMEOUT (a bounded wait gave up) or MOE_ERR_DEVICE_BOUNDS. */
moe_status_t gqa_decode_get_error(void* workspace);

#ifdef __cplusplus
}
#endif

#endif /* GQA_DECODE_H */
