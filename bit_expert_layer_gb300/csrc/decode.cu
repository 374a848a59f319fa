// decode.cu -- routing for small batches (T <= 8 tokens) as a standalone kernel, used
// by moe_route; the decode forward itself runs in decode_layers_kernel.
//
//   decode_router_kernel   33 CTAs: 32 compute 8 router logits each (one warp per
//                          expert row, 128-bit loads), the 33rd the shared-gate dot;
//                          the last CTA to finish (atomic ticket, no waiting) does the
//                          top-8, the weights, counts/offsets/stable permutation and
//                          the list of active experts with a per-token weight column.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

__device__ __forceinline__ float dot8(uint4 a, uint4 b) {
  float s = bf16lo(a.x) * bf16lo(b.x);
  s = fmaf(bf16hi(a.x), bf16hi(b.x), s);
  s = fmaf(bf16lo(a.y), bf16lo(b.y), s);
  s = fmaf(bf16hi(a.y), bf16hi(b.y), s);
  s = fmaf(bf16lo(a.z), bf16lo(b.z), s);
  s = fmaf(bf16hi(a.z), bf16hi(b.z), s);
  s = fmaf(bf16lo(a.w), bf16lo(b.w), s);
  s = fmaf(bf16hi(a.w), bf16hi(b.w), s);
  return s;
}

// inclusive scan of one int per thread over a 256-thread block
__device__ __forceinline__ int block_scan256(int v, int* sc) {
  const int i = threadIdx.x;
  sc[i] = v;
  __syncthreads();
  for (int off = 1; off < 256; off <<= 1) {
    const int o = (i >= off) ? sc[i - off] : 0;
    __syncthreads();
    sc[i] += o;
    __syncthreads();
  }
  const int r = sc[i];
  __syncthreads();
  return r;
}

}  // namespace

// ============================================================================ router
__global__ void __launch_bounds__(256) decode_router_kernel(DecodeParams p) {
  __shared__ int s_last;
  __shared__ int s_idx[DEC_MAX_T][TOPK];
  __shared__ float s_w[DEC_MAX_T][TOPK];
  __shared__ int sc[256];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.T;

  if (blockIdx.x <= NEXP / 8) {
    const bool gate_cta = blockIdx.x == NEXP / 8;
    if (!gate_cta || warp == 0) {
      const int e = gate_cta ? NEXP : blockIdx.x * 8 + warp;
      const __nv_bfloat16* row = gate_cta ? p.shared_gate_w : p.router_w + static_cast<size_t>(e) * HID;
      float acc[DEC_MAX_T];
#pragma unroll
      for (int t = 0; t < DEC_MAX_T; ++t) acc[t] = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int el = (lane + 32 * j) * 8;
        const uint4 w = ldg_nc_v4(row + el);
#pragma unroll
        for (int t = 0; t < DEC_MAX_T; ++t)
          if (t < T) acc[t] += dot8(ldg_nc_v4(p.x + static_cast<size_t>(t) * HID + el), w);
      }
#pragma unroll
      for (int t = 0; t < DEC_MAX_T; ++t) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
      }
      if (lane == 0) {
        const float b = (!gate_cta && p.router_bias) ? p.router_bias[e] : 0.0f;
#pragma unroll
        for (int t = 0; t < DEC_MAX_T; ++t)
          if (t < T) p.logits[t * (NEXP + 1) + e] = acc[t] + b;
      }
    }
  }
  __threadfence();   // every writer publishes its logits before the ticket is taken
  __syncthreads();
  if (tid == 0) {
    const unsigned prev = atomicAdd(p.counter, 1u);
    s_last = (prev == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- the last CTA: top-8 per token (one warp per token)
  if (warp < T) {
    const int t = warp;
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __ldcg(p.logits + t * (NEXP + 1) + lane + 32 * j);
    unsigned taken = 0;
    float selv[TOPK];
    int sele[TOPK];
#pragma unroll
    for (int k = 0; k < TOPK; ++k) {
      float bv = -INFINITY;
      int be = 0x7FFFFFFF;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (!((taken >> j) & 1u) && v[j] > bv) { bv = v[j]; be = lane + 32 * j; }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oe = __shfl_xor_sync(0xffffffffu, be, off);
        if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
      }
      selv[k] = bv;
      sele[k] = be;
      if (be >= 0 && be < NEXP && (be & 31) == lane) taken |= 1u << (be >> 5);
    }
    float ex[TOPK], sum = 0.0f;
#pragma unroll
    for (int k = 0; k < TOPK; ++k) { ex[k] = expf(selv[k] - selv[0]); sum += ex[k]; }
    const float inv = 1.0f / sum;
    if (lane < TOPK) {
      float wk = 0.0f;
      int ek = 0;
#pragma unroll
      for (int k = 0; k < TOPK; ++k)
        if (k == lane) { wk = ex[k] * inv; ek = sele[k]; }
      if (ek < 0 || ek >= NEXP) { atomicOr(p.err, ERRBIT_BOUNDS); ek = 0; }
      s_idx[t][lane] = ek;
      s_w[t][lane] = wk;
      p.topk_idx[t * TOPK + lane] = ek;
      p.topk_w[t * TOPK + lane] = wk;
    }
  }
  __syncthreads();

  // ---- tables: thread = expert
  const int e = tid;
  int c = 0;
  for (int t = 0; t < T; ++t)
#pragma unroll
    for (int k = 0; k < TOPK; ++k) c += (s_idx[t][k] == e);
  const int incl = block_scan256(c, sc);
  const int off = incl - c;
  p.counts[e] = c;
  p.offsets[e] = off;
  int n = 0;
  for (int s = 0; s < T * TOPK; ++s)
    if (s_idx[s / TOPK][s % TOPK] == e) p.perm[off + n++] = s;
  const int act_incl = block_scan256(c > 0 ? 1 : 0, sc);
  if (c > 0) {
    const int a = act_incl - 1;
    p.act_expert[a] = e;
#pragma unroll
    for (int t = 0; t < DEC_MAX_T; ++t) {
      float w = 0.0f;
      if (t < T)
#pragma unroll
        for (int k = 0; k < TOPK; ++k)
          if (s_idx[t][k] == e) w = s_w[t][k];
      p.act_w[a * DEC_MAX_T + t] = w;
    }
  }
  if (e == NEXP - 1) {
    const int a = act_incl;   // number of active routed experts
    p.act_expert[a] = NEXP;   // the shared expert goes last
#pragma unroll
    for (int t = 0; t < DEC_MAX_T; ++t) {
      float w = 0.0f;
      if (t < T) w = 1.0f / (1.0f + expf(-__ldcg(p.logits + t * (NEXP + 1) + NEXP)));
      p.act_w[a * DEC_MAX_T + t] = w;
    }
    *p.n_active = a + 1;
    p.counts[NEXP] = T;
    p.offsets[NEXP] = 8 * T;
    p.offsets[NEXP + 1] = 9 * T;
    *p.counter = 0u;   // ticket reset for the next call (every other CTA has arrived)
  }
}

cudaError_t launch_decode_router(const DecodeParams& p, cudaStream_t s) {
  decode_router_kernel<<<NEXP / 8 + 1, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
