// decode.cu -- the memory-bound decode path (T <= 8 tokens).  Decode reads the
// weights again at every step, so the bound moves from compute to memory bandwidth
// (aimanavo.com, "Why is Perplexity's local AI Lily faster than MLX", section
// "Prefill and decode are not treated as the same job").  Three kernels:
//
//   decode_router_kernel   33 CTAs: 32 compute 8 router logits each (one warp per
//                          expert row, 128-bit loads), the 33rd the shared-gate dot;
//                          the last CTA to finish (atomic ticket, no waiting) does the
//                          top-8, the weights, counts/offsets/stable permutation and
//                          the list of active experts with a per-token weight column.
//   decode_gateup_kernel   one CTA per (active expert, 16 rows): 8 warps split K, each
//                          streams packed gate/up rows with 128-bit loads, dequantises
//                          in registers and multiplies on the tensor cores with
//                          mma.sync m16n8k16 (all <= 8 tokens are the N=8 columns);
//                          fixed-order reduction over the K split, SwiGLU, times the
//                          token's routing weight (0 for tokens not routed here).
//   decode_down_kernel     one CTA per 16 output rows: 16 warps = 4 K splits x 4
//                          expert interleaves; the weighted h columns of every active
//                          expert are accumulated in one MMA accumulator, so the
//                          combine over the 8 routed + 1 shared experts costs nothing
//                          extra; fixed-order reduction, residual, bf16 output.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ __nv_bfloat162 bf2(uint16_t bits) {
  const uint32_t v = static_cast<uint32_t>(bits) * 0x00010001u;
  return *reinterpret_cast<const __nv_bfloat162*>(&v);
}

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

// ============================================================================ gate/up
__global__ void __launch_bounds__(256) decode_gateup_kernel(DecodeParams p) {
  __shared__ float red[8][32][8];
  const int a = blockIdx.y;
  const int n_act = __ldcg(p.n_active);
  if (n_act < 1 || n_act > DEC_MAX_ACTIVE) {   // tables not built: record, touch nothing
    if (threadIdx.x == 0 && blockIdx.x == 0 && a == 0) atomicOr(p.err, ERRBIT_BOUNDS);
    return;
  }
  if (a >= n_act) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int e = __ldcg(p.act_expert + a);
  if (e < 0 || e > NEXP) {
    if (tid == 0) atomicOr(p.err, ERRBIT_BOUNDS);
    return;
  }
  const bool sh = e == NEXP;
  const int r0 = blockIdx.x * 16 + g, r1 = r0 + 8;
  const size_t rb0 = sh ? static_cast<size_t>(r0) : static_cast<size_t>(e) * INTER + r0;
  const size_t rb1 = rb0 + 8;
  const uint32_t* gq = sh ? p.sgq : p.gq;
  const uint32_t* uq = sh ? p.suq : p.uq;
  const uint16_t* gs = sh ? p.sgs : p.gs;
  const uint16_t* gb = sh ? p.sgb : p.gb;
  const uint16_t* us = sh ? p.sus : p.us;
  const uint16_t* ub = sh ? p.sub : p.ub;
  const int T = p.T;

  uint4 wg0[2], wg1[2], wu0[2], wu1[2], xb[2][4];
  uint16_t sg0[2], sg1[2], bg0[2], bg1[2], su0[2], su1[2], bu0[2], bu1[2];
#pragma unroll
  for (int sp = 0; sp < 2; ++sp) {
    const int kbase = warp * 256 + sp * 128;
    const int wo = kbase / 8 + 4 * c;              // word offset in the row
    const int gi = (kbase + 32 * c) / GROUP;       // quantisation group
    wg0[sp] = ldg_nc_v4(gq + rb0 * (HID / 8) + wo);
    wg1[sp] = ldg_nc_v4(gq + rb1 * (HID / 8) + wo);
    wu0[sp] = ldg_nc_v4(uq + rb0 * (HID / 8) + wo);
    wu1[sp] = ldg_nc_v4(uq + rb1 * (HID / 8) + wo);
    sg0[sp] = __ldg(gs + rb0 * (HID / GROUP) + gi);
    sg1[sp] = __ldg(gs + rb1 * (HID / GROUP) + gi);
    bg0[sp] = __ldg(gb + rb0 * (HID / GROUP) + gi);
    bg1[sp] = __ldg(gb + rb1 * (HID / GROUP) + gi);
    su0[sp] = __ldg(us + rb0 * (HID / GROUP) + gi);
    su1[sp] = __ldg(us + rb1 * (HID / GROUP) + gi);
    bu0[sp] = __ldg(ub + rb0 * (HID / GROUP) + gi);
    bu1[sp] = __ldg(ub + rb1 * (HID / GROUP) + gi);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint4 v = make_uint4(0, 0, 0, 0);
      if (g < T) v = interleave8(ldg_nc_v4(p.x + static_cast<size_t>(g) * HID + kbase + 32 * c + 8 * j));
      xb[sp][j] = v;
    }
  }
  float dg[4] = {0.f, 0.f, 0.f, 0.f}, du[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int sp = 0; sp < 2; ++sp) {
    const __nv_bfloat162 mg0 = bf2(sg0[sp]), mg1 = bf2(sg1[sp]), ag0 = bf2(bg0[sp]), ag1 = bf2(bg1[sp]);
    const __nv_bfloat162 mu0 = bf2(su0[sp]), mu1 = bf2(su1[sp]), au0 = bf2(bu0[sp]), au1 = bf2(bu1[sp]);
    const uint32_t g0w[4] = {wg0[sp].x, wg0[sp].y, wg0[sp].z, wg0[sp].w};
    const uint32_t g1w[4] = {wg1[sp].x, wg1[sp].y, wg1[sp].z, wg1[sp].w};
    const uint32_t u0w[4] = {wu0[sp].x, wu0[sp].y, wu0[sp].z, wu0[sp].w};
    const uint32_t u1w[4] = {wu1[sp].x, wu1[sp].y, wu1[sp].z, wu1[sp].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 o0 = dequant8(g0w[j], mg0, ag0), o1 = dequant8(g1w[j], mg1, ag1);
      mma16816(dg, o0.x, o1.x, o0.y, o1.y, xb[sp][j].x, xb[sp][j].y);
      mma16816(dg, o0.z, o1.z, o0.w, o1.w, xb[sp][j].z, xb[sp][j].w);
      const uint4 v0 = dequant8(u0w[j], mu0, au0), v1 = dequant8(u1w[j], mu1, au1);
      mma16816(du, v0.x, v1.x, v0.y, v1.y, xb[sp][j].x, xb[sp][j].y);
      mma16816(du, v0.z, v1.z, v0.w, v1.w, xb[sp][j].z, xb[sp][j].w);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    red[warp][lane][i] = dg[i];
    red[warp][lane][4 + i] = du[i];
  }
  __syncthreads();
  if (warp == 0) {
    float sg[4] = {0.f, 0.f, 0.f, 0.f}, su[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < 8; ++w) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        sg[i] += red[w][lane][i];
        su[i] += red[w][lane][4 + i];
      }
    }
    // d[0]: (row g, token 2c), d[1]: (g, 2c+1), d[2]: (g+8, 2c), d[3]: (g+8, 2c+1)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int tok = 2 * c + (i & 1);
      const int row = (i < 2) ? r0 : r1;
      const float wt = __ldcg(p.act_w + a * DEC_MAX_T + tok);
      const float hv = sg[i] / (1.0f + __expf(-sg[i])) * su[i] * wt;
      p.hw[(static_cast<size_t>(a) * DEC_MAX_T + tok) * INTER + ilv_pos(row)] = __float2bfloat16_rn(hv);
    }
  }
}

// ============================================================================ down + combine
__global__ void __launch_bounds__(512) decode_down_kernel(DecodeParams p) {
  __shared__ float red[16][32][4];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int ks = warp & 3, eq = warp >> 2;
  const int r0 = blockIdx.x * 16 + g, r1 = r0 + 8;
  int n_act = __ldcg(p.n_active);
  if (n_act < 1 || n_act > DEC_MAX_ACTIVE) {
    if (tid == 0 && blockIdx.x == 0) atomicOr(p.err, ERRBIT_BOUNDS);
    n_act = 0;
  }
  const int wo = ks * 16 + 4 * c;                  // word offset in a down row (64 words)
  const int gi = (ks * 128 + 32 * c) / GROUP;      // quantisation group (8 per row)
  float d[4] = {0.f, 0.f, 0.f, 0.f};

  for (int a0 = eq; a0 < n_act; a0 += 8) {
    uint4 w0[2], w1[2], hb[2][4];
    uint16_t s0[2], s1[2], b0[2], b1[2];
    bool have[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int a = a0 + 4 * u;
      have[u] = a < n_act;
      if (!have[u]) continue;
      const int e = __ldcg(p.act_expert + a);
      if (e < 0 || e > NEXP) {
        if (lane == 0) atomicOr(p.err, ERRBIT_BOUNDS);
        have[u] = false;
        continue;
      }
      const bool sh = e == NEXP;
      const size_t rw0 = sh ? static_cast<size_t>(r0) : static_cast<size_t>(e) * HID + r0;
      const size_t rw1 = rw0 + 8;
      const uint32_t* dq = sh ? p.sdq : p.dq;
      const uint16_t* ds = sh ? p.sds : p.ds;
      const uint16_t* db = sh ? p.sdb : p.db;
      w0[u] = ldg_nc_v4(dq + rw0 * (INTER / 8) + wo);
      w1[u] = ldg_nc_v4(dq + rw1 * (INTER / 8) + wo);
      s0[u] = __ldg(ds + rw0 * (INTER / GROUP) + gi);
      s1[u] = __ldg(ds + rw1 * (INTER / GROUP) + gi);
      b0[u] = __ldg(db + rw0 * (INTER / GROUP) + gi);
      b1[u] = __ldg(db + rw1 * (INTER / GROUP) + gi);
      const __nv_bfloat16* hr = p.hw + (static_cast<size_t>(a) * DEC_MAX_T + g) * INTER + ks * 128 + 32 * c;
#pragma unroll
      for (int j = 0; j < 4; ++j) hb[u][j] = __ldcg(reinterpret_cast<const uint4*>(hr + 8 * j));
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (!have[u]) continue;
      const __nv_bfloat162 m0 = bf2(s0[u]), m1 = bf2(s1[u]), c0 = bf2(b0[u]), c1 = bf2(b1[u]);
      const uint32_t x0[4] = {w0[u].x, w0[u].y, w0[u].z, w0[u].w};
      const uint32_t x1[4] = {w1[u].x, w1[u].y, w1[u].z, w1[u].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 o0 = dequant8(x0[j], m0, c0), o1 = dequant8(x1[j], m1, c1);
        mma16816(d, o0.x, o1.x, o0.y, o1.y, hb[u][j].x, hb[u][j].y);
        mma16816(d, o0.z, o1.z, o0.w, o1.w, hb[u][j].z, hb[u][j].w);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) red[warp][lane][i] = d[i];
  __syncthreads();
  if (warp == 0) {
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < 16; ++w)
#pragma unroll
      for (int i = 0; i < 4; ++i) s[i] += red[w][lane][i];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int tok = 2 * c + (i & 1);
      const int row = (i < 2) ? r0 : r1;
      if (tok < p.T) {
        float o = s[i];
        const size_t off = static_cast<size_t>(tok) * HID + row;
        if (p.residual) o += __bfloat162float(p.x_resid[off]);
        p.out[off] = __float2bfloat16_rn(o);
      }
    }
  }
}

cudaError_t launch_decode_router(const DecodeParams& p, cudaStream_t s) {
  decode_router_kernel<<<NEXP / 8 + 1, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode_gateup(const DecodeParams& p, cudaStream_t s) {
  const int ny = min(8 * p.T, NEXP) + 1;
  decode_gateup_kernel<<<dim3(INTER / 16, ny), 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode_down(const DecodeParams& p, cudaStream_t s) {
  decode_down_kernel<<<HID / 16, 512, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
