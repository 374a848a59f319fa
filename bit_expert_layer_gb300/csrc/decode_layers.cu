// decode_layers.cu -- the memory-bound decode path (T <= 8 tokens) as one persistent
// kernel that runs every layer of a decode step.  Decode reads the weights again at
// every step, so the bound moves from compute to memory bandwidth (aimanavo.com, "Why
// is Perplexity's local AI Lily faster than MLX", section "Prefill and decode are not
// treated as the same job"); Lily overlaps its many small decode kernels (same page,
// section "Where the gains come from").  Here the stages of a layer are phases of one
// cooperative launch, and no launch gap or grid-wide barrier sits between them.
//
// One CTA per SM (cooperative launch: all CTAs are resident, so they may wait on one
// another), 16 warps.  Per layer:
//   phase A  every CTA reads the layer input x, forms its RMSNorm (when the layer has
//            one) in shared memory, and computes its share of the 256 router logits and
//            the shared-expert gate logit (8 warps split the 2048 inputs of one row).
//   phase B  every CTA repeats the top-8 selection from the logits (the same result in
//            every CTA), builds the list of active experts (the routed ones in id order,
//            the shared expert last) with a per-token weight column, and computes
//            gate/up units: 8 features x (gate row, up row) of one active expert, an
//            m16n8k16 tile whose two row halves are the gate and the up rows of the same
//            features, so SwiGLU needs no exchange.  The 16 warps split K; fixed-order
//            reduction; h' = weight * silu(g) * u.
//   phase C  16 output rows per CTA: the weighted h' columns of every active expert are
//            accumulated in one MMA accumulator (the combine over the 8 routed + 1
//            shared experts), fixed-order reduction over 16 warps, residual, bf16 out.
//
// Hand-off between CTAs without barriers: every value one CTA passes to another (the
// layer output x, the logits, h') travels as a 64-bit word {32-bit payload, 32-bit tag}
// written and read with single-copy-atomic relaxed accesses; the tag names the launch
// (an epoch counter kept in the scratch) and the layer.  A consumer polls the words it
// needs until every tag is current, so it waits for exactly the producers it depends
// on, one L2 round trip, instead of a grid barrier followed by a read.  The tables are
// double-buffered by layer parity: a producer can be at most one layer ahead of the
// slowest consumer of the same buffer, because every layer's phase B needs all logits,
// its phase C all of h', and its phase A all of x.
//
// Weights move into shared memory by cp.async: 16-byte pieces, consecutive threads on
// consecutive pieces of a contiguous block (8 KB of gate or up rows, 4 KB of down rows),
// which streams at the HBM rate, where per-copy costs make small bulk-engine copies slow.
// Each CTA's gate/up units come in two batches in flight; its router rows and the norm
// weights of the next layer are copied during phase C, its 16 down rows of the active
// experts (up to DL_STAGE routed ones) during phase B.  Completion is counted on
// mbarriers (one cp.async arrival per thread).  Every wait (tags, copies) gives up after
// a time limit (error bit, abort flag shared by all CTAs).
#include "common.cuh"
#include "decode_tag.h"
#include "gemm_common.cuh"
#include "internal.h"

#include <mutex>

namespace moe {

namespace {

constexpr int DL_THREADS = 512;
constexpr int DL_WARPS = DL_THREADS / 32;
constexpr int DL_ROWS_C = 16;                 // output rows per CTA in phase C
constexpr int DL_CTAS_C = HID / DL_ROWS_C;    // 128 CTAs carry phase C
constexpr int DL_STAGE = 18;                  // routed experts whose down rows are staged in shared memory
constexpr int NROW_A = NEXP + 1;              // router rows + the shared-expert gate row
constexpr unsigned DL_POLL_NS = 100;          // pause between polls of a stale tagged word
constexpr int DQ_WORDS = DL_ROWS_C * INTER / 8;        // 1024 words = 4 KB of packed down rows
constexpr int DQ_GROUPS = DL_ROWS_C * INTER / GROUP;   // 128 scales (or biases) = 256 B
// gate/up unit in shared memory: 8 gate rows, 8 up rows (1 KB each), then the scales
// and biases of both (8 x 32 bf16 each)
constexpr int U_ROWB = HID / 2;                        // 1024 bytes of packed codes per row
constexpr int U_SC = 16 * U_ROWB;                      // 16384: gate scales, gate biases, up scales, up biases
constexpr int U_BYTES = U_SC + 4 * 8 * (HID / GROUP) * 2;   // 18432
constexpr int DL_UB = 2;                               // units per batch; two batches in flight
constexpr int HS_ROWS = 2 * DL_UB * U_BYTES / (INTER * 2);  // 72 rows of h' (1 KB) in the same space

struct alignas(16) DlShared {
  uint8_t gu[2 * DL_UB][U_BYTES];               // phase B: staged units; phase C: h' rows
  __nv_bfloat16 xn[DEC_MAX_T][HID];             // normalised layer input (natural order)
  float red[DL_UB][DL_WARPS][32][4];            // K-split partials
  uint32_t dq[DL_STAGE][DQ_WORDS];              // staged down rows of routed experts
  uint16_t dsc[DL_STAGE][DQ_GROUPS];
  uint16_t dbi[DL_STAGE][DQ_GROUPS];
  uint32_t sdq[DQ_WORDS];                       // staged down rows of the shared expert
  uint16_t sdsc[DQ_GROUPS];
  uint16_t sdbi[DQ_GROUPS];
  __nv_bfloat16 rrow[2][HID];                   // this CTA's router rows
  __nv_bfloat16 normw[HID];                     // the layer's norm weights
  uint64_t mb_a, mb_c, mb_b[2];                 // bulk-copy barriers
  float xres[DEC_MAX_T][DL_ROWS_C];             // residual inputs of this CTA's output rows
  float ssp[DEC_MAX_T][8];                      // sum-of-squares partials
  float inv_rms[DEC_MAX_T];
  float rpart[DL_WARPS][DEC_MAX_T];             // router partials
  float sig[DEC_MAX_T];                         // shared-expert gate per token
  int idx[DEC_MAX_T][TOPK];
  float w[DEC_MAX_T][TOPK];
  uint32_t mask[NEXP / 32];                     // experts routed by any token
  int act_e[DEC_MAX_ACTIVE];
  float act_w[DEC_MAX_ACTIVE][DEC_MAX_T];
  int n_active;
  int abort;
  int last;                                     // this CTA is the last one out of the launch
};
static_assert(HS_ROWS >= DEC_MAX_T * 9, "h' staging must hold one batch of 9 experts at T = 8");
static_assert(DEC_MAX_LAYERS <= (1 << DEC_TAG_LAYER_BITS), "a tag holds the layer in its low bits");
static_assert(sizeof(DlShared) <= 232448, "shared memory per CTA exceeds 227 KB");
static_assert(DEC_LT_WORDS == 2ull * DEC_MAX_T * NROW_A && DEC_HT_WORDS == 2ull * DEC_MAX_ACTIVE * DEC_MAX_T * (INTER / 2) &&
                  DEC_XT_WORDS == 2ull * DEC_MAX_T * (HID / 2),
              "tagged table sizes");

struct Ctx {
  unsigned long long* trace;    // this layer's and CTA's timestamps, or nullptr
  uint32_t tag;                 // current layer's tag
  unsigned* abort_word;         // grid-wide abort flag
  unsigned* err;
  unsigned long long limit;     // time limit of a bounded wait
};

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ __nv_bfloat162 bf2h(uint16_t bits) {
  const uint32_t v = static_cast<uint32_t>(bits) * 0x00010001u;
  return *reinterpret_cast<const __nv_bfloat162*>(&v);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// 16-byte asynchronous global -> shared copy (L2 only); a CTA copies contiguous blocks
// with consecutive threads on consecutive 16-byte pieces, fully coalesced.
__device__ __forceinline__ void cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
// The calling thread's arrival on `bar` once all its earlier cp.async copies have landed
// (the barrier counts one arrival per thread of the CTA).
__device__ __forceinline__ void cp_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cta_copy(void* dst, const void* src, int bytes) {
  for (int i = threadIdx.x * 16; i < bytes; i += DL_THREADS * 16)
    cp16(static_cast<uint8_t*>(dst) + i, static_cast<const uint8_t*>(src) + i);
}

// ---- tagged words
// Published with an atomic exchange (performed at L2, its old value discarded) rather than
// a plain store: measured with per-CTA phase stamps, plain relaxed stores of the router
// logits became visible to the polling CTAs 4-7 us after they were issued (write-through,
// release and fenced stores likewise), the exchanges about 2 us after.
__device__ __forceinline__ void st_tagged(unsigned long long* p, uint32_t payload, uint32_t tag) {
  const unsigned long long v = (static_cast<unsigned long long>(tag) << 32) | payload;
  asm volatile("{\n\t.reg .b64 old;\n\tatom.relaxed.gpu.global.exch.b64 old, [%0], %1;\n\t}" ::"l"(p), "l"(v)
               : "memory");
}
__device__ __forceinline__ unsigned long long ld_tagged(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void ld_tagged2(const unsigned long long* p, unsigned long long& a,
                                           unsigned long long& b) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ bool tag_ok(unsigned long long v, uint32_t tag) {
  return static_cast<uint32_t>(v >> 32) == tag;
}

// Paces the re-polling of stale tagged words: false once the caller must give up (the
// time limit, which raises the grid's abort flag, or an abort raised elsewhere).
struct PollClock {
  unsigned long long t0 = 0;
  __device__ __forceinline__ bool tick(const Ctx& cx) {
    if (*reinterpret_cast<volatile unsigned*>(cx.abort_word) != 0u) return false;
    const unsigned long long now = globaltimer_ns();
    if (t0 == 0) {
      t0 = now;
    } else if (cx.limit < WAIT_LIMIT_IMMEDIATE_NS || now - t0 > cx.limit) {
      atomicOr(cx.err, ERRBIT_TIMEOUT);
      atomicExch(cx.abort_word, 1u);
      return false;
    }
    __nanosleep(DL_POLL_NS);   // keeps the polling of 152 CTAs from crowding the L2 slices
    return true;
  }
};

// Phase timestamp k of this layer and CTA (tracing only).
__device__ __forceinline__ void stamp(const Ctx& cx, int k) {
  if (cx.trace != nullptr && threadIdx.x == 0) cx.trace[k] = globaltimer_ns();
}

// ---- order-preserving float keys (larger float -> larger key); NaN maps below -inf
__device__ __forceinline__ uint32_t fkey(float v) {
  const uint32_t u = __float_as_uint(v);
  if (v != v) return 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float kfloat(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// bounded wait on one of this CTA's bulk-copy barriers, the same outcome in every thread
__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t parity, const Ctx& cx, DlShared& s) {
  bool ok = mbar_wait(smem_u32(bar), parity, cx.err, &s.abort, cx.limit);
  if (!ok) atomicExch(cx.abort_word, 1u);
  return __syncthreads_and(ok) != 0;
}

// ---------------------------------------------------------------- staging (all threads)
// Phase A's inputs of layer L: this CTA's router rows and the norm weights.
__device__ void issue_stage_a(const DecLayer& L, DlShared& s) {
  const int c = blockIdx.x, G = gridDim.x;
  for (int sl = 0; sl < 2; ++sl) {
    const int r = c + sl * G;
    if (r < NROW_A) cta_copy(s.rrow[sl], r < NEXP ? L.router_w + static_cast<size_t>(r) * HID : L.shared_gate_w, HID * 2);
  }
  if (L.norm_w) cta_copy(s.normw, L.norm_w, HID * 2);
  cp_arrive(&s.mb_a);
}

// Phase C's weights of layer L for this CTA's 16 output rows: the down rows of the
// shared expert and of the first DL_STAGE routed experts into shared memory (phase C
// reads the rows of any further routed experts from memory).
__device__ void issue_stage_c(const DecLayer& L, DlShared& s) {
  const int c = blockIdx.x, tid = threadIdx.x;
  if (c >= DL_CTAS_C) return;
  const int n_routed = s.n_active - 1;
  const int n_st = n_routed < DL_STAGE ? n_routed : DL_STAGE;
  constexpr int PIECES = (DQ_WORDS * 4 + 2 * DQ_GROUPS * 2) / 16;   // 288 per expert
  for (int k = tid; k < (n_st + 1) * PIECES; k += DL_THREADS) {
    const int i = k / PIECES, off = k % PIECES;
    const bool sh = i == n_st;
    const size_t r0 = (sh ? 0 : static_cast<size_t>(s.act_e[i]) * HID) + static_cast<size_t>(c) * DL_ROWS_C;
    if (off < DQ_WORDS / 4) {
      cp16((sh ? s.sdq : s.dq[i]) + off * 4, (sh ? L.sdq : L.dq) + r0 * (INTER / 8) + off * 4);
    } else if (off < DQ_WORDS / 4 + DQ_GROUPS / 8) {
      const int o = (off - DQ_WORDS / 4) * 8;
      cp16((sh ? s.sdsc : s.dsc[i]) + o, (sh ? L.sds : L.ds) + r0 * (INTER / GROUP) + o);
    } else {
      const int o = (off - DQ_WORDS / 4 - DQ_GROUPS / 8) * 8;
      cp16((sh ? s.sdbi : s.dbi[i]) + o, (sh ? L.sdb : L.db) + r0 * (INTER / GROUP) + o);
    }
  }
  cp_arrive(&s.mb_c);
}

// Gate/up batch b of this CTA (units blockIdx.x + (DL_UB*b + j) * G) into buffer b & 1:
// per unit 8 KB of gate rows, 8 KB of up rows, 4 x 512 B of scales and biases.
__device__ void issue_units(const DecLayer& L, DlShared& s, int b, int n_units) {
  const int tid = threadIdx.x, G = gridDim.x, buf = b & 1;
  constexpr int SB = 8 * (HID / GROUP) * 2;   // 512 B of scales (or biases) for 8 rows
  for (int j = 0; j < DL_UB; ++j) {
    const int u = blockIdx.x + (DL_UB * b + j) * G;
    if (u >= n_units) break;
    const int a = u / (INTER / 8), f0 = (u % (INTER / 8)) * 8;
    const int e = s.act_e[a];
    const bool sh = e == NEXP;
    const size_t row = (sh ? 0 : static_cast<size_t>(e) * INTER) + f0;
    uint8_t* dst = s.gu[buf * DL_UB + j];
    static_assert(8 * U_ROWB == DL_THREADS * 16, "one 16-byte piece of each 8-row block per thread");
    cp16(dst + tid * 16, reinterpret_cast<const uint8_t*>((sh ? L.sgq : L.gq) + row * (HID / 8)) + tid * 16);
    cp16(dst + 8 * U_ROWB + tid * 16, reinterpret_cast<const uint8_t*>((sh ? L.suq : L.uq) + row * (HID / 8)) + tid * 16);
    if (tid < 4 * SB / 16) {
      const int part = tid / (SB / 16), o = (tid % (SB / 16)) * 16;
      const uint16_t* src = part == 0 ? (sh ? L.sgs : L.gs) : part == 1 ? (sh ? L.sgb : L.gb)
                          : part == 2 ? (sh ? L.sus : L.us) : (sh ? L.sub : L.ub);
      cp16(dst + U_SC + part * SB + o, reinterpret_cast<const uint8_t*>(src + row * (HID / GROUP)) + o);
    }
  }
  cp_arrive(&s.mb_b[buf]);
}

// ---------------------------------------------------------------- phase A
// x -> xn in shared memory (RMSNorm with the layer's weights, or a copy), then this CTA's
// router logits.  Layer 0 reads the caller's x; later layers the tagged output of the
// layer before.
__device__ bool phase_a(const DecLayersParams& p, const DecLayer& L, int l, const Ctx& cx, DlShared& s) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.T, c = blockIdx.x, G = gridDim.x;
  // thread chunk q = 8 inputs of token q / 256; a warp-iteration covers 32 chunks of one token
  constexpr int CH_PER_THREAD = DEC_MAX_T * (HID / 8) / DL_THREADS;   // 4
  uint4 v[CH_PER_THREAD];
  bool ok = true;
  if (l == 0) {
#pragma unroll
    for (int i = 0; i < CH_PER_THREAD; ++i) {
      const int q = tid + DL_THREADS * i;
      v[i] = make_uint4(0, 0, 0, 0);
      if (q / (HID / 8) < T) v[i] = ldg_nc_v4(p.x + static_cast<size_t>(q) * 8);
    }
  } else {
    const unsigned long long* xt = p.xt + static_cast<size_t>(l & 1) * DEC_MAX_T * (HID / 2);
    unsigned long long e[CH_PER_THREAD][4];
#pragma unroll
    for (int i = 0; i < CH_PER_THREAD; ++i) {
      const int q = tid + DL_THREADS * i;
      if (q / (HID / 8) < T) {
        ld_tagged2(xt + static_cast<size_t>(q) * 4, e[i][0], e[i][1]);
        ld_tagged2(xt + static_cast<size_t>(q) * 4 + 2, e[i][2], e[i][3]);
      }
    }
    // re-poll every stale word of this thread together: one L2 round trip per poll
    PollClock pc;
    while (true) {
      bool stale = false;
#pragma unroll
      for (int i = 0; i < CH_PER_THREAD; ++i)
        if ((tid + DL_THREADS * i) / (HID / 8) < T)
#pragma unroll
          for (int k = 0; k < 4; ++k) stale |= !tag_ok(e[i][k], cx.tag);
      if (!stale) break;
      if (!pc.tick(cx)) { ok = false; break; }
#pragma unroll
      for (int i = 0; i < CH_PER_THREAD; ++i) {
        const int q = tid + DL_THREADS * i;
        if (q / (HID / 8) < T) {
          if (!tag_ok(e[i][0], cx.tag) || !tag_ok(e[i][1], cx.tag))
            ld_tagged2(xt + static_cast<size_t>(q) * 4, e[i][0], e[i][1]);
          if (!tag_ok(e[i][2], cx.tag) || !tag_ok(e[i][3], cx.tag))
            ld_tagged2(xt + static_cast<size_t>(q) * 4 + 2, e[i][2], e[i][3]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < CH_PER_THREAD; ++i)
      v[i] = ((tid + DL_THREADS * i) / (HID / 8) < T)
                 ? make_uint4(static_cast<uint32_t>(e[i][0]), static_cast<uint32_t>(e[i][1]),
                              static_cast<uint32_t>(e[i][2]), static_cast<uint32_t>(e[i][3]))
                 : make_uint4(0, 0, 0, 0);
  }
  if (!__syncthreads_and(ok)) return false;
  stamp(cx, 1);
  // residual inputs of this CTA's phase-C rows (chunks 2c, 2c+1 of every token)
  if (p.residual && c < DL_CTAS_C) {
#pragma unroll
    for (int i = 0; i < CH_PER_THREAD; ++i) {
      const int q = tid + DL_THREADS * i;
      const int t = q / (HID / 8), ch = q % (HID / 8);
      if (t < T && (ch >> 1) == c) {
        const uint32_t u[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          s.xres[t][(ch & 1) * 8 + 2 * j] = bf16lo(u[j]);
          s.xres[t][(ch & 1) * 8 + 2 * j + 1] = bf16hi(u[j]);
        }
      }
    }
  }
  if (!cta_wait(&s.mb_a, l & 1, cx, s)) return false;
  stamp(cx, 2);
  if (L.norm_w) {
#pragma unroll
    for (int i = 0; i < CH_PER_THREAD; ++i) {
      const int t = (tid + DL_THREADS * i) / (HID / 8);
      const uint32_t u[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
      float ss = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        ss = fmaf(bf16lo(u[j]), bf16lo(u[j]), ss);
        ss = fmaf(bf16hi(u[j]), bf16hi(u[j]), ss);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      if (lane == 0 && t < T) s.ssp[t][warp & 7] = ss;
    }
    __syncthreads();
    if (tid < T) {
      float ss = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) ss += s.ssp[tid][j];
      s.inv_rms[tid] = 1.0f / sqrtf(ss / static_cast<float>(HID) + 1e-6f);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < CH_PER_THREAD; ++i) {
    const int q = tid + DL_THREADS * i;
    const int t = q / (HID / 8), k = (q % (HID / 8)) * 8;
    uint4 o = v[i];
    if (L.norm_w && t < T) {
      const float r = s.inv_rms[t];
      const uint4 g = *reinterpret_cast<const uint4*>(&s.normw[k]);
      const uint32_t u[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
      const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
      uint32_t ov[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        ov[j] = pack_bf16x2(bf16lo(u[j]) * r * bf16lo(gw[j]), bf16hi(u[j]) * r * bf16hi(gw[j]));
      o = make_uint4(ov[0], ov[1], ov[2], ov[3]);
    }
    *reinterpret_cast<uint4*>(&s.xn[t][k]) = o;
  }
  __syncthreads();

  // router rows: 8 warps per row, each 256 inputs (8 per lane)
  const int slot = warp >> 3, ks = (warp & 7) * 256 + lane * 8;
  const int r = c + slot * G;
  float acc[DEC_MAX_T];
#pragma unroll
  for (int t = 0; t < DEC_MAX_T; ++t) acc[t] = 0.0f;
  if (r < NROW_A) {
    const uint4 wv = *reinterpret_cast<const uint4*>(&s.rrow[slot][ks]);
    const uint32_t wu[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int t = 0; t < DEC_MAX_T; ++t) {
      if (t < T) {
        const uint4 xv = *reinterpret_cast<const uint4*>(&s.xn[t][ks]);
        const uint32_t xu[4] = {xv.x, xv.y, xv.z, xv.w};
        float a = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          a = fmaf(bf16lo(xu[j]), bf16lo(wu[j]), a);
          a = fmaf(bf16hi(xu[j]), bf16hi(wu[j]), a);
        }
        acc[t] = a;
      }
    }
  }
#pragma unroll
  for (int t = 0; t < DEC_MAX_T; ++t) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
  }
  if (lane == 0) {
#pragma unroll
    for (int t = 0; t < DEC_MAX_T; ++t) s.rpart[warp][t] = acc[t];
  }
  __syncthreads();
  if (tid < 2 * DEC_MAX_T) {
    const int sl = tid / DEC_MAX_T, t = tid % DEC_MAX_T;
    const int rr = c + sl * G;
    if (rr < NROW_A && t < T) {
      float a = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) a += s.rpart[sl * 8 + j][t];
      if (rr < NEXP && L.router_bias) a += L.router_bias[rr];
      st_tagged(p.lt + (static_cast<size_t>(l & 1) * DEC_MAX_T + t) * NROW_A + rr, __float_as_uint(a), cx.tag);
    }
  }
  stamp(cx, 3);
  return true;
}

// ---------------------------------------------------------------- phase B
// Top-8 per token (one warp per token; the arg-max of each round by warp reductions on
// order-preserving keys, ties to the lowest expert id), renormalised weights, and the
// list of active experts from a bitmap of the routed ids.
__device__ bool phase_b_route(const DecLayersParams& p, const DecLayer& L, int l, const Ctx& cx, DlShared& s,
                              bool write_topk) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.T;
  for (int i = tid; i < DEC_MAX_ACTIVE * DEC_MAX_T; i += DL_THREADS) (&s.act_w[0][0])[i] = 0.0f;
  if (tid < NEXP / 32) s.mask[tid] = 0u;
  bool ok = true;
  if (warp < T) {
    const int t = warp;
    const unsigned long long* lt = p.lt + (static_cast<size_t>(l & 1) * DEC_MAX_T + t) * NROW_A;
    unsigned long long e[9];
#pragma unroll
    for (int j = 0; j < 8; ++j) e[j] = ld_tagged(lt + lane + 32 * j);
    e[8] = lane == 0 ? ld_tagged(lt + NEXP) : 0ull;
    PollClock pc;
    while (true) {
      bool stale = lane == 0 && !tag_ok(e[8], cx.tag);
#pragma unroll
      for (int j = 0; j < 8; ++j) stale |= !tag_ok(e[j], cx.tag);
      if (!stale) break;
      if (!pc.tick(cx)) { ok = false; break; }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (!tag_ok(e[j], cx.tag)) e[j] = ld_tagged(lt + lane + 32 * j);
      if (lane == 0 && !tag_ok(e[8], cx.tag)) e[8] = ld_tagged(lt + NEXP);
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      if (lane == 0) s.sig[t] = 1.0f / (1.0f + expf(-__uint_as_float(static_cast<uint32_t>(e[8]))));
      // key + 1: 0 marks an expert already taken (+inf's key + 1 does not wrap)
      uint32_t key[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) key[j] = fkey(__uint_as_float(static_cast<uint32_t>(e[j]))) + 1u;
      float selv[TOPK];
      int sele[TOPK];
#pragma unroll
      for (int k = 0; k < TOPK; ++k) {
        uint32_t bk = 0u;
        int bj = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (key[j] > bk) { bk = key[j]; bj = j; }
        const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t ex =
            __reduce_min_sync(0xffffffffu, bk == m ? static_cast<uint32_t>(lane + 32 * bj) : 0xFFFFFFFFu);
        if ((ex & 31u) == static_cast<uint32_t>(lane)) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (j == static_cast<int>(ex >> 5)) key[j] = 0u;
        }
        selv[k] = kfloat(m - 1u);
        sele[k] = static_cast<int>(ex);
      }
      float exv[TOPK], sum = 0.0f;
#pragma unroll
      for (int k = 0; k < TOPK; ++k) { exv[k] = expf(selv[k] - selv[0]); sum += exv[k]; }
      const float inv = 1.0f / sum;
      if (lane < TOPK) {
        float wk = 0.0f, vk = 0.0f;
        int ek = 0;
#pragma unroll
        for (int k = 0; k < TOPK; ++k)
          if (k == lane) { wk = exv[k] * inv; ek = sele[k]; vk = selv[k]; }
        if (!isfinite(vk) && blockIdx.x == 0) atomicOr(L.err, ERRBIT_BOUNDS);   // non-finite logits
        s.idx[t][lane] = ek;
        s.w[t][lane] = wk;
        if (write_topk) {
          p.topk_idx[t * TOPK + lane] = ek;
          p.topk_w[t * TOPK + lane] = wk;
        }
      }
    }
  }
  if (!__syncthreads_and(ok)) return false;
  stamp(cx, 4);
  if (tid < T * TOPK) {
    const int e = s.idx[tid / TOPK][tid % TOPK];
    atomicOr(&s.mask[e >> 5], 1u << (e & 31));
  }
  __syncthreads();
  // position of expert e in the active list = number of routed ids below it
  auto pos = [&](int e) {
    int n = __popc(s.mask[e >> 5] & ((1u << (e & 31)) - 1u));
    for (int w = 0; w < (e >> 5); ++w) n += __popc(s.mask[w]);
    return n;
  };
  if (tid < T * TOPK) {
    const int t = tid / TOPK, e = s.idx[t][tid % TOPK];
    s.act_w[pos(e)][t] = s.w[t][tid % TOPK];
  } else if (tid >= DL_THREADS - NEXP) {
    const int e = tid - (DL_THREADS - NEXP);
    if ((s.mask[e >> 5] >> (e & 31)) & 1u) s.act_e[pos(e)] = e;
  }
  if (tid < DEC_MAX_T) {
    int n = 0;
#pragma unroll
    for (int w = 0; w < NEXP / 32; ++w) n += __popc(s.mask[w]);
    if (tid == 0) {
      s.act_e[n] = NEXP;
      s.n_active = n + 1;
    }
    if (tid < T) s.act_w[n][tid] = s.sig[tid];
  }
  __syncthreads();
  stamp(cx, 5);
  return true;
}

__device__ bool phase_b_gateup(const DecLayersParams& p, const DecLayer& L, int l, const Ctx& cx, DlShared& s,
                               uint32_t (&bphase)[2]) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c4 = lane & 3;
  const int T = p.T, G = gridDim.x;
  const int kbase = warp * (HID / DL_WARPS);           // 128 inputs per warp
  const int wo = kbase / 8 + 4 * c4;                   // word offset in a gate/up row
  const int gi = (kbase + 32 * c4) / GROUP;            // quantisation group
  const int n_units = s.n_active * (INTER / 8);
  const int my_units = blockIdx.x < n_units ? (n_units - 1 - blockIdx.x) / G + 1 : 0;
  const int nb = (my_units + DL_UB - 1) / DL_UB;
  for (int b = 0; b < 2 && b < nb; ++b) issue_units(L, s, b, n_units);
  issue_stage_c(L, s);   // phase C's copies queue behind the first batches
  stamp(cx, 6);
  // B fragments (token g, this lane's 32 inputs), the same for every unit
  uint4 xb[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    xb[j] = make_uint4(0, 0, 0, 0);
    if (g < T) xb[j] = interleave8(*reinterpret_cast<const uint4*>(&s.xn[g][kbase + 32 * c4 + 8 * j]));
  }
  unsigned long long* ht = p.ht + static_cast<size_t>(l & 1) * DEC_MAX_ACTIVE * DEC_MAX_T * (INTER / 2);
  for (int b = 0; b < nb; ++b) {
    const int buf = b & 1;
    if (!cta_wait(&s.mb_b[buf], bphase[buf] & 1, cx, s)) return false;
    ++bphase[buf];
    if (b == 0) stamp(cx, 7);
#pragma unroll
    for (int j = 0; j < DL_UB; ++j) {
      const int u = blockIdx.x + (DL_UB * b + j) * G;
      if (u >= n_units) break;
      const uint8_t* U = s.gu[buf * DL_UB + j];
      const uint4 wg = *reinterpret_cast<const uint4*>(U + g * U_ROWB + wo * 4);
      const uint4 wu = *reinterpret_cast<const uint4*>(U + (8 + g) * U_ROWB + wo * 4);
      const uint16_t* sc = reinterpret_cast<const uint16_t*>(U + U_SC);
      const __nv_bfloat162 mg = bf2h(sc[g * 32 + gi]), ag = bf2h(sc[256 + g * 32 + gi]);
      const __nv_bfloat162 mu = bf2h(sc[512 + g * 32 + gi]), au = bf2h(sc[768 + g * 32 + gi]);
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t gw[4] = {wg.x, wg.y, wg.z, wg.w};
      const uint32_t uw[4] = {wu.x, wu.y, wu.z, wu.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 o0 = dequant8(gw[k], mg, ag), o1 = dequant8(uw[k], mu, au);
        mma16816(d, o0.x, o1.x, o0.y, o1.y, xb[k].x, xb[k].y);
        mma16816(d, o0.z, o1.z, o0.w, o1.w, xb[k].z, xb[k].w);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) s.red[j][warp][lane][k] = d[k];
    }
    if (b == 0) stamp(cx, 12);
    __syncthreads();
    if (b + 2 < nb) issue_units(L, s, b + 2, n_units);   // buffer b & 1 is free
    if (tid < DL_UB * 32) {
      const int j = tid >> 5, ln = tid & 31;
      const int u = blockIdx.x + (DL_UB * b + j) * G;   // warp-uniform
      if (u < n_units) {
        float q[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int w = 0; w < DL_WARPS; ++w)
#pragma unroll
          for (int k = 0; k < 4; ++k) q[k] += s.red[j][w][ln][k];
        // q[0], q[1]: gate of feature f0 + ln/4 for tokens 2(ln%4), 2(ln%4)+1; q[2], q[3]: up
        const int a = u / (INTER / 8), fi = ln >> 2, t0 = 2 * (ln & 3);
        float hv[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float gv = q[h], uv = q[2 + h];
          hv[h] = gv / (1.0f + __expf(-gv)) * uv * s.act_w[a][t0 + h];
        }
        // interleaved pair (2i, 2i+1) of the unit holds features (i, i + 4)
        const float h0 = __shfl_down_sync(0xffffffffu, hv[0], 16);
        const float h1 = __shfl_down_sync(0xffffffffu, hv[1], 16);
        if (fi < 4) {
          const size_t pair = (u % (INTER / 8)) * 4 + fi;
#pragma unroll
          for (int h = 0; h < 2; ++h)
            if (t0 + h < T)
              st_tagged(ht + (static_cast<size_t>(a) * DEC_MAX_T + t0 + h) * (INTER / 2) + pair,
                        pack_bf16x2(hv[h], h ? h1 : h0), cx.tag);
        }
      }
    }
    if (b == 0) stamp(cx, 13);
    __syncthreads();
  }
  stamp(cx, 8);
  return true;
}

// ---------------------------------------------------------------- phase C
__device__ __forceinline__ void down_mma(float (&d)[4], uint4 w0, uint4 w1, uint16_t s0, uint16_t s1, uint16_t b0,
                                         uint16_t b1, uint4 (&hb)[4]) {
  const __nv_bfloat162 m0 = bf2h(s0), m1 = bf2h(s1), c0 = bf2h(b0), c1 = bf2h(b1);
  const uint32_t x0[4] = {w0.x, w0.y, w0.z, w0.w};
  const uint32_t x1[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 o0 = dequant8(x0[j], m0, c0), o1 = dequant8(x1[j], m1, c1);
    mma16816(d, o0.x, o1.x, o0.y, o1.y, hb[j].x, hb[j].y);
    mma16816(d, o0.z, o1.z, o0.w, o1.w, hb[j].z, hb[j].w);
  }
}

__device__ bool phase_c(const DecLayersParams& p, const DecLayer& L, int l, const Ctx& cx, DlShared& s) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c4 = lane & 3;
  const int ks = warp & 3, eq = warp >> 2;
  const int T = p.T;
  if (blockIdx.x >= DL_CTAS_C) return true;            // uniform per CTA
  const int r0 = blockIdx.x * DL_ROWS_C + g, r1 = r0 + 8;
  const int n_act = s.n_active, n_routed = n_act - 1;
  const int n_st = n_routed < DL_STAGE ? n_routed : DL_STAGE;
  const int wo = ks * 16 + 4 * c4;                     // word offset in a down row (64 words)
  const int gi = (ks * 128 + 32 * c4) / GROUP;         // quantisation group (8 per row)
  const unsigned long long* ht = p.ht + static_cast<size_t>(l & 1) * DEC_MAX_ACTIVE * DEC_MAX_T * (INTER / 2);
  uint32_t* hs = reinterpret_cast<uint32_t*>(&s.gu[0][0]);   // h' rows [expert-in-batch * T + t][256 pairs]
  if (!cta_wait(&s.mb_c, l & 1, cx, s)) return false;
  stamp(cx, 9);
  float d[4] = {0.f, 0.f, 0.f, 0.f};
  const int eb = HS_ROWS / T;                          // experts per batch
  for (int a0 = 0; a0 < n_act; a0 += eb) {
    const int na = n_act - a0 < eb ? n_act - a0 : eb;
    // h' of experts a0 .. a0+na-1, tokens < T, from the tagged table into shared memory
    const int n_pairs = na * T * (INTER / 2);
    bool ok = true;
    constexpr int PG = 4;   // pieces of 2 words per thread polled together
    for (int g0 = 2 * tid; g0 < n_pairs && ok; g0 += PG * 2 * DL_THREADS) {
      unsigned long long w[PG][2];
      auto src = [&](int k) {
        const int i0 = g0 + k * 2 * DL_THREADS;
        const int row = i0 / (INTER / 2), pr = i0 % (INTER / 2);
        return ht + (static_cast<size_t>(a0 + row / T) * DEC_MAX_T + row % T) * (INTER / 2) + pr;
      };
#pragma unroll
      for (int k = 0; k < PG; ++k)
        if (g0 + k * 2 * DL_THREADS < n_pairs) ld_tagged2(src(k), w[k][0], w[k][1]);
      PollClock pc;
      while (true) {
        bool stale = false;
#pragma unroll
        for (int k = 0; k < PG; ++k)
          if (g0 + k * 2 * DL_THREADS < n_pairs) stale |= !tag_ok(w[k][0], cx.tag) || !tag_ok(w[k][1], cx.tag);
        if (!stale) break;
        if (!pc.tick(cx)) { ok = false; break; }
#pragma unroll
        for (int k = 0; k < PG; ++k)
          if (g0 + k * 2 * DL_THREADS < n_pairs && (!tag_ok(w[k][0], cx.tag) || !tag_ok(w[k][1], cx.tag)))
            ld_tagged2(src(k), w[k][0], w[k][1]);
      }
#pragma unroll
      for (int k = 0; k < PG; ++k) {
        const int i0 = g0 + k * 2 * DL_THREADS;
        if (i0 < n_pairs)
          *reinterpret_cast<uint2*>(hs + i0) = make_uint2(static_cast<uint32_t>(w[k][0]), static_cast<uint32_t>(w[k][1]));
      }
    }
    if (!__syncthreads_and(ok)) return false;
    if (a0 == 0) stamp(cx, 10);
    for (int ai = eq; ai < na; ai += 4) {
      const int a = a0 + ai;
      uint4 hb[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        hb[j] = (g < T) ? *reinterpret_cast<const uint4*>(hs + (ai * T + g) * (INTER / 2) + ks * 64 + 16 * c4 + 4 * j)
                        : make_uint4(0, 0, 0, 0);
      const bool sh = a == n_routed;
      if (sh || a < n_st) {
        const uint32_t* q = sh ? s.sdq : s.dq[a];
        const uint16_t* sc = sh ? s.sdsc : s.dsc[a];
        const uint16_t* bi = sh ? s.sdbi : s.dbi[a];
        const uint4 w0 = *reinterpret_cast<const uint4*>(q + g * (INTER / 8) + wo);
        const uint4 w1 = *reinterpret_cast<const uint4*>(q + (g + 8) * (INTER / 8) + wo);
        down_mma(d, w0, w1, sc[g * (INTER / GROUP) + gi], sc[(g + 8) * (INTER / GROUP) + gi],
                 bi[g * (INTER / GROUP) + gi], bi[(g + 8) * (INTER / GROUP) + gi], hb);
      } else {   // beyond the staging capacity: straight from memory
        const size_t rw0 = static_cast<size_t>(s.act_e[a]) * HID + r0, rw1 = rw0 + 8;
        const uint4 w0 = ldg_nc_v4(L.dq + rw0 * (INTER / 8) + wo);
        const uint4 w1 = ldg_nc_v4(L.dq + rw1 * (INTER / 8) + wo);
        down_mma(d, w0, w1, __ldg(L.ds + rw0 * (INTER / GROUP) + gi), __ldg(L.ds + rw1 * (INTER / GROUP) + gi),
                 __ldg(L.db + rw0 * (INTER / GROUP) + gi), __ldg(L.db + rw1 * (INTER / GROUP) + gi), hb);
      }
    }
    __syncthreads();   // the h' rows are rewritten by the next batch
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) s.red[0][warp][lane][k] = d[k];
  stamp(cx, 14);
  __syncthreads();
  if (warp == 0) {
    float q[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < DL_WARPS; ++w)
#pragma unroll
      for (int k = 0; k < 4; ++k) q[k] += s.red[0][w][lane][k];
    // q[0]: (row r0, token 2c), q[1]: (r0, 2c+1), q[2]: (r1, 2c), q[3]: (r1, 2c+1)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int tok = 2 * c4 + (k & 1);
      if (p.residual && tok < T) q[k] += s.xres[tok][(k < 2) ? g : g + 8];
    }
    stamp(cx, 15);
    if (l + 1 == p.n_layers) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int tok = 2 * c4 + (k & 1);
        if (tok < T) p.out[static_cast<size_t>(tok) * HID + ((k < 2) ? r0 : r1)] = __float2bfloat16_rn(q[k]);
      }
    } else {
      // the next layer's input, as tagged pairs of adjacent rows (lanes g and g + 1)
      unsigned long long* xt = p.xt + static_cast<size_t>((l + 1) & 1) * DEC_MAX_T * (HID / 2);
      const uint32_t tag = cx.tag + 1u;
      float nb[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) nb[k] = __shfl_down_sync(0xffffffffu, q[k], 4);
      if ((g & 1) == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int tok = 2 * c4 + (k & 1);
          const int row = (k < 2) ? r0 : r1;
          if (tok < T) st_tagged(xt + static_cast<size_t>(tok) * (HID / 2) + row / 2, pack_bf16x2(q[k], nb[k]), tag);
        }
      }
    }
  }
  stamp(cx, 11);
  return true;
}

}  // namespace

__global__ void __launch_bounds__(DL_THREADS, 1) decode_layers_kernel(const __grid_constant__ DecLayersParams p) {
  extern __shared__ __align__(128) uint8_t dl_smem[];
  DlShared& s = *reinterpret_cast<DlShared*>(dl_smem);
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&s.mb_a), DL_THREADS);   // one cp.async arrival per thread
    mbar_init(smem_u32(&s.mb_c), DL_THREADS);
    mbar_init(smem_u32(&s.mb_b[0]), DL_THREADS);
    mbar_init(smem_u32(&s.mb_b[1]), DL_THREADS);
    s.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // tags: dec_tag(launch epoch, layer); the epoch advances when a launch ends
  const uint32_t epoch = *reinterpret_cast<volatile unsigned*>(p.sync + 3);
  Ctx cx;
  cx.trace = nullptr;
  cx.abort_word = p.sync + 2;
  cx.limit = p.wait_ns;
  uint32_t bphase[2] = {0u, 0u};
  issue_stage_a(p.layer[0], s);
  for (int l = 0; l < p.n_layers; ++l) {
    const DecLayer& L = p.layer[l];
    cx.tag = dec_tag(epoch, l);
    cx.err = L.err;
    cx.trace = (p.trace != nullptr && blockIdx.x < DEC_TRACE_CTAS)
                   ? p.trace + (static_cast<size_t>(l) * DEC_TRACE_CTAS + blockIdx.x) * DEC_TRACE_STAMPS
                   : nullptr;
    stamp(cx, 0);
    if (!phase_a(p, L, l, cx, s)) break;
    if (!phase_b_route(p, L, l, cx, s, l == p.n_layers - 1 && blockIdx.x == 0 && p.topk_idx != nullptr)) break;
    if (!phase_b_gateup(p, L, l, cx, s, bphase)) break;
    if (l + 1 < p.n_layers) {
      issue_stage_a(p.layer[l + 1], s);
    }
    if (!phase_c(p, L, l, cx, s)) break;
  }
  // leaving early: this thread's copies still in flight land before the CTA exits
  asm volatile("cp.async.wait_all;" ::: "memory");
  // the last CTA out clears the exit count and the abort flag and advances the epoch;
  // at the end of an epoch period it first clears every tagged word (see decode_tag.h)
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s.last = atomicAdd(p.sync + 1, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (s.last) {
    __threadfence();
    const uint32_t next = dec_next_epoch(epoch);
    if (next == 0u) {
      for (size_t i = threadIdx.x; i < DEC_LT_WORDS; i += DL_THREADS) p.lt[i] = 0ull;
      for (size_t i = threadIdx.x; i < DEC_HT_WORDS; i += DL_THREADS) p.ht[i] = 0ull;
      for (size_t i = threadIdx.x; i < DEC_XT_WORDS; i += DL_THREADS) p.xt[i] = 0ull;
      __threadfence();
      __syncthreads();
    }
    if (threadIdx.x == 0) {
      atomicExch(p.sync + 2, 0u);
      atomicExch(p.sync + 3, next);
      __threadfence();
      atomicExch(p.sync + 1, 0u);
    }
  }
}

cudaError_t launch_decode_layers(const DecLayersParams& p, cudaStream_t s) {
  // per device: the kernel's shared-memory attribute is a setting of the current device,
  // and the grid is that device's SM count
  constexpr int kMaxDevices = 64;
  struct DevInit {
    std::once_flag once;
    int grid = 0;
    cudaError_t err = cudaSuccess;
  };
  static DevInit init[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  DevInit& d = init[dev];
  std::call_once(d.once, [&d, dev] {
    int nsm = 0, per_sm = 0;
    cudaError_t e2 = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e2 == cudaSuccess)
      e2 = cudaFuncSetAttribute(decode_layers_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(sizeof(DlShared)));
    if (e2 == cudaSuccess)
      e2 = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_layers_kernel, DL_THREADS, sizeof(DlShared));
    if (e2 == cudaSuccess && per_sm < 1) e2 = cudaErrorCooperativeLaunchTooLarge;
    if (e2 == cudaSuccess && nsm < DL_CTAS_C) e2 = cudaErrorCooperativeLaunchTooLarge;
    d.err = e2;
    d.grid = nsm;   // one CTA per SM: all resident, as the cross-CTA waits require
  });
  if (d.err != cudaSuccess) return d.err;
  void* args[] = {const_cast<DecLayersParams*>(&p)};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(decode_layers_kernel), dim3(d.grid),
                                     dim3(DL_THREADS), args, sizeof(DlShared), s);
}

}  // namespace moe
