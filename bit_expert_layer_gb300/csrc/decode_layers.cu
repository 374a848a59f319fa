// decode_layers.cu -- the memory-bound decode path (T <= 8 tokens) as one persistent
// kernel that runs every layer of a decode step.  Decode reads the weights again at
// every step, so the bound moves from compute to memory bandwidth (aimanavo.com, "Why
// is Perplexity's local AI Lily faster than MLX", section "Prefill and decode are not
// treated as the same job"); Lily overlaps its many small decode kernels (same page,
// section "Where the gains come from").  Here the stages of a layer are phases of one
// cooperative launch, and no launch gap or grid-wide barrier sits between them.
//
// One CTA per SM (cooperative launch: all CTAs are resident, so they may wait on one
// another): 16 compute warps and 4 copy warps.  Per layer:
//   phase A  every CTA reads the layer input x, forms its RMSNorm (when the layer has
//            one) in shared memory, and computes its share of the 256 router logits and
//            the shared-expert gate logit (8 warps split the 2048 inputs of one row).
//   phase B  every CTA repeats the top-8 selection from the logits (the same result in
//            every CTA), builds the list of active experts (the routed ones in id order,
//            the shared expert last) with a per-token weight column and token mask, and
//            computes its gate/up units: 8 features x (gate row, up row) of one active
//            expert, an m16n8k16 tile whose two row halves are the gate and the up rows
//            of the same features, so SwiGLU needs no exchange.  Two units per round, the
//            16 warps splitting K; the 4-bit codes enter the MMAs as 128 + q and each
//            quantisation group's scale and bias are applied to its partial sum in fp32;
//            a fixed-order reduction gives h' = weight * silu(g) * u, published only for
//            the tokens that chose the expert (h' is zero otherwise).
//   phase C  16 output rows per CTA (128 CTAs): the weighted h' columns of every active
//            expert, four experts per job, accumulate in one MMA accumulator per warp
//            (four warps split the K of one expert: the combine over the 8 routed + 1
//            shared experts), a fixed-order reduction over the 16 warps, residual, bf16
//            out.  Only the nonzero h' rows are fetched.
//
// Hand-off between CTAs without barriers: every value one CTA passes to another (the
// layer output x, the logits, h') travels as a 64-bit word {32-bit payload, 32-bit tag}
// written and read with single-copy-atomic relaxed accesses; the tag names the launch
// (an epoch counter kept in the scratch) and the layer.  A consumer polls the words it
// needs until every tag is current, so it waits for exactly the producers it depends
// on, one L2 round trip, instead of a grid barrier followed by a read.  The tables are
// double-buffered by layer parity: a producer can be at most one layer ahead of the
// slowest consumer of the same buffer, because every layer's phase B needs all logits,
// its phase C all of h', and its phase A all of x.  Each publishing thread issues at most
// one such word per phase (a thread's exchanges would otherwise wait on one another).
//
// Weights stream through one ring of NSLOT shared-memory slots of 18 KB: a job is one
// gate/up unit (8 KB of gate rows, 8 KB of up rows, their scales and biases) or the down
// rows of four experts for the CTA's 16 output rows (4 KB each, with scales and biases).
// The four copy warps queue the CTA's job list as soon as the routing is known -- its
// gate/up units, then its down rows -- each into a slot the compute warps have released
// (full / empty mbarriers per slot), so the weights stream while the compute warps work.
// Copies are 16-byte cp.async (consecutive threads on consecutive pieces of a contiguous
// block, which streams at the HBM rate, where per-copy costs make small bulk-engine
// copies slow), counted on the slot's mbarrier; one copy warp alone issues too slowly to
// keep up, four do.  The 16-byte chunks of every weight row are stored XOR-swizzled by the
// row (chunk c of row r at c ^ (r & 7)), so the MMA fragments' loads, eight rows at a
// time, hit distinct banks.  The copy warps also fetch the next layer's router rows and
// norm weights.  The compute warps synchronise on a named barrier of their own; the copy
// warps hand their registers to them (setmaxnreg).  Every wait (tags, copies, slots)
// gives up after a time limit (error bit, abort flags shared by the CTA's warps and by all
// CTAs).
#include "common.cuh"
#include "decode_tag.h"
#include "gemm_common.cuh"
#include "internal.h"

#include <mutex>

namespace moe {

namespace {

constexpr int DL_THREADS = 512;                // compute threads (16 warps)
constexpr int DL_WARPS = DL_THREADS / 32;
constexpr int DL_COPY = 128;                   // copy threads (4 warps) that stream the weights
constexpr int DL_BLOCK = DL_THREADS + DL_COPY;
// Registers per thread after the split (setmaxnreg): the copy warpgroup hands registers to
// the four compute warpgroups.  The split needs DL_BLOCK * (registers at launch) >= its sum;
// the host checks that before the first launch.
constexpr int DL_REGS_COMPUTE = 104;
constexpr int DL_REGS_COPY = 32;
constexpr int DL_REGS_SPLIT = DL_THREADS * DL_REGS_COMPUTE + DL_COPY * DL_REGS_COPY;   // 57,344
constexpr int DL_ROWS_C = 16;                 // output rows per CTA in phase C
constexpr int DL_CTAS_C = HID / DL_ROWS_C;    // 128 CTAs carry phase C
constexpr int NROW_A = NEXP + 1;              // router rows + the shared-expert gate row
constexpr unsigned DL_POLL_NS = 0;            // pause between polls of a stale tagged word (none:
                                               // 17.40 against 17.55 us per layer at T = 1 with 100 ns)
// gate/up unit in a slot: 8 gate rows, 8 up rows (1 KB each), then the scales and biases of
// both (8 x 32 bf16 each)
constexpr int U_ROWB = HID / 2;                        // 1024 bytes of packed codes per row
constexpr int U_SC = 16 * U_ROWB;                      // 16384: gate scales, gate biases, up scales, up biases
constexpr int SLOT_BYTES = U_SC + 4 * 8 * (HID / GROUP) * 2;   // 18432
constexpr int NSLOT = 8;                               // weight ring depth
constexpr int UNITS_PER_ROUND = 2;                     // gate/up units computed together
// down rows of one expert in a slot: 16 rows x 256 bytes of codes, then 16 x 8 scales and biases
constexpr int DQ_WORDS = DL_ROWS_C * INTER / 8;        // 1024 words = 4 KB
constexpr int DQ_GROUPS = DL_ROWS_C * INTER / GROUP;   // 128 scales (or biases) = 256 B
constexpr int C_EXP_BYTES = DQ_WORDS * 4 + 2 * DQ_GROUPS * 2;   // 4608
constexpr int C_EXP_PER_JOB = SLOT_BYTES / C_EXP_BYTES;         // 4

struct alignas(16) DlShared {
  uint8_t ring[NSLOT][SLOT_BYTES];              // weight jobs
  __nv_bfloat16 xn[DEC_MAX_T][HID];             // normalised layer input (natural order); in
                                                // phase C the h' rows of one down job
  float red[2][UNITS_PER_ROUND][DL_WARPS][32][4];   // K-split partials of a round (by round parity)
  __nv_bfloat16 rrow[2][HID];                   // this CTA's router rows
  __nv_bfloat16 normw[HID];                     // the layer's norm weights
  float xg[DEC_MAX_T][HID / GROUP];             // sum of each token's xn over each quantisation group
  uint64_t mb_a;                                // router rows / norm weights of the layer landed
  uint64_t mb_full[NSLOT], mb_empty[NSLOT];     // weight slots: landed / released by the 16 compute warps
  uint64_t mb_route;                            // the layer's routing tables are built
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
  uint8_t tmask[DEC_MAX_ACTIVE];                // tokens routed to each active expert
  uint8_t rowbase[DEC_MAX_ACTIVE + 1];          // first compact h' row of each active expert
  uint16_t rowinfo[DEC_MAX_T * (TOPK + 1)];     // compact h' row -> active expert * 8 + token
  int n_active;
  int abort;
  int last;                                     // this CTA is the last one out of the launch
};
static_assert(C_EXP_PER_JOB * 4 == DL_WARPS, "four experts per down job, four warps per expert");
static_assert(UNITS_PER_ROUND % 2 == 0, "units are computed in pairs");
constexpr int HS_ROWS = DEC_MAX_T * HID * 2 / (INTER * 2);   // 32 h' rows (1 KB) fit in the xn buffer
static_assert(C_EXP_PER_JOB * DEC_MAX_T <= HS_ROWS, "the h' rows of one down job fit in the xn buffer");
static_assert(NSLOT >= 2 * UNITS_PER_ROUND, "two rounds of units in flight");
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

// The eight 4-bit codes of a packed word as bf16 pairs of 128 + q (exact), in the pair
// order of the K-interleave (q0,q4), (q1,q5), (q2,q6), (q3,q7).  The affine map of the
// codes is applied after the MMA, once per quantisation group and output element:
// sum_k (s q_k + b) x_k = s * sum_k (128 + q_k) x_k + (b - 128 s) * sum_k x_k.
__device__ __forceinline__ uint4 codes8(uint32_t w) {
  return make_uint4((w & 0x000F000Fu) | 0x43004300u, ((w >> 4) & 0x000F000Fu) | 0x43004300u,
                    ((w >> 8) & 0x000F000Fu) | 0x43004300u, ((w >> 12) & 0x000F000Fu) | 0x43004300u);
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
    if (DL_POLL_NS != 0) __nanosleep(DL_POLL_NS);
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

// Barriers of the 16 compute warps (named barrier 1; the copy warps never join them).
__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"n"(DL_THREADS) : "memory"); }
__device__ __forceinline__ bool cbar_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "n"(DL_THREADS)
      : "memory");
  return r != 0;
}

// Barrier of the copy warps (named barrier 2), with an AND of their votes.
__device__ __forceinline__ bool copy_bar_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 2, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "n"(DL_COPY)
      : "memory");
  return r != 0;
}

// bounded wait of the compute warps on one of this CTA's copy barriers, the same outcome
// in every compute thread
__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t parity, const Ctx& cx, DlShared& s) {
  bool ok = mbar_wait(smem_u32(bar), parity, cx.err, &s.abort, cx.limit);
  if (!ok) atomicExch(cx.abort_word, 1u);
  return cbar_and(ok);
}

// ---------------------------------------------------------------- staging (all threads)
// Phase A's inputs of layer L (copy warps): this CTA's router rows and the norm weights.
__device__ void issue_stage_a(const DecLayer& L, DlShared& s) {
  const int c = blockIdx.x, G = gridDim.x, ct = threadIdx.x - DL_THREADS;
  constexpr int RP = HID * 2 / 16;   // 256 pieces per row
  for (int k = ct; k < 3 * RP; k += DL_COPY) {
    const int part = k / RP, off = (k % RP) * 16;
    if (part < 2) {
      const int r = c + part * G;
      if (r < NROW_A)
        cp16(reinterpret_cast<uint8_t*>(s.rrow[part]) + off,
             reinterpret_cast<const uint8_t*>(r < NEXP ? L.router_w + static_cast<size_t>(r) * HID : L.shared_gate_w) + off);
    } else if (L.norm_w) {
      cp16(reinterpret_cast<uint8_t*>(s.normw) + off, reinterpret_cast<const uint8_t*>(L.norm_w) + off);
    }
  }
  cp_arrive(&s.mb_a);
}

// This CTA's weight jobs of a layer: n_units gate/up units (unit blockIdx.x + i * G of
// the layer's n_active * 64), then (phase-C CTAs) ceil(n_active / 4) jobs of down rows.
struct Jobs {
  int nb;      // gate/up units of this CTA
  int nc;      // down jobs of this CTA
  int n;       // nb + nc
  uint32_t j0; // ring position of the layer's first job
};

__device__ __forceinline__ Jobs layer_jobs(const DlShared& s, uint32_t j0) {
  const int G = gridDim.x;
  const int n_units = s.n_active * (INTER / 8);
  Jobs J;
  J.nb = blockIdx.x < n_units ? (n_units - 1 - static_cast<int>(blockIdx.x)) / G + 1 : 0;
  J.nc = blockIdx.x < DL_CTAS_C ? (s.n_active + C_EXP_PER_JOB - 1) / C_EXP_PER_JOB : 0;
  J.n = J.nb + J.nc;
  J.j0 = j0;
  return J;
}

// Copy job j (copy warps): its 16-byte pieces into slot (j0 + j) % NSLOT, chunk c of row r
// at c ^ (r & 7), then one arrival per copy thread on the slot's barrier.
__device__ void issue_job(const DecLayer& L, DlShared& s, const Jobs& J, int j) {
  const int ct = threadIdx.x - DL_THREADS, G = gridDim.x;
  const int slot = static_cast<int>((J.j0 + j) % NSLOT);
  uint8_t* dst = s.ring[slot];
  if (j < J.nb) {
    const int u = blockIdx.x + j * G;
    const int a = u / (INTER / 8), f0 = (u % (INTER / 8)) * 8;
    const int e = s.act_e[a];
    const bool sh = e == NEXP;
    const size_t row = (sh ? 0 : static_cast<size_t>(e) * INTER) + f0;
    const uint8_t* gsrc = reinterpret_cast<const uint8_t*>((sh ? L.sgq : L.gq) + row * (HID / 8));
    const uint8_t* usrc = reinterpret_cast<const uint8_t*>((sh ? L.suq : L.uq) + row * (HID / 8));
    constexpr int RP = 8 * U_ROWB / 16;         // 512 pieces of 8 rows
    constexpr int SB = 8 * (HID / GROUP) * 2;   // 512 B of scales (or biases) for 8 rows
    for (int k = ct; k < 2 * RP + 4 * SB / 16; k += DL_COPY) {
      if (k < 2 * RP) {
        const int m = k / RP, q = k % RP;        // matrix (gate, up), piece
        const int r = q >> 6, c = q & 63;        // row r of the 8, chunk c of its 64
        cp16(dst + m * 8 * U_ROWB + r * U_ROWB + ((c ^ (r & 7)) << 4), (m ? usrc : gsrc) + q * 16);
      } else {
        const int q = k - 2 * RP;
        const int part = q / (SB / 16), o = (q % (SB / 16)) * 16;
        const uint16_t* src = part == 0 ? (sh ? L.sgs : L.gs) : part == 1 ? (sh ? L.sgb : L.gb)
                            : part == 2 ? (sh ? L.sus : L.us) : (sh ? L.sub : L.ub);
        cp16(dst + U_SC + part * SB + o, reinterpret_cast<const uint8_t*>(src + row * (HID / GROUP)) + o);
      }
    }
  } else {
    const int a0 = (j - J.nb) * C_EXP_PER_JOB;
    const int ne = min(C_EXP_PER_JOB, s.n_active - a0);
    constexpr int PIECES = C_EXP_BYTES / 16;   // 288 per expert
    for (int k = ct; k < ne * PIECES; k += DL_COPY) {
      const int i = k / PIECES, off = k % PIECES;
      const int e = s.act_e[a0 + i];
      const bool sh = e == NEXP;
      const size_t r0 = (sh ? 0 : static_cast<size_t>(e) * HID) + static_cast<size_t>(blockIdx.x) * DL_ROWS_C;
      uint8_t* d = dst + i * C_EXP_BYTES;
      if (off < DQ_WORDS / 4) {                 // codes: 16 rows x 16 chunks
        const int r = off >> 4, c = off & 15;
        cp16(d + r * (INTER / 2) + ((c ^ (r & 7)) << 4),
             reinterpret_cast<const uint8_t*>((sh ? L.sdq : L.dq) + r0 * (INTER / 8)) + off * 16);
      } else if (off < DQ_WORDS / 4 + DQ_GROUPS / 8) {
        const int o = (off - DQ_WORDS / 4) * 8;
        cp16(d + DQ_WORDS * 4 + o * 2, (sh ? L.sds : L.ds) + r0 * (INTER / GROUP) + o);
      } else {
        const int o = (off - DQ_WORDS / 4 - DQ_GROUPS / 8) * 8;
        cp16(d + DQ_WORDS * 4 + DQ_GROUPS * 2 + o * 2, (sh ? L.sdb : L.db) + r0 * (INTER / GROUP) + o);
      }
    }
  }
  cp_arrive(&s.mb_full[slot]);
}

// The copy warps' work for one layer: every job of this CTA in order, each into a slot the
// compute warps have released, then the next layer's phase-A inputs.  False if a wait gave up.
__device__ bool copy_layer(const DecLayersParams& p, int l, const Ctx& cx, DlShared& s, const Jobs& J) {
  // The down rows follow the gate/up units at once (holding them back until the first
  // round of units had landed measured 0.1-0.7 % slower at T = 1 and 8).
  for (int j = 0; j < J.n; ++j) {
    const uint32_t q = J.j0 + static_cast<uint32_t>(j);
    // the slot's previous job has been released (its first use needs no wait)
    if (!copy_bar_and(mbar_wait(smem_u32(&s.mb_empty[q % NSLOT]), ((q / NSLOT) & 1) ^ 1, cx.err, &s.abort,
                                cx.limit)))
      return false;
    issue_job(p.layer[l], s, J, j);
  }
  if (l + 1 < p.n_layers) issue_stage_a(p.layer[l + 1], s);
  return true;
}

// This thread's bounded wait for job j's data (no barrier: the caller's next compute barrier
// makes the outcome uniform); a give-up raises the grid's abort flag.
__device__ __forceinline__ bool wait_job(const Jobs& J, int j, const Ctx& cx, DlShared& s) {
  const uint32_t q = J.j0 + static_cast<uint32_t>(j);
  const bool ok = mbar_wait(smem_u32(&s.mb_full[q % NSLOT]), (q / NSLOT) & 1, cx.err, &s.abort, cx.limit);
  if (!ok) atomicExch(cx.abort_word, 1u);
  return ok;
}
// this warp is done with job j's slot (16 arrivals free it for the copy warps)
__device__ __forceinline__ void release_job(const Jobs& J, int j, DlShared& s) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(smem_u32(&s.mb_empty[(J.j0 + static_cast<uint32_t>(j)) % NSLOT]));
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
  if (!cbar_and(ok)) return false;
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
    cbar();
    if (tid < T) {
      float ss = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) ss += s.ssp[tid][j];
      s.inv_rms[tid] = 1.0f / sqrtf(ss / static_cast<float>(HID) + 1e-6f);
    }
    cbar();
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
  cbar();

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
    if (t < T) {   // uniform
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int t = 0; t < DEC_MAX_T; ++t) s.rpart[warp][t] = acc[t];
  }
  cbar();
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
  // each token's xn summed over each quantisation group (zero for tokens past T), for the
  // bias terms of phase B; the upper warps do it while the lower ones poll the logits (the
  // barriers of the routing separate it from its readers)
  static_assert(DEC_MAX_T * (HID / GROUP) <= DL_THREADS / 2, "one sum per thread of the upper half");
  if (tid >= DL_THREADS - DEC_MAX_T * (HID / GROUP)) {
    const int i = tid - (DL_THREADS - DEC_MAX_T * (HID / GROUP));
    const int t = i / (HID / GROUP), gq = i % (HID / GROUP);
    const uint4* src = reinterpret_cast<const uint4*>(&s.xn[t][gq * GROUP]);
    float a = 0.0f;
#pragma unroll
    for (int j = 0; j < GROUP / 8; ++j) {
      const uint4 v = src[j];
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) a += bf16lo(u[k]) + bf16hi(u[k]);
    }
    s.xg[t][gq] = a;
  }
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
  if (tid < DEC_MAX_ACTIVE) s.tmask[tid] = 0;
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
  if (!cbar_and(ok)) return false;
  stamp(cx, 4);
  if (tid < T * TOPK) {
    const int e = s.idx[tid / TOPK][tid % TOPK];
    atomicOr(&s.mask[e >> 5], 1u << (e & 31));
  }
  cbar();
  // position of expert e in the active list = number of routed ids below it
  auto pos = [&](int e) {
    int n = __popc(s.mask[e >> 5] & ((1u << (e & 31)) - 1u));
    for (int w = 0; w < (e >> 5); ++w) n += __popc(s.mask[w]);
    return n;
  };
  if (tid < T * TOPK) {
    // weight column and token mask of the active expert (the shared one's are set below)
    const int t = tid / TOPK, e = s.idx[t][tid % TOPK];
    const int a = pos(e);
    s.act_w[a][t] = s.w[t][tid % TOPK];
    atomicOr(reinterpret_cast<unsigned*>(&s.tmask[0]) + (a >> 2), (1u << t) << (8 * (a & 3)));
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
      atomicOr(reinterpret_cast<unsigned*>(&s.tmask[0]) + (n >> 2), ((1u << T) - 1u) << (8 * (n & 3)));
    }
    if (tid < T) s.act_w[n][tid] = s.sig[tid];
  }
  cbar();
  stamp(cx, 5);
  return true;
}

// Gate/up units, UNITS_PER_ROUND per round, the 16 warps splitting K (128 inputs, two
// quantisation groups each); the K partials are reduced in a fixed order and
// h' = weight * silu(g) * u is published as tagged words.
//
// Each MMA's K lies inside one quantisation group: lane quarter c4 feeds words 2 c4 and
// 2 c4 + 1 of the warp's first group (eight inputs each, K-interleaved) to the first four
// MMAs and words 8 + 2 c4, 9 + 2 c4 of its second group to the last four, as the codes
// 128 + q; each group's accumulator is then scaled into the running sum with the group's
// scale s and bias term (b - 128 s) * sum(x) of the output row (see codes8).
__device__ bool phase_b_gateup(const DecLayersParams& p, const DecLayer& L, int l, const Ctx& cx, DlShared& s,
                               const Jobs& J) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c4 = lane & 3;
  const int T = p.T, G = gridDim.x;
  const int kbase = warp * (HID / DL_WARPS);           // 128 inputs per warp
  const int gq0 = kbase / GROUP;                       // its first quantisation group (even)
  // 16-byte chunk of a row holding words 2 c4, 2 c4 + 1, and their offset in it (the
  // second group's pair sits two chunks on)
  const int c0 = kbase / 32 + (c4 >> 1), o8 = (c4 & 1) * 8;
  unsigned long long* ht = p.ht + static_cast<size_t>(l & 1) * DEC_MAX_ACTIVE * DEC_MAX_T * (INTER / 2);
  // B fragments (token g; word slot k = word 2 c4 + k of the first group, 8 + 2 c4 + k - 2
  // of the second), the same for every unit
  uint4 xb[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int wd = (k < 2 ? 0 : 6) + 2 * c4 + k;
    xb[k] = make_uint4(0, 0, 0, 0);
    if (g < T) xb[k] = interleave8(*reinterpret_cast<const uint4*>(&s.xn[g][kbase + 8 * wd]));
  }
  // group sums of x for this lane's output tokens 2 c4, 2 c4 + 1 (zero past T)
  float xs[2][2];
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int i = 0; i < 2; ++i) xs[q][i] = s.xg[2 * c4 + i][gq0 + q];
  const int nr = (J.nb + UNITS_PER_ROUND - 1) / UNITS_PER_ROUND;
  for (int r = 0; r < nr; ++r) {
    const int jlo = r * UNITS_PER_ROUND, jhi = min(J.nb, jlo + UNITS_PER_ROUND);
    bool ok = true;
    for (int jj = jlo; jj < jhi && ok; ++jj) ok = wait_job(J, jj, cx, s);
    ok = __all_sync(0xffffffffu, ok);   // the warp computes together or not at all
    if (r == 0) stamp(cx, 7);
    float (*red)[DL_WARPS][32][4] = s.red[r & 1];
    // every warp: its 128 inputs of each unit of the round, two units at a time with their
    // MMAs interleaved (two independent accumulator chains)
#pragma unroll
    for (int u2 = 0; u2 < UNITS_PER_ROUND; u2 += 2) {
      if (!ok || jlo + u2 >= jhi) break;
      const bool two = jlo + u2 + 1 < jhi;                 // uniform
      uint32_t gw[2][4], uw[2][4];
      uint32_t ms[2], mb[2], ns[2], nb[2];                 // [unit]: bf16 pairs of groups gq0, gq0 + 1
#pragma unroll
      for (int v = 0; v < 2; ++v) {
        const uint8_t* U = s.ring[(J.j0 + jlo + u2 + (two ? v : 0)) % NSLOT];
        const uint16_t* sc = reinterpret_cast<const uint16_t*>(U + U_SC);
        const uint8_t* rg = U + g * U_ROWB;
        const uint8_t* ru = U + (8 + g) * U_ROWB;
        const uint2 g0 = *reinterpret_cast<const uint2*>(rg + ((c0 ^ g) << 4) + o8);
        const uint2 g1 = *reinterpret_cast<const uint2*>(rg + (((c0 + 2) ^ g) << 4) + o8);
        const uint2 u0 = *reinterpret_cast<const uint2*>(ru + ((c0 ^ g) << 4) + o8);
        const uint2 u1 = *reinterpret_cast<const uint2*>(ru + (((c0 + 2) ^ g) << 4) + o8);
        gw[v][0] = g0.x; gw[v][1] = g0.y; gw[v][2] = g1.x; gw[v][3] = g1.y;
        uw[v][0] = u0.x; uw[v][1] = u0.y; uw[v][2] = u1.x; uw[v][3] = u1.y;
        // scales and biases of rows g (gate) and g (up) for groups gq0, gq0 + 1 (adjacent)
        ms[v] = *reinterpret_cast<const uint32_t*>(sc + g * 32 + gq0);
        mb[v] = *reinterpret_cast<const uint32_t*>(sc + 256 + g * 32 + gq0);
        ns[v] = *reinterpret_cast<const uint32_t*>(sc + 512 + g * 32 + gq0);
        nb[v] = *reinterpret_cast<const uint32_t*>(sc + 768 + g * 32 + gq0);
      }
      float t[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int q = 0; q < 2; ++q) {   // quantisation group gq0 + q: word slots 2q, 2q + 1
        float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int k = 2 * q; k < 2 * q + 2; ++k) {
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            const uint4 o0 = codes8(gw[v][k]), o1 = codes8(uw[v][k]);
            mma16816(d[v], o0.x, o1.x, o0.y, o1.y, xb[k].x, xb[k].y);
            mma16816(d[v], o0.z, o1.z, o0.w, o1.w, xb[k].z, xb[k].w);
          }
        }
        // d[v][0..1]: gate row g, tokens 2 c4 and 2 c4 + 1; d[v][2..3]: up row g
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          const float sg = q ? bf16hi(ms[v]) : bf16lo(ms[v]), su = q ? bf16hi(ns[v]) : bf16lo(ns[v]);
          const float bg = fmaf(-128.0f, sg, q ? bf16hi(mb[v]) : bf16lo(mb[v]));
          const float bu = fmaf(-128.0f, su, q ? bf16hi(nb[v]) : bf16lo(nb[v]));
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            t[v][i] = fmaf(sg, d[v][i], fmaf(bg, xs[q][i], t[v][i]));
            t[v][2 + i] = fmaf(su, d[v][2 + i], fmaf(bu, xs[q][i], t[v][2 + i]));
          }
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) red[u2][warp][lane][k] = t[0][k];
      if (two) {
#pragma unroll
        for (int k = 0; k < 4; ++k) red[u2 + 1][warp][lane][k] = t[1][k];
      }
    }
    for (int jj = jlo; jj < jhi; ++jj) release_job(J, jj, s);
    if (r == 0) stamp(cx, 12);
    // one barrier per round: every warp's partials are written (and every wait succeeded);
    // the partials are double-buffered by round parity, so the next round's writes cannot
    // meet this round's reduction
    if (!cbar_and(ok)) return false;
    // warp ui reduces unit ui of the round in a fixed order (the next round's partials are
    // written only after its copy wait, which every thread reaches after this)
    if (warp < UNITS_PER_ROUND && jlo + warp < jhi) {
      const int u = blockIdx.x + (jlo + warp) * G;
      float q[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int w = 0; w < DL_WARPS; ++w)
#pragma unroll
        for (int k = 0; k < 4; ++k) q[k] += red[warp][w][lane][k];
      // q[0], q[1]: gate of feature f0 + lane/4 for tokens 2(lane%4), 2(lane%4)+1; q[2], q[3]: up
      const int a = u / (INTER / 8), fi = lane >> 2, t0 = 2 * (lane & 3);
      float hv[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float gv = q[h], uv = q[2 + h];
        hv[h] = gv / (1.0f + __expf(-gv)) * uv * s.act_w[a][t0 + h];
      }
      // interleaved pair (2i, 2i+1) of the unit holds features (i, i + 4): lanes 0-15 (features
      // 0-3) publish token t0, lanes 16-31 (features 4-7) token t0 + 1, one word each, and
      // only for tokens that chose the expert
      const float other0 = __shfl_down_sync(0xffffffffu, hv[0], 16);   // for lanes 0-15
      const float other1 = __shfl_up_sync(0xffffffffu, hv[1], 16);     // for lanes 16-31
      const bool lo = fi < 4;
      const int t = lo ? t0 : t0 + 1;
      if (t < T && ((s.tmask[a] >> t) & 1u)) {
        const size_t pair = (u % (INTER / 8)) * 4 + (fi & 3);
        st_tagged(ht + (static_cast<size_t>(a) * DEC_MAX_T + t) * (INTER / 2) + pair,
                  lo ? pack_bf16x2(hv[0], other0) : pack_bf16x2(other1, hv[1]), cx.tag);
      }
    }
    if (r == 0) stamp(cx, 13);
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

// Down rows, four experts per job: warp quarter wg takes expert 4i + wg of job i, its four
// warps split K (512) into quarters; every warp keeps its accumulator across the jobs, and
// the 16 warps' partials are reduced once, in a fixed order.
__device__ bool phase_c(const DecLayersParams& p, const DecLayer& L, int l, const Ctx& cx, DlShared& s,
                        const Jobs& J) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c4 = lane & 3;
  const int wg = warp >> 2, kq = warp & 3;
  const int T = p.T;
  if (blockIdx.x >= DL_CTAS_C) return true;            // uniform per CTA
  // compact h' rows of each active expert (the shared expert: every token): h' is zero for a
  // token that did not choose the expert, so those rows are neither published nor read
  if (warp == 0) {
    // exclusive scan of the token counts over the (at most 65) active experts, 32 at a time
    const int n = s.n_active;
    int carry = 0;
    for (int a0 = 0; a0 < n; a0 += 32) {
      const int a = a0 + lane;
      const uint32_t tm = a < n ? s.tmask[a] : 0u;
      const int c = __popc(tm);
      int incl = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      if (a < n) {
        const int base = carry + incl - c;
        s.rowbase[a] = static_cast<uint8_t>(base);
        int k = base;
        for (int t = 0; t < T; ++t)
          if ((tm >> t) & 1u) s.rowinfo[k++] = static_cast<uint16_t>(a * DEC_MAX_T + t);
        if (a == n - 1) s.rowbase[n] = static_cast<uint8_t>(base + c);
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  cbar();
  const int r0 = blockIdx.x * DL_ROWS_C + g, r1 = r0 + 8;
  const unsigned long long* ht = p.ht + static_cast<size_t>(l & 1) * DEC_MAX_ACTIVE * DEC_MAX_T * (INTER / 2);
  uint32_t* hs = reinterpret_cast<uint32_t*>(&s.xn[0][0]);   // h' rows [expert in job * T + t][256 pairs]
  const int ch = kq * 4 + c4;                         // this lane's 16-byte chunk of a down row
  const int gi = (kq * 128 + 32 * c4) / GROUP;        // its quantisation group (8 per row)
  float d[4] = {0.f, 0.f, 0.f, 0.f};
  const int n_act = s.n_active;
  int i = 0;
  while (i < J.nc) {
    // a batch of jobs whose compact h' rows (only tokens that chose the expert) fit in hs
    const int lo = s.rowbase[i * C_EXP_PER_JOB];
    int i2 = i + 1;
    while (i2 < J.nc && s.rowbase[min((i2 + 1) * C_EXP_PER_JOB, n_act)] - lo <= HS_ROWS) ++i2;
    const int n_pairs = (s.rowbase[min(i2 * C_EXP_PER_JOB, n_act)] - lo) * (INTER / 2);
    bool ok = true;
    constexpr int PG = 4;   // pieces of 2 words per thread polled together
    for (int g0 = 2 * tid; g0 < n_pairs && ok; g0 += PG * 2 * DL_THREADS) {
      unsigned long long w[PG][2];
      auto src = [&](int k) {
        const int q0 = g0 + k * 2 * DL_THREADS;
        const int ri = s.rowinfo[lo + q0 / (INTER / 2)], pr = q0 % (INTER / 2);
        return ht + static_cast<size_t>(ri) * (INTER / 2) + pr;   // ri = active expert * 8 + token
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
        const int q0 = g0 + k * 2 * DL_THREADS;
        if (q0 < n_pairs)
          *reinterpret_cast<uint2*>(hs + q0) = make_uint2(static_cast<uint32_t>(w[k][0]), static_cast<uint32_t>(w[k][1]));
      }
    }
    if (!cbar_and(ok)) return false;
    if (i == 0) stamp(cx, 10);
    // the batch's jobs, each as soon as its data is in; one barrier at the end of the batch
    bool okc = true;
    if (i == 0) stamp(cx, 9);
    for (; i < i2; ++i) {
      const int j = J.nb + i;
      const int a = i * C_EXP_PER_JOB + wg;
      if (okc) okc = __all_sync(0xffffffffu, wait_job(J, j, cx, s));
      if (okc && a < n_act) {
        // B fragments: token g's h' row if it chose the expert, else zero
        const uint32_t tm = s.tmask[a];
        const bool on = g < T && ((tm >> g) & 1u);
        const int hr = s.rowbase[a] - lo + __popc(tm & ((1u << g) - 1u));
        uint4 hb[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          hb[k] = on ? *reinterpret_cast<const uint4*>(hs + hr * (INTER / 2) + kq * 64 + 16 * c4 + 4 * k)
                     : make_uint4(0, 0, 0, 0);
        const uint8_t* D = s.ring[(J.j0 + j) % NSLOT] + wg * C_EXP_BYTES;
        const uint16_t* sc = reinterpret_cast<const uint16_t*>(D + DQ_WORDS * 4);
        const uint16_t* bi = sc + DQ_GROUPS;
        const uint4 w0 = *reinterpret_cast<const uint4*>(D + g * (INTER / 2) + ((ch ^ g) << 4));
        const uint4 w1 = *reinterpret_cast<const uint4*>(D + (g + 8) * (INTER / 2) + ((ch ^ g) << 4));
        down_mma(d, w0, w1, sc[g * (INTER / GROUP) + gi], sc[(g + 8) * (INTER / GROUP) + gi],
                 bi[g * (INTER / GROUP) + gi], bi[(g + 8) * (INTER / GROUP) + gi], hb);
      }
      release_job(J, j, s);
    }
    if (!cbar_and(okc)) return false;   // the batch's h' rows are free
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) s.red[0][0][warp][lane][k] = d[k];
  stamp(cx, 14);
  cbar();
  // warp k sums component k of the 16 warps' accumulators (row r0 or r1, token 2c or 2c+1)
  if (warp < 4) {
    const int k = warp;
    float q = 0.f;
#pragma unroll
    for (int w = 0; w < DL_WARPS; ++w) q += s.red[0][0][w][lane][k];
    const int tok = 2 * c4 + (k & 1);
    const int row = (k < 2) ? r0 : r1;
    if (p.residual && tok < T) q += s.xres[tok][(k < 2) ? g : g + 8];
    if (k == 0) stamp(cx, 15);
    if (l + 1 == p.n_layers) {
      if (tok < T) p.out[static_cast<size_t>(tok) * HID + row] = __float2bfloat16_rn(q);
    } else {
      // the next layer's input, as tagged pairs of adjacent rows (lanes g and g + 1)
      unsigned long long* xt = p.xt + static_cast<size_t>((l + 1) & 1) * DEC_MAX_T * (HID / 2);
      const float nb = __shfl_down_sync(0xffffffffu, q, 4);
      if ((g & 1) == 0 && tok < T)
        st_tagged(xt + static_cast<size_t>(tok) * (HID / 2) + row / 2, pack_bf16x2(q, nb), cx.tag + 1u);
    }
  }
  stamp(cx, 11);
  return true;
}

}  // namespace

__global__ void __launch_bounds__(DL_BLOCK, 1) decode_layers_kernel(const __grid_constant__ DecLayersParams p) {
  extern __shared__ __align__(128) uint8_t dl_smem[];
  DlShared& s = *reinterpret_cast<DlShared*>(dl_smem);
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&s.mb_a), DL_COPY);      // one cp.async arrival per copy thread
    for (int k = 0; k < NSLOT; ++k) {
      mbar_init(smem_u32(&s.mb_full[k]), DL_COPY);
      mbar_init(smem_u32(&s.mb_empty[k]), DL_WARPS);
    }
    mbar_init(smem_u32(&s.mb_route), 1);
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
  uint32_t jpos = 0;   // ring position of the next job
  static_assert(DL_THREADS % 128 == 0 && DL_COPY == 128, "whole warpgroups for the register split");
  if (threadIdx.x < DL_THREADS) {
    // ------------------------------------------------ compute warps
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(DL_REGS_COMPUTE));
    bool done = true;
    for (int l = 0; l < p.n_layers; ++l) {
      const DecLayer& L = p.layer[l];
      cx.tag = dec_tag(epoch, l);
      cx.err = L.err;
      cx.trace = (p.trace != nullptr && blockIdx.x < DEC_TRACE_CTAS)
                     ? p.trace + (static_cast<size_t>(l) * DEC_TRACE_CTAS + blockIdx.x) * DEC_TRACE_STAMPS
                     : nullptr;
      stamp(cx, 0);
      done = false;
      if (!phase_a(p, L, l, cx, s)) break;
      if (!phase_b_route(p, L, l, cx, s, l == p.n_layers - 1 && blockIdx.x == 0 && p.topk_idx != nullptr)) break;
      if (threadIdx.x == 0) mbar_arrive(smem_u32(&s.mb_route));   // the copy warps may start
      const Jobs J = layer_jobs(s, jpos);
      stamp(cx, 6);
      if (!phase_b_gateup(p, L, l, cx, s, J)) break;
      if (!phase_c(p, L, l, cx, s, J)) break;
      jpos += static_cast<uint32_t>(J.n);
      done = true;
    }
    if (!done && threadIdx.x == 0) s.abort = 1;   // the copy warps stop waiting
  } else {
    // ------------------------------------------------ copy warps
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(DL_REGS_COPY));
    issue_stage_a(p.layer[0], s);
    for (int l = 0; l < p.n_layers; ++l) {
      cx.err = p.layer[l].err;
      if (!copy_bar_and(mbar_wait(smem_u32(&s.mb_route), l & 1, cx.err, &s.abort, cx.limit))) break;
      const Jobs J = layer_jobs(s, jpos);
      if (!copy_layer(p, l, cx, s, J)) break;
      jpos += static_cast<uint32_t>(J.n);
    }
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
      for (size_t i = threadIdx.x; i < DEC_LT_WORDS; i += DL_BLOCK) p.lt[i] = 0ull;
      for (size_t i = threadIdx.x; i < DEC_HT_WORDS; i += DL_BLOCK) p.ht[i] = 0ull;
      for (size_t i = threadIdx.x; i < DEC_XT_WORDS; i += DL_BLOCK) p.xt[i] = 0ull;
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
      e2 = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_layers_kernel, DL_BLOCK, sizeof(DlShared));
    if (e2 == cudaSuccess && per_sm < 1) e2 = cudaErrorCooperativeLaunchTooLarge;
    // the register split inside the kernel draws on the registers allocated at launch: a
    // build whose allocation is smaller than the split is refused here (it would stall)
    cudaFuncAttributes fa;
    if (e2 == cudaSuccess) e2 = cudaFuncGetAttributes(&fa, decode_layers_kernel);
    if (e2 == cudaSuccess && fa.numRegs * DL_BLOCK < DL_REGS_SPLIT) e2 = cudaErrorInvalidConfiguration;
    if (e2 == cudaSuccess && nsm < DL_CTAS_C) e2 = cudaErrorCooperativeLaunchTooLarge;
    d.err = e2;
    d.grid = nsm;   // one CTA per SM: all resident, as the cross-CTA waits require
  });
  if (d.err != cudaSuccess) return d.err;
  void* args[] = {const_cast<DecLayersParams*>(&p)};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(decode_layers_kernel), dim3(d.grid),
                                     dim3(DL_BLOCK), args, sizeof(DlShared), s);
}

}  // namespace moe
