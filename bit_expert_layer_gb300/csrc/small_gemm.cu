// small_gemm.cu -- the grouped expert GEMMs of the prefill path for few tokens per expert
// (T up to about a thousand), as weight-streaming dequant-GEMV kernels.  At these sizes an
// expert owns one or two dozen rows, and the weights (455.8 MB per layer when every expert
// is touched) are the cost: the layer is memory-bound (Lily treats prefill and decode as
// different jobs with different bottlenecks: aimanavo.com, "Why is Perplexity's local AI
// Lily faster than MLX", section "Prefill and decode are not treated as the same job").
// A tcgen05 MMA of 128 weight rows costs the same issue time at N = 16 tokens as at
// N = 256, so the tile-based kernels of expert_gemm.cu and down.cu waste most of it here;
// these kernels stream each weight row once per 16 tokens through registers instead.
//
//   small_gateup_kernel  h = silu(W_gate x) * (W_up x) per permuted row (same layout as
//                        gateup_kernel writes: K-interleaved columns)
//   small_down_kernel    y = W_down h per permuted row (same layout as down_kernel)
//
// Work items (per expert, in expert order, the shared expert last):
//   gate/up  8 features (8 gate rows + 8 up rows, 16 KB of codes + 2 KB of scales and
//            biases) x up to SM_TB groups of 8 of the expert's rows
//   down     64 output rows (16 KB + 2 KB) x up to SM_TB groups of 8 rows
// Each CTA takes a contiguous range of items.  Weights reach shared memory by coalesced
// 16-byte cp.async into a ring of SM_NST stages (one mbarrier each, one arrival per
// thread), issued SM_NST items ahead.  Each thread turns its own packed words into the A
// fragments of mma.sync m16n8k16 (bf16, fp32 accumulate): the m16 tile is 8 gate rows on
// top of the same 8 up rows, so SwiGLU needs no exchange; the 8 token columns are the N
// side.  K is split over the warps and reduced in a fixed order (deterministic).
#include "common.cuh"
#include "gemm_common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int SM_THREADS = 512;
constexpr int SM_WARPS = SM_THREADS / 32;
constexpr int SM_NST = 4;                                  // weight stages in flight
constexpr int SM_TB = 2;                                   // groups of 8 rows per item
constexpr int SM_STAGE = 18432;                            // 16 KB of codes + 2 KB of scales/biases
// gate/up stage: [gate 8 rows][up 8 rows] x 1024 B, then gate scales, gate biases, up
// scales, up biases (8 rows x 32 groups x 2 B each)
constexpr int SG_ROWB = HID / 2;
constexpr int SG_SCB = 8 * (HID / GROUP) * 2;
static_assert(16 * SG_ROWB + 4 * SG_SCB == SM_STAGE, "gate/up stage size");
// down stage: 64 rows x 256 B, then 64 x 8 scales, 64 x 8 biases
constexpr int SD_ROWS = 64;
constexpr int SD_ROWB = INTER / 2;
constexpr int SD_SCB = SD_ROWS * (INTER / GROUP) * 2;
static_assert(SD_ROWS * SD_ROWB + 2 * SD_SCB == SM_STAGE, "down stage size");
constexpr int SM_PIECES = SM_STAGE / 16;                   // 1152 16-byte pieces per stage

struct alignas(16) SmShared {
  uint8_t stage[SM_NST][SM_STAGE];
  float red[SM_TB][SM_WARPS][32][4];                      // K-split partial sums
  uint16_t ytile[SM_TB * 8][SD_ROWS];                      // down: one item's outputs, bf16
  uint64_t bar[SM_NST];
  int pre[NEXP + 2];                                       // exclusive prefix of items per expert
  int off[NEXP + 2];
  int cnt[NEXP + 2];
  int abort;
};

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Items per expert: units x ceil(groups of 8 rows / SM_TB); the shared expert is 256.
// Stages the row offsets and counts, writes the exclusive prefix of items; returns the
// total.  All threads.
__device__ int stage_items(SmShared& s, const int* offsets, const int* counts, int units) {
  const int tid = threadIdx.x;
  for (int i = tid; i < NEXP + 2; i += SM_THREADS) {
    s.off[i] = __ldg(offsets + i);
    s.cnt[i] = i <= NEXP ? __ldg(counts + i) : 0;
  }
  __syncthreads();
  if (tid < 32) {
    // 257 experts over one warp: 9 per lane, then a warp scan of the lane sums
    int loc[9], sum = 0;
#pragma unroll
    for (int j = 0; j < 9; ++j) {
      const int e = tid * 9 + j;
      int v = 0;
      if (e <= NEXP) {
        const int c = max(s.cnt[e], 0);
        v = units * ((c + 8 * SM_TB - 1) / (8 * SM_TB));
      }
      loc[j] = sum;
      sum += v;
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (tid >= o) incl += n;
    }
    const int excl = incl - sum;
#pragma unroll
    for (int j = 0; j < 9; ++j) {
      const int e = tid * 9 + j;
      if (e <= NEXP + 1) s.pre[e] = excl + loc[j];
    }
  }
  __syncthreads();
  return s.pre[NEXP + 1];
}

struct Item {
  int e, unit, g0;   // expert, unit in the expert, first group of 8 rows
};

// item -> (expert, unit, first row group); `e` walks forward (a CTA's items ascend)
__device__ __forceinline__ Item item_at(const SmShared& s, int item, int& e, int units) {
  while (e < NEXP && item >= s.pre[e + 1]) ++e;
  const int local = item - s.pre[e];
  const int nb = (max(s.cnt[e], 0) + 8 * SM_TB - 1) / (8 * SM_TB);
  Item it;
  it.e = e;
  it.unit = local / nb;
  it.g0 = (local - it.unit * nb) * SM_TB;
  (void)units;
  return it;
}

__device__ __forceinline__ bool sm_wait(uint64_t* bar, uint32_t parity, unsigned int* err, SmShared& s) {
  const bool ok = mbar_wait(smem_u32(bar), parity, err, &s.abort);
  return __syncthreads_and(ok) != 0;
}

}  // namespace

// ============================================================================ gate/up
__global__ void __launch_bounds__(SM_THREADS, 1) small_gateup_kernel(SmallParams p) {
  extern __shared__ uint8_t smem_raw[];
  SmShared& s = *reinterpret_cast<SmShared*>((reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~uintptr_t(15));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c4 = lane & 3;
  constexpr int UNITS = INTER / 8;   // 64 units of 8 features per expert
  if (tid == 0) {
    for (int i = 0; i < SM_NST; ++i) mbar_init(smem_u32(&s.bar[i]), SM_THREADS);
    s.abort = 0;
    fence_mbar_init();
  }
  const int total = stage_items(s, p.offsets, p.counts, UNITS);
  const long long G = gridDim.x;
  const int i0 = static_cast<int>(total * static_cast<long long>(blockIdx.x) / G);
  const int i1 = static_cast<int>(total * static_cast<long long>(blockIdx.x + 1) / G);
  const int n = i1 - i0;
  const int n8 = 8 * p.T, n9 = 9 * p.T;

  // weights of item k into stage k % SM_NST
  int e_issue = 0;
  auto issue = [&](int k) {
    if (k < n) {
      const Item it = item_at(s, i0 + k, e_issue, UNITS);
      const bool sh = it.e == NEXP;
      const size_t row = (sh ? 0 : static_cast<size_t>(it.e) * INTER) + it.unit * 8;
      uint8_t* dst = s.stage[k % SM_NST];
      for (int q = tid; q < SM_PIECES; q += SM_THREADS) {
        const uint8_t* src;
        if (q < 512) {   // gate rows (8 KB), then up rows
          src = reinterpret_cast<const uint8_t*>((sh ? p.sgq : p.gq) + row * (HID / 8)) + q * 16;
        } else if (q < 1024) {
          src = reinterpret_cast<const uint8_t*>((sh ? p.suq : p.uq) + row * (HID / 8)) + (q - 512) * 16;
        } else {
          const int part = (q - 1024) >> 5, o = ((q - 1024) & 31) * 16;
          const uint16_t* b = part == 0 ? (sh ? p.sgs : p.gs) : part == 1 ? (sh ? p.sgb : p.gb)
                            : part == 2 ? (sh ? p.sus : p.us) : (sh ? p.sub : p.ub);
          src = reinterpret_cast<const uint8_t*>(b + row * (HID / GROUP)) + o;
        }
        cp16(dst + q * 16, src);
      }
    }
    cp_arrive(&s.bar[k % SM_NST]);   // every thread arrives on every stage use, also past the end
  };
  for (int k = 0; k < SM_NST; ++k) issue(k);

  const int kbase = warp * (HID / SM_WARPS);   // 128 inputs per warp
  const int wo = kbase / 8 + 4 * c4;           // this lane's 4 words (32 inputs) of a row
  const int gi = (kbase + 32 * c4) / GROUP;    // their quantisation group
  int e_tok = 0, e_cur = 0;
  // token of this lane's row (row g of each group) of item k, fetched one item ahead
  auto tokens = [&](int k, int (&tk)[SM_TB]) {
#pragma unroll
    for (int j = 0; j < SM_TB; ++j) tk[j] = -1;
    if (k >= n) return;
    int e = e_tok;
    const Item it = item_at(s, i0 + k, e, UNITS);
    e_tok = e;
    const int c = max(s.cnt[it.e], 0);
#pragma unroll
    for (int j = 0; j < SM_TB; ++j) {
      const int r = (it.g0 + j) * 8 + g;
      if (r < c) {
        const int row = s.off[it.e] + r;
        int t = (row >= n8) ? row - n8 : (row >= 0 && row < n8 ? (__ldg(p.row_dst + row) >> 3) : -2);
        if (t < 0 || t >= p.T || row >= n9) { atomicOr(p.err, ERRBIT_BOUNDS); t = 0; }
        tk[j] = t;
      }
    }
  };
  int tk_next[SM_TB];
  tokens(0, tk_next);
  for (int k = 0; k < n; ++k) {
    const Item it = item_at(s, i0 + k, e_cur, UNITS);
    int tk[SM_TB];
#pragma unroll
    for (int j = 0; j < SM_TB; ++j) tk[j] = tk_next[j];
    // B fragments of this item's rows (token g of each group, this lane's 32 inputs)
    uint4 xb[SM_TB][4];
#pragma unroll
    for (int j = 0; j < SM_TB; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q)
        xb[j][q] = tk[j] >= 0 ? ldg_nc_v4(p.x_ilv + static_cast<size_t>(tk[j]) * HID + kbase + 32 * c4 + 8 * q)
                              : make_uint4(0, 0, 0, 0);
    tokens(k + 1, tk_next);
    if (!sm_wait(&s.bar[k % SM_NST], (k / SM_NST) & 1, p.err, s)) break;
    const uint8_t* U = s.stage[k % SM_NST];
    const uint4 wg = *reinterpret_cast<const uint4*>(U + g * SG_ROWB + wo * 4);
    const uint4 wu = *reinterpret_cast<const uint4*>(U + (8 + g) * SG_ROWB + wo * 4);
    const uint16_t* sc = reinterpret_cast<const uint16_t*>(U + 16 * SG_ROWB);
    const __nv_bfloat162 mg = bf2(sc[g * 32 + gi]), ag = bf2(sc[256 + g * 32 + gi]);
    const __nv_bfloat162 mu = bf2(sc[512 + g * 32 + gi]), au = bf2(sc[768 + g * 32 + gi]);
    const uint32_t gw[4] = {wg.x, wg.y, wg.z, wg.w};
    const uint32_t uw[4] = {wu.x, wu.y, wu.z, wu.w};
    float d[SM_TB][4];
#pragma unroll
    for (int j = 0; j < SM_TB; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = 0.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 o0 = dequant8(gw[q], mg, ag), o1 = dequant8(uw[q], mu, au);
#pragma unroll
      for (int j = 0; j < SM_TB; ++j) {
        mma16816(d[j], o0.x, o1.x, o0.y, o1.y, xb[j][q].x, xb[j][q].y);
        mma16816(d[j], o0.z, o1.z, o0.w, o1.w, xb[j][q].z, xb[j][q].w);
      }
    }
#pragma unroll
    for (int j = 0; j < SM_TB; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) s.red[j][warp][lane][q] = d[j][q];
    __syncthreads();
    issue(k + SM_NST);   // the stage of item k is free
    if (tid < SM_TB * 32) {
      // q[0], q[1]: gate of feature unit*8 + ln/4 for rows 2(ln%4), +1 of group j; q[2], q[3]: up
      const int j = tid >> 5, ln = tid & 31;
      float q[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int w = 0; w < SM_WARPS; ++w)
#pragma unroll
        for (int i = 0; i < 4; ++i) q[i] += s.red[j][w][ln][i];
      const int fi = ln >> 2, r0 = (it.g0 + j) * 8 + 2 * (ln & 3);
      float hv[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        // silu(g) = g/2 + (g/2) tanh(g/2), the hardware tanh (relative error 2^-10.99)
        const float hg = 0.5f * q[h];
        float th;
        asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(hg));
        hv[h] = fmaf(hg, th, hg) * q[2 + h];
      }
      // interleaved pair (2i, 2i+1) of the 8 features holds features (i, i + 4)
      const float h0 = __shfl_down_sync(0xffffffffu, hv[0], 16);
      const float h1 = __shfl_down_sync(0xffffffffu, hv[1], 16);
      const int c = max(s.cnt[it.e], 0);
      if (fi < 4) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int r = r0 + h;
          if (r < c) {
            const int row = s.off[it.e] + r;
            if (row >= 0 && row < n9) {
              const __nv_bfloat162 v = __floats2bfloat162_rn(hv[h], h ? h1 : h0);
              *reinterpret_cast<__nv_bfloat162*>(p.h + static_cast<size_t>(row) * INTER + it.unit * 8 + 2 * fi) = v;
            }
          }
        }
      }
    }
    __syncthreads();   // red is free again
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// ============================================================================ down
__global__ void __launch_bounds__(SM_THREADS, 1) small_down_kernel(SmallParams p) {
  extern __shared__ uint8_t smem_raw[];
  SmShared& s = *reinterpret_cast<SmShared*>((reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~uintptr_t(15));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c4 = lane & 3;
  constexpr int UNITS = HID / SD_ROWS;   // 32 blocks of 64 output rows per expert
  if (tid == 0) {
    for (int i = 0; i < SM_NST; ++i) mbar_init(smem_u32(&s.bar[i]), SM_THREADS);
    s.abort = 0;
    fence_mbar_init();
  }
  const int total = stage_items(s, p.offsets, p.counts, UNITS);
  const long long G = gridDim.x;
  const int i0 = static_cast<int>(total * static_cast<long long>(blockIdx.x) / G);
  const int i1 = static_cast<int>(total * static_cast<long long>(blockIdx.x + 1) / G);
  const int n = i1 - i0;
  const int n9 = 9 * p.T;

  int e_issue = 0;
  auto issue = [&](int k) {
    if (k < n) {
      const Item it = item_at(s, i0 + k, e_issue, UNITS);
      const bool sh = it.e == NEXP;
      const size_t row = (sh ? 0 : static_cast<size_t>(it.e) * HID) + it.unit * SD_ROWS;
      uint8_t* dst = s.stage[k % SM_NST];
      for (int q = tid; q < SM_PIECES; q += SM_THREADS) {
        const uint8_t* src;
        if (q < 1024) {   // 64 rows x 256 B of codes, contiguous
          src = reinterpret_cast<const uint8_t*>((sh ? p.sdq : p.dq) + row * (INTER / 8)) + q * 16;
        } else {
          const int part = (q - 1024) >> 6, o = ((q - 1024) & 63) * 16;
          const uint16_t* b = part == 0 ? (sh ? p.sds : p.ds) : (sh ? p.sdb : p.db);
          src = reinterpret_cast<const uint8_t*>(b + row * (INTER / GROUP)) + o;
        }
        cp16(dst + q * 16, src);
      }
    }
    cp_arrive(&s.bar[k % SM_NST]);
  };
  for (int k = 0; k < SM_NST; ++k) issue(k);

  const int rb = warp >> 2, kq = warp & 3;     // 16-row block, K quarter (128 inputs)
  const int wo = kq * 16 + 4 * c4;             // this lane's 4 words of a row
  const int gi = (kq * 128 + 32 * c4) / GROUP;
  int e_cur = 0;
  for (int k = 0; k < n; ++k) {
    const Item it = item_at(s, i0 + k, e_cur, UNITS);
    const int c = max(s.cnt[it.e], 0), off = s.off[it.e];
    // B fragments: h of row g of each group, this lane's 32 inputs
    uint4 hb[SM_TB][4];
#pragma unroll
    for (int j = 0; j < SM_TB; ++j) {
      const int r = (it.g0 + j) * 8 + g, row = off + r;
      const bool ok = r < c && row >= 0 && row < n9;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        hb[j][q] = ok ? ldg_nc_v4(p.h + static_cast<size_t>(row) * INTER + kq * 128 + 32 * c4 + 8 * q)
                      : make_uint4(0, 0, 0, 0);
    }
    if (!sm_wait(&s.bar[k % SM_NST], (k / SM_NST) & 1, p.err, s)) break;
    const uint8_t* U = s.stage[k % SM_NST];
    const int ra = rb * 16 + g, rc = ra + 8;   // the two weight rows of this lane
    const uint4 w0 = *reinterpret_cast<const uint4*>(U + ra * SD_ROWB + wo * 4);
    const uint4 w1 = *reinterpret_cast<const uint4*>(U + rc * SD_ROWB + wo * 4);
    const uint16_t* sc = reinterpret_cast<const uint16_t*>(U + SD_ROWS * SD_ROWB);
    const __nv_bfloat162 m0 = bf2(sc[ra * 8 + gi]), b0 = bf2(sc[SD_ROWS * 8 + ra * 8 + gi]);
    const __nv_bfloat162 m1 = bf2(sc[rc * 8 + gi]), b1 = bf2(sc[SD_ROWS * 8 + rc * 8 + gi]);
    const uint32_t x0[4] = {w0.x, w0.y, w0.z, w0.w};
    const uint32_t x1[4] = {w1.x, w1.y, w1.z, w1.w};
    float d[SM_TB][4];
#pragma unroll
    for (int j = 0; j < SM_TB; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = 0.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 o0 = dequant8(x0[q], m0, b0), o1 = dequant8(x1[q], m1, b1);
#pragma unroll
      for (int j = 0; j < SM_TB; ++j) {
        mma16816(d[j], o0.x, o1.x, o0.y, o1.y, hb[j][q].x, hb[j][q].y);
        mma16816(d[j], o0.z, o1.z, o0.w, o1.w, hb[j][q].z, hb[j][q].w);
      }
    }
#pragma unroll
    for (int j = 0; j < SM_TB; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) s.red[j][warp][lane][q] = d[j][q];
    __syncthreads();
    issue(k + SM_NST);
    if (tid < SM_TB * 4 * 32) {
      // (group j, row block rb2, lane ln): sum the 4 K quarters; rows rb2*16 + ln/4 (+8) of
      // the item, tokens 2(ln%4), +1 of group j
      const int j = tid >> 7, rb2 = (tid >> 5) & 3, ln = tid & 31;
      float q[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int i = 0; i < 4; ++i) q[i] += s.red[j][rb2 * 4 + kk][ln][i];
      const int f = rb2 * 16 + (ln >> 2), t0 = j * 8 + 2 * (ln & 3);
      const __nv_bfloat16 v0 = __float2bfloat16_rn(q[0]), v1 = __float2bfloat16_rn(q[1]);
      const __nv_bfloat16 v2 = __float2bfloat16_rn(q[2]), v3 = __float2bfloat16_rn(q[3]);
      s.ytile[t0][f] = *reinterpret_cast<const uint16_t*>(&v0);
      s.ytile[t0 + 1][f] = *reinterpret_cast<const uint16_t*>(&v1);
      s.ytile[t0][f + 8] = *reinterpret_cast<const uint16_t*>(&v2);
      s.ytile[t0 + 1][f + 8] = *reinterpret_cast<const uint16_t*>(&v3);
    }
    __syncthreads();
    if (tid < SM_TB * 8 * (SD_ROWS / 8)) {
      // one 16-byte piece (8 outputs) of one row per thread
      const int t = tid / (SD_ROWS / 8), pc = tid % (SD_ROWS / 8);
      const int r = it.g0 * 8 + t, row = off + r;
      if (r < c && row >= 0 && row < n9)
        *reinterpret_cast<uint4*>(p.y + static_cast<size_t>(row) * HID + it.unit * SD_ROWS + pc * 8) =
            *reinterpret_cast<const uint4*>(&s.ytile[t][pc * 8]);
    }
    __syncthreads();   // red and ytile are free again
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

cudaError_t launch_small_gemms(const SmallParams& p, int grid, cudaStream_t s, int which) {
  const size_t smem = sizeof(SmShared) + 16;
  if (which == 0) small_gateup_kernel<<<grid, SM_THREADS, smem, s>>>(p);
  else small_down_kernel<<<grid, SM_THREADS, smem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t set_small_attributes() {
  const int smem = static_cast<int>(sizeof(SmShared) + 16);
  cudaError_t e = cudaFuncSetAttribute(small_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(small_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  return e;
}

}  // namespace moe
