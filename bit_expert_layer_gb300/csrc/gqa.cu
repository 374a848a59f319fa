// gqa.cu -- grouped-query decode attention over a bf16 KV cache, for the model's
// full-attention layers: 16 query heads share 2 key/value heads (aimanavo.com, "Why is
// Perplexity's local AI Lily faster than MLX", section "Qwen3.6's 256 experts and two layer
// kinds make the MLX/Lily gap").  Decode reads the whole KV cache at every step, so it is
// bound by memory bandwidth, and Lily packs the query heads of a group so that each KV row
// is read once for all of them (same page, section "Prefill and decode are not treated as
// the same job"; dzen.guru, "Perplexity opened the Lily engine", section "Where the
// speed-up comes from").  Here the 8 query heads of a group are the rows of one MMA tile:
// every key and value row crosses HBM once and feeds all 8 heads.
//
// One new query token per sequence; per (sequence b, KV head g) the cached positions are
// split over `nsplit` CTAs (flash-decoding), one CTA per SM.  A CTA streams its positions in
// chunks of 128 keys (K and V, 64 KB per stage, four TMA boxes of 16 KB with the 128-byte
// swizzle: few, large copies, since each bulk copy has a fixed cost) through a ring of
// GQ_STAGES stages; 8 consumer warps take 16 keys each per stage:
//   S^T = Q K^T   mma.sync m16n8k16: A = the 8 query heads (rows 8..15 zero), B = K rows
//                 (ldmatrix), fp32 scores
//   online softmax in base 2 per head (running max and sum), probabilities rounded to
//                 bf16 (the sum is taken over the rounded values)
//   O += P V      A = P straight from the score fragments, B = V (ldmatrix.trans)
// The warps' partial (max, sum, O) merge in shared memory, each CTA writes its split's
// partial to the workspace, and the last CTA of a (b, g) pair (an atomic ticket, no waiting)
// merges the splits in split order and writes the 8 heads' outputs as bf16.  The MMAs are
// the legacy warp-level ones: the contraction has 8 useful rows and is bound by HBM (4
// multiply-adds per byte), where they cost about a fifth of the run time.
#include <cstring>

#include "common.cuh"
#include "gqa_decode.h"
#include "internal.h"
#include "moe_layer.h"

namespace moe {

namespace {

constexpr int GQ_STAGE_K = 0;                          // K: two boxes of GQ_CH keys x 64 dims
constexpr int GQ_STAGE_V = 2 * GQ_CH * 64 * 2;         // V: the same, after K
constexpr int GQ_SMEM = GQ_STAGES * GQ_STAGE_BYTES + 1024 /* align */ + 256 /* barriers */;
constexpr int GQ_WARPS = GQ_CH / 16;                  // consumers (16 keys each); the last warp is the TMA producer
constexpr int GQ_PS = GQ_D + 4;   // floats per partial row: O[128], max (base 2), sum, 2 unused (16-byte rows)
constexpr int GQ_FS_OFF = GQ_STAGE_BYTES;   // merge weights [8][GQ_MAX_SPLIT] in the second stage
static_assert(GQ_WARPS * GQ_G * (GQ_D + 2) * 4 <= GQ_FS_OFF, "warp-merge scratch fits the first stage");
static_assert(GQ_FS_OFF + GQ_G * GQ_MAX_SPLIT * 4 <= GQ_STAGES * GQ_STAGE_BYTES, "split weights fit the stages");

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  // rows 8..15 of A (a1, a3) are zero: the 8 query heads of a group fill rows 0..7
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// Byte offset of (key r, 16-byte chunk cd of the 256-byte row) in a stage's K or V half:
// box cd / 8 (dims 0-63 or 64-127), 128-byte swizzle inside the box.
__device__ __forceinline__ uint32_t kv_off(int r, int cd) {
  return static_cast<uint32_t>((cd >> 3) * (GQ_CH * 128) + r * 128 + (((cd & 7) ^ (r & 7)) << 4));
}

}  // namespace

__global__ void __launch_bounds__((GQ_WARPS + 1) * 32)
    gqa_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ GqaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + GQ_STAGES * GQ_STAGE_BYTES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * GQ_STAGES);
  int* s_last = const_cast<int*>(abort_flag) + 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + GQ_STAGES);

  const int len = p.lens[b];
  const int kps = ((len + p.nsplit - 1) / p.nsplit + GQ_CH - 1) / GQ_CH * GQ_CH;   // keys per split
  const int k0 = split * kps;
  const int k1 = min(len, k0 + kps);
  const int nch = k1 > k0 ? (k1 - k0 + GQ_CH - 1) / GQ_CH : 0;
  const int row0 = (b * GQ_HKV + g) * p.S_max + k0;    // tensor-map row of this split's first key

  if (tid == 0) {
    for (int s = 0; s < GQ_STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, GQ_WARPS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  int issued = 0;   // producer: chunks whose loads it issued
  // per consumer warp: running max (base 2), this thread's share of the sum, O fragments
  float m_run = -INFINITY, l_part = 0.0f;
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;

  if (warp == GQ_WARPS) {
    if (lane == 0 && nch > 0) {
      // ------------------------------------------------ TMA producer
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const uint64_t pol = l2_policy_evict_first();   // every KV row is read once
      for (int c = 0; c < nch; ++c) {
        const int s = c % GQ_STAGES;
        if (!mbar_wait(empty0 + 8 * s, ((c / GQ_STAGES) & 1) ^ 1, p.err, abort_flag, p.wait_ns)) break;
        const uint32_t st = smem_u32(smem + s * GQ_STAGE_BYTES);
        mbar_arrive_expect_tx(full0 + 8 * s, GQ_STAGE_BYTES);
        const int y = row0 + c * GQ_CH;
        tma_load_2d_hint(st + GQ_STAGE_K, &tm_k, full0 + 8 * s, 0, y, pol);
        tma_load_2d_hint(st + GQ_STAGE_K + GQ_CH * 128, &tm_k, full0 + 8 * s, 64, y, pol);
        tma_load_2d_hint(st + GQ_STAGE_V, &tm_v, full0 + 8 * s, 0, y, pol);
        tma_load_2d_hint(st + GQ_STAGE_V + GQ_CH * 128, &tm_v, full0 + 8 * s, 64, y, pol);
        issued = c + 1;
      }
    }
  } else {
    // ------------------------------------------------ consumers: 16 keys per warp and stage
    const int g4 = lane >> 2, c2 = (lane & 3) * 2;
    // A fragments of Q: head g4 of the group, dims 16j + c2 (+1) and 16j + 8 + c2 (+1)
    uint32_t qa[8][2];
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(p.q + (static_cast<size_t>(b) * GQ_HQ + g * GQ_G + g4) * GQ_D);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      qa[j][0] = __ldg(qrow + (16 * j + c2) / 2);
      qa[j][1] = __ldg(qrow + (16 * j + 8 + c2) / 2);
    }
    const float sc = p.scale_log2;
    for (int c = 0; c < nch; ++c) {
      const int s = c % GQ_STAGES;
      // the whole warp goes on or stops together (ldmatrix and mma.sync are warp-collective)
      if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * s, (c / GQ_STAGES) & 1, p.err, abort_flag, p.wait_ns))) break;
      const uint32_t st = smem_u32(smem + s * GQ_STAGE_BYTES);
      const int kw = warp * 16;                         // this warp's first key in the chunk
      // ---- scores of keys kw .. kw+15 (two n8 blocks) for the 8 heads
      float sv[2][4];
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
        sv[nb][0] = sv[nb][1] = sv[nb][2] = sv[nb][3] = 0.0f;
        const int r = kw + 8 * nb + (lane & 7);         // the key whose row this thread addresses
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {                // dims 32jj .. 32jj+31
          uint32_t b0, b1, b2, b3;
          ldsm_x4(st + GQ_STAGE_K + kv_off(r, 4 * jj + (lane >> 3)), b0, b1, b2, b3);
          mma_bf16_16816(sv[nb], qa[2 * jj][0], qa[2 * jj][1], b0, b1);
          mma_bf16_16816(sv[nb], qa[2 * jj + 1][0], qa[2 * jj + 1][1], b2, b3);
        }
      }
      // ---- online softmax (base 2); keys at or past the length are masked
      const int kg = k0 + c * GQ_CH + kw;               // global position of key kw
      float x[4];
      x[0] = (kg + c2 < k1) ? sv[0][0] * sc : -INFINITY;
      x[1] = (kg + c2 + 1 < k1) ? sv[0][1] * sc : -INFINITY;
      x[2] = (kg + 8 + c2 < k1) ? sv[1][0] * sc : -INFINITY;
      x[3] = (kg + 8 + c2 + 1 < k1) ? sv[1][1] * sc : -INFINITY;
      float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run, mx);
      // every key so far masked: nothing to add, nothing to rescale
      const float corr = (m_new == -INFINITY) ? 1.0f : exp2f(m_run - m_new);
      float pr[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pr[i] = (m_new == -INFINITY) ? 0.0f : exp2f(x[i] - m_new);
      const uint32_t pa0 = pack2_bf16(pr[0], pr[1]);    // keys c2, c2+1
      const uint32_t pa2 = pack2_bf16(pr[2], pr[3]);    // keys 8+c2, 8+c2+1
      l_part = l_part * corr + bf16lo(pa0) + bf16hi(pa0) + bf16lo(pa2) + bf16hi(pa2);
      m_run = m_new;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        o[i][0] *= corr;
        o[i][1] *= corr;
      }
      // ---- O += P V over the 128 dims (16 n8 blocks, two per ldmatrix.x4.trans)
      const int rv = kw + 8 * ((lane >> 3) & 1) + (lane & 7);
#pragma unroll
      for (int dn = 0; dn < 16; dn += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(st + GQ_STAGE_V + kv_off(rv, dn + (lane >> 4)), b0, b1, b2, b3);
        mma_bf16_16816(o[dn], pa0, pa2, b0, b1);
        mma_bf16_16816(o[dn + 1], pa0, pa2, b2, b3);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }
    l_part += __shfl_xor_sync(0xffffffffu, l_part, 1);
    l_part += __shfl_xor_sync(0xffffffffu, l_part, 2);
  }

  // ------------------------------------------------ merge the warps, then the splits
  __syncthreads();
  if (warp == GQ_WARPS && lane == 0 && *abort_flag) {
    // a launch that gave up: loads still in flight land before the shared memory goes away
    for (int c = (issued > GQ_STAGES ? issued - GQ_STAGES : 0); c < issued; ++c) {
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(full0 + 8 * (c % GQ_STAGES), (c / GQ_STAGES) & 1) && globaltimer_ns() - t0 < WAIT_LIMIT_NS) {
      }
    }
  }
  __syncthreads();
  // the stages are free now: per warp m[8], l[8], o[8][128] (fp32)
  float* wm = reinterpret_cast<float*>(smem);
  float* wl = wm + GQ_WARPS * GQ_G;
  float* wo = wl + GQ_WARPS * GQ_G;
  if (warp < GQ_WARPS) {
    const int g4 = lane >> 2, c2 = (lane & 3) * 2;
    if ((lane & 3) == 0) {
      wm[warp * GQ_G + g4] = m_run;
      wl[warp * GQ_G + g4] = l_part;
    }
#pragma unroll
    for (int dn = 0; dn < 16; ++dn) {
      wo[(warp * GQ_G + g4) * GQ_D + 8 * dn + c2] = o[dn][0];
      wo[(warp * GQ_G + g4) * GQ_D + 8 * dn + c2 + 1] = o[dn][1];
    }
  }
  __syncthreads();
  // 128 threads: head h = tid / 16, dims 8 (tid % 16) .. +7; this split's partial
  if (tid < GQ_G * 16) {
    const int h = tid >> 4, d0 = (tid & 15) * 8;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < GQ_WARPS; ++w) M = fmaxf(M, wm[w * GQ_G + h]);
    float L = 0.0f, O[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int w = 0; w < GQ_WARPS; ++w) {
      const float f = (M == -INFINITY) ? 0.0f : exp2f(wm[w * GQ_G + h] - M);
      L += f * wl[w * GQ_G + h];
#pragma unroll
      for (int i = 0; i < 8; ++i) O[i] += f * wo[(w * GQ_G + h) * GQ_D + d0 + i];
    }
    float* dst = p.part + ((static_cast<size_t>(b) * GQ_HQ + g * GQ_G + h) * p.nsplit + split) * GQ_PS;
    *reinterpret_cast<float4*>(dst + d0) = make_float4(O[0], O[1], O[2], O[3]);
    *reinterpret_cast<float4*>(dst + d0 + 4) = make_float4(O[4], O[5], O[6], O[7]);
    if (d0 == 0) *reinterpret_cast<float2*>(dst + GQ_D) = make_float2(M, L);
  }
  __threadfence();   // publish the partial before the ticket is taken
  __syncthreads();
  unsigned* ticket = p.ticket + b * GQ_HKV + g;
  if (tid == 0) *s_last = (atomicAdd(ticket, 1u) == static_cast<unsigned>(p.nsplit) - 1u);
  __syncthreads();
  if (!*s_last) return;
  __threadfence();
  // The last CTA of (b, g) merges the splits.  Every load below is independent of the
  // others, so they are issued together rather than as one chain of L2 round trips:
  // (1) the 16 threads of head h read the splits' (max, sum) pairs, split j, j + 16, ...
  //     each, and reduce the maximum and the rescaled sum across the 16;
  // (2) each thread sums its 8 dims of O over the splits with the weights from (1).
  const int ns = p.nsplit;
  float* fs = reinterpret_cast<float*>(smem + GQ_FS_OFF);   // [8][GQ_MAX_SPLIT] split weights
  float L = 0.0f;
  if (tid < GQ_G * 16) {
    const int h = tid >> 4, j = tid & 15;
    const float* src = p.part + (static_cast<size_t>(b) * GQ_HQ + g * GQ_G + h) * ns * GQ_PS;
    float2 ml[GQ_MAX_SPLIT / 16];
#pragma unroll
    for (int i = 0; i < GQ_MAX_SPLIT / 16; ++i)
      ml[i] = (j + 16 * i < ns) ? __ldcg(reinterpret_cast<const float2*>(src + (j + 16 * i) * GQ_PS + GQ_D))
                                : make_float2(-INFINITY, 0.0f);
    float M = -INFINITY;
#pragma unroll
    for (int i = 0; i < GQ_MAX_SPLIT / 16; ++i)
      if (ml[i].y > 0.0f) M = fmaxf(M, ml[i].x);
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
#pragma unroll
    for (int i = 0; i < GQ_MAX_SPLIT / 16; ++i) {
      const float f = (ml[i].y > 0.0f) ? exp2f(ml[i].x - M) : 0.0f;   // empty splits weigh nothing
      L += f * ml[i].y;
      if (j + 16 * i < ns) fs[h * GQ_MAX_SPLIT + j + 16 * i] = f;
    }
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  }
  __syncthreads();
  if (tid < GQ_G * 16) {
    const int h = tid >> 4, d0 = (tid & 15) * 8;
    const float* src = p.part + (static_cast<size_t>(b) * GQ_HQ + g * GQ_G + h) * ns * GQ_PS + d0;
    const float* fh = fs + h * GQ_MAX_SPLIT;
    float O[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    int sp = 0;
    for (; sp + 4 <= ns; sp += 4) {   // four splits' loads in flight at once
      float4 a[4], c[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        a[u] = __ldcg(reinterpret_cast<const float4*>(src + (sp + u) * GQ_PS));
        c[u] = __ldcg(reinterpret_cast<const float4*>(src + (sp + u) * GQ_PS + 4));
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float f = fh[sp + u];
        O[0] += f * a[u].x, O[1] += f * a[u].y, O[2] += f * a[u].z, O[3] += f * a[u].w;
        O[4] += f * c[u].x, O[5] += f * c[u].y, O[6] += f * c[u].z, O[7] += f * c[u].w;
      }
    }
    for (; sp < ns; ++sp) {
      const float4 a = __ldcg(reinterpret_cast<const float4*>(src + sp * GQ_PS));
      const float4 c = __ldcg(reinterpret_cast<const float4*>(src + sp * GQ_PS + 4));
      const float f = fh[sp];
      O[0] += f * a.x, O[1] += f * a.y, O[2] += f * a.z, O[3] += f * a.w;
      O[4] += f * c.x, O[5] += f * c.y, O[6] += f * c.z, O[7] += f * c.w;
    }
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    if (!(L > 0.0f)) atomicOr(p.err, ERRBIT_BOUNDS);   // no key at all: cannot happen for len >= 1
    uint4 r;
    r.x = pack2_bf16(O[0] * inv, O[1] * inv);
    r.y = pack2_bf16(O[2] * inv, O[3] * inv);
    r.z = pack2_bf16(O[4] * inv, O[5] * inv);
    r.w = pack2_bf16(O[6] * inv, O[7] * inv);
    *reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(b) * GQ_HQ + g * GQ_G + h) * GQ_D + d0) = r;
  }
  if (tid == 0) *ticket = 0u;   // ready for the next call (every CTA of this pair has taken its ticket)
}

cudaError_t launch_gqa_decode(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const GqaParams& p, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(gqa_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GQ_SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  gqa_decode_kernel<<<dim3(p.nsplit, GQ_HKV, p.B), (GQ_WARPS + 1) * 32, GQ_SMEM, s>>>(tm_k, tm_v, p);
  return cudaGetLastError();
}

}  // namespace moe

// ============================================================================ C ABI
namespace moe {
namespace {

constexpr size_t GQ_PART_FLOATS_PER_SEQ = static_cast<size_t>(GQ_HQ) * GQ_MAX_SPLIT * GQ_PS;

struct GqaWorkspace {
  unsigned* err;
  unsigned* ticket;
  float* part;
};

// error word (256 B), tickets [GQ_MAX_B][2] (512 B), partials
constexpr size_t GQ_WS_TICKETS = 256;
constexpr size_t GQ_WS_PART = GQ_WS_TICKETS + GQ_MAX_B * GQ_HKV * 4;
static_assert(GQ_WS_PART % 256 == 0, "partials 256-byte aligned");

GqaWorkspace gqa_carve(void* ws) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  return GqaWorkspace{reinterpret_cast<unsigned*>(b), reinterpret_cast<unsigned*>(b + GQ_WS_TICKETS),
                      reinterpret_cast<float*>(b + GQ_WS_PART)};
}

size_t gqa_ws_bytes(int B) {
  if (B < 1 || B > GQ_MAX_B) return 0;
  return GQ_WS_PART + static_cast<size_t>(B) * GQ_PART_FLOATS_PER_SEQ * 4;
}

int sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 148;
  }
  return cached[dev];
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t gqa_decode_workspace_bytes(int B) { return gqa_ws_bytes(B); }

extern "C" moe_status_t gqa_decode_attention(const void* q, const void* k, const void* v, const int32_t* lens, int B,
                                             int S_max, void* out, void* workspace, size_t workspace_bytes,
                                             moe_stream_t stream) {
  if (!q || !k || !v || !lens || !out || !workspace) return MOE_ERR_INVALID_ARG;
  if (B < 1 || B > GQ_MAX_B || S_max < 1 || S_max > (1 << 20)) return MOE_ERR_INVALID_ARG;
  const uintptr_t al = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                       reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out);
  if ((al & 15u) != 0 || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MOE_ERR_ALIGNMENT;
  if (workspace_bytes < gqa_ws_bytes(B)) return MOE_ERR_WORKSPACE;
  GqaParams p;
  std::memset(&p, 0, sizeof p);
  int max_len = 0;
  for (int b = 0; b < B; ++b) {
    if (lens[b] < 1 || lens[b] > S_max) return MOE_ERR_INVALID_ARG;
    p.lens[b] = lens[b];
    max_len = lens[b] > max_len ? lens[b] : max_len;
  }
  const GqaWorkspace w = gqa_carve(workspace);
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.part = w.part;
  p.ticket = w.ticket;
  p.err = w.err;
  p.B = B;
  p.S_max = S_max;
  // one CTA per SM over all (sequence, KV head) pairs in a single wave, no more splits
  // than chunks
  int ns = sm_count() / (GQ_HKV * B);
  const int chunks = (max_len + GQ_CH - 1) / GQ_CH;
  ns = ns < chunks ? ns : chunks;
  ns = ns < GQ_MAX_SPLIT ? ns : GQ_MAX_SPLIT;
  p.nsplit = ns < 1 ? 1 : ns;
  p.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(GQ_D));
  p.wait_ns = wait_limit_ns();
  CUtensorMap tk, tv;
  const uint64_t rows = static_cast<uint64_t>(B) * GQ_HKV * S_max;
  if (!encode_bf16_sw128(&tk, k, GQ_D, rows, GQ_CH) || !encode_bf16_sw128(&tv, v, GQ_D, rows, GQ_CH))
    return MOE_ERR_CUDA;
  const cudaError_t e = launch_gqa_decode(tk, tv, p, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    set_error_detail("gqa_decode_attention: launch", e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

extern "C" moe_status_t gqa_decode_get_error(void* workspace) {
  if (!workspace) return MOE_ERR_INVALID_ARG;
  const GqaWorkspace w = gqa_carve(workspace);
  unsigned v = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(&v, w.err, 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(w.err, 0, 4);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    set_error_detail("gqa_decode_get_error", e);
    return MOE_ERR_CUDA;
  }
  if (v & ERRBIT_TIMEOUT) return MOE_ERR_TIMEOUT;
  if (v & ERRBIT_BOUNDS) return MOE_ERR_DEVICE_BOUNDS;
  return MOE_OK;
}
