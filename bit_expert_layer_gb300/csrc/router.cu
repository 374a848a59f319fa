// router.cu -- on-device routing for the prefill path, with no host synchronisation
// anywhere (Lily keeps mixture-of-experts routing on the GPU and drops the per-layer
// CPU sync: aimanavo.com, "Why is Perplexity's local AI Lily faster than MLX",
// section "Prefill and decode are not treated as the same job"; dzen.guru,
// "Perplexity opened the Lily engine", section "Where the speed-up comes from").
//
//   router_prefill_kernel  logits = x W_r^T on tcgen05 (bf16 in, fp32 accumulate in
//                          TMEM); per token: top-8 by logit with lowest-index ties (four
//                          warps per token quarter, each over 64 experts, then a merge),
//                          weights exp(l_k - l_1) / sum (equal to softmax over all 256
//                          followed by renormalisation over the 8), and a per-CTA
//                          expert histogram.
//   router_cluster_kernel  the same up to 8192 tokens with each 128-token block's K
//                          split over a cluster of 2 or 4 CTAs (partials through
//                          distributed shared memory).
//   route_scan_kernel      per-expert counts, exclusive-scan offsets, the first
//                          permuted row of every (router block, expert), and the
//                          ordered token blocks that both grouped GEMMs deal as tiles
//                          (above 16384 tokens; up to that the scatter does this work).
//   route_scatter_kernel   stable permutation of the slots t*8+k into expert order and
//                          the per-row weight (first CTA of each router block), one
//                          K-interleaved copy of x per token (the gate/up GEMM gathers
//                          its rows from it by token) and, on the same read of x, the
//                          shared-expert gate sigmoid(g_s . x) (in a stack, the previous
//                          layer's combine writes these two instead); up to 16384
//                          tokens also the scan's tables (one extra CTA) and the first
//                          rows straight from the histograms.
#include "common.cuh"
#include "internal.h"

namespace moe {

__global__ void __launch_bounds__(RT_THREADS, 1)
    router_prefill_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_wr,
                          RouteParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + RT_STAGES * RT_STAGE_BYTES);  // full[4] empty[4] done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  int* hist_s = reinterpret_cast<int*>(tmem_slot + 4);
  float* bias_s = reinterpret_cast<float*>(hist_s + NEXP);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bias_s + NEXP);
  // top-8 lists of expert segments 1-3: values [seg-1][k][row], then expert ids
  float* cand_v = reinterpret_cast<float*>(smem + RT_STAGES * RT_STAGE_BYTES + 3072);
  int* cand_e = reinterpret_cast<int*>(cand_v + (RT_SEGS - 1) * TOPK * RT_BM);
  static_assert(RT_STAGES * RT_STAGE_BYTES + 3072 + RT_CAND_BYTES + 1024 <= RT_SMEM, "router shared memory");
  static_assert(NEXP == RT_SEGS * 64 && RT_THREADS == RT_SEGS * RT_BM, "one warp per (token quarter, segment)");

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m0 = blockIdx.x * RT_BM;
  const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[4]), done = smem_u32(&bars[8]);

  if (tid == 0) {
    for (int s = 0; s < RT_STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = tid; i < NEXP; i += RT_THREADS) {
    hist_s[i] = 0;
    bias_s[i] = p.router_bias ? p.router_bias[i] : 0.0f;
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_wait();   // x (and, in a stack, the workspace) come from the kernels before this one
  constexpr int NKB = HID / 64;
  int issued = 0;   // TMA producer: K steps whose loads it issued

  if (warp == 0 && lane == 0) {
    // ---- TMA producer
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_wr);
    for (int kb = 0; kb < NKB; ++kb) {
      const int s = kb % RT_STAGES;
      const uint32_t ph = (kb / RT_STAGES) & 1;
      if (!mbar_wait(empty0 + 8 * s, ph ^ 1, p.err, abort_flag, p.wait_ns)) break;
      uint8_t* st = smem + s * RT_STAGE_BYTES;
      mbar_arrive_expect_tx(full0 + 8 * s, RT_STAGE_BYTES);
      // the CTAs start at different K steps (7 is prime to the 32 steps), so that they do
      // not all read the same 32 KB of the router matrix from the same L2 slices at once
      const int kr = (kb + static_cast<int>(blockIdx.x) * 7) % NKB;
      tma_load_2d(smem_u32(st), &tm_x, full0 + 8 * s, kr * 64, m0);
      tma_load_2d(smem_u32(st + RT_A_BYTES), &tm_wr, full0 + 8 * s, kr * 64, 0);
      issued = kb + 1;
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer
    const uint32_t id_r = idesc_bf16(128, 256);
    for (int kb = 0; kb < NKB; ++kb) {
      const int s = kb % RT_STAGES;
      const uint32_t ph = (kb / RT_STAGES) & 1;
      if (!mbar_wait(full0 + 8 * s, ph, p.err, abort_flag, p.wait_ns)) break;
      tc_fence_after();
      const uint32_t a = smem_u32(smem + s * RT_STAGE_BYTES);
      const uint32_t b = a + RT_A_BYTES;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        umma_bf16(tmem, sdesc_sw128(a + kk * 32), sdesc_sw128(b + kk * 32), id_r, (kb | kk) != 0);
      umma_commit(empty0 + 8 * s);
    }
    umma_commit(done);   // also covers an early exit: all issued MMAs complete first
  }
  __syncwarp();

  // ---- epilogue: warp w reads TMEM lane quarter w % 4 (32 token rows) and the 64
  // expert columns of segment w / 4 and keeps its top 8; the segment-0 warps then take
  // the other segments' lists in segment order.  Insertion is strictly-greater and the
  // candidates of equal logit arrive in ascending expert order, so ties go to the lowest
  // index exactly as in one pass over all 256 experts.
  bool ok = mbar_wait(done, 0, p.err, abort_flag, p.wait_ns);
  ok = __syncthreads_and(ok && !*abort_flag) != 0;   // the merge reads every warp's list
  tc_fence_after();
  const int seg = warp >> 2, row = (warp & 3) * 32 + lane;
  const int t = m0 + row;
  float tv[TOPK];
  int ti[TOPK];
#pragma unroll
  for (int k = 0; k < TOPK; ++k) { tv[k] = -INFINITY; ti[k] = NEXP; }
  auto insert = [&](float v, int e) {
    if (v > tv[TOPK - 1]) {          // strictly greater: equal logits keep the lower index
      tv[TOPK - 1] = v;
      ti[TOPK - 1] = e;
#pragma unroll
      for (int k = TOPK - 1; k > 0; --k) {
        if (tv[k] > tv[k - 1]) {
          const float fv = tv[k]; tv[k] = tv[k - 1]; tv[k - 1] = fv;
          const int iv = ti[k]; ti[k] = ti[k - 1]; ti[k - 1] = iv;
        }
      }
    }
  };
  if (ok) {
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
      const int col = seg * 64 + c * 32;
      uint32_t r[32];
      tmem_ld32(lane_base + col, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) insert(__uint_as_float(r[j]) + bias_s[col + j], col + j);
    }
    if (seg > 0) {
#pragma unroll
      for (int k = 0; k < TOPK; ++k) {
        cand_v[((seg - 1) * TOPK + k) * RT_BM + row] = tv[k];
        cand_e[((seg - 1) * TOPK + k) * RT_BM + row] = ti[k];
      }
    }
  }
  __syncthreads();
  if (ok && seg == 0) {
#pragma unroll 1
    for (int sg = 0; sg < RT_SEGS - 1; ++sg)
#pragma unroll
      for (int k = 0; k < TOPK; ++k) insert(cand_v[(sg * TOPK + k) * RT_BM + row], cand_e[(sg * TOPK + k) * RT_BM + row]);
    if (t < p.T) {
      // fewer than 8 ordered logits (NaN input): record it and route to expert 0
      if (ti[TOPK - 1] >= NEXP) {
        atomicOr(p.err, ERRBIT_BOUNDS);
#pragma unroll
        for (int k = 0; k < TOPK; ++k)
          if (ti[k] >= NEXP) { ti[k] = k; tv[k] = tv[0]; }
      }
      float ex[TOPK], sum = 0.0f;
#pragma unroll
      for (int k = 0; k < TOPK; ++k) { ex[k] = expf(tv[k] - tv[0]); sum += ex[k]; }
      const float inv = 1.0f / sum;
#pragma unroll
      for (int k = 0; k < TOPK; ++k) {
        p.topk_idx[t * TOPK + k] = ti[k];
        p.topk_w[t * TOPK + k] = ex[k] * inv;
        atomicAdd(&hist_s[ti[k]], 1);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  for (int i = tid; i < NEXP; i += RT_THREADS) p.hist[blockIdx.x * NEXP + i] = hist_s[i];
  if (warp == 0 && lane == 0 && *abort_flag) {
    // a launch that gave up (whichever thread did): copies still in flight land before
    // the CTA's shared memory goes away (the latest phase of each stage)
    for (int kb = (issued > RT_STAGES ? issued - RT_STAGES : 0); kb < issued; ++kb) {
      const int s = kb % RT_STAGES;
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(full0 + 8 * s, (kb / RT_STAGES) & 1) && globaltimer_ns() - t0 < WAIT_LIMIT_NS) {
      }
    }
  }
  if (warp == 1) {
    tc_fence_after();
    if (lane == 0 && *abort_flag) {
      // MMAs issued before an abort finish before their columns are released
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(done, 0) && globaltimer_ns() - t0 < WAIT_LIMIT_NS) {
      }
    }
    __syncwarp();
    tmem_dealloc(tmem, 256);
  }
}

// router_cluster_kernel<S>: the same routing where one CTA per 128 tokens would leave
// SMs idle.  The contraction over the 2048 hidden columns is cut in S parts: a cluster of
// S CTAs per token block, CTA r accumulating part r of K for all 256 experts (MMA N = 256,
// 32/S K steps).  The partial logits move through distributed shared memory -- CTA r
// sends the rows of tokens (128/S) j.. to CTA j -- and CTA j adds the S partials in part
// order (a fixed order, so the result does not depend on timing), adds the bias and keeps
// the top 8 of each of its 128/S tokens as router_prefill_kernel does: four 64-expert
// segments with strictly-greater insertion over ascending experts, merged in segment
// order.  S = 4 up to RC_MAX_T tokens, S = 2 up to RC2_MAX_T (measured per-launch: T =
// 8192 25 us against 31 for router_prefill_kernel; at T = 16384, 3.4 waves of clusters,
// 48 against 35).  Rank 0
// clears the block's histogram row before the first cluster barrier; every CTA adds its
// tokens' counts after the second.  Every thread passes both cluster barriers on every
// path (a launch that gave up included), so no CTA waits for a peer that has left.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The address of the same shared-memory location in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(addr), "r"(rank));
  return d;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
// Every thread of every CTA of the cluster arrives; writes before it (shared::cluster and
// global) are visible to every thread of the cluster after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int S>
__global__ void __cluster_dims__(1, S, 1) __launch_bounds__(rc_threads(S), 1)
    router_cluster_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_wr,
                          RouteParams p) {
  constexpr int TPO = RT_BM / S;        // tokens whose top 8 this CTA selects
  constexpr int NTH = rc_threads(S);    // 4 segments x TPO tokens
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* misc = smem + RC_STAGES * RT_STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);                  // full[4] empty[4] done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 132);
  float* bias_s = reinterpret_cast<float*>(misc + 256);                // [256]
  int* hist_s = reinterpret_cast<int*>(misc + 256 + NEXP * 4);         // [256]
  float* cand_v = reinterpret_cast<float*>(misc + 256 + NEXP * 8);     // [4 segments][8][TPO tokens]
  int* cand_e = reinterpret_cast<int*>(cand_v + 4 * TOPK * TPO);
  // the S partials of this CTA's TPO tokens over the stage buffers once every MMA of the
  // cluster is done: float4 [part][expert / 4][token], so that a warp's 16-byte stores
  // into a peer, and its loads here, cover 512 contiguous bytes
  float4* recv = reinterpret_cast<float4*>(smem);
  static_assert(S * (NEXP / 4) * TPO * 16 <= RC_STAGES * RT_STAGE_BYTES, "partials fit the stage buffers");
  static_assert(rc_misc(S) + 1024 <= rc_smem(S) - RC_STAGES * RT_STAGE_BYTES, "router smem");
  static_assert((S == 2 || S == 4) && NEXP == 4 * 64 && TPO % 32 == 0, "whole warps per token group and segment");

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x, m0 = b * RT_BM;
  const uint32_t rank = cluster_ctarank();
  const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[RC_STAGES]), done = smem_u32(&bars[2 * RC_STAGES]);
  if (tid == 0) {
    for (int s = 0; s < RC_STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = tid; i < NEXP; i += NTH) {
    bias_s[i] = p.router_bias ? p.router_bias[i] : 0.0f;
    hist_s[i] = 0;
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_wait();   // x (and, in a stack, the workspace) come from the kernels before this one
  if (rank == 0)   // the other CTAs add to the block's histogram row after the cluster barriers
    for (int i = tid; i < NEXP; i += NTH) p.hist[b * NEXP + i] = 0;
  constexpr int NK = HID / 64 / S;   // K steps of this CTA's part
  const int kb0 = static_cast<int>(rank) * NK;
  int issued = 0;   // TMA producer: K steps whose loads it issued

  if (warp == 0 && lane == 0) {
    // ---- TMA producer: the block's x rows and all 256 router rows, K part `rank`
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_wr);
    for (int i = 0; i < NK; ++i) {
      const int s = i % RC_STAGES;
      if (!mbar_wait(empty0 + 8 * s, ((i / RC_STAGES) & 1) ^ 1, p.err, abort_flag, p.wait_ns)) break;
      uint8_t* st = smem + s * RT_STAGE_BYTES;
      mbar_arrive_expect_tx(full0 + 8 * s, RT_STAGE_BYTES);
      // the clusters start at different K steps of their part, so that the CTAs of one
      // part do not all read the same router rows from the same L2 slices at once
      const int kr = kb0 + (i + static_cast<int>(blockIdx.x)) % NK;
      tma_load_2d(smem_u32(st), &tm_x, full0 + 8 * s, kr * 64, m0);
      tma_load_2d(smem_u32(st + RT_A_BYTES), &tm_wr, full0 + 8 * s, kr * 64, 0);
      issued = i + 1;
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer
    const uint32_t id_r = idesc_bf16(128, 256);
    for (int i = 0; i < NK; ++i) {
      const int s = i % RC_STAGES;
      if (!mbar_wait(full0 + 8 * s, (i / RC_STAGES) & 1, p.err, abort_flag, p.wait_ns)) break;
      tc_fence_after();
      const uint32_t a = smem_u32(smem + s * RT_STAGE_BYTES);
      const uint32_t bb = a + RT_A_BYTES;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        umma_bf16(tmem, sdesc_sw128(a + kk * 32), sdesc_sw128(bb + kk * 32), id_r, (i | kk) != 0);
      umma_commit(empty0 + 8 * s);
    }
    umma_commit(done);   // also covers an early exit: all issued MMAs complete first
  }
  __syncwarp();
  bool ok = mbar_wait(done, 0, p.err, abort_flag, p.wait_ns);
  ok = __syncthreads_and(ok && !*abort_flag) != 0;
  if (!ok) {
    // a launch that gave up: copies and MMAs still in flight finish before the stage
    // buffers are handed to the peers (the latest phase of each stage; bounded waits)
    if (warp == 0 && lane == 0)
      for (int i = (issued > RC_STAGES ? issued - RC_STAGES : 0); i < issued; ++i) {
        const unsigned long long t0 = globaltimer_ns();
        while (!mbar_try_wait(full0 + 8 * (i % RC_STAGES), (i / RC_STAGES) & 1) &&
               globaltimer_ns() - t0 < WAIT_LIMIT_NS) {
        }
      }
    if (warp == 1 && lane == 0) {
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(done, 0) && globaltimer_ns() - t0 < WAIT_LIMIT_NS) {
      }
    }
    __syncwarp();
  }
  tc_fence_after();
  // ---- every CTA of the cluster is done with its stage buffers
  cluster_sync();
  if (ok && warp < 4) {
    // warp w holds TMEM lanes 32w..32w+31 = tokens 32w.. of the block, owned by CTA
    // 32w / TPO (local tokens 32w % TPO ..)
    const int tq = 32 * warp + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t dst = mapa_shared(smem_u32(recv + rank * (NEXP / 4) * TPO + tq % TPO), static_cast<uint32_t>(tq / TPO));
#pragma unroll 1
    for (int c = 0; c < NEXP / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(lane_base + c * 32, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 8; ++j)   // experts 32c + 4j .. + 3
        st_cluster_v4(dst + (c * 8 + j) * TPO * 16, r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
    }
  }
  tc_fence_before();
  // ---- every partial has arrived
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
  // ---- thread: expert segment tid / TPO, local token tid % TPO (token TPO rank + that)
  float tv[TOPK];
  int ti[TOPK];
#pragma unroll
  for (int k = 0; k < TOPK; ++k) { tv[k] = -INFINITY; ti[k] = NEXP; }
  auto insert = [&](float v, int e) {
    if (v > tv[TOPK - 1]) {          // strictly greater: equal logits keep the lower index
      tv[TOPK - 1] = v;
      ti[TOPK - 1] = e;
#pragma unroll
      for (int k = TOPK - 1; k > 0; --k) {
        if (tv[k] > tv[k - 1]) {
          const float fv = tv[k]; tv[k] = tv[k - 1]; tv[k - 1] = fv;
          const int iv = ti[k]; ti[k] = ti[k - 1]; ti[k - 1] = iv;
        }
      }
    }
  };
  const int lt = tid % TPO, seg = tid / TPO;
  const int t = m0 + static_cast<int>(rank) * TPO + lt;
  // eight experts per pass, all loads first: the four quarters summed in order, then the bias
#pragma unroll 1
  for (int e8 = 0; e8 < 64; e8 += 8) {
    const int e = seg * 64 + e8;
    float4 a[2][S];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int q = 0; q < S; ++q) a[h][q] = recv[(q * (NEXP / 4) + e / 4 + h) * TPO + lt];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float4 acc = a[h][0];
#pragma unroll
      for (int q = 1; q < S; ++q) {
        acc.x += a[h][q].x; acc.y += a[h][q].y; acc.z += a[h][q].z; acc.w += a[h][q].w;
      }
      const float4 bv = *reinterpret_cast<const float4*>(bias_s + e + 4 * h);
      insert(acc.x + bv.x, e + 4 * h);
      insert(acc.y + bv.y, e + 4 * h + 1);
      insert(acc.z + bv.z, e + 4 * h + 2);
      insert(acc.w + bv.w, e + 4 * h + 3);
    }
  }
#pragma unroll
  for (int k = 0; k < TOPK; ++k) {
    cand_v[(seg * TOPK + k) * TPO + lt] = tv[k];
    cand_e[(seg * TOPK + k) * TPO + lt] = ti[k];
  }
  __syncthreads();
  if (seg == 0 && t < p.T) {
    // the four segments' lists (each in descending order, equal logits by ascending
    // expert) merged: each step takes the largest head, the lowest segment on equal
    // values -- the order of one strictly-greater insertion pass over all 256 experts
    int p0 = 0, p1 = 0, p2 = 0, p3 = 0;
    float h0 = cand_v[(0 * TOPK) * TPO + lt], h1 = cand_v[(1 * TOPK) * TPO + lt];
    float h2 = cand_v[(2 * TOPK) * TPO + lt], h3 = cand_v[(3 * TOPK) * TPO + lt];
#pragma unroll
    for (int k = 0; k < TOPK; ++k) {
      int bs = 0;
      float bv = h0;
      if (h1 > bv) { bv = h1; bs = 1; }
      if (h2 > bv) { bv = h2; bs = 2; }
      if (h3 > bv) { bv = h3; bs = 3; }
      const int pk = bs == 0 ? p0 : bs == 1 ? p1 : bs == 2 ? p2 : p3;
      tv[k] = bv;
      ti[k] = cand_e[(bs * TOPK + pk) * TPO + lt];
      const int nx = pk + 1;
      const float hn = nx < TOPK ? cand_v[(bs * TOPK + nx) * TPO + lt] : -INFINITY;
      if (bs == 0) { p0 = nx; h0 = hn; } else if (bs == 1) { p1 = nx; h1 = hn; } else if (bs == 2) { p2 = nx; h2 = hn; } else { p3 = nx; h3 = hn; }
    }
    // fewer than 8 ordered logits (NaN input): record it and route to expert 0 ..
    if (ti[TOPK - 1] >= NEXP) {
      atomicOr(p.err, ERRBIT_BOUNDS);
#pragma unroll
      for (int k = 0; k < TOPK; ++k)
        if (ti[k] >= NEXP) { ti[k] = k; tv[k] = tv[0]; }
    }
    float ex[TOPK], sum = 0.0f;
#pragma unroll
    for (int k = 0; k < TOPK; ++k) { ex[k] = expf(tv[k] - tv[0]); sum += ex[k]; }
    const float inv = 1.0f / sum;
#pragma unroll
    for (int k = 0; k < TOPK; ++k) {
      p.topk_idx[t * TOPK + k] = ti[k];
      p.topk_w[t * TOPK + k] = ex[k] * inv;
      atomicAdd(&hist_s[ti[k]], 1);
    }
  }
  __syncthreads();
  for (int i = tid; i < NEXP; i += NTH)
    if (hist_s[i] != 0) atomicAdd(p.hist + b * NEXP + i, hist_s[i]);
}

// The routing tables from the router's per-block histograms, on Q * 256 threads: thread
// (q, e) = expert e's router blocks of part q (the per-expert sums and prefixes over the
// blocks run Q ways in parallel); the per-expert steps below run on the q = 0 threads,
// every thread reaching the barriers.  route_scan_kernel runs it on 1024 threads; a
// short prefill runs it on one extra CTA of the scatter (256 threads).
template <int SCAN_Q>
__device__ __forceinline__ void scan_tables(const ScanParams& p) {
  __shared__ int sc[NEXP];      // inclusive scan of the experts' row counts
  __shared__ int sf[NEXP];      // inclusive scan of their numbers of full blocks
  __shared__ int s_wtot[2][NEXP / 32];
  __shared__ int s_seg[SCAN_Q][NEXP];
  __shared__ int s_part[NEXP + 1];   // each expert's partial block (the shared expert last)
  const int e = threadIdx.x % NEXP, q = threadIdx.x / NEXP, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool lead = q == 0;
  const int per_q = (p.nblk + SCAN_Q - 1) / SCAN_Q;
  const int b_lo = q * per_q, b_hi = min(p.nblk, b_lo + per_q);
  constexpr int CH = 8;    // histogram entries loaded together (independent loads in flight)
  constexpr int HC = 32;   // from 33 to 128 router blocks (4096 < T <= 16384) a thread's
                           // quarter stays in registers: one round of loads, none in the
                           // second pass (at fewer blocks one round of CH loads is enough,
                           // and the unrolled 32 measured 2 us slower)
  const bool cached = per_q > CH && per_q <= HC;
  int hc[HC];
  int cq = 0;
  if (cached) {
#pragma unroll
    for (int i = 0; i < HC; ++i) hc[i] = (b_lo + i < b_hi) ? __ldg(p.hist + (b_lo + i) * NEXP + e) : 0;
#pragma unroll
    for (int i = 0; i < HC; ++i) cq += hc[i];
  } else {
    for (int b0 = b_lo; b0 < b_hi; b0 += CH) {
      int h[CH];
#pragma unroll
      for (int i = 0; i < CH; ++i) h[i] = (b0 + i < b_hi) ? __ldg(p.hist + (b0 + i) * NEXP + e) : 0;
#pragma unroll
      for (int i = 0; i < CH; ++i) cq += h[i];
    }
  }
  s_seg[q][e] = cq;
  __syncthreads();
  int c = 0, pre = 0;   // expert e's count; the count of its blocks before quarter q
#pragma unroll
  for (int j = 0; j < SCAN_Q; ++j) {
    pre += (j < q) ? s_seg[j][e] : 0;
    c += s_seg[j][e];
  }
  // block-wide inclusive scans of the counts and of the numbers of full blocks: warp
  // shuffles over 32 experts, then the 8 warp totals (the lead threads are warps 0-7)
  const int full = c / GX_BN, part = c % GX_BN;
  if (lead) {
    int ic = c, ifl = full;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, ic, o), f = __shfl_up_sync(0xffffffffu, ifl, o);
      if (lane >= o) {
        ic += a;
        ifl += f;
      }
    }
    if (lane == 31) {
      s_wtot[0][warp] = ic;
      s_wtot[1][warp] = ifl;
    }
    __syncwarp();
    sc[e] = ic;
    sf[e] = ifl;
    s_part[e] = part;
  }
  if (threadIdx.x == 0) s_part[NEXP] = p.T % GX_BN;
  __syncthreads();
  if (lead && warp > 0) {
    int ac = 0, af = 0;
    for (int w = 0; w < warp; ++w) {
      ac += s_wtot[0][w];
      af += s_wtot[1][w];
    }
    sc[e] += ac;
    sf[e] += af;
  }
  __syncthreads();
  const int excl = sc[e] - c;
  // first permuted row of (block, expert): the expert's offset plus earlier blocks' counts
  int run = excl + pre;
  if (cached) {
#pragma unroll
    for (int i = 0; i < HC; ++i) {
      if (b_lo + i < b_hi) p.base[(b_lo + i) * NEXP + e] = run;
      run += hc[i];
    }
  } else {
    for (int b0 = b_lo; b0 < b_hi; b0 += CH) {
      int h[CH];
#pragma unroll
      for (int i = 0; i < CH; ++i) h[i] = (b0 + i < b_hi) ? __ldg(p.hist + (b0 + i) * NEXP + e) : 0;
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        if (b0 + i < b_hi) p.base[(b0 + i) * NEXP + e] = run;
        run += h[i];
      }
    }
  }
  if (lead) {
    p.counts[e] = c;
    p.offsets[e] = excl;
  }
  // Token blocks of the grouped GEMMs (a block = up to 256 consecutive permuted rows of
  // one expert; every tile is a block x one row block of the weights): all full blocks
  // first (expert order, the shared expert last), then each expert's partial last block,
  // largest first (ties: lower expert first).  The GEMMs deal their tiles in this order,
  // so the smallest tiles are the last ones dealt and the CTAs' loads even out.  Entries
  // expert | (block index << 9) from blocks[2]; blocks[0] = their number, blocks[1] = the
  // number of blocks of more than GX_SMALL rows.
  const int full_routed = sf[NEXP - 1], full_sh = p.T / GX_BN;
  const int n_full = full_routed + full_sh;
  int* blk = p.blocks + 2;
  if (lead)
    for (int k = 0; k < full; ++k) blk[sf[e] - full + k] = e | (k << 9);
  for (int k = threadIdx.x; k < full_sh; k += blockDim.x) blk[full_routed + k] = NEXP | (k << 9);
  // rank of a partial block among all partial blocks (four independent counts in flight)
  auto prank = [&](int x) {
    const int px = s_part[x];
    int r[4] = {0, 0, 0, 0};
#pragma unroll 4
    for (int y = 0; y < NEXP; ++y) {
      const int py = s_part[y];
      r[y & 3] += (py > px) || (py == px && y < x);
    }
    return r[0] + r[1] + r[2] + r[3] + (s_part[NEXP] > px);   // the shared expert sorts last among equals
  };
  if (lead && part > 0) blk[n_full + prank(e)] = e | (full << 9);
  // the shared expert's partial block: thread 256 (a q = 1 thread), or thread 0 after its own
  if (threadIdx.x == (SCAN_Q > 1 ? NEXP : 0) && s_part[NEXP] > 0) blk[n_full + prank(NEXP)] = NEXP | (full_sh << 9);
  const int np = __syncthreads_count(lead && part > 0) + (s_part[NEXP] > 0);
  // the big blocks (more than GX_SMALL rows): every full block and the partial blocks
  // above GX_SMALL rows, which the order puts right after them
  const int np_big = __syncthreads_count(lead && part > GX_SMALL) + (s_part[NEXP] > GX_SMALL);
  if (threadIdx.x == 0) {
    p.counts[NEXP] = p.T;
    p.offsets[NEXP] = 8 * p.T;
    p.offsets[NEXP + 1] = 9 * p.T;
    p.blocks[0] = n_full + np;
    p.blocks[1] = n_full + np_big;
  }
}

constexpr int SCAN_Q = 4;
__global__ void __launch_bounds__(SCAN_Q * NEXP) route_scan_kernel(ScanParams p) {
  grid_dep_wait();   // the histograms come from the router
  scan_tables<SCAN_Q>(p);
}

// Expert e's (= this thread's) first permuted row in router block b, straight from the
// histograms: the exclusive scan of the experts' totals plus e's rows in the earlier
// blocks (the same integers route_scan_kernel writes to base).  Every thread of the CTA
// (256) calls it.
__device__ __forceinline__ int fused_base(const int* hist, int nblk, int b) {
  __shared__ int s_w[NEXP / 32];
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
  int tot = 0, pre = 0;
  for (int bb = 0; bb < nblk; ++bb) {
    const int h = __ldg(hist + bb * NEXP + e);
    tot += h;
    pre += bb < b ? h : 0;
  }
  int inc = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) s_w[warp] = inc;
  __syncthreads();
  int add = 0;
  for (int w = 0; w < warp; ++w) add += s_w[w];
  return add + inc - tot + pre;
}

__global__ void __launch_bounds__(SC_THREADS) route_scatter_kernel(ScatterParams p) {
  constexpr int SLOTS = RT_BM * TOPK;   // 1024 slots per router block
  __shared__ int wh[8][NEXP];
  const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  grid_dep_wait();   // the routing and the bases come from the kernels before this one
  if (p.fused && b == p.scan.nblk) {   // the extra CTA column of a short prefill: the scan's tables
    static_assert(SC_THREADS == NEXP, "the scan's tables on one thread per expert");
    if (blockIdx.y == 0) scan_tables<1>(p.scan);
    return;
  }
  const int slot0 = b * SLOTS;
  const int nslots = min(SLOTS, p.T * TOPK - slot0);
  const int n8 = 8 * p.T;
  if (blockIdx.y == 0) {
  // this thread's four slots (warp * 128 + j * 32 + lane, the order of pass 3), their
  // routing weights and its expert's block base: every global read up front
  int ev[4];
  float wv[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int sl = warp * 128 + j * 32 + lane;
    ev[j] = (sl < nslots) ? __ldg(p.topk_idx + slot0 + sl) : -1;
    wv[j] = (sl < nslots) ? __ldg(p.topk_w + slot0 + sl) : 0.0f;
  }
  const int base_e = p.fused ? fused_base(p.scan.hist, p.scan.nblk, b) : __ldg(p.base + b * NEXP + tid);
  for (int i = tid; i < 8 * NEXP; i += SC_THREADS) (&wh[0][0])[i] = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (ev[j] >= NEXP || ev[j] < -1) {   // never index shared memory with a bad expert id
      atomicOr(p.err, ERRBIT_BOUNDS);
      ev[j] = -1;
    }
  }
  __syncthreads();
  // pass 1: histogram of each warp's 128 consecutive slots
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (ev[j] >= 0) atomicAdd(&wh[warp][ev[j]], 1);
  __syncthreads();
  // pass 2: per expert, each warp's first global row (block base + earlier warps)
  {
    const int e = tid;
    int run = base_e;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const int c = wh[w][e];
      wh[w][e] = run;
      run += c;
    }
  }
  __syncthreads();
  // pass 3: stable ranks, slot order inside each warp's range
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int s = warp * 128 + j * 32 + lane;
    const int e = ev[j];
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    int pos = -1;
    if (e >= 0) pos = wh[warp][e] + rank;
    __syncwarp();
    if (e >= 0 && rank == 0) wh[warp][e] += __popc(peers);
    __syncwarp();
    if (e >= 0 && (pos < 0 || pos >= n8)) {
      atomicOr(p.err, ERRBIT_BOUNDS);
      pos = -1;
    }
    if (pos >= 0) {
      p.row_dst[pos] = slot0 + s;
      p.row_w[pos] = wv[j];
    }
    if (s < nslots) p.slot_row[slot0 + s] = pos;   // -1 for a slot that failed validation
  }
  }   // blockIdx.y == 0
  if (!p.gather) return;
  // one warp per token: one read of x, one K-interleaved copy (the gate/up GEMM gathers
  // its rows from it by token), and the shared-expert gate on the same read
  constexpr int TPC = RT_BM / SC_SPLIT;   // tokens of this CTA
  const int t0 = b * RT_BM + blockIdx.y * TPC;
  const uint4* gsv = reinterpret_cast<const uint4*>(p.shared_gate_w);
  // the shared-gate vector is the same for every token: read once per warp; a token's
  // eight x chunks are all requested before any is used
  uint4 gw[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) gw[c] = ldg_nc_v4(gsv + lane + 32 * c);
#pragma unroll 1
  for (int tl = warp; tl < TPC; tl += SC_THREADS / 32) {
    const int t = t0 + tl;
    if (t >= p.T) break;
    const uint4* src = reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(t) * HID);
    uint4 cur[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) cur[c] = ldg_nc_v4(src + lane + 32 * c);
    uint4* dst = reinterpret_cast<uint4*>(p.x_ilv + static_cast<size_t>(t) * HID);
    // the summation order of row_dot (chunk lane + 32c is "thread" lane of "warp" c), so
    // the combine, which computes this dot for the next stacked layer, gets the same bits
    float dot = 0.0f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 raw = cur[c];
      const uint4 g = gw[c];
      float d = 0.0f;
      d = fmaf(bf16lo(raw.x), bf16lo(g.x), d);
      d = fmaf(bf16hi(raw.x), bf16hi(g.x), d);
      d = fmaf(bf16lo(raw.y), bf16lo(g.y), d);
      d = fmaf(bf16hi(raw.y), bf16hi(g.y), d);
      d = fmaf(bf16lo(raw.z), bf16lo(g.z), d);
      d = fmaf(bf16hi(raw.z), bf16hi(g.z), d);
      d = fmaf(bf16lo(raw.w), bf16lo(g.w), d);
      d = fmaf(bf16hi(raw.w), bf16hi(g.w), d);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
      dot += d;
      dst[lane + 32 * c] = interleave8(raw);
    }
    if (lane == 0) {
      const int srow = n8 + t;
      p.row_dst[srow] = srow;
      p.row_w[srow] = 1.0f / (1.0f + expf(-dot));
    }
  }
}

// Input RMSNorm of a stacked layer: xn = bf16(x / sqrt(mean(x^2) + 1e-6) * w), one CTA
// of 256 threads per token row (the fixed summation order of row_inv_rms, which the
// combine uses when it normalises the next layer's input itself).
__global__ void __launch_bounds__(256) rmsnorm_kernel(const __nv_bfloat16* __restrict__ x,
                                                      const __nv_bfloat16* __restrict__ w,
                                                      __nv_bfloat16* __restrict__ xn, int T) {
  __shared__ float s_warp[8];
  const int row = blockIdx.x, c = threadIdx.x;
  grid_dep_wait();   // x may come from the kernel before this one
  const uint4 v = ldg_nc_v4(x + static_cast<size_t>(row) * HID + c * 8);
  const float r = row_inv_rms(v, s_warp);
  *reinterpret_cast<uint4*>(xn + static_cast<size_t>(row) * HID + c * 8) = rms_scale8(v, ldg_nc_v4(w + c * 8), r);
}

cudaError_t launch_rmsnorm(const __nv_bfloat16* x, const __nv_bfloat16* w, __nv_bfloat16* xn, int T,
                           cudaStream_t s) {
  return launch_pdl(rmsnorm_kernel, T, 256, 0, s, x, w, xn, T);
}

cudaError_t launch_router_prefill(const CUtensorMap& tm_x, const CUtensorMap& tm_wr, const RouteParams& p,
                                  cudaStream_t s) {
  const int nblk = (p.T + RT_BM - 1) / RT_BM;
  return launch_pdl(router_prefill_kernel, nblk, RT_THREADS, RT_SMEM, s, tm_x, tm_wr, p);
}

cudaError_t launch_router_cluster(const CUtensorMap& tm_x, const CUtensorMap& tm_wr, const RouteParams& p,
                                  cudaStream_t s) {
  const int nblk = (p.T + RT_BM - 1) / RT_BM;
  if (p.T <= RC_MAX_T)
    return launch_pdl(router_cluster_kernel<4>, dim3(nblk, 4), rc_threads(4), rc_smem(4), s, tm_x, tm_wr, p);
  return launch_pdl(router_cluster_kernel<2>, dim3(nblk, 2), rc_threads(2), rc_smem(2), s, tm_x, tm_wr, p);
}

cudaError_t launch_scan(const ScanParams& p, cudaStream_t s) {
  return launch_pdl(route_scan_kernel, 1, SCAN_Q * NEXP, 0, s, p);
}

cudaError_t launch_scatter(const ScatterParams& p, int nblk, cudaStream_t s) {
  return launch_pdl(route_scatter_kernel, dim3(nblk, p.gather ? SC_SPLIT : 1), SC_THREADS, 0, s, p);
}

cudaError_t set_router_attributes() {
  cudaError_t e = cudaFuncSetAttribute(router_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, RT_SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(router_cluster_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, rc_smem(4));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(router_cluster_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, rc_smem(2));
  return e;
}

}  // namespace moe
