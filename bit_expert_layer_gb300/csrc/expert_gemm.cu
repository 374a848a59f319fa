// expert_gemm.cu -- the grouped expert GEMMs of the prefill path, with the 4-bit
// dequantisation fused into the GEMM: packed weights go from HBM to shared memory by
// TMA, dequant warps expand them to bf16 tiles in shared memory, and tcgen05 MMAs
// accumulate into TMEM; the dequantised weights never touch device memory (Lily fuses
// the 4-bit restore into its grouped GEMM and keeps the result in on-chip memory:
// aimanavo.com, "Why is Perplexity's local AI Lily faster than MLX", section "Prefill
// and decode are not treated as the same job"; dzen.guru, "Perplexity opened the Lily
// engine", section "Where the speed-up comes from").
//
// Orientation: weight rows are the MMA's M side (128 per tile), tokens its N side (up
// to 256 per tile, rounded up to 16), K steps of 64 = one quantisation group, so each
// dequantised row needs exactly one scale and one bias per K step.
//
//   gateup_kernel  h = silu(W_gate x) * (W_up x) for every (expert, token) pair of the
//                  permuted activations; the shared expert is expert 256 over all T
//                  tokens.  Two TMEM accumulators (gate, up), SwiGLU in the epilogue.
//   down_kernel    y[row_dst] = row_w * (W_down h): each routed row is scaled by its
//                  renormalised routing weight, each shared row by sigmoid(g_s . x).
//                  Double-buffered TMEM accumulator so the epilogue overlaps the next
//                  tile's MMAs.
//   combine_kernel out[t] = sum_k y[8t+k] + y[8T+t] (+ x[t]) in a fixed order.
//
// Persistent kernels: grid = number of SMs, tiles taken in a static stride from the
// device-side tile tables built by route_scan_kernel (no host readback).
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

// gate/up stage layout
constexpr int GU_AG = 0;
constexpr int GU_AU = GX_A_BYTES;
constexpr int GU_X = 2 * GX_A_BYTES;
constexpr int GU_PG = GU_X + GX_X_BYTES;
constexpr int GU_PU = GU_PG + GX_P_BYTES;
// down stage layout
constexpr int DN_A = 0;
constexpr int DN_X = GX_A_BYTES;
constexpr int DN_P = GX_A_BYTES + GX_X_BYTES;

struct TileInfo {
  int e, mb, row0, n_rows;
  bool ok;   // tables consistent: every role skips a bad tile the same way
};

__device__ __forceinline__ TileInfo tile_info(const int* tiles, const int* offsets, const int* counts, int tile,
                                              int mblk, int T) {
  int lo = 0, hi = NEXP;   // largest e in [0, 256] with tiles[e] <= tile
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(tiles + mid) <= tile) lo = mid;
    else hi = mid - 1;
  }
  TileInfo ti;
  ti.e = lo;
  const int local = tile - __ldg(tiles + lo);
  const int nb = local / mblk;
  ti.mb = local - nb * mblk;
  ti.row0 = __ldg(offsets + lo) + nb * GX_BN;
  ti.n_rows = min(GX_BN, __ldg(counts + lo) - nb * GX_BN);
  ti.ok = ti.n_rows >= 1 && ti.row0 >= 0 && ti.row0 + ti.n_rows <= 9 * T && local >= 0;
  return ti;
}

__device__ __forceinline__ __nv_bfloat162 bf2(uint32_t bits16) {
  const uint32_t v = (bits16 & 0xFFFFu) * 0x00010001u;
  return *reinterpret_cast<const __nv_bfloat162*>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint8_t* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

// Bounded wait used only while tearing down after an abort (ignores the abort flag).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity) && globaltimer_ns() - t0 < WAIT_LIMIT_NS) {
  }
}

}  // namespace

// ============================================================================ gate/up
__global__ void __launch_bounds__(GU_THREADS, 1)
    gateup_kernel(const __grid_constant__ CUtensorMap tm_qg, const __grid_constant__ CUtensorMap tm_qu,
                  const __grid_constant__ CUtensorMap tm_sqg, const __grid_constant__ CUtensorMap tm_squ,
                  const __grid_constant__ CUtensorMap tm_x, GateUpParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + GU_STAGES * GU_STAGE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t bar0 = smem_u32(bars);
  // full[s] = 0..2, afull[s] = 3..5, empty[s] = 6..8, accf 9, acce 10, drain 11
#define FULL(s) (bar0 + 8u * (s))
#define AFULL(s) (bar0 + 8u * (3 + (s)))
#define EMPTY(s) (bar0 + 8u * (6 + (s)))
  const uint32_t ACCF = bar0 + 72, ACCE = bar0 + 80, DRAIN = bar0 + 88;

  if (tid == 0) {
    for (int s = 0; s < GU_STAGES; ++s) {
      mbar_init(FULL(s), 1);
      mbar_init(AFULL(s), 256);
      mbar_init(EMPTY(s), 1);
    }
    mbar_init(ACCF, 1);
    mbar_init(ACCE, 256);
    mbar_init(DRAIN, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = __ldg(p.tiles + NEXP + 1);
  constexpr int NKB = HID / 64;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      tma_prefetch_desc(&tm_qg);
      tma_prefetch_desc(&tm_qu);
      tma_prefetch_desc(&tm_x);
      uint32_t it = 0;
      bool alive = true;
      for (int tile = blockIdx.x; tile < total && alive; tile += gridDim.x) {
        const TileInfo ti = tile_info(p.tiles, p.offsets, p.counts, tile, GU_MBLK, p.T);
        if (!ti.ok) { if (threadIdx.x == 0) atomicOr(p.err, ERRBIT_BOUNDS); continue; }
        const bool sh = ti.e == SHARED_E;
        const CUtensorMap* mg = sh ? &tm_sqg : &tm_qg;
        const CUtensorMap* mu = sh ? &tm_squ : &tm_qu;
        const int wrow = (sh ? 0 : ti.e * INTER) + ti.mb * GX_BM;
        const int nbox = (ti.n_rows + GX_XBOX - 1) / GX_XBOX;
        const uint32_t bytes = 2 * GX_P_BYTES + nbox * GX_XBOX * 128;
        for (int kb = 0; kb < NKB; ++kb, ++it) {
          const int s = it % GU_STAGES;
          const uint32_t ph = (it / GU_STAGES) & 1;
          if (!mbar_wait(EMPTY(s), ph ^ 1, p.err, abort_flag)) { alive = false; break; }
          const uint32_t st = smem_u32(smem + s * GU_STAGE_BYTES);
          mbar_arrive_expect_tx(FULL(s), bytes);
          tma_load_2d(st + GU_PG, mg, FULL(s), kb * 8, wrow);
          tma_load_2d(st + GU_PU, mu, FULL(s), kb * 8, wrow);
          for (int j = 0; j < nbox; ++j)
            tma_load_2d(st + GU_X + j * GX_XBOX * 128, &tm_x, FULL(s), kb * 64, ti.row0 + j * GX_XBOX);
        }
      }
      if (!alive) {
        for (uint32_t i = (it > GU_STAGES ? it - GU_STAGES : 0); i < it; ++i)
          drain_wait(FULL(i % GU_STAGES), (i / GU_STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      uint32_t it = 0, tc = 0;
      for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        const TileInfo ti = tile_info(p.tiles, p.offsets, p.counts, tile, GU_MBLK, p.T);
        if (!ti.ok) { if (threadIdx.x == 0) atomicOr(p.err, ERRBIT_BOUNDS); continue; }
        const int N = max(16, (ti.n_rows + 15) & ~15);
        const uint32_t idesc = idesc_bf16(128, N);
        if (!mbar_wait(ACCE, (tc & 1) ^ 1, p.err, abort_flag)) break;
        tc_fence_after();
        bool alive = true;
        for (int kb = 0; kb < NKB; ++kb, ++it) {
          const int s = it % GU_STAGES;
          const uint32_t ph = (it / GU_STAGES) & 1;
          if (!mbar_wait(AFULL(s), ph, p.err, abort_flag) || !mbar_wait(FULL(s), ph, p.err, abort_flag)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + s * GU_STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = sdesc_sw128(st + GU_X + kk * 32);
            const uint32_t acc = (kb | kk) != 0;
            umma_bf16(tmem, sdesc_sw128(st + GU_AG + kk * 32), bd, idesc, acc);
            umma_bf16(tmem + 256, sdesc_sw128(st + GU_AU + kk * 32), bd, idesc, acc);
          }
          umma_commit(EMPTY(s));
        }
        if (!alive) break;
        umma_commit(ACCF);
        ++tc;
      }
      umma_commit(DRAIN);
    }
  } else {
    // ------------------------------------------------ dequant (8 warps) + epilogue
    const int dt = tid - 64;           // 0..255
    const int mat = dt >> 7;           // 0: gate rows, 1: up rows
    const int r = dt & 127;            // row inside the tile
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;  // which half of the token columns this warp drains
    uint32_t it = 0, tc = 0;
    bool alive = true;
    for (int tile = blockIdx.x; tile < total && alive; tile += gridDim.x) {
      const TileInfo ti = tile_info(p.tiles, p.offsets, p.counts, tile, GU_MBLK, p.T);
        if (!ti.ok) { if (threadIdx.x == 0) atomicOr(p.err, ERRBIT_BOUNDS); continue; }
      const bool sh = ti.e == SHARED_E;
      const size_t srow = sh ? static_cast<size_t>(ti.mb * GX_BM + r)
                             : static_cast<size_t>(ti.e) * INTER + ti.mb * GX_BM + r;
      const uint16_t* sc = (mat == 0 ? (sh ? p.sg_scales : p.g_scales) : (sh ? p.su_scales : p.u_scales)) +
                           srow * (HID / GROUP);
      const uint16_t* bi = (mat == 0 ? (sh ? p.sg_biases : p.g_biases) : (sh ? p.su_biases : p.u_biases)) +
                           srow * (HID / GROUP);
      const int p_off = mat ? GU_PU : GU_PG;
      const int a_off = mat ? GU_AU : GU_AG;
      for (int kc = 0; kc < NKB / 8 && alive; ++kc) {
        const uint4 sv = ldg_nc_v4(sc + kc * 8);
        const uint4 bv = ldg_nc_v4(bi + kc * 8);
        const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
        const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int s = it % GU_STAGES;
          const uint32_t ph = (it / GU_STAGES) & 1;
          if (!mbar_wait(FULL(s), ph, p.err, abort_flag)) { alive = false; break; }
          ++it;
          const __nv_bfloat162 ms = bf2((j & 1) ? (sw[j >> 1] >> 16) : sw[j >> 1]);
          const __nv_bfloat162 mbv = bf2((j & 1) ? (bw[j >> 1] >> 16) : bw[j >> 1]);
          uint8_t* st = smem + s * GU_STAGE_BYTES;
          const uint4* P = reinterpret_cast<const uint4*>(st + p_off + r * 32);
          const uint4 w0 = P[0], w1 = P[1];
          uint8_t* A = st + a_off;
          st_shared_v4(A + sw128_off(r, 0), dequant8(w0.x, ms, mbv));
          st_shared_v4(A + sw128_off(r, 1), dequant8(w0.y, ms, mbv));
          st_shared_v4(A + sw128_off(r, 2), dequant8(w0.z, ms, mbv));
          st_shared_v4(A + sw128_off(r, 3), dequant8(w0.w, ms, mbv));
          st_shared_v4(A + sw128_off(r, 4), dequant8(w1.x, ms, mbv));
          st_shared_v4(A + sw128_off(r, 5), dequant8(w1.y, ms, mbv));
          st_shared_v4(A + sw128_off(r, 6), dequant8(w1.z, ms, mbv));
          st_shared_v4(A + sw128_off(r, 7), dequant8(w1.w, ms, mbv));
          fence_proxy_async_smem();
          mbar_arrive(AFULL(s));
        }
      }
      if (!alive) break;
      // ---- epilogue: SwiGLU of this warp's quarter of rows and half of the columns
      bool ok = mbar_wait(ACCF, tc & 1, p.err, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) { alive = false; break; }
      tc_fence_after();
      const int f = ti.mb * GX_BM + q * 32 + lane;   // intermediate feature of this lane
      const int hcol = ilv_pos(f);
      const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        const int col0 = half * 128 + cc * 32;
        if (col0 >= ti.n_rows) break;
        uint32_t g[32], u[32];
        tmem_ld32(tl + col0, g);
        tmem_ld32(tl + 256 + col0, u);
        tmem_ld_wait();
        __nv_bfloat16* hp = p.h + static_cast<size_t>(ti.row0 + col0) * INTER + hcol;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (col0 + j < ti.n_rows) {
            const float gv = __uint_as_float(g[j]), uv = __uint_as_float(u[j]);
            const float hv = gv / (1.0f + __expf(-gv)) * uv;
            hp[static_cast<size_t>(j) * INTER] = __float2bfloat16_rn(hv);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(ACCE);
      ++tc;
    }
  }

  // ------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if (lane == 0) drain_wait(DRAIN, 0);
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
#undef FULL
#undef AFULL
#undef EMPTY
}

// ============================================================================ down
__global__ void __launch_bounds__(DN_THREADS, 1)
    down_kernel(const __grid_constant__ CUtensorMap tm_qd, const __grid_constant__ CUtensorMap tm_sqd,
                const __grid_constant__ CUtensorMap tm_h, DownParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + DN_STAGES * DN_STAGE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 24);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t bar0 = smem_u32(bars);
  // full 0..3, afull 4..7, empty 8..11, accf 12..13, acce 14..15, drain 16
#define FULL(s) (bar0 + 8u * (s))
#define AFULL(s) (bar0 + 8u * (4 + (s)))
#define EMPTY(s) (bar0 + 8u * (8 + (s)))
#define ACCF(b) (bar0 + 8u * (12 + (b)))
#define ACCE(b) (bar0 + 8u * (14 + (b)))
  const uint32_t DRAIN = bar0 + 8u * 16;

  if (tid == 0) {
    for (int s = 0; s < DN_STAGES; ++s) {
      mbar_init(FULL(s), 1);
      mbar_init(AFULL(s), 128);
      mbar_init(EMPTY(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(ACCF(b), 1);
      mbar_init(ACCE(b), 128);
    }
    mbar_init(DRAIN, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = __ldg(p.tiles + NEXP + 1);
  constexpr int NKB = INTER / 64;   // 8

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_qd);
      tma_prefetch_desc(&tm_h);
      uint32_t it = 0;
      bool alive = true;
      for (int tile = blockIdx.x; tile < total && alive; tile += gridDim.x) {
        const TileInfo ti = tile_info(p.tiles, p.offsets, p.counts, tile, DN_MBLK, p.T);
        if (!ti.ok) { if (threadIdx.x == 0) atomicOr(p.err, ERRBIT_BOUNDS); continue; }
        const bool sh = ti.e == SHARED_E;
        const CUtensorMap* mq = sh ? &tm_sqd : &tm_qd;
        const int wrow = (sh ? 0 : ti.e * HID) + ti.mb * GX_BM;
        const int nbox = (ti.n_rows + GX_XBOX - 1) / GX_XBOX;
        const uint32_t bytes = GX_P_BYTES + nbox * GX_XBOX * 128;
        for (int kb = 0; kb < NKB; ++kb, ++it) {
          const int s = it % DN_STAGES;
          const uint32_t ph = (it / DN_STAGES) & 1;
          if (!mbar_wait(EMPTY(s), ph ^ 1, p.err, abort_flag)) { alive = false; break; }
          const uint32_t st = smem_u32(smem + s * DN_STAGE_BYTES);
          mbar_arrive_expect_tx(FULL(s), bytes);
          tma_load_2d(st + DN_P, mq, FULL(s), kb * 8, wrow);
          for (int j = 0; j < nbox; ++j)
            tma_load_2d(st + DN_X + j * GX_XBOX * 128, &tm_h, FULL(s), kb * 64, ti.row0 + j * GX_XBOX);
        }
      }
      if (!alive) {
        for (uint32_t i = (it > DN_STAGES ? it - DN_STAGES : 0); i < it; ++i)
          drain_wait(FULL(i % DN_STAGES), (i / DN_STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t it = 0, tc = 0;
      for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        const TileInfo ti = tile_info(p.tiles, p.offsets, p.counts, tile, DN_MBLK, p.T);
        if (!ti.ok) { if (threadIdx.x == 0) atomicOr(p.err, ERRBIT_BOUNDS); continue; }
        const int N = max(16, (ti.n_rows + 15) & ~15);
        const uint32_t idesc = idesc_bf16(128, N);
        const int buf = tc & 1;
        if (!mbar_wait(ACCE(buf), ((tc >> 1) & 1) ^ 1, p.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * 256;
        bool alive = true;
        for (int kb = 0; kb < NKB; ++kb, ++it) {
          const int s = it % DN_STAGES;
          const uint32_t ph = (it / DN_STAGES) & 1;
          if (!mbar_wait(AFULL(s), ph, p.err, abort_flag) || !mbar_wait(FULL(s), ph, p.err, abort_flag)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + s * DN_STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(d, sdesc_sw128(st + DN_A + kk * 32), sdesc_sw128(st + DN_X + kk * 32), idesc,
                      (kb | kk) != 0);
          umma_commit(EMPTY(s));
        }
        if (!alive) break;
        umma_commit(ACCF(buf));
        ++tc;
      }
      umma_commit(DRAIN);
    }
  } else if (warp < 6) {
    // ------------------------------------------------ dequant (4 warps, one row each)
    const int r = tid - 64;   // 0..127
    uint32_t it = 0;
    bool alive = true;
    for (int tile = blockIdx.x; tile < total && alive; tile += gridDim.x) {
      const TileInfo ti = tile_info(p.tiles, p.offsets, p.counts, tile, DN_MBLK, p.T);
        if (!ti.ok) { if (threadIdx.x == 0) atomicOr(p.err, ERRBIT_BOUNDS); continue; }
      const bool sh = ti.e == SHARED_E;
      const size_t srow = sh ? static_cast<size_t>(ti.mb * GX_BM + r)
                             : static_cast<size_t>(ti.e) * HID + ti.mb * GX_BM + r;
      const uint4 sv = ldg_nc_v4((sh ? p.sd_scales : p.d_scales) + srow * (INTER / GROUP));
      const uint4 bv = ldg_nc_v4((sh ? p.sd_biases : p.d_biases) + srow * (INTER / GROUP));
      const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
      const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int kb = 0; kb < NKB; ++kb) {
        const int s = it % DN_STAGES;
        const uint32_t ph = (it / DN_STAGES) & 1;
        if (!mbar_wait(FULL(s), ph, p.err, abort_flag)) { alive = false; break; }
        ++it;
        const __nv_bfloat162 ms = bf2((kb & 1) ? (sw[kb >> 1] >> 16) : sw[kb >> 1]);
        const __nv_bfloat162 mbv = bf2((kb & 1) ? (bw[kb >> 1] >> 16) : bw[kb >> 1]);
        uint8_t* st = smem + s * DN_STAGE_BYTES;
        const uint4* P = reinterpret_cast<const uint4*>(st + DN_P + r * 32);
        const uint4 w0 = P[0], w1 = P[1];
        uint8_t* A = st + DN_A;
        st_shared_v4(A + sw128_off(r, 0), dequant8(w0.x, ms, mbv));
        st_shared_v4(A + sw128_off(r, 1), dequant8(w0.y, ms, mbv));
        st_shared_v4(A + sw128_off(r, 2), dequant8(w0.z, ms, mbv));
        st_shared_v4(A + sw128_off(r, 3), dequant8(w0.w, ms, mbv));
        st_shared_v4(A + sw128_off(r, 4), dequant8(w1.x, ms, mbv));
        st_shared_v4(A + sw128_off(r, 5), dequant8(w1.y, ms, mbv));
        st_shared_v4(A + sw128_off(r, 6), dequant8(w1.z, ms, mbv));
        st_shared_v4(A + sw128_off(r, 7), dequant8(w1.w, ms, mbv));
        fence_proxy_async_smem();
        mbar_arrive(AFULL(s));
      }
    }
  } else {
    // ------------------------------------------------ epilogue (4 warps)
    const int q = warp & 3;
    const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const int nrows_all = 9 * p.T;
    uint32_t tc = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const TileInfo ti = tile_info(p.tiles, p.offsets, p.counts, tile, DN_MBLK, p.T);
        if (!ti.ok) { if (threadIdx.x == 0) atomicOr(p.err, ERRBIT_BOUNDS); continue; }
      const int buf = tc & 1;
      bool ok = mbar_wait(ACCF(buf), (tc >> 1) & 1, p.err, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int f = ti.mb * GX_BM + q * 32 + lane;   // output feature of this lane
#pragma unroll 1
      for (int cc = 0; cc < GX_BN / 32; ++cc) {
        const int col0 = cc * 32;
        if (col0 >= ti.n_rows) break;
        uint32_t d[32];
        tmem_ld32(tl + buf * 256 + col0, d);
        const bool valid = col0 + lane < ti.n_rows;
        int dst = valid ? __ldg(p.row_dst + ti.row0 + col0 + lane) : -1;
        const float wt = valid ? __ldg(p.row_w + ti.row0 + col0 + lane) : 0.0f;
        if (valid && (dst < 0 || dst >= nrows_all)) {
          atomicOr(p.err, ERRBIT_BOUNDS);
          dst = -1;
        }
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int dj = __shfl_sync(0xffffffffu, dst, j);
          const float wj = __shfl_sync(0xffffffffu, wt, j);
          if (dj >= 0)
            p.y[static_cast<size_t>(dj) * HID + f] = __float2bfloat16_rn(wj * __uint_as_float(d[j]));
        }
      }
      tc_fence_before();
      mbar_arrive(ACCE(buf));
      ++tc;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if (lane == 0) drain_wait(DRAIN, 0);
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
#undef FULL
#undef AFULL
#undef EMPTY
#undef ACCF
#undef ACCE
}

// ============================================================================ combine
// One CTA per token, 256 threads x 8 features; fixed summation order: the 8 routed
// slots in rank order, then the shared expert, then the residual.
__global__ void __launch_bounds__(256) combine_kernel(const __nv_bfloat16* __restrict__ y,
                                                      const __nv_bfloat16* x, __nv_bfloat16* out, int T,
                                                      int residual) {
  const int t = blockIdx.x, c = threadIdx.x;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
  for (int k = 0; k <= TOPK; ++k) {
    const size_t row = (k < TOPK) ? static_cast<size_t>(t) * TOPK + k : static_cast<size_t>(8 * T + t);
    const uint4 v = ldg_nc_v4(y + row * HID + c * 8);
    acc[0] += bf16lo(v.x); acc[1] += bf16hi(v.x);
    acc[2] += bf16lo(v.y); acc[3] += bf16hi(v.y);
    acc[4] += bf16lo(v.z); acc[5] += bf16hi(v.z);
    acc[6] += bf16lo(v.w); acc[7] += bf16hi(v.w);
  }
  const size_t o = static_cast<size_t>(t) * HID + c * 8;
  if (residual) {
    const uint4 v = *reinterpret_cast<const uint4*>(x + o);
    acc[0] += bf16lo(v.x); acc[1] += bf16hi(v.x);
    acc[2] += bf16lo(v.y); acc[3] += bf16hi(v.y);
    acc[4] += bf16lo(v.z); acc[5] += bf16hi(v.z);
    acc[6] += bf16lo(v.w); acc[7] += bf16hi(v.w);
  }
  uint4 r;
  uint32_t* rp = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    rp[i] = *reinterpret_cast<const uint32_t*>(&b2);
  }
  *reinterpret_cast<uint4*>(out + o) = r;
}

cudaError_t launch_gateup(const CUtensorMap& qg, const CUtensorMap& qu, const CUtensorMap& sqg,
                          const CUtensorMap& squ, const CUtensorMap& xperm, const GateUpParams& p, int grid,
                          cudaStream_t s) {
  gateup_kernel<<<grid, GU_THREADS, GU_SMEM, s>>>(qg, qu, sqg, squ, xperm, p);
  return cudaGetLastError();
}

cudaError_t launch_down(const CUtensorMap& qd, const CUtensorMap& sqd, const CUtensorMap& hmap,
                        const DownParams& p, int grid, cudaStream_t s) {
  down_kernel<<<grid, DN_THREADS, DN_SMEM, s>>>(qd, sqd, hmap, p);
  return cudaGetLastError();
}

cudaError_t launch_combine(const __nv_bfloat16* y, const __nv_bfloat16* x, __nv_bfloat16* out, int T,
                           int residual, cudaStream_t s) {
  combine_kernel<<<T, 256, 0, s>>>(y, x, out, T, residual);
  return cudaGetLastError();
}

cudaError_t set_gemm_attributes() {
  cudaError_t e = cudaFuncSetAttribute(gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GU_SMEM);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, DN_SMEM);
}

}  // namespace moe
