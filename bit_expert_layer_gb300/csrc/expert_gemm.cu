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
#include "gemm_common.cuh"
#include "internal.h"

namespace moe {

namespace {

// gate/up stage layout
constexpr int GU_AG = 0;
constexpr int GU_AU = GX_A_BYTES;
constexpr int GU_X = 2 * GX_A_BYTES;
constexpr int GU_PG = GU_X + GX_X_BYTES;
constexpr int GU_PU = GU_PG + GX_P_BYTES;

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
  int* s_tiles = reinterpret_cast<int*>(bars + 32);
  int* s_off = s_tiles + (NEXP + 2);
  int* s_cnt = s_off + (NEXP + 2);
  stage_tables(s_tiles, p.tiles, p.offsets, p.counts);

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
    mbar_init(ACCE, 128);
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
  const int total = s_tiles[NEXP + 1];
  constexpr int NKB = HID / 64;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      const bool pp = p.pipe != nullptr;
      unsigned long long pc[1] = {0};
      const unsigned long long t_role = pp ? clock64() : 0;
      tma_prefetch_desc(&tm_qg);
      tma_prefetch_desc(&tm_qu);
      tma_prefetch_desc(&tm_x);
      uint32_t it = 0;
      bool alive = true;
      for (int tile = blockIdx.x; tile < total && alive; tile += gridDim.x) {
        const TileInfo ti = tile_info(s_tiles, s_off, s_cnt, tile, GU_MBLK, p.T);
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
          if (!mbar_wait_t(EMPTY(s), ph ^ 1, p.err, abort_flag, pc[0], pp)) { alive = false; break; }
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
      if (pp) pipe_flush(p.pipe, 4, pc, 1, clock64() - t_role, 5);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      const bool pp = p.pipe != nullptr;
      unsigned long long pc[3] = {0, 0, 0};
      const unsigned long long t_role = pp ? clock64() : 0;
      uint32_t it = 0, tc = 0;
      for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        const TileInfo ti = tile_info(s_tiles, s_off, s_cnt, tile, GU_MBLK, p.T);
        if (!ti.ok) { if (threadIdx.x == 0) atomicOr(p.err, ERRBIT_BOUNDS); continue; }
        const int N = max(16, (ti.n_rows + 15) & ~15);
        const uint32_t idesc = idesc_bf16(128, N);
        if (!mbar_wait_t(ACCE, (tc & 1) ^ 1, p.err, abort_flag, pc[0], pp)) break;
        tc_fence_after();
        bool alive = true;
        for (int kb = 0; kb < NKB; ++kb, ++it) {
          const int s = it % GU_STAGES;
          const uint32_t ph = (it / GU_STAGES) & 1;
          if (!mbar_wait_t(AFULL(s), ph, p.err, abort_flag, pc[1], pp) ||
              !mbar_wait_t(FULL(s), ph, p.err, abort_flag, pc[2], pp)) {
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
      if (pp) {
        pipe_flush(p.pipe, 0, pc, 3, clock64() - t_role, 3);
        atomicAdd(p.pipe + 10, static_cast<unsigned long long>(tc));
      }
    }
  } else if (warp < 10) {
    // ------------------------------------------------ dequant (8 warps)
    const int dt = tid - 64;           // 0..255
    const bool pp = p.pipe != nullptr;
    unsigned long long pc[1] = {0};
    const unsigned long long t_role = pp ? clock64() : 0;
    const int mat = dt >> 7;           // 0: gate rows, 1: up rows
    const int r = dt & 127;            // row inside the tile
    const int p_off = mat ? GU_PU : GU_PG;
    const int a_off = mat ? GU_AU : GU_AG;
    uint32_t it = 0;
    bool alive = true;
    // The scales and biases of 8 K steps (16 bytes each) are loaded one chunk ahead,
    // across tile boundaries, so their DRAM latency overlaps the previous chunk.
    TileInfo ti;
    ti.ok = false;
    const uint16_t *sc = nullptr, *bi = nullptr;
    uint4 nsv = make_uint4(0, 0, 0, 0), nbv = nsv;
    auto load_next = [&](int t) {
      if (t >= total) return;
      ti = tile_info(s_tiles, s_off, s_cnt, t, GU_MBLK, p.T);
      if (!ti.ok) return;
      const bool sh = ti.e == SHARED_E;
      const size_t srow = sh ? static_cast<size_t>(ti.mb * GX_BM + r)
                             : static_cast<size_t>(ti.e) * INTER + ti.mb * GX_BM + r;
      sc = (mat == 0 ? (sh ? p.sg_scales : p.g_scales) : (sh ? p.su_scales : p.u_scales)) + srow * (HID / GROUP);
      bi = (mat == 0 ? (sh ? p.sg_biases : p.g_biases) : (sh ? p.su_biases : p.u_biases)) + srow * (HID / GROUP);
      nsv = ldg_nc_v4(sc);
      nbv = ldg_nc_v4(bi);
    };
    load_next(blockIdx.x);
    for (int tile = blockIdx.x; tile < total && alive; tile += gridDim.x) {
      const TileInfo cur = ti;
      const uint16_t* csc = sc;
      const uint16_t* cbi = bi;
      if (!cur.ok) {
        if (threadIdx.x == 64) atomicOr(p.err, ERRBIT_BOUNDS);
        load_next(tile + gridDim.x);
        continue;
      }
      for (int kc = 0; kc < NKB / 8 && alive; ++kc) {
        const uint4 sv = nsv, bv = nbv;
        if (kc + 1 < NKB / 8) {
          nsv = ldg_nc_v4(csc + (kc + 1) * 8);
          nbv = ldg_nc_v4(cbi + (kc + 1) * 8);
        } else {
          load_next(tile + gridDim.x);
        }
        const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
        const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int s = it % GU_STAGES;
          const uint32_t ph = (it / GU_STAGES) & 1;
          if (!mbar_wait_t(FULL(s), ph, p.err, abort_flag, pc[0], pp)) { alive = false; break; }
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
    }
    if (pp && dt == 0) pipe_flush(p.pipe, 6, pc, 1, clock64() - t_role, 7);
  } else {
    // ------------------------------------------------ epilogue (4 warps): SwiGLU
    // While these warps drain TMEM, the dequant warps already fill the next tile's stages.
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const bool pp = p.pipe != nullptr;
    unsigned long long pc[1] = {0};
    const unsigned long long t_role = pp ? clock64() : 0;
    uint32_t tc = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const TileInfo ti = tile_info(s_tiles, s_off, s_cnt, tile, GU_MBLK, p.T);
      if (!ti.ok) continue;
      // each row's weight (routing weight, or the shared-expert gate) is applied here,
      // W_down (w h) = w (W_down h), so the down GEMM's epilogue has no per-row scaling;
      // the weights are fetched before waiting for the accumulator
      float wv[GX_BN / 32];
#pragma unroll
      for (int c = 0; c < GX_BN / 32; ++c) {
        const int j = c * 32 + lane;
        wv[c] = (j < ti.n_rows) ? __ldg(p.row_w + ti.row0 + j) : 0.0f;
      }
      bool ok = mbar_wait_t(ACCF, tc & 1, p.err, abort_flag, pc[0], pp);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int f = ti.mb * GX_BM + q * 32 + lane;   // intermediate feature of this lane
      const int hcol = ilv_pos(f);
#pragma unroll
      for (int cc = 0; cc < GX_BN / 32; ++cc) {
        const int col0 = cc * 32;
        if (col0 >= ti.n_rows) break;
        uint32_t g[32], u[32];
        tmem_ld32(tl + col0, g);
        tmem_ld32(tl + 256 + col0, u);
        tmem_ld_wait();
        __nv_bfloat16* hp = p.h + static_cast<size_t>(ti.row0 + col0) * INTER + hcol;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float wj = __shfl_sync(0xffffffffu, wv[cc], j);
          if (col0 + j < ti.n_rows) {
            const float gv = __uint_as_float(g[j]), uv = __uint_as_float(u[j]);
            // silu(g) = g * sigmoid(g), sigmoid(g) = (1 + tanh(g/2)) / 2 with the hardware
            // tanh (max relative error 2^-10.99, below the bf16 rounding of h)
            float th;
            asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(0.5f * gv));
            const float hv = gv * fmaf(0.5f, th, 0.5f) * uv * wj;
            hp[static_cast<size_t>(j) * INTER] = __float2bfloat16_rn(hv);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(ACCE);
      ++tc;
    }
    if (pp && warp == 10 && lane == 0) pipe_flush(p.pipe, 8, pc, 1, clock64() - t_role, 9);
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

cudaError_t launch_combine(const __nv_bfloat16* y, const __nv_bfloat16* x, __nv_bfloat16* out, int T,
                           int residual, cudaStream_t s) {
  combine_kernel<<<T, 256, 0, s>>>(y, x, out, T, residual);
  return cudaGetLastError();
}

cudaError_t set_gemm_attributes() {
  cudaError_t e = cudaFuncSetAttribute(gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GU_SMEM);
  if (e != cudaSuccess) return e;
  return set_down_attributes();
}

}  // namespace moe
