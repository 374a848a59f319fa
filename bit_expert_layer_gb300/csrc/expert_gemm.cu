// expert_gemm.cu -- the grouped gate/up GEMM of the prefill path with the 4-bit
// dequantisation fused into it, and the combine.  Packed weights go from HBM to shared
// memory by TMA, dequant warps expand them to bf16 tiles in shared memory, and tcgen05
// MMAs accumulate into TMEM; the dequantised weights never touch device memory (Lily
// fuses the 4-bit restore into its grouped GEMM and keeps the result in on-chip memory:
// aimanavo.com, "Why is Perplexity's local AI Lily faster than MLX", section "Prefill
// and decode are not treated as the same job"; dzen.guru, "Perplexity opened the Lily
// engine", section "Where the speed-up comes from").
//
// Orientation: weight rows are the MMA's M side (128 per tile), tokens its N side (up
// to 256 per tile, rounded up to 16), K steps of 64 = one quantisation group, so each
// dequantised row needs exactly one scale and one bias per K step.
//
//   gateup_kernel  h = silu(W_gate x) * (W_up x) for every (expert, token) pair of the
//                  permuted activations (the shared expert is expert 256 over all T
//                  tokens).  Two TMEM accumulators (gate, up), SwiGLU in the epilogue.
//   combine_kernel out[t] = sum_k w_k y[row(t,k)] + g_s y[8T+t] (+ x[t]) in a fixed
//                  order, row(t,k) = the permuted row of slot t*8+k, w_k its routing
//                  weight, g_s = sigmoid(g_s . x) the shared-expert gate; the weights are
//                  applied here, where they cost nothing in a memory-bound pass.
//
// Warp roles of gateup_kernel (20 warps, one role per warpgroup but the first):
//   warp 0      TMA producer of the packed 4-bit tiles (ring of GU_NP)
//   warp 1      TMEM allocator and MMA issuer
//   warps 2-7   activation gather (GU_GW warps, ring of GU_NX): the tile's rows are tokens in expert
//               order; each row is copied from the K-interleaved copy of x by token id
//               with 16-byte cp.async into the 128-byte-swizzled layout the MMA reads,
//               so the nine permuted copies of x are never written to memory; the
//               activation rows are kept in L2 (evict-last), the weights streamed
//               through it (evict-first)
//   warps 8-15  dequant: packed tile -> 128-byte-swizzled bf16 tiles (ring of GU_NA)
//   warps 16-19 epilogue, one per TMEM lane quarter: SwiGLU; per 32-row
//               chunk, bf16 pairs transposed into a 32 x 32 staging tile with stmatrix
//               and written with one TMA store (the dequant permutes the weight rows
//               so that lane order is h column order)
// The rings are separate so the HBM-bound packed tiles can be fetched further ahead than
// the large activation tiles fit.  A tile of at most GU_SWAP_ROWS tokens runs with the
// operands swapped (tokens on M, its gate and up rows together on N = 256).
//
// Persistent kernel: grid = number of SMs, tiles dealt from the size-ordered token-block
// list that route_scan_kernel builds on the device (no host readback).
#include "common.cuh"
#include "gemm_common.cuh"
#include "internal.h"

namespace moe {

namespace {
// shared-memory layout (1024-byte aligned base)
constexpr int OFF_A = 0;                                     // [GU_NA][gate 16 KB | up 16 KB]
constexpr int OFF_X = OFF_A + GU_NA * GU_A_STAGE;            // [GU_NX][32 KB]
constexpr int OFF_P = OFF_X + GU_NX * GX_X_BYTES;            // [GU_NP][gate 4 KB | up 4 KB]
constexpr int OFF_MISC = OFF_P + GU_NP * GU_P_STAGE;
static_assert(OFF_X % 1024 == 0 && OFF_P % 1024 == 0, "swizzled tiles need 1024-byte alignment");
constexpr int STG_ROW = 32 * 2;                      // bytes of one staged row (32 bf16)
constexpr int STG_BUF = 32 * STG_ROW;                // one 32 x 32 staging tile
static_assert(4 * GU_STG_BUFS * STG_BUF == GU_STG_BYTES, "staging size");
static_assert((512 + GX_TAB_BYTES + GU_GW * GU_GROWS * 4) % 16 == 0, "schedule alignment");
// the epilogue's staging tiles are 64-byte-swizzled TMA-store sources: 1024-byte aligned
// (misc is 1024-aligned)
constexpr int STG_OFF = (512 + GX_TAB_BYTES + GU_GW * GU_GROWS * 4 + GU_SCHED_CAP * 16 + 1023) / 1024 * 1024;
static_assert(STG_OFF % 1024 == 0 && OFF_MISC % 1024 == 0 && STG_BUF % 1024 == 0, "staging alignment");
}  // namespace

// kLimit: the bounded waits take their time limit from the launch (p.wait_ns) instead of
// the default; the launcher picks that instance only for a non-default limit, so the
// default instance keeps the limit a compile-time constant (the down GEMM measured 3%
// slower with a run-time limit).
template <bool kLimit>
__global__ void __launch_bounds__(GU_THREADS, 1)
    gateup_kernel(const __grid_constant__ CUtensorMap tm_qg, const __grid_constant__ CUtensorMap tm_qu,
                  const __grid_constant__ CUtensorMap tm_sqg, const __grid_constant__ CUtensorMap tm_squ,
                  const __grid_constant__ CUtensorMap tm_hs, GateUpParams p) {
  const unsigned long long wlim = kLimit ? p.wait_ns : WAIT_LIMIT_NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* misc = smem + OFF_MISC;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);                   // 32 barriers
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 260);
  int* s_off = reinterpret_cast<int*>(misc + 512);   // row tables (GX_TAB_BYTES reserved)
  int* s_cnt = s_off + (NEXP + 2);
  int* s_tok = reinterpret_cast<int*>(misc + 512 + GX_TAB_BYTES);   // [GU_GW][GU_GROWS] token ids
  int4* sched = reinterpret_cast<int4*>(s_tok + GU_GW * GU_GROWS);   // [GU_SCHED_CAP] this CTA's tiles
  uint8_t* stg = misc + STG_OFF;                                       // [4 warps][GU_STG_BUFS][32][32] bf16

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t bar0 = smem_u32(bars);
#define PFULL(s) (bar0 + 8u * (s))
#define PEMPTY(s) (bar0 + 8u * (GU_NP + (s)))
#define XEMPTY(s) (bar0 + 8u * (2 * GU_NP + (s)))
#define AEMPTY(s) (bar0 + 8u * (2 * GU_NP + GU_NX + (s)))
  // One READY barrier per K step: the dequant threads arrive on it after writing the
  // weight stage, the gather threads once their copies into the activation stage landed,
  // so the MMA issuer polls one barrier per step.  With a ring of max(GU_NX, GU_NA), the
  // arrivals for step it + GU_NR wait for stages that the MMAs of step it or later free,
  // and those MMAs follow the completion of step it's phase: phases never overlap.
  constexpr int GU_NR = GU_NX > GU_NA ? GU_NX : GU_NA;
#define READY(s) (bar0 + 8u * (2 * GU_NP + GU_NX + GU_NA + (s)))
  constexpr int NB = 2 * GU_NP + GU_NX + GU_NA + GU_NR;
  static_assert(8 * (NB + 3) <= 256, "barriers overlap the TMEM slot");
  const uint32_t ACCF = bar0 + 8u * NB, ACCE = bar0 + 8u * (NB + 1), DRAIN = bar0 + 8u * (NB + 2);

  if (tid == 0) {
    for (int s = 0; s < GU_NP; ++s) {
      mbar_init(PFULL(s), 1);
      mbar_init(PEMPTY(s), 256);
    }
    for (int s = 0; s < GU_NX; ++s) mbar_init(XEMPTY(s), 1);
    for (int s = 0; s < GU_NA; ++s) mbar_init(AEMPTY(s), 1);
    // one arrival per dequant thread and per gather thread (after its copies landed)
    for (int s = 0; s < GU_NR; ++s) mbar_init(READY(s), 256 + GU_GW * 32);
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
  grid_dep_wait();   // the routing tables and activations come from the kernels before this one
  stage_tables(s_off, p.offsets, p.counts);
  __syncthreads();
  const int ntiles = build_schedule(sched, GU_SCHED_CAP, p.blocks, s_off, s_cnt, GU_MBLK, p.T, p.err, true, BLOCKS_ALL);
  __syncthreads();
  constexpr int NKB = HID / 64;
  const bool pp = p.pipe != nullptr;

  // Registers by warpgroup (setmaxnreg, executed by all four warps of a group at the
  // top of its branch): the copy and MMA-issue warpgroups 0-1 hand theirs to the dequant
  // and epilogue warpgroups 2-4.  Launch: 640 x 96 = 61,440; after: 128 x (64 + 64 +
  // 112 + 112 + 112) = 59,392.
  static_assert(GU_THREADS == 640 && GU_GW == 6, "register split assumes 5 warpgroups");
  if (warp < 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 64;");
    if (warp == 0) {
      if (lane == 0) {
        // ------------------------------------------------ packed-tile producer
        unsigned long long pc[1] = {0};
        const unsigned long long t_role = pp ? clock64() : 0;
        tma_prefetch_desc(&tm_qg);
        tma_prefetch_desc(&tm_qu);
        const uint64_t pol = l2_policy_evict_first();   // each weight tile is read by one CTA once
        uint32_t it = 0;
        bool alive = true;
        for (int tix = 0; tix < ntiles && alive; ++tix) {
          const TileInfo ti = sched_tile(sched, tix);
          if (!ti.ok) { atomicOr(p.err, ERRBIT_BOUNDS); continue; }
          const bool sh = ti.e == SHARED_E;
          const CUtensorMap* mg = sh ? &tm_sqg : &tm_qg;
          const CUtensorMap* mu = sh ? &tm_squ : &tm_qu;
          const int wrow = (sh ? 0 : ti.e * INTER) + ti.mb * GX_BM;
          for (int kb = 0; kb < NKB; ++kb, ++it) {
            const int s = it % GU_NP;
            if (!mbar_wait_t(PEMPTY(s), ((it / GU_NP) & 1) ^ 1, p.err, abort_flag, wlim, pc[0], pp)) {
              alive = false;
              break;
            }
            const uint32_t st = smem_u32(smem + OFF_P + s * GU_P_STAGE);
            mbar_arrive_expect_tx(PFULL(s), GU_P_STAGE);
            tma_load_2d_hint(st, mg, PFULL(s), kb * 8, wrow, pol);
            tma_load_2d_hint(st + GX_P_BYTES, mu, PFULL(s), kb * 8, wrow, pol);
          }
        }
        // the packed tiles still in flight land before this thread leaves (a launch that
        // gave up may end before anyone consumes them; the latest phase of each stage)
        for (uint32_t i = (it > GU_NP ? it - GU_NP : 0); i < it; ++i) drain_wait(PFULL(i % GU_NP), (i / GU_NP) & 1);
        if (pp) pipe_flush(p.pipe, 4, pc, 1, clock64() - t_role, 5);
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // ------------------------------------------------ MMA issuer
        unsigned long long pc[3] = {0, 0, 0};
        const unsigned long long t_role = pp ? clock64() : 0;
        uint32_t it = 0, tc = 0;
        uint32_t rdy = 0;   // bit 0: READY of step `it` seen complete by the last poll
        for (int tix = 0; tix < ntiles; ++tix) {
          const TileInfo ti = sched_tile(sched, tix);
          if (!ti.ok) continue;
          const int N = max(16, (ti.n_rows + 15) & ~15);
          // a tile of at most GU_SWAP_ROWS tokens: one M = 128 (tokens) x N = 256 (gate and
          // up rows) MMA per K slice instead of a gate and an up MMA of N tokens each
          const bool swp = ti.n_rows <= GU_SWAP_ROWS;
          const uint32_t idesc = swp ? idesc_bf16(128, 2 * GX_BM) : idesc_bf16(128, N);
          if (!mbar_wait_t(ACCE, (tc & 1) ^ 1, p.err, abort_flag, wlim, pc[0], pp)) break;
          tc_fence_after();
          bool alive = true;
          for (int kb = 0; kb < NKB; ++kb, ++it) {
            const int sa = it % GU_NA, sx = it % GU_NX;
            if (!(rdy & 1u) && !mbar_wait_t(READY(it % GU_NR), (it / GU_NR) & 1, p.err, abort_flag, wlim, pc[1], pp)) {
              alive = false;
              break;
            }
            fence_proxy_async_smem();   // the activation stage was written by cp.async (generic proxy)
            tc_fence_after();
            const uint32_t a = smem_u32(smem + OFF_A + sa * GU_A_STAGE);
            const uint32_t x = smem_u32(smem + OFF_X + sx * GX_X_BYTES);
            // gate and up MMAs of this K step; the next step's stages are polled meanwhile
            const uint32_t nx = it + 1;
            if (swp)
              rdy = umma_k64_poll1(tmem, sdesc_sw128(x), sdesc_sw128(a), idesc, kb != 0, READY(nx % GU_NR),
                                   (nx / GU_NR) & 1);
            else
              rdy = umma_k64_x2_poll(tmem, tmem + 256, sdesc_sw128(a), sdesc_sw128(a + GX_A_BYTES), sdesc_sw128(x),
                                     idesc, kb != 0, READY(nx % GU_NR), (nx / GU_NR) & 1);
            umma_commit(AEMPTY(sa));
            umma_commit(XEMPTY(sx));
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
    } else {
      // ------------------------------------------------ activation gather (GU_GW warps)
      // Warp g copies rows g, g + GU_GW, g + 2 GU_GW, ... of every tile, so the gather
      // warps never wait on each other (each decides alone to stop on an abort).
      const int gw = warp - 2;
      int* tok = s_tok + gw * GU_GROWS;
      const int n8 = 8 * p.T;
      const uint64_t pol = l2_policy_evict_last();   // every token row is read by about nine tiles
      uint32_t it = 0;
      bool alive = true;
      for (int tix = 0; tix < ntiles && alive; ++tix) {
        const TileInfo ti = sched_tile(sched, tix);
        if (!ti.ok) continue;
        const int N = max(16, (ti.n_rows + 15) & ~15);
        const int nr = (N - gw + GU_GW - 1) / GU_GW;   // this warp's rows
        // token of each of this warp's rows (rows past n_rows repeat the first, unused)
        __syncwarp();   // the previous tile's reads of tok are done
        for (int i = lane; i < nr; i += 32) {
          const int r = gw + GU_GW * i;
          const int row = ti.row0 + (r < ti.n_rows ? r : 0);
          int t = row >= n8 ? row - n8 : (__ldg(p.row_dst + row) >> 3);
          if (t < 0 || t >= p.T) { atomicOr(p.err, ERRBIT_BOUNDS); t = 0; }
          tok[i] = t;
        }
        __syncwarp();
        for (int kb = 0; kb < NKB; ++kb, ++it) {
          const int s = it % GU_NX;
          alive = __all_sync(0xffffffffu, mbar_wait(XEMPTY(s), ((it / GU_NX) & 1) ^ 1, p.err, abort_flag, wlim));
          if (!alive) break;
          uint8_t* st = smem + OFF_X + s * GX_X_BYTES;
          for (int q = lane; q < nr * 8; q += 32) {
            const int i = q >> 3, c = q & 7;
            const __nv_bfloat16* src = p.x_ilv + static_cast<size_t>(tok[i]) * HID + kb * 64 + c * 8;
            asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(
                             smem_u32(st + sw128_off(gw + GU_GW * i, c))),
                         "l"(src), "l"(pol)
                         : "memory");
          }
          // one arrival per thread once its copies into the stage have landed; the MMA
          // issuer fences them into the async proxy after its wait
          asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(READY(it % GU_NR)) : "memory");
        }
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
    }
  } else if (warp < 16) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 112;");
    // ------------------------------------------------ dequant (8 warps)
    const int dt = tid - (2 + GU_GW) * 32;   // 0..255
    const int mat = dt >> 7;           // 0: gate rows, 1: up rows
    const int r = dt & 127;            // row inside the tile
    const int wr = ilv_row(r);         // the weight row it holds
    unsigned long long pc[1] = {0};
    const unsigned long long t_role = pp ? clock64() : 0;
    uint32_t it = 0;
    bool alive = true;
    // The scales and biases of 8 K steps (16 bytes each) are loaded one chunk ahead,
    // across tile boundaries, so their DRAM latency overlaps the previous chunk.
    TileInfo ti;
    ti.ok = false;
    const uint16_t *sc = nullptr, *bi = nullptr;
    uint4 nsv = make_uint4(0, 0, 0, 0), nbv = nsv;
    auto load_next = [&](int t) {
      if (t >= ntiles) return;
      ti = sched_tile(sched, t);
      if (!ti.ok) return;
      const bool sh = ti.e == SHARED_E;
      const size_t srow = sh ? static_cast<size_t>(ti.mb * GX_BM + wr)
                             : static_cast<size_t>(ti.e) * INTER + ti.mb * GX_BM + wr;
      sc = (mat == 0 ? (sh ? p.sg_scales : p.g_scales) : (sh ? p.su_scales : p.u_scales)) + srow * (HID / GROUP);
      bi = (mat == 0 ? (sh ? p.sg_biases : p.g_biases) : (sh ? p.su_biases : p.u_biases)) + srow * (HID / GROUP);
      nsv = ldg_nc_v4(sc);
      nbv = ldg_nc_v4(bi);
    };
    load_next(0);
    for (int tix = 0; tix < ntiles && alive; ++tix) {
      const TileInfo cur = ti;
      const uint16_t* csc = sc;
      const uint16_t* cbi = bi;
      if (!cur.ok) {
        load_next(tix + 1);
        continue;
      }
      for (int kc = 0; kc < NKB / 8 && alive; ++kc) {
        const uint4 sv = nsv, bv = nbv;
        if (kc + 1 < NKB / 8) {
          nsv = ldg_nc_v4(csc + (kc + 1) * 8);
          nbv = ldg_nc_v4(cbi + (kc + 1) * 8);
        } else {
          load_next(tix + 1);
        }
        const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
        const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int sp = it % GU_NP, sa = it % GU_NA, sr = it % GU_NR;
          if (!mbar_wait_t(PFULL(sp), (it / GU_NP) & 1, p.err, abort_flag, wlim, pc[0], pp) ||
              !mbar_wait(AEMPTY(sa), ((it / GU_NA) & 1) ^ 1, p.err, abort_flag, wlim)) {
            alive = false;
            break;
          }
          ++it;
          const __nv_bfloat162 ms = bf2((j & 1) ? (sw[j >> 1] >> 16) : sw[j >> 1]);
          const __nv_bfloat162 mbv = bf2((j & 1) ? (bw[j >> 1] >> 16) : bw[j >> 1]);
          // the row's two 16-byte halves, stored 32-byte swizzled (half c at c ^ bit 2 of the row)
          const uint8_t* P = smem + OFF_P + sp * GU_P_STAGE + mat * GX_P_BYTES + wr * 32;
          const int hs = ((wr >> 2) & 1) << 4;
          const uint4 w0 = *reinterpret_cast<const uint4*>(P + hs), w1 = *reinterpret_cast<const uint4*>(P + (16 ^ hs));
          // the packed words are in registers; the next TMA write into this stage is an
          // async-proxy access, so the generic reads are fenced before the release
          fence_proxy_async_smem();
          mbar_arrive(PEMPTY(sp));
          uint8_t* A = smem + OFF_A + sa * GU_A_STAGE + mat * GX_A_BYTES;
          st_shared_v4(A + sw128_off(r, 0), dequant8(w0.x, ms, mbv));
          st_shared_v4(A + sw128_off(r, 1), dequant8(w0.y, ms, mbv));
          st_shared_v4(A + sw128_off(r, 2), dequant8(w0.z, ms, mbv));
          st_shared_v4(A + sw128_off(r, 3), dequant8(w0.w, ms, mbv));
          st_shared_v4(A + sw128_off(r, 4), dequant8(w1.x, ms, mbv));
          st_shared_v4(A + sw128_off(r, 5), dequant8(w1.y, ms, mbv));
          st_shared_v4(A + sw128_off(r, 6), dequant8(w1.z, ms, mbv));
          st_shared_v4(A + sw128_off(r, 7), dequant8(w1.w, ms, mbv));
          fence_proxy_async_smem();
          mbar_arrive(READY(sr));
        }
      }
    }
    if (pp && dt == 0) pipe_flush(p.pipe, 6, pc, 1, clock64() - t_role, 7);
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 112;");
    // ------------------------------------------------ epilogue (4 warps): SwiGLU
    // While these warps drain TMEM, the dequant warps already fill the next tile's stages.
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
    uint8_t* wst = stg + q * (GU_STG_BUFS * STG_BUF);
    unsigned long long pc[1] = {0};
    const unsigned long long t_role = pp ? clock64() : 0;
    if (lane == 0) tma_prefetch_desc(&tm_hs);
    uint32_t tc = 0, nst = 0;   // tiles done; staging tiles used (warp-uniform)
    for (int tix = 0; tix < ntiles; ++tix) {
      const TileInfo ti = sched_tile(sched, tix);
      if (!ti.ok) continue;
      bool ok = mbar_wait_t(ACCF, tc & 1, p.err, abort_flag, wlim, pc[0], pp);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      if (ti.n_rows <= GU_SWAP_ROWS) {
        // swapped tile: TMEM lane = the tile's row 32q + lane (a token), columns 0-127 the
        // gate and 128-255 the up outputs of the tile's 128 h columns, in h column order
        // (the dequant permuted the weight rows); each thread writes its row's 256 bytes
        const int row = 32 * q + lane;
        __nv_bfloat16* hrow = p.h + static_cast<size_t>(ti.row0 + row) * INTER + ti.mb * GX_BM;
#pragma unroll 1
        for (int c0 = 0; c0 < GX_BM; c0 += 16) {
          uint32_t g[16], u[16];
          tmem_ld16(tl + c0, g);
          tmem_ld16(tl + GX_BM + c0, u);
          tmem_ld_wait();
          if (c0 + 16 == GX_BM) {   // last read: the MMA may overwrite the accumulator
            tc_fence_before();
            mbar_arrive(ACCE);
          }
          uint32_t w[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            float hv[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const float hg = 0.5f * __uint_as_float(g[2 * k + i]);
              float th;
              asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(hg));
              hv[i] = fmaf(hg, th, hg) * __uint_as_float(u[2 * k + i]);
            }
            w[k] = pack_bf16x2(__float_as_uint(hv[0]), __float_as_uint(hv[1]));
          }
          if (row < ti.n_rows) {
            *reinterpret_cast<uint4*>(hrow + c0) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(hrow + c0 + 8) = make_uint4(w[4], w[5], w[6], w[7]);
          }
        }
        ++tc;
        continue;
      }
      const int hcol = ti.mb * GX_BM + q * 32;   // h column of this warp's first lane
      // One 32-row chunk: gate and up read as 16-lane fragments (lanes 0-15, then 16-31
      // of this warp), SwiGLU, rounded to bf16 pairs (rows j, j+1) and
      // staged transposed with stmatrix: staged row j = the tile's row col0 + j, its 32
      // bf16 in lane order = h column order (the dequant permuted the weight rows).
      // Thread t holds rows 8g + 2(t%4) + {0,1}, g = 0..3, of lanes t/4 and 8 + t/4.
#pragma unroll 1
      for (int cc = 0; cc < GX_BN / 32; ++cc) {
        const int col0 = cc * 32;
        if (col0 >= ti.n_rows) break;
        uint32_t m[2][4][2];   // [lane half][g][lane t/4 or 8 + t/4]
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t g[16], u[16];
          tmem_ld16x256(tl + (static_cast<uint32_t>(16 * hh) << 16) + col0, g);
          tmem_ld16x256(tl + (static_cast<uint32_t>(16 * hh) << 16) + 256 + col0, u);
          tmem_ld_wait();
          if (hh == 1 && col0 + 32 >= ti.n_rows) {   // last read: the MMA may overwrite the accumulator
            tc_fence_before();
            mbar_arrive(ACCE);
          }
          float hv[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            // silu(g) = g sigmoid(g) = g/2 + (g/2) tanh(g/2), with the hardware tanh (max
            // relative error 2^-10.99, below the bf16 rounding of h)
            const float hg = 0.5f * __uint_as_float(g[k]);
            float th;
            asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(hg));
            hv[k] = fmaf(hg, th, hg) * __uint_as_float(u[k]);
          }
#pragma unroll
          for (int gg = 0; gg < 4; ++gg) {
            m[hh][gg][0] = pack_bf16x2(__float_as_uint(hv[4 * gg]), __float_as_uint(hv[4 * gg + 1]));
            m[hh][gg][1] = pack_bf16x2(__float_as_uint(hv[4 * gg + 2]), __float_as_uint(hv[4 * gg + 3]));
          }
        }
        uint8_t* sb = wst + (nst % GU_STG_BUFS) * STG_BUF;
        // the TMA store issued from this staging tile GU_STG_BUFS stores ago has read it
        if (lane == 0 && nst >= GU_STG_BUFS) tma_store_wait_read<GU_STG_BUFS - 1>();
        __syncwarp();
        // matrix lane/8, row lane%8; the staging tile is 64-byte swizzled like the TMA box
        const uint32_t ra = smem_u32(sb) + (lane & 7) * STG_ROW + ((((lane >> 3) ^ ((lane >> 1) & 3))) << 4);
#pragma unroll
        for (int gg = 0; gg < 4; ++gg)   // rows 8g..8g+7; matrices = lanes 0-7, 8-15, 16-23, 24-31
          stmatrix_x4_trans(ra + gg * 8 * STG_ROW, m[0][gg][0], m[0][gg][1], m[1][gg][0], m[1][gg][1]);
        const int rows = min(32, ti.n_rows - col0);
        if (rows == 32) {
          fence_proxy_async_smem();   // the generic writes, before the TMA reads them
          __syncwarp();
          // h goes out evict-first, so that it does not push out of L2 the activation
          // rows that later tiles gather again (measured at T=16384: 130 MB less DRAM
          // read per launch, same time)
          if (lane == 0) tma_store_2d_hint(&tm_hs, smem_u32(sb), hcol, ti.row0 + col0, l2_policy_evict_first());
          ++nst;
        } else {
          // ragged last chunk: only its own rows (the next rows belong to other tiles)
          __syncwarp();
          for (int item = lane; item < rows * 4; item += 32) {
            const int j = item >> 2, seg = item & 3;
            const uint4 v = *reinterpret_cast<const uint4*>(sb + j * STG_ROW + ((seg ^ ((j >> 1) & 3)) << 4));
            *reinterpret_cast<uint4*>(p.h + static_cast<size_t>(ti.row0 + col0 + j) * INTER + hcol + seg * 8) = v;
          }
          __syncwarp();   // this staging tile is free again
        }
      }
      ++tc;
    }
    if (lane == 0) tma_store_wait_all();
    if (pp && warp == 2 + GU_GW + 8 && lane == 0) pipe_flush(p.pipe, 8, pc, 1, clock64() - t_role, 9);
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
#undef PFULL
#undef PEMPTY
#undef XEMPTY
#undef AEMPTY
#undef READY
}

// ============================================================================ combine
// One CTA per token, 256 threads x 8 features; fixed summation order: the 8 routed
// slots in rank order, then the shared expert, then the residual.
__global__ void __launch_bounds__(256) combine_kernel(const __nv_bfloat16* __restrict__ y,
                                                      const int* __restrict__ slot_row,
                                                      const float* __restrict__ row_w,
                                                      const __nv_bfloat16* x, __nv_bfloat16* out, int T,
                                                      int residual, NextLayerIn nx) {
  const int t = blockIdx.x, c = threadIdx.x;
  grid_dep_wait();   // y, the slot tables and x come from the kernels before this one
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  // the token's eight routed rows (y is in permuted-row order), then its shared-expert row
  int rows[TOPK + 1];
#pragma unroll
  for (int k = 0; k < TOPK; ++k) rows[k] = __ldg(slot_row + static_cast<size_t>(t) * TOPK + k);
  rows[TOPK] = 8 * T + t;
#pragma unroll
  for (int k = 0; k <= TOPK; ++k) {
    if (rows[k] < 0 || rows[k] >= 9 * T) continue;   // a slot the scatter rejected (error recorded)
    const float w = __ldg(row_w + rows[k]);   // routing weight, or the shared-expert gate
    const uint4 v = ldg_nc_v4(y + static_cast<size_t>(rows[k]) * HID + c * 8);
    acc[0] = fmaf(w, bf16lo(v.x), acc[0]); acc[1] = fmaf(w, bf16hi(v.x), acc[1]);
    acc[2] = fmaf(w, bf16lo(v.y), acc[2]); acc[3] = fmaf(w, bf16hi(v.y), acc[3]);
    acc[4] = fmaf(w, bf16lo(v.z), acc[4]); acc[5] = fmaf(w, bf16hi(v.z), acc[5]);
    acc[6] = fmaf(w, bf16lo(v.w), acc[6]); acc[7] = fmaf(w, bf16hi(v.w), acc[7]);
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
  if (nx.norm_w) {
    // The next stacked layer's inputs from this output row while it is in registers: its
    // RMSNorm, the K-interleaved copy its gate/up GEMM gathers, and its shared-expert gate
    // (the work its scatter does otherwise, in the same summation order).
    __shared__ float s_warp[8];
    const float rr = row_inv_rms(r, s_warp);
    const uint4 xn = rms_scale8(r, ldg_nc_v4(nx.norm_w + c * 8), rr);
    *reinterpret_cast<uint4*>(nx.xn + o) = xn;
    *reinterpret_cast<uint4*>(nx.x_ilv + o) = interleave8(xn);
    const float dot = row_dot(xn, ldg_nc_v4(nx.gate_w + c * 8), s_warp);
    if (c == 0) {
      const int srow = 8 * T + t;
      nx.row_dst[srow] = srow;
      nx.row_w[srow] = 1.0f / (1.0f + expf(-dot));
    }
  }
}

cudaError_t launch_gateup(const CUtensorMap& qg, const CUtensorMap& qu, const CUtensorMap& sqg,
                          const CUtensorMap& squ, const CUtensorMap& hs, const GateUpParams& p, int grid,
                          cudaStream_t s) {
  return launch_pdl(p.wait_ns == WAIT_LIMIT_NS ? gateup_kernel<false> : gateup_kernel<true>, grid, GU_THREADS,
                    GU_SMEM, s, qg, qu, sqg, squ, hs, p);
}

cudaError_t launch_combine(const __nv_bfloat16* y, const int* slot_row, const float* row_w, const __nv_bfloat16* x,
                           __nv_bfloat16* out, int T, int residual, const NextLayerIn& nx, cudaStream_t s) {
  return launch_pdl(combine_kernel, T, 256, 0, s, y, slot_row, row_w, x, out, T, residual, nx);
}

cudaError_t set_gemm_attributes() {
  cudaError_t e = cudaFuncSetAttribute(gateup_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, GU_SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gateup_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, GU_SMEM);
  if (e != cudaSuccess) return e;
  return set_down_attributes();
}

}  // namespace moe
