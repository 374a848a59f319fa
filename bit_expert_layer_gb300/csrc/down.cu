// down.cu -- the grouped down GEMM of the prefill path: y[row] = W_down h[row] for every
// permuted row (8 routed slots and 1 shared row per token; the rows' weights are applied
// by the combine), with the 4-bit weights dequantised inside the kernel (Lily restores
// the 4-bit weights inside its grouped GEMM: aimanavo.com, "Why is Perplexity's local AI
// Lily faster than MLX", section "Prefill and decode are not treated as the same job").
//
// A tile is 128 output features (M) x up to 256 permuted rows (N); K = 512 is only 8
// steps of 64, so one tile's MMAs take ~2 us and the dequant and epilogue have to keep
// pace with that.  Warp w runs on scheduler w % 4.  A single thread issues the MMAs and
// each tcgen05.mma holds it for ~100 cycles of issue; sharing its scheduler with the
// ALU-bound dequant warps slowed the MMA stream by ~40%, so no dequant warp runs on
// scheduler 1.  Warp roles (16 warps):
//   warp 0      TMA producer of the packed 4-bit tiles (ring of DN_NP, 4 KB stages)
//   warp 1      TMEM allocator and MMA issuer (double-buffered 128 x 256 accumulator)
//   warp 5      TMA producer of the activation rows h (ring of DN_NX, 32 KB stages)
//   warps 2-4, 6-8, 10, 11
//               dequant: two threads per weight row, four packed words each (ring of
//               DN_NA dequantised 16 KB tiles)
//   warps 12-15 epilogue, one per TMEM lane quarter (32 features), each on its own:
//               per 32-row chunk, round to bf16 pairs, transpose into a 32 x 32 staging
//               tile with stmatrix and write it with one TMA store (y is kept in
//               permuted-row order, so a chunk is one box; the combine reads each
//               token's nine rows through the slot -> row map); DN_STG_BUFS staging
//               tiles per warp rotate; a ragged last chunk is written with 16-byte stores
//   warp 9      none
// The rings are separate so the small packed tiles, which come from HBM, run further
// ahead than the activation tiles, which each expert's 16 row blocks re-read from L2
// (evict-last) while the weights stream through it (evict-first).
#include "common.cuh"
#include "gemm_common.cuh"
#include "internal.h"

namespace moe {

namespace {
// shared-memory layout (1024-byte aligned base)
constexpr int OFF_A = 0;                                   // [DN_NA][16 KB]
constexpr int OFF_X = OFF_A + DN_NA * GX_A_BYTES;          // [DN_NX][32 KB]
constexpr int OFF_P = OFF_X + DN_NX * GX_X_BYTES;          // [DN_NP][4 KB]
constexpr int OFF_MISC = OFF_P + DN_NP * GX_P_BYTES;
static_assert(OFF_X % 1024 == 0 && OFF_P % 1024 == 0, "swizzled tiles need 1024-byte alignment");
constexpr int STG_ROW = 32 * 2;                      // bytes of one staged row (32 bf16)
constexpr int STG_BUF = 32 * STG_ROW;                // one 32 x 32 staging tile
static_assert(4 * DN_STG_BUFS * STG_BUF == DN_STG_BYTES, "staging size");
}  // namespace

// kLimit: the bounded waits take their time limit from the launch (p.wait_ns) instead of
// the default; the launcher picks that instance only for a non-default limit, so the
// default instance keeps the limit a compile-time constant.
template <bool kLimit>
__global__ void __launch_bounds__(DN_THREADS, 1)
    down_kernel(const __grid_constant__ CUtensorMap tm_qd, const __grid_constant__ CUtensorMap tm_sqd,
                const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_y,
                DownParams p) {
  extern __shared__ uint8_t smem_raw[];
  const unsigned long long wlim = kLimit ? p.wait_ns : WAIT_LIMIT_NS;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* misc = smem + OFF_MISC;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);                       // 40 barriers
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 512);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 516);
  uint8_t* stg = misc + 1024;                                     // [4 warps][DN_STG_BUFS][32][32] bf16
  int* s_off = reinterpret_cast<int*>(stg + DN_STG_BYTES);   // row tables (GX_TAB_BYTES reserved)
  int* s_cnt = s_off + (NEXP + 2);
  constexpr int SCHED_OFF = (1024 + DN_STG_BYTES + GX_TAB_BYTES + 15) / 16 * 16;
  int4* sched = reinterpret_cast<int4*>(misc + SCHED_OFF);   // [DN_SCHED_CAP] this CTA's tiles

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t bar0 = smem_u32(bars);
#define PFULL(s) (bar0 + 8u * (s))
#define PEMPTY(s) (bar0 + 8u * (DN_NP + (s)))
#define XFULL(s) (bar0 + 8u * (2 * DN_NP + (s)))
#define XEMPTY(s) (bar0 + 8u * (2 * DN_NP + DN_NX + (s)))
#define AFULL(s) (bar0 + 8u * (2 * DN_NP + 2 * DN_NX + (s)))
#define AEMPTY(s) (bar0 + 8u * (2 * DN_NP + 2 * DN_NX + DN_NA + (s)))
  constexpr int NB = 2 * DN_NP + 2 * DN_NX + 2 * DN_NA;
  static_assert(NB + 5 <= 64, "barrier space");
#define ACCF(b) (bar0 + 8u * (NB + (b)))
#define ACCE(b) (bar0 + 8u * (NB + 2 + (b)))
  const uint32_t DRAIN = bar0 + 8u * (NB + 4);

  if (tid == 0) {
    for (int s = 0; s < DN_NP; ++s) {
      mbar_init(PFULL(s), 1);
      mbar_init(PEMPTY(s), 256);
    }
    for (int s = 0; s < DN_NX; ++s) {
      mbar_init(XFULL(s), 1);
      mbar_init(XEMPTY(s), 1);
    }
    for (int s = 0; s < DN_NA; ++s) {
      mbar_init(AFULL(s), 256);
      mbar_init(AEMPTY(s), 1);
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
  grid_dep_wait();   // the routing tables and activations come from the kernels before this one
  stage_tables(s_off, p.offsets, p.counts);
  __syncthreads();
  const int ntiles = build_schedule(sched, DN_SCHED_CAP, p.blocks, s_off, s_cnt, DN_MBLK, p.T, p.err, false,
                                    p.small_apart ? BLOCKS_BIG : BLOCKS_ALL);
  __syncthreads();
  constexpr int NKB = INTER / 64;   // 8
  uint32_t p_issued = 0;   // packed-tile producer (warp 0) / activation producer (warp 5): K steps issued

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ packed-tile producer
      const bool pp = p.pipe != nullptr;
      unsigned long long pc[1] = {0};
      const unsigned long long t_role = pp ? clock64() : 0;
      tma_prefetch_desc(&tm_qd);
      tma_prefetch_desc(&tm_sqd);
      const uint64_t pol = l2_policy_evict_first();   // each weight tile is read once
      uint32_t it = 0;
      bool alive = true;
      for (int tix = 0; tix < ntiles && alive; ++tix) {
        const TileInfo ti = sched_tile(sched, tix);
        if (!ti.ok) { atomicOr(p.err, ERRBIT_BOUNDS); continue; }
        const bool sh = ti.e == SHARED_E;
        const CUtensorMap* mq = sh ? &tm_sqd : &tm_qd;
        const int wrow = (sh ? 0 : ti.e * HID) + ti.mb * GX_BM;
        for (int kb = 0; kb < NKB; ++kb, ++it) {
          const int s = it % DN_NP;
          if (!mbar_wait_t(PEMPTY(s), ((it / DN_NP) & 1) ^ 1, p.err, abort_flag, wlim, pc[0], pp)) { alive = false; break; }
          mbar_arrive_expect_tx(PFULL(s), GX_P_BYTES);
          tma_load_2d_hint(smem_u32(smem + OFF_P + s * GX_P_BYTES), mq, PFULL(s), kb * 8, wrow, pol);
        }
      }
      p_issued = it;
      if (pp) pipe_flush(p.pipe, 4, pc, 1, clock64() - t_role, 5);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      // ------------------------------------------------ activation-tile producer
      tma_prefetch_desc(&tm_h);
      const uint64_t pol = l2_policy_evict_last();    // each h block is read by 16 row blocks
      uint32_t it = 0;
      bool alive = true;
      for (int tix = 0; tix < ntiles && alive; ++tix) {
        const TileInfo ti = sched_tile(sched, tix);
        if (!ti.ok) continue;
        const int nbox = (ti.n_rows + GX_XBOX - 1) / GX_XBOX;
        for (int kb = 0; kb < NKB; ++kb, ++it) {
          const int s = it % DN_NX;
          if (!mbar_wait(XEMPTY(s), ((it / DN_NX) & 1) ^ 1, p.err, abort_flag, wlim)) { alive = false; break; }
          const uint32_t st = smem_u32(smem + OFF_X + s * GX_X_BYTES);
          mbar_arrive_expect_tx(XFULL(s), nbox * GX_XBOX * 128);
          for (int j = 0; j < nbox; ++j)
            tma_load_2d_hint(st + j * GX_XBOX * 128, &tm_h, XFULL(s), kb * 64, ti.row0 + j * GX_XBOX, pol);
        }
      }
      p_issued = it;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      const bool pp = p.pipe != nullptr;
      unsigned long long pc[3] = {0, 0, 0};
      const unsigned long long t_role = pp ? clock64() : 0;
      uint32_t it = 0, tc = 0;
      uint32_t rdy = 0;   // bit 0 / 1: AFULL / XFULL of step `it` seen complete by the last poll
      for (int tix = 0; tix < ntiles; ++tix) {
        const TileInfo ti = sched_tile(sched, tix);
        if (!ti.ok) continue;
        const int N = max(16, (ti.n_rows + 15) & ~15);
        const uint32_t idesc = idesc_bf16(128, N);
        const int buf = tc & 1;
        if (!mbar_wait_t(ACCE(buf), ((tc >> 1) & 1) ^ 1, p.err, abort_flag, wlim, pc[0], pp)) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * 256;
        bool alive = true;
        for (int kb = 0; kb < NKB; ++kb, ++it) {
          const int sa = it % DN_NA, sx = it % DN_NX;
          if ((!(rdy & 1u) && !mbar_wait_t(AFULL(sa), (it / DN_NA) & 1, p.err, abort_flag, wlim, pc[1], pp)) ||
              (!(rdy & 2u) && !mbar_wait_t(XFULL(sx), (it / DN_NX) & 1, p.err, abort_flag, wlim, pc[2], pp))) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = smem_u32(smem + OFF_A + sa * GX_A_BYTES);
          const uint32_t x = smem_u32(smem + OFF_X + sx * GX_X_BYTES);
          const uint32_t nx = it + 1;   // the next step's stages are polled while these issue
          rdy = umma_k64_poll(d, sdesc_sw128(a), sdesc_sw128(x), idesc, kb != 0, AFULL(nx % DN_NA),
                              (nx / DN_NA) & 1, XFULL(nx % DN_NX), (nx / DN_NX) & 1);
          umma_commit(AEMPTY(sa));
          umma_commit(XEMPTY(sx));
        }
        if (!alive) break;
        umma_commit(ACCF(buf));
        ++tc;
      }
      umma_commit(DRAIN);
      if (pp) {
        pipe_flush(p.pipe, 0, pc, 3, clock64() - t_role, 3);
        atomicAdd(p.pipe + 10, static_cast<unsigned long long>(tc));
      }
    }
  } else if (warp < 12 && warp != 9) {
    // ------------------------------------------------ dequant (8 warps, 2 threads per row)
    const int dt = (warp - 2 - (warp - 2) / 4) * 32 + lane;   // warps 2-4, 6-8, 10, 11 -> 0..255
    const int r = dt & 127;        // row inside the tile
    const int hw = dt >> 7;        // which four of the row's eight packed words
    const bool pp = p.pipe != nullptr;
    unsigned long long pc[1] = {0};
    const unsigned long long t_role = pp ? clock64() : 0;
    uint32_t it = 0;
    bool alive = true;
    // a row's 8 scales and 8 biases (one per K step) are loaded one tile ahead
    TileInfo ti;
    ti.ok = false;
    uint4 nsv = make_uint4(0, 0, 0, 0), nbv = nsv;
    auto load_next = [&](int t) {
      if (t >= ntiles) return;
      ti = sched_tile(sched, t);
      if (!ti.ok) return;
      const bool sh = ti.e == SHARED_E;
      const size_t srow = sh ? static_cast<size_t>(ti.mb * GX_BM + r)
                             : static_cast<size_t>(ti.e) * HID + ti.mb * GX_BM + r;
      nsv = ldg_nc_v4((sh ? p.sd_scales : p.d_scales) + srow * (INTER / GROUP));
      nbv = ldg_nc_v4((sh ? p.sd_biases : p.d_biases) + srow * (INTER / GROUP));
    };
    load_next(0);
    for (int tix = 0; tix < ntiles && alive; ++tix) {
      const bool cur_ok = ti.ok;
      const uint4 sv = nsv, bv = nbv;
      load_next(tix + 1);
      if (!cur_ok) continue;
      const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
      const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int kb = 0; kb < NKB; ++kb) {
        const int sp = it % DN_NP, sa = it % DN_NA;
        if (!mbar_wait_t(PFULL(sp), (it / DN_NP) & 1, p.err, abort_flag, wlim, pc[0], pp)) {
          alive = false;
          break;
        }
        const __nv_bfloat162 ms = bf2((kb & 1) ? (sw[kb >> 1] >> 16) : sw[kb >> 1]);
        const __nv_bfloat162 mbv = bf2((kb & 1) ? (bw[kb >> 1] >> 16) : bw[kb >> 1]);
        // this thread's 16-byte half of the row, stored 32-byte swizzled (half c at c ^ bit 2 of the row)
        const uint4 w = *reinterpret_cast<const uint4*>(smem + OFF_P + sp * GX_P_BYTES + r * 32 +
                                                        ((hw ^ ((r >> 2) & 1)) << 4));
        // the packed words are in registers; the next TMA write into this stage is an
        // async-proxy access, so the generic reads are fenced before the release
        fence_proxy_async_smem();
        mbar_arrive(PEMPTY(sp));
        // dequantise into registers before waiting for the weight stage (two stages only):
        // the stores alone then sit between the MMAs that free it and the MMAs that read it
        // again (measured 1.5% faster; in the gate/up GEMM the same order was slower)
        const uint4 d0 = dequant8(w.x, ms, mbv), d1 = dequant8(w.y, ms, mbv), d2 = dequant8(w.z, ms, mbv),
                    d3 = dequant8(w.w, ms, mbv);
        if (!mbar_wait(AEMPTY(sa), ((it / DN_NA) & 1) ^ 1, p.err, abort_flag, wlim)) {
          alive = false;
          break;
        }
        ++it;
        uint8_t* A = smem + OFF_A + sa * GX_A_BYTES;
        st_shared_v4(A + sw128_off(r, 4 * hw + 0), d0);
        st_shared_v4(A + sw128_off(r, 4 * hw + 1), d1);
        st_shared_v4(A + sw128_off(r, 4 * hw + 2), d2);
        st_shared_v4(A + sw128_off(r, 4 * hw + 3), d3);
        fence_proxy_async_smem();
        mbar_arrive(AFULL(sa));
      }
    }
    if (pp && dt == 0) pipe_flush(p.pipe, 6, pc, 1, clock64() - t_role, 7);
  } else if (warp >= 12) {
    // ------------------------------------------------ epilogue (4 warps, independent)
    const int q = warp & 3;                       // TMEM lane quarter = features q*32..q*32+31
    const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
    uint8_t* wst = stg + q * (DN_STG_BUFS * STG_BUF);
    const bool pp = p.pipe != nullptr;
    unsigned long long pc[1] = {0};
    const unsigned long long t_role = pp ? clock64() : 0;
    if (lane == 0) tma_prefetch_desc(&tm_y);
    uint32_t tc = 0, nst = 0;                     // tiles done; staging tiles used (warp-uniform)
    for (int tix = 0; tix < ntiles; ++tix) {
      const TileInfo ti = sched_tile(sched, tix);
      if (!ti.ok) continue;
      const int buf = tc & 1;
      const bool got = mbar_wait_t(ACCF(buf), (tc >> 1) & 1, p.err, abort_flag, wlim, pc[0], pp);
      if (!__all_sync(0xffffffffu, got)) break;   // tcgen05.ld below needs the whole warp
      tc_fence_after();
      const int fcol = ti.mb * GX_BM + q * 32;    // this warp's first output feature
      const uint32_t tb = tl + buf * 256;
      // One 32-row chunk, read as two 16-lane fragments (features 0-15 and 16-31 of this
      // warp): round to bf16 pairs and stage it transposed with stmatrix, so staged row j
      // (the tile's row c0 + j) holds the warp's 32 features in order; then one TMA store.
      auto stage = [&](const uint32_t (&fa)[16], const uint32_t (&fb)[16], int c0) {
        uint8_t* sb = wst + (nst % DN_STG_BUFS) * STG_BUF;
        // the TMA store issued from this staging tile DN_STG_BUFS stores ago has read it
        if (lane == 0 && nst >= DN_STG_BUFS) tma_store_wait_read<DN_STG_BUFS - 1>();
        __syncwarp();
        // matrix lane/8, row lane%8; the staging tile is 64-byte swizzled like the TMA box
        const uint32_t ra = smem_u32(sb) + (lane & 7) * STG_ROW + ((((lane >> 3) ^ ((lane >> 1) & 3))) << 4);
#pragma unroll
        for (int g = 0; g < 4; ++g)   // rows 8g..8g+7; matrices = features 0-7, 8-15, 16-23, 24-31
          stmatrix_x4_trans(ra + g * 8 * STG_ROW, pack_bf16x2(fa[4 * g], fa[4 * g + 1]),
                            pack_bf16x2(fa[4 * g + 2], fa[4 * g + 3]), pack_bf16x2(fb[4 * g], fb[4 * g + 1]),
                            pack_bf16x2(fb[4 * g + 2], fb[4 * g + 3]));
        const int rows = min(32, ti.n_rows - c0);
        if (rows == 32) {
          fence_proxy_async_smem();               // the generic writes, before the TMA reads them
          __syncwarp();
          if (lane == 0) tma_store_2d(&tm_y, smem_u32(sb), fcol, ti.row0 + c0);
          ++nst;
        } else {
          // ragged last chunk: only its own rows (the next rows belong to other tiles)
          __syncwarp();
          for (int item = lane; item < rows * 4; item += 32) {
            const int j = item >> 2, seg = item & 3;
            const uint4 v = *reinterpret_cast<const uint4*>(sb + j * STG_ROW + ((seg ^ ((j >> 1) & 3)) << 4));
            *reinterpret_cast<uint4*>(p.y + static_cast<size_t>(ti.row0 + c0 + j) * HID + fcol + seg * 8) = v;
          }
          __syncwarp();                           // this staging tile is free again
        }
      };
#pragma unroll 1
      for (int col0 = 0; col0 < ti.n_rows; col0 += 64) {
        const bool two = col0 + 32 < ti.n_rows;   // warp-uniform
        uint32_t a0[16], b0[16], a1[16], b1[16];
        tmem_ld16x256(tb + col0, a0);
        tmem_ld16x256(tb + (16u << 16) + col0, b0);
        if (two) {
          tmem_ld16x256(tb + col0 + 32, a1);
          tmem_ld16x256(tb + (16u << 16) + col0 + 32, b1);
        }
        tmem_ld_wait();
        if (col0 + 64 >= ti.n_rows) {             // last read of this buffer: the MMA may reuse it
          tc_fence_before();
          mbar_arrive(ACCE(buf));
        }
        stage(a0, b0, col0);
        if (two) stage(a1, b1, col0 + 32);
      }
      ++tc;
    }
    if (lane == 0) tma_store_wait_all();
    if (pp && q == 0 && lane == 0) pipe_flush(p.pipe, 8, pc, 1, clock64() - t_role, 9);
  }
  // warp 9 has no role

  tc_fence_before();
  __syncthreads();
  if ((warp == 0 || warp == 5) && lane == 0 && *abort_flag) {
    // a launch that gave up (whichever role did): the tiles still in flight land before
    // the CTA's shared memory goes away (the latest phase of each stage)
    if (warp == 0)
      for (uint32_t i = (p_issued > DN_NP ? p_issued - DN_NP : 0); i < p_issued; ++i)
        drain_wait(PFULL(i % DN_NP), (i / DN_NP) & 1);
    else
      for (uint32_t i = (p_issued > DN_NX ? p_issued - DN_NX : 0); i < p_issued; ++i)
        drain_wait(XFULL(i % DN_NX), (i / DN_NX) & 1);
  }
  if (warp == 1) {
    tc_fence_after();
    if (lane == 0) drain_wait(DRAIN, 0);
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
#undef PFULL
#undef PEMPTY
#undef XFULL
#undef XEMPTY
#undef AFULL
#undef AEMPTY
#undef ACCF
#undef ACCE
}

// ============================================================================ small blocks
// down_swap_kernel: the token blocks of at most GX_SMALL rows (an expert's partial last
// block) with the operands swapped, for T <= DS_MAX_T.  The block's rows are the MMA's M
// side (128; rows past the block's end are computed but never stored) and 256 weight
// rows -- two row blocks, 256 output features -- its N side, so one MMA covers 256
// features instead of 128 features of a handful of rows and a block needs half the K
// steps.  A swapped K step takes about twice as long as a narrow one (measured: ~1.9 K
// against ~1 K cycles), so this pays only while most blocks are small; above DS_MAX_T
// down_kernel runs every block.  A tile is (small block, feature pair pb = 0..7); the K
// loop is 8 steps of 64.
//
// Warp roles (16 warps), as in down_kernel where not said:
//   warp 0      TMA producer of the packed 4-bit tiles (two 4 KB boxes: weight rows
//               256 pb .. +127 and +128 .. +255)
//   warp 1      TMEM allocator and MMA issuer (double-buffered 128 x 256 accumulator)
//   warp 5      TMA producer of the block's activation rows (up to four 32-row boxes)
//   warps 2-4, 6-8, 10, 11
//               dequant: one thread per weight row (256), its 64 weights of the K step
//   warps 12-15 epilogue, one per TMEM lane quarter (32 block rows): each thread rounds
//               its row's 256 outputs to bf16 and writes them to y, 64 bytes a chunk
namespace {
constexpr int DS_OFF_W = 0;                                       // [DS_NW][32 KB]
constexpr int DS_OFF_H = DS_OFF_W + DS_NW * DS_W_STAGE;           // [DS_NH][16 KB]
constexpr int DS_OFF_P = DS_OFF_H + DS_NH * DS_H_STAGE;           // [DS_NP][8 KB]
constexpr int DS_OFF_MISC = DS_OFF_P + DS_NP * DS_P_STAGE;
static_assert(DS_OFF_H % 1024 == 0 && DS_OFF_P % 1024 == 0 && DS_OFF_MISC % 1024 == 0, "1024-byte alignment");
static_assert(DS_SMEM >= DS_OFF_MISC + 1024 + (GX_TAB_BYTES + 15) / 16 * 16 + DS_SCHED_CAP * 16 + 1024,
              "shared-memory budget (the last 1024: slack for aligning the base)");
}  // namespace

template <bool kLimit>
__global__ void __launch_bounds__(DN_THREADS, 1)
    down_swap_kernel(const __grid_constant__ CUtensorMap tm_qd, const __grid_constant__ CUtensorMap tm_sqd,
                     const __grid_constant__ CUtensorMap tm_h, DownParams p) {
  extern __shared__ uint8_t smem_raw[];
  const unsigned long long wlim = kLimit ? p.wait_ns : WAIT_LIMIT_NS;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* misc = smem + DS_OFF_MISC;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 512);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 516);
  int* s_off = reinterpret_cast<int*>(misc + 1024);                   // row tables (GX_TAB_BYTES)
  int* s_cnt = s_off + (NEXP + 2);
  int4* sched = reinterpret_cast<int4*>(misc + 1024 + (GX_TAB_BYTES + 15) / 16 * 16);   // [DS_SCHED_CAP]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t bar0 = smem_u32(bars);
#define PFULL(s) (bar0 + 8u * (s))
#define PEMPTY(s) (bar0 + 8u * (DS_NP + (s)))
#define WFULL(s) (bar0 + 8u * (2 * DS_NP + (s)))
#define WEMPTY(s) (bar0 + 8u * (2 * DS_NP + DS_NW + (s)))
#define HFULL(s) (bar0 + 8u * (2 * DS_NP + 2 * DS_NW + (s)))
#define HEMPTY(s) (bar0 + 8u * (2 * DS_NP + 2 * DS_NW + DS_NH + (s)))
  constexpr int NB = 2 * DS_NP + 2 * DS_NW + 2 * DS_NH;
  static_assert(8 * (NB + 5) <= 512, "barriers overlap the TMEM slot");
#define ACCF(b) (bar0 + 8u * (NB + (b)))
#define ACCE(b) (bar0 + 8u * (NB + 2 + (b)))
  const uint32_t DRAIN = bar0 + 8u * (NB + 4);

  if (tid == 0) {
    for (int s = 0; s < DS_NP; ++s) {
      mbar_init(PFULL(s), 1);
      mbar_init(PEMPTY(s), 256);
    }
    for (int s = 0; s < DS_NW; ++s) {
      mbar_init(WFULL(s), 256);
      mbar_init(WEMPTY(s), 1);
    }
    for (int s = 0; s < DS_NH; ++s) {
      mbar_init(HFULL(s), 1);
      mbar_init(HEMPTY(s), 1);
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
  grid_dep_wait();   // the routing tables and activations come from the kernels before this one
  stage_tables(s_off, p.offsets, p.counts);
  __syncthreads();
  const int ntiles =
      build_schedule(sched, DS_SCHED_CAP, p.blocks, s_off, s_cnt, DS_PAIRS, p.T, p.err, false, BLOCKS_SMALL);
  __syncthreads();
  constexpr int NKB = INTER / 64;   // 8
  uint32_t p_issued = 0;   // packed-tile producer (warp 0) / activation producer (warp 5): K steps issued

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ packed-tile producer
      tma_prefetch_desc(&tm_qd);
      tma_prefetch_desc(&tm_sqd);
      const uint64_t pol = l2_policy_evict_first();   // each weight tile is read once
      uint32_t it = 0;
      bool alive = true;
      for (int tix = 0; tix < ntiles && alive; ++tix) {
        const TileInfo ti = sched_tile(sched, tix);
        if (!ti.ok) { atomicOr(p.err, ERRBIT_BOUNDS); continue; }
        const bool sh = ti.e == SHARED_E;
        const CUtensorMap* mq = sh ? &tm_sqd : &tm_qd;
        const int wrow = (sh ? 0 : ti.e * HID) + ti.mb * (2 * GX_BM);
        for (int kb = 0; kb < NKB; ++kb, ++it) {
          const int s = it % DS_NP;
          if (!mbar_wait(PEMPTY(s), ((it / DS_NP) & 1) ^ 1, p.err, abort_flag, wlim)) { alive = false; break; }
          const uint32_t st = smem_u32(smem + DS_OFF_P + s * DS_P_STAGE);
          mbar_arrive_expect_tx(PFULL(s), DS_P_STAGE);
          tma_load_2d_hint(st, mq, PFULL(s), kb * 8, wrow, pol);
          tma_load_2d_hint(st + GX_P_BYTES, mq, PFULL(s), kb * 8, wrow + GX_BM, pol);
        }
      }
      p_issued = it;
    }
  } else if (warp == 5) {
    if (lane == 0) {
      // ------------------------------------------------ activation-row producer
      tma_prefetch_desc(&tm_h);
      const uint64_t pol = l2_policy_evict_last();    // each block's rows are read by 8 feature pairs
      uint32_t it = 0;
      bool alive = true;
      for (int tix = 0; tix < ntiles && alive; ++tix) {
        const TileInfo ti = sched_tile(sched, tix);
        if (!ti.ok) continue;
        const int nbox = (min(ti.n_rows, GX_SMALL) + GX_XBOX - 1) / GX_XBOX;
        for (int kb = 0; kb < NKB; ++kb, ++it) {
          const int s = it % DS_NH;
          if (!mbar_wait(HEMPTY(s), ((it / DS_NH) & 1) ^ 1, p.err, abort_flag, wlim)) { alive = false; break; }
          const uint32_t st = smem_u32(smem + DS_OFF_H + s * DS_H_STAGE);
          mbar_arrive_expect_tx(HFULL(s), nbox * GX_XBOX * 128);
          for (int j = 0; j < nbox; ++j)
            tma_load_2d_hint(st + j * GX_XBOX * 128, &tm_h, HFULL(s), kb * 64, ti.row0 + j * GX_XBOX, pol);
        }
      }
      p_issued = it;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      const uint32_t idesc = idesc_bf16(128, 2 * GX_BM);
      uint32_t it = 0, tc = 0;
      uint32_t rdy = 0;   // bit 0 / 1: WFULL / HFULL of step `it` seen complete by the last poll
      for (int tix = 0; tix < ntiles; ++tix) {
        const TileInfo ti = sched_tile(sched, tix);
        if (!ti.ok) continue;
        const int buf = tc & 1;
        if (!mbar_wait(ACCE(buf), ((tc >> 1) & 1) ^ 1, p.err, abort_flag, wlim)) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * 256;
        bool alive = true;
        for (int kb = 0; kb < NKB; ++kb, ++it) {
          const int sw = it % DS_NW, sh = it % DS_NH;
          if ((!(rdy & 1u) && !mbar_wait(WFULL(sw), (it / DS_NW) & 1, p.err, abort_flag, wlim)) ||
              (!(rdy & 2u) && !mbar_wait(HFULL(sh), (it / DS_NH) & 1, p.err, abort_flag, wlim))) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = smem_u32(smem + DS_OFF_H + sh * DS_H_STAGE);   // block rows (M)
          const uint32_t b = smem_u32(smem + DS_OFF_W + sw * DS_W_STAGE);   // 256 weight rows (N)
          const uint32_t nx = it + 1;   // the next step's stages are polled while these issue
          rdy = umma_k64_poll(d, sdesc_sw128(a), sdesc_sw128(b), idesc, kb != 0, WFULL(nx % DS_NW),
                              (nx / DS_NW) & 1, HFULL(nx % DS_NH), (nx / DS_NH) & 1);
          umma_commit(WEMPTY(sw));
          umma_commit(HEMPTY(sh));
        }
        if (!alive) break;
        umma_commit(ACCF(buf));
        ++tc;
      }
      umma_commit(DRAIN);
    }
  } else if (warp < 12 && warp != 9) {
    // ------------------------------------------------ dequant (8 warps, one thread per weight row)
    const int wr = (warp - 2 - (warp - 2) / 4) * 32 + lane;   // warps 2-4, 6-8, 10, 11 -> rows 0..255
    const int box = wr >> 7, r = wr & 127;                    // packed box and row inside it
    uint32_t it = 0;
    bool alive = true;
    // the row's 8 scales and 8 biases (one per K step) are loaded one tile ahead
    TileInfo ti;
    ti.ok = false;
    uint4 nsv = make_uint4(0, 0, 0, 0), nbv = nsv;
    auto load_next = [&](int t) {
      if (t >= ntiles) return;
      ti = sched_tile(sched, t);
      if (!ti.ok) return;
      const bool sh = ti.e == SHARED_E;
      const size_t srow = (sh ? 0 : static_cast<size_t>(ti.e) * HID) + static_cast<size_t>(ti.mb) * (2 * GX_BM) + wr;
      nsv = ldg_nc_v4((sh ? p.sd_scales : p.d_scales) + srow * (INTER / GROUP));
      nbv = ldg_nc_v4((sh ? p.sd_biases : p.d_biases) + srow * (INTER / GROUP));
    };
    load_next(0);
    for (int tix = 0; tix < ntiles && alive; ++tix) {
      const bool cur_ok = ti.ok;
      const uint4 sv = nsv, bv = nbv;
      load_next(tix + 1);
      if (!cur_ok) continue;
      const uint32_t swd[4] = {sv.x, sv.y, sv.z, sv.w};
      const uint32_t bwd[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int kb = 0; kb < NKB; ++kb) {
        const int sp = it % DS_NP, sw = it % DS_NW;
        if (!mbar_wait(PFULL(sp), (it / DS_NP) & 1, p.err, abort_flag, wlim) ||
            !mbar_wait(WEMPTY(sw), ((it / DS_NW) & 1) ^ 1, p.err, abort_flag, wlim)) {
          alive = false;
          break;
        }
        ++it;
        const __nv_bfloat162 ms = bf2((kb & 1) ? (swd[kb >> 1] >> 16) : swd[kb >> 1]);
        const __nv_bfloat162 mbv = bf2((kb & 1) ? (bwd[kb >> 1] >> 16) : bwd[kb >> 1]);
        // the row's two 16-byte halves, stored 32-byte swizzled (half c at c ^ bit 2 of the row)
        const uint8_t* P = smem + DS_OFF_P + sp * DS_P_STAGE + box * GX_P_BYTES + r * 32;
        const int hs = ((r >> 2) & 1) << 4;
        const uint4 w0 = *reinterpret_cast<const uint4*>(P + hs), w1 = *reinterpret_cast<const uint4*>(P + (16 ^ hs));
        // the packed words are in registers; the next TMA write into this stage is an
        // async-proxy access, so the generic reads are fenced before the release
        fence_proxy_async_smem();
        mbar_arrive(PEMPTY(sp));
        uint8_t* W = smem + DS_OFF_W + sw * DS_W_STAGE;
        st_shared_v4(W + sw128_off(wr, 0), dequant8(w0.x, ms, mbv));
        st_shared_v4(W + sw128_off(wr, 1), dequant8(w0.y, ms, mbv));
        st_shared_v4(W + sw128_off(wr, 2), dequant8(w0.z, ms, mbv));
        st_shared_v4(W + sw128_off(wr, 3), dequant8(w0.w, ms, mbv));
        st_shared_v4(W + sw128_off(wr, 4), dequant8(w1.x, ms, mbv));
        st_shared_v4(W + sw128_off(wr, 5), dequant8(w1.y, ms, mbv));
        st_shared_v4(W + sw128_off(wr, 6), dequant8(w1.z, ms, mbv));
        st_shared_v4(W + sw128_off(wr, 7), dequant8(w1.w, ms, mbv));
        fence_proxy_async_smem();
        mbar_arrive(WFULL(sw));
      }
    }
  } else if (warp >= 12) {
    // ------------------------------------------------ epilogue (4 warps): y rows straight from TMEM
    const int q = warp & 3;                       // TMEM lane quarter = block rows 32q .. 32q+31
    const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const int row = 32 * q + lane;
    uint32_t tc = 0;
    for (int tix = 0; tix < ntiles; ++tix) {
      const TileInfo ti = sched_tile(sched, tix);
      if (!ti.ok) continue;
      const int buf = tc & 1;
      const bool got = mbar_wait(ACCF(buf), (tc >> 1) & 1, p.err, abort_flag, wlim);
      if (!__all_sync(0xffffffffu, got)) break;   // tcgen05.ld below needs the whole warp
      tc_fence_after();
      __nv_bfloat16* yrow = p.y + static_cast<size_t>(ti.row0 + row) * HID + ti.mb * (2 * GX_BM);
      const bool mine = row < ti.n_rows;          // rows past the block's end belong to other blocks
#pragma unroll 1
      for (int c0 = 0; c0 < 2 * GX_BM; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tl + buf * 256 + c0, v);
        tmem_ld_wait();
        if (c0 + 32 == 2 * GX_BM) {               // last read: the MMA may reuse this buffer
          tc_fence_before();
          mbar_arrive(ACCE(buf));
        }
        if (mine) {
          uint32_t w[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) w[k] = pack_bf16x2(v[2 * k], v[2 * k + 1]);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            *reinterpret_cast<uint4*>(yrow + c0 + 8 * k) = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
        }
      }
      ++tc;
    }
  }
  // warp 9 has no role

  tc_fence_before();
  __syncthreads();
  if ((warp == 0 || warp == 5) && lane == 0 && *abort_flag) {
    // a launch that gave up (whichever role did): the tiles still in flight land before
    // the CTA's shared memory goes away (the latest phase of each stage)
    if (warp == 0)
      for (uint32_t i = (p_issued > DS_NP ? p_issued - DS_NP : 0); i < p_issued; ++i)
        drain_wait(PFULL(i % DS_NP), (i / DS_NP) & 1);
    else
      for (uint32_t i = (p_issued > DS_NH ? p_issued - DS_NH : 0); i < p_issued; ++i)
        drain_wait(HFULL(i % DS_NH), (i / DS_NH) & 1);
  }
  if (warp == 1) {
    tc_fence_after();
    if (lane == 0) drain_wait(DRAIN, 0);
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
#undef PFULL
#undef PEMPTY
#undef WFULL
#undef WEMPTY
#undef HFULL
#undef HEMPTY
#undef ACCF
#undef ACCE
}

cudaError_t launch_down(const CUtensorMap& qd, const CUtensorMap& sqd, const CUtensorMap& hmap,
                        const CUtensorMap& ymap, const DownParams& p, int grid, cudaStream_t s) {
  return launch_pdl(p.wait_ns == WAIT_LIMIT_NS ? down_kernel<false> : down_kernel<true>, grid, DN_THREADS, DN_SMEM,
                    s, qd, sqd, hmap, ymap, p);
}

cudaError_t launch_down_swap(const CUtensorMap& qd, const CUtensorMap& sqd, const CUtensorMap& hmap, const DownParams& p,
                             int grid, cudaStream_t s) {
  return launch_pdl(p.wait_ns == WAIT_LIMIT_NS ? down_swap_kernel<false> : down_swap_kernel<true>, grid, DN_THREADS,
                    DS_SMEM, s, qd, sqd, hmap, p);
}

cudaError_t set_down_attributes() {
  cudaError_t e = cudaFuncSetAttribute(down_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, DN_SMEM);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(down_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, DN_SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(down_swap_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, DS_SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(down_swap_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, DS_SMEM);
  return e;
}

}  // namespace moe
