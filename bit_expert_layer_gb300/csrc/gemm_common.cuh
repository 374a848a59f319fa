// gemm_common.cuh -- helpers shared by the grouped expert GEMM kernels (gate/up and
// down): the device-side tile lookup, staging of the tile tables in shared memory,
// bf16 pair construction, bounded teardown waits and the pipeline-trace counters.
#pragma once

#include "common.cuh"

namespace moe {

struct TileInfo {
  int e, mb, row0, n_rows;
  bool ok;   // tables consistent: every role skips a bad tile the same way
};

__device__ __forceinline__ TileInfo tile_info(const int* tiles, const int* offsets, const int* counts, int tile,
                                              int mblk, int T) {
  // the tables live in shared memory (stage_tables): a binary search over global memory
  // would be nine dependent L2 round trips per tile and role
  int lo = 0, hi = NEXP;   // largest e in [0, 256] with tiles[e] <= tile
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tiles[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  TileInfo ti;
  ti.e = lo;
  const int local = tile - tiles[lo];
  const int nb = local / mblk;
  ti.mb = local - nb * mblk;
  ti.row0 = offsets[lo] + nb * GX_BN;
  ti.n_rows = min(GX_BN, counts[lo] - nb * GX_BN);
  ti.ok = ti.n_rows >= 1 && ti.row0 >= 0 && ti.row0 + ti.n_rows <= 9 * T && local >= 0;
  return ti;
}

// Copy the tile prefix [258], row offsets [258] and row counts [257] into shared memory.
__device__ __forceinline__ void stage_tables(int* s, const int* tiles, const int* offsets, const int* counts) {
  for (int i = threadIdx.x; i < NEXP + 2; i += blockDim.x) {
    s[i] = __ldg(tiles + i);
    s[(NEXP + 2) + i] = __ldg(offsets + i);
    s[2 * (NEXP + 2) + i] = (i <= NEXP) ? __ldg(counts + i) : 0;
  }
}

__device__ __forceinline__ __nv_bfloat162 bf2(uint32_t bits16) {
  const uint32_t v = (bits16 & 0xFFFFu) * 0x00010001u;
  return *reinterpret_cast<const __nv_bfloat162*>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint8_t* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

// Pipeline tracing (MOE_PIPE_PROF=1 on the host): a role adds the clock cycles it spends
// in each barrier wait, and its whole running time, to per-kernel counters.
//   slot 0..2  MMA issuer: waiting for the accumulator to drain / dequant / TMA; 3 total
//   slot 4, 5  TMA producer: waiting for a free stage; total
//   slot 6, 7  one dequant thread: waiting for the TMA; total
//   slot 8, 9  one epilogue thread: waiting for the accumulator; total
//   slot 10    tiles processed (MMA issuer)
__device__ __forceinline__ bool mbar_wait_t(uint32_t bar, uint32_t parity, unsigned int* err,
                                            volatile int* abort_flag, unsigned long long& acc, bool on) {
  if (!on) return mbar_wait(bar, parity, err, abort_flag);
  const unsigned long long t0 = clock64();
  const bool r = mbar_wait(bar, parity, err, abort_flag);
  acc += clock64() - t0;
  return r;
}

__device__ __forceinline__ void pipe_flush(unsigned long long* pipe, int slot0, const unsigned long long* pc,
                                           int n, unsigned long long total, int total_slot) {
  if (!pipe) return;
  for (int i = 0; i < n; ++i) atomicAdd(pipe + slot0 + i, pc[i]);
  atomicAdd(pipe + total_slot, total);
}

// Bounded wait used only while tearing down after an abort (ignores the abort flag).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity) && globaltimer_ns() - t0 < WAIT_LIMIT_NS) {
  }
}

}  // namespace moe
