// gemm_common.cuh -- helpers shared by the grouped expert GEMM kernels (gate/up and
// down): the device-side tile schedule, staging of the row tables in shared memory,
// bf16 pair construction, bounded teardown waits and the pipeline-trace counters.
#pragma once

#include "common.cuh"

namespace moe {

struct TileInfo {
  int e, mb, row0, n_rows;
  bool ok;   // tables consistent: every role skips a bad tile the same way
};

// The ordered token-block list built by route_scan_kernel: blocks[0] = its length n,
// blocks[1] = n_big, the number of blocks of more than GX_SMALL rows (they come first:
// every full block, then the partial blocks largest first), entries from blocks[2]
// (expert | (block index << 9)).  Tile `tile` = token block b0 + tile / mblk x weight row
// block tile % mblk.  The offsets and counts live in shared memory (stage_tables).
__device__ __forceinline__ TileInfo tile_info(const int* blocks, const int* offsets, const int* counts, int tile,
                                              int mblk, int T, int b0 = 0) {
  const int j = b0 + tile / mblk;
  const int v = __ldg(blocks + 2 + j);
  TileInfo ti;
  ti.e = v & 511;
  ti.mb = tile - (j - b0) * mblk;
  const int nb = v >> 9;
  const int e = ti.e <= NEXP ? ti.e : 0;
  ti.row0 = offsets[e] + nb * GX_BN;
  ti.n_rows = min(GX_BN, counts[e] - nb * GX_BN);
  ti.ok = ti.e <= NEXP && nb >= 0 && ti.n_rows >= 1 && ti.row0 >= 0 && ti.row0 + ti.n_rows <= 9 * T;
  return ti;
}

// This CTA's share of a grouped GEMM's tiles, decoded once at kernel start, one thread
// per tile, into a shared-memory schedule that every role reads.  Round i gives CTA b
// tile i G + b, or with `snake` i G + G - 1 - b for odd i, so that with the token blocks
// ordered by size (full blocks first, then the partial ones largest first) each CTA's
// sum of tile sizes evens out and the last, incomplete round holds the smallest tiles
// (gate/up, about 18 tiles per CTA at T = 16384: measured faster; down, about 73 tiles
// per CTA: the straight order measured faster).  A record is {expert, row block, first row, rows};
// rows = 0 marks a tile whose tables are inconsistent, which every role skips.  More
// tiles than `cap` is a bounds error (the host sizes the grid so that it cannot
// happen).  `part` picks the blocks: all of them, the big ones (more than GX_SMALL rows)
// or the small ones.  Returns the number of records.
enum BlockPart { BLOCKS_ALL, BLOCKS_BIG, BLOCKS_SMALL };
__device__ __forceinline__ int build_schedule(int4* sched, int cap, const int* blocks, const int* s_off,
                                              const int* s_cnt, int mblk, int T, unsigned int* err,
                                              bool snake, BlockPart part) {
  int nblocks = __ldg(blocks), nbig = __ldg(blocks + 1);
  // at most ceil(8T / 256) + min(8T, 256) routed blocks and ceil(T / 256) shared ones
  if (nblocks < 0 || nblocks > (8 * T + GX_BN - 1) / GX_BN + min(8 * T, NEXP) + (T + GX_BN - 1) / GX_BN ||
      nbig < 0 || nbig > nblocks) {
    if (threadIdx.x == 0) atomicOr(err, ERRBIT_BOUNDS);
    nblocks = 0;
    nbig = 0;
  }
  const int b0 = part == BLOCKS_SMALL ? nbig : 0;
  const int b1 = part == BLOCKS_BIG ? nbig : nblocks;
  const int total = (b1 - b0) * mblk;
  const int b = static_cast<int>(blockIdx.x), g = static_cast<int>(gridDim.x);
  const int rounds = total / g, rem = total - rounds * g;
  const int n = rounds + (((snake && (rounds & 1)) ? g - 1 - b : b) < rem ? 1 : 0);
  if (n > cap && threadIdx.x == 0) atomicOr(err, ERRBIT_BOUNDS);
  const int m = min(n, cap);
  for (int i = threadIdx.x; i < m; i += blockDim.x) {
    const TileInfo ti = tile_info(blocks, s_off, s_cnt, i * g + ((snake && (i & 1)) ? g - 1 - b : b), mblk, T, b0);
    sched[i] = ti.ok ? make_int4(ti.e, ti.mb, ti.row0, ti.n_rows) : make_int4(0, 0, 0, 0);
  }
  return m;
}

__device__ __forceinline__ TileInfo sched_tile(const int4* sched, int i) {
  const int4 r = sched[i];
  TileInfo ti;
  ti.e = r.x;
  ti.mb = r.y;
  ti.row0 = r.z;
  ti.n_rows = r.w;
  ti.ok = r.w > 0;
  return ti;
}

// Copy the row offsets [258] and row counts [257] into shared memory: s[0..257], s[258..].
__device__ __forceinline__ void stage_tables(int* s, const int* offsets, const int* counts) {
  for (int i = threadIdx.x; i < NEXP + 2; i += blockDim.x) {
    s[i] = __ldg(offsets + i);
    s[(NEXP + 2) + i] = (i <= NEXP) ? __ldg(counts + i) : 0;
  }
}

__device__ __forceinline__ __nv_bfloat162 bf2(uint32_t bits16) {
  const uint32_t v = (bits16 & 0xFFFFu) * 0x00010001u;
  return *reinterpret_cast<const __nv_bfloat162*>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint8_t* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

// MMA issue with the next step's barrier polls folded in.  On sm_103a an mbarrier poll
// holds the issuing thread for about 200 cycles even when the phase completed long ago:
// polling ahead of the MMAs of the current step, and reading the result only after those
// are issued, hides part of that, and fewer barriers per K step hide the rest.  The poll
// is a non-blocking test_wait (acquire, CTA scope); a stage it finds not yet full is
// waited for in the ordinary bounded way.  Descriptors advance 32 bytes (16 bf16) of K per
// MMA: +2 in the 16-byte address field.  Returns bit 0 = the barrier already complete.
//
// One K step of 64 into two accumulators (gate, up) that share the B operand; one
// barrier covers both operands of the next step.
__device__ __forceinline__ uint32_t umma_k64_x2_poll(uint32_t d0, uint32_t d1, uint64_t a0, uint64_t a1, uint64_t b,
                                                     uint32_t idesc, uint32_t accumulate, uint32_t nbar,
                                                     uint32_t npar) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pa, pt, q0;\n\t.reg .b64 x0, x1, xb;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q0, [%8], %9;\n\t"
      "setp.ne.b32 pa, %7, 0;\n\t"
      "setp.ne.b32 pt, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], %3, %5, %6, pa;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%2], %4, %5, %6, pa;\n\t"
      "add.s64 x0, %3, 2;\n\tadd.s64 x1, %4, 2;\n\tadd.s64 xb, %5, 2;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], x0, xb, %6, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%2], x1, xb, %6, pt;\n\t"
      "add.s64 x0, %3, 4;\n\tadd.s64 x1, %4, 4;\n\tadd.s64 xb, %5, 4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], x0, xb, %6, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%2], x1, xb, %6, pt;\n\t"
      "add.s64 x0, %3, 6;\n\tadd.s64 x1, %4, 6;\n\tadd.s64 xb, %5, 6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], x0, xb, %6, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%2], x1, xb, %6, pt;\n\t"
      "selp.u32 %0, 1, 0, q0;\n\t}"
      : "=r"(r)
      : "r"(d0), "r"(d1), "l"(a0), "l"(a1), "l"(b), "r"(idesc), "r"(accumulate), "r"(nbar), "r"(npar)
      : "memory");
  return r;
}

// One K step of 64 into one accumulator; one barrier covers both operands of the next step.
__device__ __forceinline__ uint32_t umma_k64_poll1(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                                   uint32_t accumulate, uint32_t nbar, uint32_t npar) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pa, pt, q0;\n\t.reg .b64 x0, xb;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q0, [%6], %7;\n\t"
      "setp.ne.b32 pa, %5, 0;\n\t"
      "setp.ne.b32 pt, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], %2, %3, %4, pa;\n\t"
      "add.s64 x0, %2, 2;\n\tadd.s64 xb, %3, 2;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], x0, xb, %4, pt;\n\t"
      "add.s64 x0, %2, 4;\n\tadd.s64 xb, %3, 4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], x0, xb, %4, pt;\n\t"
      "add.s64 x0, %2, 6;\n\tadd.s64 xb, %3, 6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], x0, xb, %4, pt;\n\t"
      "selp.u32 %0, 1, 0, q0;\n\t}"
      : "=r"(r)
      : "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(nbar), "r"(npar)
      : "memory");
  return r;
}

// One K step of 64 into one accumulator; two barriers (weights, activations) cover the
// next step's operands: bit 0 / bit 1 of the result.
__device__ __forceinline__ uint32_t umma_k64_poll(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                                  uint32_t accumulate, uint32_t nbar0, uint32_t npar0,
                                                  uint32_t nbar1, uint32_t npar1) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pa, pt, q0, q1;\n\t.reg .b64 x0, xb;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q0, [%6], %7;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q1, [%8], %9;\n\t"
      "setp.ne.b32 pa, %5, 0;\n\t"
      "setp.ne.b32 pt, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], %2, %3, %4, pa;\n\t"
      "add.s64 x0, %2, 2;\n\tadd.s64 xb, %3, 2;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], x0, xb, %4, pt;\n\t"
      "add.s64 x0, %2, 4;\n\tadd.s64 xb, %3, 4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], x0, xb, %4, pt;\n\t"
      "add.s64 x0, %2, 6;\n\tadd.s64 xb, %3, 6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], x0, xb, %4, pt;\n\t"
      "selp.u32 %0, 1, 0, q0;\n\t"
      "@q1 or.b32 %0, %0, 2;\n\t}"
      : "=r"(r)
      : "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(nbar0), "r"(npar0), "r"(nbar1), "r"(npar1)
      : "memory");
  return r;
}

// Pipeline tracing (MOE_PIPE_PROF=1 on the host): a role adds the clock cycles it spends
// in each barrier wait, and its whole running time, to per-kernel counters.
//   slot 0..2  MMA issuer: waiting for the accumulator to drain / dequant / TMA (gate/up:
//              slot 1 = both operands, slot 2 unused); 3 total
//   slot 4, 5  TMA producer: waiting for a free stage; total
//   slot 6, 7  one dequant thread: waiting for the TMA; total
//   slot 8, 9  one epilogue thread: waiting for the accumulator; total
//   slot 10    tiles processed (MMA issuer)
__device__ __forceinline__ bool mbar_wait_t(uint32_t bar, uint32_t parity, unsigned int* err,
                                            volatile int* abort_flag, unsigned long long limit_ns,
                                            unsigned long long& acc, bool on) {
  if (!on) return mbar_wait(bar, parity, err, abort_flag, limit_ns);
  const unsigned long long t0 = clock64();
  const bool r = mbar_wait(bar, parity, err, abort_flag, limit_ns);
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
