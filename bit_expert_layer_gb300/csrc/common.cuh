// common.cuh -- sm_103a building blocks shared by the layer's kernels: mbarriers,
// TMA tile loads, tcgen05 (TMEM allocation, MMA, commit, loads), the shared-memory
// matrix descriptor for 128-byte-swizzled K-major bf16 tiles, bounded waits that
// record a timeout instead of hanging, and the constants of the one layer shape.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// ----------------------------------------------------------------- layer shape
constexpr int HID = 2048;        // hidden size
constexpr int NEXP = 256;        // routed experts
constexpr int TOPK = 8;          // experts kept per token
constexpr int INTER = 512;       // routed expert intermediate size
constexpr int SH_INTER = 512;    // shared expert intermediate size
constexpr int GROUP = 64;        // quantisation group along the input dim
constexpr int SHARED_E = NEXP;   // the shared expert's index in the row tables and token blocks

// ----------------------------------------------------------------- device error word
enum : uint32_t { ERRBIT_TIMEOUT = 1u, ERRBIT_BOUNDS = 2u };
// Default time limit of a bounded wait (2 s).  The limit of the waits a launch makes on
// the work of other threads is a launch parameter (moe_set_wait_limit_ns can shorten it,
// to exercise the give-up path); the waits of the teardown after a give-up, which let
// copies and MMAs already in flight land before the CTA exits, always use this one.
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;

// ----------------------------------------------------------------- kernel geometry
// Router (prefill): 128 tokens per CTA (M), the 256 experts on N.
constexpr int RT_BM = 128;
constexpr int RT_STAGES = 4;
constexpr int RT_A_BYTES = RT_BM * 64 * 2;          // 16 KB  x tile
constexpr int RT_B_BYTES = NEXP * 64 * 2;           // 32 KB  router tile
constexpr int RT_STAGE_BYTES = RT_A_BYTES + RT_B_BYTES;
constexpr int RT_SEGS = 4;                          // expert segments scanned by separate warps
constexpr int RT_CAND_BYTES = (RT_SEGS - 1) * 8 * RT_BM * 8;   // top-8 lists of segments 1-3
constexpr int RT_SMEM = RT_STAGES * RT_STAGE_BYTES + 1024 + 3072 + RT_CAND_BYTES;
constexpr int RT_THREADS = 128 * RT_SEGS;
// cluster router: a cluster of S CTAs per 128-token block, each over a part of K (48 KB
// stages); the partial logits meet in distributed shared memory.  S = 4 up to RC_MAX_T
// tokens, S = 2 up to RC2_MAX_T; above, router_prefill_kernel (one CTA per block, whole K)
constexpr int RC_MAX_T = 4096;
constexpr int RC2_MAX_T = 8192;
constexpr int RC_STAGES = 4;
__host__ __device__ constexpr int rc_threads(int S) { return 4 * (RT_BM / S); }
__host__ __device__ constexpr int rc_misc(int S) { return 256 + NEXP * 8 + 2 * 4 * TOPK * (RT_BM / S) * 4; }
__host__ __device__ constexpr int rc_smem(int S) { return RC_STAGES * RT_STAGE_BYTES + 1024 + rc_misc(S) + 1024; }


// Grouped expert GEMMs: 128 weight rows (M) x up to 256 tokens (N) per tile, K step 64
// (= one quantisation group).
constexpr int GX_BM = 128;
constexpr int GX_BN = 256;
constexpr int GX_XBOX = 32;                         // token rows per TMA box
constexpr int GX_A_BYTES = GX_BM * 64 * 2;          // 16 KB dequantised tile
constexpr int GX_X_BYTES = GX_BN * 64 * 2;          // 32 KB activation tile
constexpr int GX_P_BYTES = GX_BM * 32;              //  4 KB packed 4-bit tile (8 words/row)
// gate/up: three rings of different depth -- packed 4-bit tiles (gate + up, 8 KB, fetched
// from HBM, deepest), activation tiles (32 KB, mostly from L2), dequantised tiles (gate +
// up, 32 KB, only between dequant and MMA)
constexpr int GU_NP = 5;
constexpr int GU_NX = 3;
constexpr int GU_NA = 2;
constexpr int GU_P_STAGE = 2 * GX_P_BYTES;
constexpr int GU_A_STAGE = 2 * GX_A_BYTES;
constexpr int GU_RINGS = GU_NA * GU_A_STAGE + GU_NX * GX_X_BYTES + GU_NP * GU_P_STAGE;
constexpr int GX_TAB_BYTES = 3 * (NEXP + 2) * 4 + 128;   // row tables staged in shared memory (one spare)
// + alignment slack, barriers (512 B), row tables
constexpr int GU_GW = 6;                            // activation gather warps
constexpr int GU_GROWS = (GX_BN + GU_GW - 1) / GU_GW + 4;   // token ids per gather warp and tile
// per-CTA tile schedules (16 bytes a tile): tiles per CTA at the largest token count and
// 152 SMs are 68 (gate/up) and 270 (down); the host checks the bound per launch
constexpr int GU_SCHED_CAP = 96;
constexpr int DN_SCHED_CAP = 288;
// gate/up epilogue staging: per epilogue warp GU_STG_BUFS tiles of 32 rows x 32 features
constexpr int GU_STG_BUFS = 2;
constexpr int GU_STG_BYTES = 4 * GU_STG_BUFS * 32 * 32 * 2;
constexpr int GU_SMEM = GU_RINGS + 1024 + 512 + GX_TAB_BYTES + GU_GW * GU_GROWS * 4 + GU_SCHED_CAP * 16 + 1024 + GU_STG_BYTES;
constexpr int GU_THREADS = (14 + GU_GW) * 32;   // packed producer, MMA, 8 dequant, 4 epilogue, gather warps
constexpr int GU_MBLK = INTER / GX_BM;              // 4 row blocks per matrix
// gate/up tiles of at most this many tokens run with the operands swapped: tokens on the
// MMA's M side (128, padded), the tile's 128 gate and 128 up weight rows on its N side
constexpr int GU_SWAP_ROWS = 128;
// down: rings of packed tiles (4 KB), activation tiles (32 KB; the deepest ring, since the
// h blocks mostly come from DRAM: 4 stages measured 3.5% faster at T=16384 than 3) and
// dequantised tiles (16 KB); double-buffered accumulator
constexpr int DN_NP = 8;
constexpr int DN_NX = 4;
constexpr int DN_NA = 2;
constexpr int DN_RINGS = DN_NP * GX_P_BYTES + DN_NX * GX_X_BYTES + DN_NA * GX_A_BYTES;
// epilogue staging: per epilogue warp DN_STG_BUFS buffers of 32 rows x 32 features (bf16)
constexpr int DN_STG_BUFS = 2;
constexpr int DN_STG_BYTES = 4 * DN_STG_BUFS * 32 * 32 * 2;
// + alignment slack, barriers and words (1 KB), staging, row tables
constexpr int DN_SMEM = DN_RINGS + 1024 + 1024 + DN_STG_BYTES + GX_TAB_BYTES + 16 + DN_SCHED_CAP * 16;
static_assert(GU_SMEM <= 232448 && DN_SMEM <= 232448, "shared memory per CTA exceeds 227 KB");
// down GEMM of the small token blocks (at most GX_SMALL rows: an expert's partial last
// block), operands swapped: rings of packed tiles (256 weight rows, 8 KB), dequantised
// weights (256 rows, 32 KB) and activation rows (128 rows, 16 KB)
constexpr int GX_SMALL = 128;
// Token counts up to which the small blocks go to the swapped kernel: a swapped K step (4
// MMAs of 256 columns) takes about twice as long as a K step of a few columns, so halving
// the steps pays only while most blocks are small (measured: T = 32 and 512 faster, 4096
// and 16384 slower)
constexpr int DS_MAX_T = 1024;
// prefill of at most this many tokens: the expert GEMMs run as mma.sync GEMVs
// (gemv_small.cu), every expert block holding at most GV_MAX_T rows
constexpr int GV_MAX_T = 192;
constexpr int DS_NP = 8;
constexpr int DS_NW = 3;
constexpr int DS_NH = 3;
constexpr int DS_P_STAGE = 2 * GX_P_BYTES;
constexpr int DS_W_STAGE = 2 * GX_A_BYTES;
constexpr int DS_H_STAGE = GX_SMALL * 64 * 2;
constexpr int DS_PAIRS = HID / (2 * GX_BM);          // 8 pairs of row blocks (256 features)
constexpr int DS_SCHED_CAP = 64;                     // at most 257 small blocks x 8 pairs: 14 per CTA on 152 SMs
// + alignment slack, barriers and words (1 KB), row tables (16-byte rounded), schedule
constexpr int DS_SMEM = DS_NP * DS_P_STAGE + DS_NW * DS_W_STAGE + DS_NH * DS_H_STAGE + 1024 + 1024 +
                        (GX_TAB_BYTES + 15) / 16 * 16 + DS_SCHED_CAP * 16;
static_assert(DS_SMEM <= 232448, "shared memory per CTA exceeds 227 KB");
constexpr int DN_THREADS = 512;   // 16 warps: producers, MMA, 8 dequant, 4 epilogue, one spare
constexpr int DN_MBLK = HID / GX_BM;                // 16 row blocks

// scatter: per router block of 128 tokens (1024 slots), SC_SPLIT CTAs; the first also
// places the slots, all of them copy their share of the tokens
constexpr int SC_THREADS = 256;
constexpr int SC_SPLIT = 4;
constexpr int SCAN_FUSE_NBLK = 128;  // router blocks (T <= 16384) up to which the scatter does the scan's work

// decode path (T <= 8)
constexpr int DEC_MAX_T = 8;
constexpr int DEC_MAX_ACTIVE = 8 * DEC_MAX_T + 1;

// ----------------------------------------------------------------- small helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

// ----------------------------------------------------------------- dependent launch
// The prefill kernels are launched with programmatic stream serialisation: the next
// kernel of the stream is launched as the CTAs of the one before it finish, before that
// kernel's memory writes are flushed, and sets up its barriers and TMEM meanwhile.
// grid_dep_wait() holds the calling thread until every earlier kernel of the stream has
// completed and its writes are visible; each kernel calls it, in every thread, before its
// first access to memory that another kernel writes or reads (activations, routing
// tables, workspace).  (No kernel signals its dependents early: CTAs of the next kernel
// that wait on SMs while this one runs measured slower than letting them in at exit.)
// Launched without the attribute, the wait does nothing.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ----------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase of parity `parity`.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Below this limit (the device timer's resolution, about 1 us) a bounded wait gives up
// at once if its phase is not already complete.
constexpr unsigned long long WAIT_LIMIT_IMMEDIATE_NS = 1000ull;

// Wait for the phase of parity `parity` to complete.  Gives up after limit_ns (or as
// soon as another thread of the CTA has given up, via *abort): records ERRBIT_TIMEOUT in
// the device error word and returns false.  Never hangs.  Under a limit below the timer's
// resolution the thread is not suspended at all: the wait gives up unless the phase is
// already complete.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned int* err,
                                          volatile int* abort_flag, unsigned long long limit_ns) {
  const bool imm = limit_ns < WAIT_LIMIT_IMMEDIATE_NS;
  if (imm ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    if (!imm) {
#pragma unroll 1
      for (int i = 0; i < 32; ++i)
        if (mbar_try_wait(bar, parity)) return true;
      if (*abort_flag) return false;
    }
    if (imm || globaltimer_ns() - t0 > limit_ns) {
      atomicOr(err, ERRBIT_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}

// ----------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 2-D tiled load into shared memory, completion counted on `bar` (bytes).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0,
                                            int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
      "[%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// The same load with an L2 eviction-priority policy (from l2_policy_*).
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0,
                                                 int c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, "
      "%4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}
// Shared -> global 2D tile store (bulk group); the smem source must stay untouched until
// tma_store_wait_read says the copy has read it.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(c0), "r"(c1)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// The same store with an L2 eviction-priority policy (from l2_policy_*).
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap* map, uint32_t src, int c0, int c1,
                                                  uint64_t policy) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(c0), "r"(c1), "l"(policy)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void tma_store_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// L2 policies: data read once (streamed weights) and data read again soon (activations)
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ----------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate, one CTA.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 consecutive fp32 columns: thread i gets lane (base lane + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr));
}
// 16 lanes x 32 columns in the MMA fragment layout: thread t gets lanes base + t/4 and
// base + 8 + t/4, columns 8g + 2(t%4) and 8g + 2(t%4) + 1 for g = 0..3, in the order
// r[4g] = (t/4, 8g+2(t%4)), r[4g+1] = (t/4, +1), r[4g+2] = (8+t/4, 8g+2(t%4)), r[4g+3] = (8+t/4, +1).
__device__ __forceinline__ void tmem_ld16x256(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// Four 8x8 bf16 matrices stored transposed: register i of thread t holds row t/4,
// columns 2(t%4), 2(t%4)+1 of matrix i; thread 8i + k gives the shared address of stored
// row k of matrix i, which receives column k of the source.
__device__ __forceinline__ void stmatrix_x4_trans(uint32_t addr, uint32_t m0, uint32_t m1, uint32_t m2, uint32_t m3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(m0), "r"(m1),
               "r"(m2), "r"(m3)
               : "memory");
}
// Two fp32 values (raw bits) rounded to a bf16 pair, `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ void tmem_ld1(uint32_t taddr, uint32_t& r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
}

// Shared-memory matrix descriptor for a K-major bf16 tile stored with the 128-byte
// swizzle: rows of 128 bytes (64 elements), 8-row atoms of 1024 bytes, atoms
// contiguous.  The tile base must be 1024-byte aligned; advancing along K inside the
// 128-byte row is done by adding the byte offset to the start address.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address, 16-byte units
  d |= static_cast<uint64_t>(1) << 16;                    // leading-dim offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;            // stride between 8-row atoms
  d |= static_cast<uint64_t>(1) << 46;                    // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;                    // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16 with bf16 A and B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Byte offset of 16-byte chunk `c` (0..7) of row `r` in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

// ----------------------------------------------------------------- 4-bit dequant
// One packed word holds codes q0..q7 (low nibble first).  Returns the eight weights
// w = scale * q + bias as bf16, each rounded once (fma.rn.bf16x2 of the exact code),
// stored in the order (q0,q4),(q1,q5),(q2,q6),(q3,q7): the same K interleave that the
// activation tiles are written in.  `ms` = (scale, scale), `mb` = (bias, bias).
__device__ __forceinline__ uint4 dequant8(uint32_t w, __nv_bfloat162 ms, __nv_bfloat162 mb) {
  const __nv_bfloat162 k128 = __halves2bfloat162(__ushort_as_bfloat16(0x4300), __ushort_as_bfloat16(0x4300));
  uint32_t p[4];
  p[0] = (w & 0x000F000Fu) | 0x43004300u;
  p[1] = ((w >> 4) & 0x000F000Fu) | 0x43004300u;
  p[2] = ((w >> 8) & 0x000F000Fu) | 0x43004300u;
  p[3] = ((w >> 12) & 0x000F000Fu) | 0x43004300u;
  uint4 o;
  uint32_t* op = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&p[i]);   // 128 + q, exact
    v = __hsub2(v, k128);                                              // q, exact
    __nv_bfloat162 r = __hfma2(v, ms, mb);                             // one rounding
    op[i] = *reinterpret_cast<uint32_t*>(&r);
  }
  return o;
}

// Reorder eight consecutive bf16 (e0..e7 in four words) into the interleave above.
__device__ __forceinline__ uint4 interleave8(uint4 v) {
  uint4 o;
  o.x = __byte_perm(v.x, v.z, 0x5410);   // e0, e4
  o.y = __byte_perm(v.x, v.z, 0x7632);   // e1, e5
  o.z = __byte_perm(v.y, v.w, 0x5410);   // e2, e6
  o.w = __byte_perm(v.y, v.w, 0x7632);   // e3, e7
  return o;
}

// Column position of feature f inside an interleaved row (inverse of the order above).
__host__ __device__ __forceinline__ int ilv_pos(int f) {
  const int i = f & 7;
  return (f & ~7) | (i < 4 ? 2 * i : 2 * (i - 4) + 1);
}

// Weight row held by row r of a dequantised gate/up tile: rows are permuted inside each
// group of 8 so that the accumulator's lanes come out in the order of ilv_pos (lane r
// holds the feature whose interleaved column is r): lanes 0..7 of a group hold features
// 0, 4, 1, 5, 2, 6, 3, 7.
__host__ __device__ __forceinline__ int ilv_row(int r) { return (r & ~7) | ((r & 1) << 2) | ((r & 7) >> 1); }

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// RMSNorm of one token row over a CTA of 256 threads, thread c holding elements
// 8c..8c+7 (bf16 pairs in v): returns 1 / sqrt(mean(x^2) + 1e-6) in every thread.  The
// fp32 sum of squares has one fixed order (each thread's 8 elements in order, a
// butterfly over the lanes, the 8 warps in order), shared by every kernel that
// normalises a layer input, so they all give the same bits.  s_warp: 8 floats of shared
// memory; contains two __syncthreads.
__device__ __forceinline__ float row_inv_rms(const uint4& v, float* s_warp) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    ss = fmaf(bf16lo(u[i]), bf16lo(u[i]), ss);
    ss = fmaf(bf16hi(u[i]), bf16hi(u[i]), ss);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = ss;
  __syncthreads();
  float t = 0.0f;
#pragma unroll
  for (int w = 0; w < 8; ++w) t += s_warp[w];
  __syncthreads();
  return 1.0f / sqrtf(t / static_cast<float>(HID) + 1e-6f);
}
// Dot product of one token row with a weight row over a CTA of 256 threads, thread c
// holding elements 8c..8c+7 of both: the same fixed order as row_inv_rms (each thread's 8
// products in order, a butterfly over the lanes, the 8 warps in order); the result in
// every thread.  s_warp: 8 floats of shared memory; contains two __syncthreads.
__device__ __forceinline__ float row_dot(const uint4& v, const uint4& g, float* s_warp) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
  const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
  float d = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    d = fmaf(bf16lo(u[i]), bf16lo(gw[i]), d);
    d = fmaf(bf16hi(u[i]), bf16hi(gw[i]), d);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
  if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = d;
  __syncthreads();
  float t = 0.0f;
#pragma unroll
  for (int w = 0; w < 8; ++w) t += s_warp[w];
  __syncthreads();
  return t;
}
// bf16(x * r * w) for the 8 elements of v and of the matching norm weights g.
__device__ __forceinline__ uint4 rms_scale8(const uint4& v, const uint4& g, float r) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
  const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 b2 = __floats2bfloat162_rn(bf16lo(u[i]) * r * bf16lo(gw[i]), bf16hi(u[i]) * r * bf16hi(gw[i]));
    o[i] = *reinterpret_cast<const uint32_t*>(&b2);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

}  // namespace moe
