// gemv_small.cu -- the grouped expert GEMMs of a short prefill (at most GV_MAX_T tokens) as
// weight-streaming GEMVs on mma.sync.  With so few tokens every expert holds one to a few
// rows, and the expert weights must still be read once from HBM (aimanavo.com, "Why is
// Perplexity's local AI Lily faster than MLX", section "Prefill and decode are not
// treated as the same job": the 4-bit restore runs inside the grouped GEMM).  A tcgen05
// tile of M = 128 tokens is then almost all padding and its cost does not shrink with the
// rows (one instruction costs the same at any N); an m16n8k16 MMA takes eight token
// columns at a time, so the weights are dequantised in registers and streamed through
// the MMAs once per group of eight tokens.
//
// gateup_gemv_kernel: one CTA per (token block, chunk of 32 of its rows, 64 h columns),
// one warp per 8 columns:
// the warp's A rows 0-7 are the gate rows and 8-15 the up rows of the features whose
// K-interleaved h columns are pos0 .. pos0 + 7, so that the accumulator pairs gate and up
// of the same feature (SwiGLU needs no exchange).  Lane quarter c4 takes words 2 c4 and
// 2 c4 + 1 of each quantisation group (eight inputs each); the B fragments are the same
// words of the K-interleaved activation rows.  down_gemv_kernel: one CTA per (token
// block, chunk of 32 rows, 128 output rows), one warp per 16 rows, B = the h rows.
//
// Both read every weight word once per pass of up to 8 rows (one pass unless the chunk
// holds more rows), with the next words of a warp in flight while it computes; the pass's
// activation (or h) rows are staged in shared memory first.  The dequantised weight is
// bf16(scale * q + bias), one rounding, as in the tcgen05 kernels.  No waits beyond the
// CTA's own barriers: the kernels only read what the kernels before them wrote.
#include "common.cuh"
#include "gemm_common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int GV_WARPS = 8;
constexpr int GV_THREADS = GV_WARPS * 32;
constexpr int GV_GU_SLICES = INTER / (8 * GV_WARPS);  // 8 slices of 64 h columns per token block
constexpr int GV_DN_SLICES = HID / (16 * GV_WARPS);   // 16 slices of 128 output rows per token block
constexpr int GV_NG = HID / GROUP;                    // 32 quantisation groups along a gate/up row
constexpr int GV_CHUNK = 4;                           // gate/up groups whose words are loaded together
constexpr int GV_RC = 32;                             // rows of a block per CTA (four passes of 8)

// Row chunks of GV_RC rows per token block: the grid has room for the largest block
// T tokens can make, and CTAs past their block's rows leave at once.
__host__ __device__ __forceinline__ int gv_chunks(int T) { return ((T < GX_BN ? T : GX_BN) + GV_RC - 1) / GV_RC; }

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint2 ldg_nc_v2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// bf16 element j (0..3) of a uint2 of four bf16
__device__ __forceinline__ uint32_t bf16_at(uint2 v, int j) {
  const uint32_t w = j < 2 ? v.x : v.y;
  return (j & 1) ? (w >> 16) : (w & 0xFFFFu);
}

// The CTA's token block (the same for every slice of it); false when the CTA has none.
// The row tables are read straight from global memory (two entries per CTA).
__device__ __forceinline__ bool gv_block(const int* blocks, const int* offsets, const int* counts, int bi, int T,
                                         unsigned int* err, TileInfo& ti) {
  const int nblocks = __ldg(blocks);
  if (nblocks < 0 || nblocks > (8 * T + GX_BN - 1) / GX_BN + min(8 * T, NEXP) + (T + GX_BN - 1) / GX_BN) {
    if (threadIdx.x == 0) atomicOr(err, ERRBIT_BOUNDS);
    return false;
  }
  if (bi >= nblocks) return false;
  ti = tile_info(blocks, offsets, counts, bi, 1, T);
  if (!ti.ok) {
    if (threadIdx.x == 0) atomicOr(err, ERRBIT_BOUNDS);
    return false;
  }
  return true;
}

// Token of permuted row `row`: routed rows through the permutation, shared rows directly.
__device__ __forceinline__ int gv_token(const int* row_dst, int row, int T, unsigned int* err) {
  const int n8 = 8 * T;
  int t = row >= n8 ? row - n8 : (__ldg(row_dst + row) >> 3);
  if (t < 0 || t >= T) {
    atomicOr(err, ERRBIT_BOUNDS);
    t = 0;
  }
  return t;
}

// Stage the pass's rows into shared memory: rows 0 .. nr - 1 of `chunks` 16-byte chunks,
// chunk c of row r at c ^ (r & 7) so that a warp's B-fragment reads, eight rows at a time,
// hit distinct banks.  The source row of pass row r: the token of permuted row row0 + r in
// the activations (by_token), else permuted row row0 + r itself (h).
__device__ __forceinline__ void gv_stage_rows(uint4* dst, int* s_tok, const __nv_bfloat16* src, int chunks, int row0,
                                              int nr, const int* row_dst, int T, unsigned int* err, bool by_token) {
  __syncthreads();   // the previous pass's reads of dst and s_tok are done
  if (threadIdx.x < 8)
    s_tok[threadIdx.x] = static_cast<int>(threadIdx.x) < nr
                             ? (by_token ? gv_token(row_dst, row0 + threadIdx.x, T, err) : row0 + threadIdx.x)
                             : 0;
  __syncthreads();
  for (int q = threadIdx.x; q < nr * chunks; q += blockDim.x) {
    const int r = q / chunks, c = q % chunks;
    const __nv_bfloat16* from = src + static_cast<size_t>(s_tok[r]) * (chunks * 8) + 8 * c;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst + r * chunks + (c ^ (r & 7)))),
                 "l"(from)
                 : "memory");
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
}

}  // namespace

__global__ void __launch_bounds__(GV_THREADS, 2)
    gateup_gemv_kernel(GateUpParams p, const uint32_t* __restrict__ gq, const uint32_t* __restrict__ uq,
                       const uint32_t* __restrict__ sgq, const uint32_t* __restrict__ suq) {
  __shared__ __align__(16) uint4 xs[8 * (HID / 8)];   // the pass's eight activation rows (32 KB)
  __shared__ int s_tok[8];
  grid_dep_wait();   // the routing tables and activations come from the kernels before this one
  TileInfo ti;
  const int nch = gv_chunks(p.T), bc = static_cast<int>(blockIdx.x) / GV_GU_SLICES;   // block * nch + chunk
  if (!gv_block(p.blocks, p.offsets, p.counts, bc / nch, p.T, p.err, ti)) return;
  const int r_lo = (bc % nch) * GV_RC, r_hi = min(ti.n_rows, r_lo + GV_RC);
  if (r_lo >= r_hi) return;   // uniform: this chunk lies past the block's rows
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c4 = lane & 3;
  const int pos0 = (static_cast<int>(blockIdx.x) % GV_GU_SLICES) * (8 * GV_WARPS) + warp * 8;
  const bool sh = ti.e == SHARED_E;
  // A row g: the gate (and up) row of the feature whose interleaved h column is pos0 + g
  const size_t wrow = (sh ? 0 : static_cast<size_t>(ti.e) * INTER) + ilv_row(pos0 + g);
  const uint32_t* gr = (sh ? sgq : gq) + wrow * (HID / 8) + 2 * c4;
  const uint32_t* ur = (sh ? suq : uq) + wrow * (HID / 8) + 2 * c4;
  const uint16_t* gs = (sh ? p.sg_scales : p.g_scales) + wrow * GV_NG;
  const uint16_t* gb = (sh ? p.sg_biases : p.g_biases) + wrow * GV_NG;
  const uint16_t* us = (sh ? p.su_scales : p.u_scales) + wrow * GV_NG;
  const uint16_t* ub = (sh ? p.su_biases : p.u_biases) + wrow * GV_NG;

  for (int c0 = r_lo; c0 < r_hi; c0 += 8) {
    const int nr = min(8, r_hi - c0);   // rows of this pass: B columns 0 .. nr - 1
    // this lane's words of groups G .. G + GV_CHUNK - 1 (the first chunk's requested before
    // the rows are staged), the next chunk's in flight while a chunk computes
    uint2 wg[GV_CHUNK], wu[GV_CHUNK], sgs, sgb, sus, sub;
#pragma unroll
    for (int j = 0; j < GV_CHUNK; ++j) {
      wg[j] = ldg_nc_v2(gr + 8 * j);
      wu[j] = ldg_nc_v2(ur + 8 * j);
    }
    sgs = ldg_nc_v2(gs); sgb = ldg_nc_v2(gb); sus = ldg_nc_v2(us); sub = ldg_nc_v2(ub);
    gv_stage_rows(xs, s_tok, p.x_ilv, HID / 8, ti.row0 + c0, nr, p.row_dst, p.T, p.err, true);
    const bool on = g < nr;
    const uint4* xrow = xs + g * (HID / 8);
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 1
    for (int G0 = 0; G0 < GV_NG; G0 += GV_CHUNK) {
      uint2 ng[GV_CHUNK], nu[GV_CHUNK], ngs, ngb, nus, nub;
      const int Gn = G0 + GV_CHUNK < GV_NG ? G0 + GV_CHUNK : G0;   // the last chunk reloads itself (unused)
#pragma unroll
      for (int j = 0; j < GV_CHUNK; ++j) {
        ng[j] = ldg_nc_v2(gr + 8 * (Gn + j));
        nu[j] = ldg_nc_v2(ur + 8 * (Gn + j));
      }
      ngs = ldg_nc_v2(gs + Gn); ngb = ldg_nc_v2(gb + Gn); nus = ldg_nc_v2(us + Gn); nub = ldg_nc_v2(ub + Gn);
#pragma unroll
      for (int j = 0; j < GV_CHUNK; ++j) {
        const int G = G0 + j;
        const __nv_bfloat162 msg = bf2(bf16_at(sgs, j)), mbg = bf2(bf16_at(sgb, j));
        const __nv_bfloat162 msu = bf2(bf16_at(sus, j)), mbu = bf2(bf16_at(sub, j));
        const uint4 a0 = dequant8(wg[j].x, msg, mbg), b0 = dequant8(wu[j].x, msu, mbu);   // word 2 c4
        const uint4 a1 = dequant8(wg[j].y, msg, mbg), b1 = dequant8(wu[j].y, msu, mbu);   // word 2 c4 + 1
        const int ch = 8 * G + 2 * c4;   // the two 16-byte chunks (words) of the B fragments
        const uint4 z = make_uint4(0, 0, 0, 0);
        const uint4 x0 = on ? xrow[ch ^ g] : z, x1 = on ? xrow[(ch + 1) ^ g] : z;
        mma16816(acc, a0.x, b0.x, a0.y, b0.y, x0.x, x0.y);
        mma16816(acc, a0.z, b0.z, a0.w, b0.w, x0.z, x0.w);
        mma16816(acc, a1.x, b1.x, a1.y, b1.y, x1.x, x1.y);
        mma16816(acc, a1.z, b1.z, a1.w, b1.w, x1.z, x1.w);
      }
#pragma unroll
      for (int j = 0; j < GV_CHUNK; ++j) {
        wg[j] = ng[j];
        wu[j] = nu[j];
      }
      sgs = ngs; sgb = ngb; sus = nus; sub = nub;
    }
    // SwiGLU: acc[i] = gate, acc[2 + i] = up of h column pos0 + g for block row c0 + 2 c4 + i;
    // lanes g and g + 1 (lane + 4) store a pair of columns
    float hv[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      // silu(g) = g/2 + (g/2) tanh(g/2), the hardware tanh, as in the tcgen05 gate/up epilogue
      const float hg = 0.5f * acc[i];
      float th;
      asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(hg));
      hv[i] = fmaf(hg, th, hg) * acc[2 + i];
    }
    const float n0 = __shfl_down_sync(0xffffffffu, hv[0], 4), n1 = __shfl_down_sync(0xffffffffu, hv[1], 4);
    if ((g & 1) == 0) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r = 2 * c4 + i;
        if (r < nr)
          *reinterpret_cast<uint32_t*>(p.h + static_cast<size_t>(ti.row0 + c0 + r) * INTER + pos0 + g) =
              pack2(hv[i], i ? n1 : n0);
      }
    }
  }
}

__global__ void __launch_bounds__(GV_THREADS, 2)
    down_gemv_kernel(DownParams p, const __nv_bfloat16* __restrict__ h, const uint32_t* __restrict__ dq,
                     const uint32_t* __restrict__ sdq) {
  __shared__ __align__(16) uint4 hs[8 * (INTER / 8)];   // the pass's eight h rows (8 KB)
  __shared__ int s_tok[8];
  grid_dep_wait();   // h comes from the gate/up kernel before this one
  TileInfo ti;
  const int nch = gv_chunks(p.T), bc = static_cast<int>(blockIdx.x) / GV_DN_SLICES;   // block * nch + chunk
  if (!gv_block(p.blocks, p.offsets, p.counts, bc / nch, p.T, p.err, ti)) return;
  const int r_lo = (bc % nch) * GV_RC, r_hi = min(ti.n_rows, r_lo + GV_RC);
  if (r_lo >= r_hi) return;   // uniform: this chunk lies past the block's rows
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c4 = lane & 3;
  const int R0 = (static_cast<int>(blockIdx.x) % GV_DN_SLICES) * (16 * GV_WARPS) + warp * 16;   // rows R0 + g, R0 + g + 8
  const bool sh = ti.e == SHARED_E;
  const size_t w0 = (sh ? 0 : static_cast<size_t>(ti.e) * HID) + R0 + g, w1 = w0 + 8;
  const uint32_t* q = sh ? sdq : dq;
  const uint16_t* sc = sh ? p.sd_scales : p.d_scales;
  const uint16_t* bi = sh ? p.sd_biases : p.d_biases;
  constexpr int NGD = INTER / GROUP;   // 8 groups along a down row
  const uint32_t* qr0 = q + w0 * (INTER / 8) + 2 * c4;
  const uint32_t* qr1 = q + w1 * (INTER / 8) + 2 * c4;
  const uint4 s0 = ldg_nc_v4(sc + w0 * NGD), b0 = ldg_nc_v4(bi + w0 * NGD);
  const uint4 s1 = ldg_nc_v4(sc + w1 * NGD), b1 = ldg_nc_v4(bi + w1 * NGD);
  const uint32_t s0w[4] = {s0.x, s0.y, s0.z, s0.w}, b0w[4] = {b0.x, b0.y, b0.z, b0.w};
  const uint32_t s1w[4] = {s1.x, s1.y, s1.z, s1.w}, b1w[4] = {b1.x, b1.y, b1.z, b1.w};

  for (int c0 = r_lo; c0 < r_hi; c0 += 8) {
    const int nr = min(8, r_hi - c0);   // rows of this pass: B columns 0 .. nr - 1
    // the two halves of the row (four groups each): the first requested before the rows are
    // staged, the second in flight while the first computes
    uint2 q0[GV_CHUNK], q1[GV_CHUNK];
#pragma unroll
    for (int j = 0; j < GV_CHUNK; ++j) {
      q0[j] = ldg_nc_v2(qr0 + 8 * j);
      q1[j] = ldg_nc_v2(qr1 + 8 * j);
    }
    gv_stage_rows(hs, s_tok, h, INTER / 8, ti.row0 + c0, nr, nullptr, p.T, p.err, false);
    const bool on = g < nr;
    const uint4* hrow = hs + g * (INTER / 8);
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int G0 = 0; G0 < NGD; G0 += GV_CHUNK) {
      uint2 n0[GV_CHUNK], n1[GV_CHUNK];
      if (G0 + GV_CHUNK < NGD) {
#pragma unroll
        for (int j = 0; j < GV_CHUNK; ++j) {
          n0[j] = ldg_nc_v2(qr0 + 8 * (G0 + GV_CHUNK + j));
          n1[j] = ldg_nc_v2(qr1 + 8 * (G0 + GV_CHUNK + j));
        }
      }
#pragma unroll
      for (int j = 0; j < GV_CHUNK; ++j) {
        const int G = G0 + j;
        const int hw = G >> 1, sh16 = (G & 1) * 16;   // group G's scale: bf16 G of the row's eight
        const __nv_bfloat162 m0 = bf2(s0w[hw] >> sh16), c0v = bf2(b0w[hw] >> sh16);
        const __nv_bfloat162 m1 = bf2(s1w[hw] >> sh16), c1v = bf2(b1w[hw] >> sh16);
        const uint4 a0 = dequant8(q0[j].x, m0, c0v), a1 = dequant8(q1[j].x, m1, c1v);   // word 2 c4
        const uint4 e0 = dequant8(q0[j].y, m0, c0v), e1 = dequant8(q1[j].y, m1, c1v);   // word 2 c4 + 1
        const int ch = 8 * G + 2 * c4;
        const uint4 z = make_uint4(0, 0, 0, 0);
        const uint4 x0 = on ? hrow[ch ^ g] : z, x1 = on ? hrow[(ch + 1) ^ g] : z;
        mma16816(acc, a0.x, a1.x, a0.y, a1.y, x0.x, x0.y);
        mma16816(acc, a0.z, a1.z, a0.w, a1.w, x0.z, x0.w);
        mma16816(acc, e0.x, e1.x, e0.y, e1.y, x1.x, x1.y);
        mma16816(acc, e0.z, e1.z, e0.w, e1.w, x1.z, x1.w);
      }
      if (G0 + GV_CHUNK < NGD) {
#pragma unroll
        for (int j = 0; j < GV_CHUNK; ++j) {
          q0[j] = n0[j];
          q1[j] = n1[j];
        }
      }
    }
    // acc[i]: output row R0 + g, acc[2 + i]: R0 + g + 8, of block row c0 + 2 c4 + i; lanes
    // g and g + 1 store a pair of adjacent output columns
    float nb[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) nb[k] = __shfl_down_sync(0xffffffffu, acc[k], 4);
    if ((g & 1) == 0) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r = 2 * c4 + i;
        if (r < nr) {
          __nv_bfloat16* yr = p.y + static_cast<size_t>(ti.row0 + c0 + r) * HID + R0 + g;
          *reinterpret_cast<uint32_t*>(yr) = pack2(acc[i], nb[i]);
          *reinterpret_cast<uint32_t*>(yr + 8) = pack2(acc[2 + i], nb[2 + i]);
        }
      }
    }
  }
}

// the most token blocks T tokens can make (the bound the scan's list obeys)
int gemv_blocks_max(int T) { return (8 * T + GX_BN - 1) / GX_BN + min(8 * T, NEXP) + (T + GX_BN - 1) / GX_BN; }

cudaError_t launch_gateup_gemv(const GateUpParams& p, const void* gq, const void* uq, const void* sgq,
                               const void* suq, cudaStream_t s) {
  return launch_pdl(gateup_gemv_kernel, dim3(gemv_blocks_max(p.T) * gv_chunks(p.T) * GV_GU_SLICES), dim3(GV_THREADS),
                    0, s, p,
                    static_cast<const uint32_t*>(gq), static_cast<const uint32_t*>(uq),
                    static_cast<const uint32_t*>(sgq), static_cast<const uint32_t*>(suq));
}

cudaError_t launch_down_gemv(const DownParams& p, const __nv_bfloat16* h, const void* dq, const void* sdq,
                             cudaStream_t s) {
  return launch_pdl(down_gemv_kernel, dim3(gemv_blocks_max(p.T) * gv_chunks(p.T) * GV_DN_SLICES), dim3(GV_THREADS),
                    0, s, p, h,
                    static_cast<const uint32_t*>(dq), static_cast<const uint32_t*>(sdq));
}

}  // namespace moe
