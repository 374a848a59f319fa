// internal.h -- parameter blocks and launch entry points shared by the library's
// translation units (host side).  Not part of the public C ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace moe {

// Launch with programmatic stream serialisation: the kernel is launched as the previous
// kernel of the stream finishes, before its writes are flushed, and waits for them in
// grid_dep_wait() (every prefill kernel calls that before touching memory that other
// kernels use).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct RouteParams {
  const __nv_bfloat16* x;
  int T;
  const float* router_bias;  // [256] or nullptr (staged by the kernel)
  int* topk_idx;             // [T][8]
  float* topk_w;             // [T][8]
  int* hist;                 // [nblk][256] per-router-block expert histogram
  unsigned int* err;
  unsigned long long wait_ns;  // time limit of a bounded wait
};

struct ScanParams {
  const int* hist;    // [nblk][256]
  int nblk;
  int T;
  int* base;          // [nblk][256] first permuted row of (block, expert)
  int* counts;        // [257]: 256 experts + shared (= T)
  int* offsets;       // [258]: exclusive scan; [256] = 8T, [257] = 9T
  int* blocks;        // [0] = number of token blocks, [1] = those of > GX_SMALL rows, then the blocks (see route_scan_kernel)
};

struct ScatterParams {
  const int* topk_idx;
  const float* topk_w;
  const int* base;
  int T;
  int* row_dst;       // [9T] routed part: the permutation of slot ids; shared part: 8T+t
  int* slot_row;      // [8T] inverse: the permuted row of slot t*8+k
  float* row_w;       // [9T] routing weight (routed rows) or shared-gate sigmoid (shared rows)
  const __nv_bfloat16* x;
  const __nv_bfloat16* shared_gate_w;   // [2048]
  __nv_bfloat16* x_ilv;    // [T][2048] copy of x with K-interleaved rows (read by the gate/up gather)
  int gather;              // 0: routing tables only (moe_route; or the previous stacked layer's
                           // combine already wrote x_ilv and the shared rows)
  unsigned int* err;
  int fused;               // 1: no scan launch; the bases come from the histograms and one
                           // extra CTA column writes the scan's tables (scan below)
  ScanParams scan;
};

struct GateUpParams {
  const int* blocks;     // token blocks: [0] = count, [1] = blocks of > GX_SMALL rows, then expert | (block << 9)
  const int* offsets;    // [258]
  const int* counts;     // [257]
  const uint16_t* g_scales; const uint16_t* g_biases;    // [256][512][32]
  const uint16_t* u_scales; const uint16_t* u_biases;
  const uint16_t* sg_scales; const uint16_t* sg_biases;  // [512][32]
  const uint16_t* su_scales; const uint16_t* su_biases;
  __nv_bfloat16* h;      // [9T][512] silu(gate) * up, K-interleaved columns
  int T;
  unsigned int* err;
  unsigned long long* pipe;   // 16 pipeline-trace counters, or nullptr
  const __nv_bfloat16* x_ilv; // [T][2048] K-interleaved activations, gathered by token
  const int* row_dst;         // [9T] slot id (t*8+k) of each routed permuted row
  unsigned long long wait_ns; // time limit of a bounded wait
};

struct DownParams {
  const int* blocks;     // token blocks: [0] = count, [1] = blocks of > GX_SMALL rows, then expert | (block << 9)
  const int* offsets;
  const int* counts;
  const uint16_t* d_scales; const uint16_t* d_biases;    // [256][2048][8]
  const uint16_t* sd_scales; const uint16_t* sd_biases;  // [2048][8]
  __nv_bfloat16* y;      // [9T][2048] by permuted row (written through a TMA map)
  int T;
  unsigned int* err;
  unsigned long long* pipe;   // 16 pipeline-trace counters, or nullptr
  unsigned long long wait_ns; // time limit of a bounded wait
  int small_apart;            // down_kernel: 1 = leave the small blocks to down_swap_kernel
};

struct DecodeParams {
  const __nv_bfloat16* x;
  int T;
  const __nv_bfloat16* router_w;
  const float* router_bias;
  const __nv_bfloat16* shared_gate_w;
  float* logits;         // [8][257]
  unsigned int* counter;
  int* topk_idx;         // [T][8]
  float* topk_w;
  int* counts;           // [257]
  int* offsets;          // [258]
  int* perm;             // [8T]
  int* act_expert;       // [65]
  float* act_w;          // [65][8]
  int* n_active;
  // expert weights (packed words / bf16 bits)
  const uint32_t* gq; const uint16_t* gs; const uint16_t* gb;     // routed gate
  const uint32_t* uq; const uint16_t* us; const uint16_t* ub;     // routed up
  const uint32_t* dq; const uint16_t* ds; const uint16_t* db;     // routed down
  const uint32_t* sgq; const uint16_t* sgs; const uint16_t* sgb;  // shared gate
  const uint32_t* suq; const uint16_t* sus; const uint16_t* sub;  // shared up
  const uint32_t* sdq; const uint16_t* sds; const uint16_t* sdb;  // shared down
  __nv_bfloat16* hw;     // [65][8][512] weighted, K-interleaved
  __nv_bfloat16* out;    // [T][2048]
  const __nv_bfloat16* x_resid;   // [T][2048] residual input (the un-normalised x)
  int residual;
  unsigned int* err;
};

// One layer of the fused decode kernel: the layer's weights and its error word.
struct DecLayer {
  const __nv_bfloat16* router_w;      // [256][2048]
  const float* router_bias;           // [256] or nullptr
  const __nv_bfloat16* shared_gate_w; // [2048]
  const __nv_bfloat16* norm_w;        // [2048] input RMSNorm weights, or nullptr (no norm)
  const uint32_t* gq; const uint16_t* gs; const uint16_t* gb;     // routed gate
  const uint32_t* uq; const uint16_t* us; const uint16_t* ub;     // routed up
  const uint32_t* dq; const uint16_t* ds; const uint16_t* db;     // routed down
  const uint32_t* sgq; const uint16_t* sgs; const uint16_t* sgb;  // shared gate
  const uint32_t* suq; const uint16_t* sus; const uint16_t* sub;  // shared up
  const uint32_t* sdq; const uint16_t* sds; const uint16_t* sdb;  // shared down
  unsigned int* err;
};

constexpr int DEC_MAX_LAYERS = 48;   // layers per launch of the fused decode kernel
constexpr size_t DEC_LT_WORDS = 2ull * 8 * 257;
constexpr size_t DEC_HT_WORDS = 2ull * 65 * 8 * 256;
constexpr size_t DEC_XT_WORDS = 2ull * 8 * 1024;
constexpr int DEC_TRACE_STAMPS = 16;           // timestamps per layer and CTA
constexpr int DEC_TRACE_CTAS = 256;            // CTAs the trace has room for
constexpr size_t DEC_TRACE_WORDS = static_cast<size_t>(DEC_MAX_LAYERS) * DEC_TRACE_CTAS * DEC_TRACE_STAMPS;

struct DecLayersParams {
  const __nv_bfloat16* x;   // [T][2048] input of the first layer
  __nv_bfloat16* out;       // [T][2048] output of every layer (may alias x)
  int T;                    // 1..8
  int n_layers;             // 1..DEC_MAX_LAYERS
  int residual;             // out = x + MoE(x) when set
  // scratch, zeroed once when the workspace is bound; tagged words {payload, tag}
  unsigned long long* lt;   // [2][8][257] router and shared-gate logits
  unsigned long long* ht;   // [2][65][8][256] weighted h' (pairs of interleaved features)
  unsigned long long* xt;   // [2][8][1024] layer outputs between layers (pairs of features)
  unsigned int* sync;       // [4]: [1] exit count, [2] abort flag, [3] launch epoch
  int* topk_idx;            // [T][8] routing of the last layer, or nullptr
  float* topk_w;
  unsigned long long wait_ns;   // time limit of a bounded wait
  unsigned long long* trace;    // phase timestamps [layer][CTA][DEC_TRACE_STAMPS], or nullptr
  DecLayer layer[DEC_MAX_LAYERS];
};

// ---- grouped-query decode attention (gqa.cu)
constexpr int GQ_HQ = 16;        // query heads
constexpr int GQ_HKV = 2;        // key/value heads
constexpr int GQ_G = GQ_HQ / GQ_HKV;
constexpr int GQ_D = 128;        // head size
constexpr int GQ_CH = 128;       // cached positions per pipeline stage
constexpr int GQ_STAGES = 3;
constexpr int GQ_STAGE_BYTES = 2 * GQ_CH * GQ_D * 2;   // K and V rows of one stage
constexpr int GQ_MAX_B = 64;     // sequences per call
constexpr int GQ_MAX_SPLIT = 160;

struct GqaParams {
  const __nv_bfloat16* q;   // [B][16][128]
  __nv_bfloat16* out;       // [B][16][128]
  float* part;              // [B][16][nsplit][132]: unnormalised O[128], max (base 2), sum, 2 unused
  unsigned* ticket;         // [B][2] splits done (the last one merges, then clears it)
  unsigned* err;
  int B, S_max, nsplit;
  float scale_log2;         // log2(e) / sqrt(128)
  unsigned long long wait_ns;
  int lens[GQ_MAX_B];       // cached positions per sequence (1..S_max)
};

// launchers (return the first launch error)
cudaError_t launch_router_cluster(const CUtensorMap& tm_x, const CUtensorMap& tm_wr, const RouteParams& p,
                                  cudaStream_t s);
cudaError_t launch_router_prefill(const CUtensorMap& tm_x, const CUtensorMap& tm_wr, const RouteParams& p,
                                  cudaStream_t s);
cudaError_t launch_rmsnorm(const __nv_bfloat16* x, const __nv_bfloat16* w, __nv_bfloat16* xn, int T,
                           cudaStream_t s);
cudaError_t launch_scan(const ScanParams& p, cudaStream_t s);
cudaError_t launch_scatter(const ScatterParams& p, int nblk, cudaStream_t s);
cudaError_t launch_gateup(const CUtensorMap& qg, const CUtensorMap& qu, const CUtensorMap& sqg,
                          const CUtensorMap& squ, const CUtensorMap& hs, const GateUpParams& p, int grid,
                          cudaStream_t s);
cudaError_t launch_down(const CUtensorMap& qd, const CUtensorMap& sqd, const CUtensorMap& hmap,
                        const CUtensorMap& ymap, const DownParams& p, int grid, cudaStream_t s);
// The next stacked layer's inputs that the combine writes from its output rows (norm_w
// == nullptr: none): the RMSNorm xn, its K-interleaved copy and the shared-expert rows'
// index and gate, in that layer's workspace.
struct NextLayerIn {
  const __nv_bfloat16* norm_w;
  const __nv_bfloat16* gate_w;
  __nv_bfloat16* xn;
  __nv_bfloat16* x_ilv;
  int* row_dst;
  float* row_w;
};
cudaError_t launch_combine(const __nv_bfloat16* y, const int* slot_row, const float* row_w, const __nv_bfloat16* x,
                           __nv_bfloat16* out, int T, int residual, const NextLayerIn& nx, cudaStream_t s);
cudaError_t launch_decode_router(const DecodeParams& p, cudaStream_t s);
cudaError_t launch_decode_layers(const DecLayersParams& p, cudaStream_t s);
cudaError_t launch_gqa_decode(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const GqaParams& p, cudaStream_t s);
// A 2-D bf16 tensor map over rows of `cols` elements with a box of 64 x box_rows and the
// 128-byte swizzle (false, with the failure detail recorded, if encoding fails).
bool encode_bf16_sw128(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows);
cudaError_t set_kernel_attributes();
// The time limit of the bounded device waits of the next launches (moe_set_wait_limit_ns).
unsigned long long wait_limit_ns();
// Record the calling thread's failure description that moe_last_error_detail returns:
// `what`, followed by the CUDA error's name when e is not cudaSuccess.
void set_error_detail(const char* what, cudaError_t e);
cudaError_t launch_gateup_gemv(const GateUpParams& p, const void* gq, const void* uq, const void* sgq,
                               const void* suq, cudaStream_t s);
cudaError_t launch_down_gemv(const DownParams& p, const __nv_bfloat16* h, const void* dq, const void* sdq,
                             cudaStream_t s);
cudaError_t launch_down_swap(const CUtensorMap& qd, const CUtensorMap& sqd, const CUtensorMap& hmap, const DownParams& p,
                             int grid, cudaStream_t s);
cudaError_t set_down_attributes();

}  // namespace moe
