// moe_layer.cu -- the C ABI (include/moe_layer.h): load-time validation, workspace
// carving, TMA descriptors and the launch sequences of the prefill and decode paths.
//
// Lily accepts exactly one model layout and refuses every other one when it loads
// (aimanavo.com, "Why is Perplexity's local AI Lily faster than MLX", section "Only one
// 4-bit checkpoint of a pinned revision runs"; news.mantis.guru, "Perplexity opened
// Lily", section "Rust drives the model, Metal computes"): moe_layer_create does the
// same for the layer's shape and quantisation, and for pointer alignment.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "moe_layer.h"

namespace moe {
cudaError_t set_router_attributes();
cudaError_t set_gemm_attributes();

namespace {
std::atomic<unsigned long long> g_wait_ns{WAIT_LIMIT_NS};
}
unsigned long long wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
}  // namespace moe

namespace {
thread_local char g_detail[256] = "";
}

void moe::set_error_detail(const char* what, cudaError_t e) {
  if (e == cudaSuccess)
    snprintf(g_detail, sizeof g_detail, "%s", what);
  else
    snprintf(g_detail, sizeof g_detail, "%s: %s", what, cudaGetErrorString(e));
}

using namespace moe;

struct moe_layer {
  moe_config_t cfg;
  moe_weights_t w;
  uint8_t* ws;
  size_t ws_bytes;
  int num_sms;
  // workspace segments
  unsigned int* err;
  unsigned int* dec_counter;
  int *hist, *base, *counts, *offsets, *blocks;
  int* topk_idx;
  float* topk_w;
  int* row_dst;
  int* slot_row;
  float* row_w;
  __nv_bfloat16 *x_ilv, *h, *y, *x_io, *xn;
  float* dec_logits;
  int* dec_act_expert;
  float* dec_act_w;
  int* dec_n_active;
  __nv_bfloat16* dec_hw;
  unsigned int* dec_sync;          // fused decode: exit count, abort flag, launch epoch
  unsigned long long* dec_lt;      // fused decode: tagged logits, h', layer outputs
  unsigned long long* dec_ht;
  unsigned long long* dec_xt;
  unsigned long long* dec_trace;   // fused decode: phase timestamps (MOE_DECODE_TRACE=1)
  unsigned long long* pipe;   // 32 pipeline-trace counters (gate/up 0..15, down 16..31)
  // TMA descriptors of the weights and of the workspace buffers
  CUtensorMap tm_wr, tm_qg, tm_qu, tm_sqg, tm_squ, tm_qd, tm_sqd, tm_h, tm_y, tm_hs;
};

namespace {

void set_detail(const char* what, cudaError_t e) {
  snprintf(g_detail, sizeof g_detail, "%s: %s", what, cudaGetErrorString(e));
}

// ------------------------------------------------------------------ kernel profiler
// While enabled, every launch is bracketed by two CUDA events on its own stream; the
// durations are resolved (and the record cleared) by moe_profiler_read.
enum KernelId {
  K_ROUTER, K_SCAN, K_SCATTER, K_GATEUP, K_DOWN, K_COMBINE, K_DEC_ROUTER, K_DEC_LAYERS, K_NORM, K_DOWN_SWAP,
  K_COUNT
};
const char* const kKernelNames[K_COUNT] = {"router_prefill", "route_scan",    "route_scatter",
                                           "gateup",         "down",          "combine",
                                           "decode_router",  "decode_layers",
                                           "rmsnorm",        "down_swap"};
struct ProfRec {
  int id;
  cudaEvent_t a, b;
};
struct Profiler {
  bool on = false;
  std::mutex m;
  std::vector<ProfRec> recs;
  std::vector<cudaEvent_t> pool;
} g_prof;

cudaEvent_t prof_event() {
  if (!g_prof.pool.empty()) {
    cudaEvent_t e = g_prof.pool.back();
    g_prof.pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// MOE_DEBUG_SYNC=1 (read once): synchronise after every launch, and turn a CUDA error
// or a bit in the device error word into cudaErrorUnknown naming the kernel.
bool debug_sync() {
  static const bool on = [] {
    const char* v = getenv("MOE_DEBUG_SYNC");
    return v && v[0] == '1';
  }();
  return on;
}

// MOE_DECODE_TRACE=1 (read once): the fused decode kernel records the global timer at
// its phase boundaries (moe_decode_trace).
bool decode_trace() {
  static const bool on = [] {
    const char* v = getenv("MOE_DECODE_TRACE");
    return v && v[0] == '1';
  }();
  return on;
}

// MOE_PIPE_PROF=1 (read once): the grouped GEMMs add their barrier-wait cycles to the
// layer's pipeline counters (moe_pipeline_counters).
bool pipe_trace() {
  static const bool on = [] {
    const char* v = getenv("MOE_PIPE_PROF");
    return v && v[0] == '1';
  }();
  return on;
}

template <typename F>
cudaError_t timed(int id, cudaStream_t s, const unsigned int* err_word, F&& launch) {
  cudaError_t e;
  if (!g_prof.on) {
    e = launch();
  } else {
    std::lock_guard<std::mutex> lk(g_prof.m);
    ProfRec r{id, prof_event(), prof_event()};
    cudaEventRecord(r.a, s);
    e = launch();
    cudaEventRecord(r.b, s);
    g_prof.recs.push_back(r);
  }
  if (e == cudaSuccess && debug_sync()) {
    e = cudaStreamSynchronize(s);
    unsigned int w = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&w, err_word, 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) {
      snprintf(g_detail, sizeof g_detail, "kernel %s: %s", kKernelNames[id], cudaGetErrorString(e));
      fprintf(stderr, "[moe debug] %s\n", g_detail);
    } else if (w) {
      snprintf(g_detail, sizeof g_detail, "kernel %s set device error bits 0x%x", kKernelNames[id], w);
      fprintf(stderr, "[moe debug] %s\n", g_detail);
      e = cudaErrorUnknown;
    }
  }
  return e;
}

constexpr int MAX_TOKENS = 65536;

// Upper bound of a grouped GEMM's tile count at T tokens: every touched expert adds at
// most one partial token block to the full ones.
long long gemm_tiles_bound(int T, int mblk) {
  const long long blocks = (8ll * T + GX_BN - 1) / GX_BN + (8ll * T < NEXP ? 8ll * T : NEXP) + (T + GX_BN - 1) / GX_BN;
  return blocks * mblk;
}
// Persistent grid: one CTA per SM, fewer when there are fewer tiles.
int gemm_grid(int T, int mblk, int num_sms) {
  const long long t = gemm_tiles_bound(T, mblk);
  return static_cast<int>(t < num_sms ? t : num_sms);
}
// Each CTA decodes its tiles into a fixed-size schedule; T <= Tm must fit it.
bool schedules_fit(int Tm, int num_sms) {
  auto per_cta = [&](int mblk) {
    const long long t = gemm_tiles_bound(Tm, mblk), g = gemm_grid(Tm, mblk, num_sms);
    return (t + g - 1) / g;
  };
  // the small blocks: at most one per expert and the shared expert
  const long long small = (NEXP + 1) * DS_PAIRS, gs = small < num_sms ? small : num_sms;
  return per_cta(GU_MBLK) <= GU_SCHED_CAP && per_cta(DN_MBLK) <= DN_SCHED_CAP && (small + gs - 1) / gs <= DS_SCHED_CAP;
}

struct Carver {
  uint8_t* base;
  size_t off = 0;
  template <typename T>
  T* take(size_t bytes) {
    off = (off + 255) & ~size_t(255);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += bytes;
    return p;
  }
};

// Lays out the workspace for max_tokens Tm; with L == nullptr only sizes it.
size_t carve(int Tm, uint8_t* base, moe_layer* L) {
  Carver c{base};
  moe_layer tmp;
  moe_layer* d = L ? L : &tmp;
  const size_t nblk = (Tm + RT_BM - 1) / RT_BM;
  const size_t rows = 9ull * Tm;
  d->err = c.take<unsigned int>(256);
  d->dec_counter = c.take<unsigned int>(256);
  d->hist = c.take<int>(nblk * NEXP * 4);
  d->base = c.take<int>(nblk * NEXP * 4);
  d->counts = c.take<int>((NEXP + 1) * 4);
  d->offsets = c.take<int>((NEXP + 2) * 4);
  d->blocks = c.take<int>((gemm_tiles_bound(Tm, 1) + 2) * 4);
  d->topk_idx = c.take<int>(static_cast<size_t>(Tm) * TOPK * 4);
  d->topk_w = c.take<float>(static_cast<size_t>(Tm) * TOPK * 4);
  d->row_dst = c.take<int>(rows * 4);
  d->row_w = c.take<float>(rows * 4);
  d->slot_row = c.take<int>(static_cast<size_t>(Tm) * TOPK * 4);
  d->x_ilv = c.take<__nv_bfloat16>(static_cast<size_t>(Tm) * HID * 2);
  d->h = c.take<__nv_bfloat16>(rows * INTER * 2);
  d->y = c.take<__nv_bfloat16>(rows * HID * 2);
  d->x_io = c.take<__nv_bfloat16>(static_cast<size_t>(Tm) * HID * 2);
  d->xn = c.take<__nv_bfloat16>(static_cast<size_t>(Tm) * HID * 2);
  d->dec_logits = c.take<float>(DEC_MAX_T * (NEXP + 1) * 4);
  d->dec_act_expert = c.take<int>(DEC_MAX_ACTIVE * 4);
  d->dec_act_w = c.take<float>(DEC_MAX_ACTIVE * DEC_MAX_T * 4);
  d->dec_n_active = c.take<int>(4);
  d->dec_hw = c.take<__nv_bfloat16>(static_cast<size_t>(DEC_MAX_ACTIVE) * DEC_MAX_T * INTER * 2);
  d->pipe = c.take<unsigned long long>(32 * 8);
  d->dec_sync = c.take<unsigned int>(256);
  d->dec_lt = c.take<unsigned long long>(DEC_LT_WORDS * 8);
  d->dec_ht = c.take<unsigned long long>(DEC_HT_WORDS * 8);
  d->dec_xt = c.take<unsigned long long>(DEC_XT_WORDS * 8);
  d->dec_trace = c.take<unsigned long long>(DEC_TRACE_WORDS * 8);
  return (c.off + 255) & ~size_t(255);
}

bool config_ok(const moe_config_t* c) {
  return c->hidden == HID && c->n_experts == NEXP && c->top_k == TOPK && c->inter == INTER &&
         c->shared_inter == SH_INTER && c->group_size == GROUP && c->bits == 4 && c->max_tokens >= 1 &&
         c->max_tokens <= MAX_TOKENS;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = g_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) snprintf(g_detail, sizeof g_detail, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return r == CUDA_SUCCESS;
}

bool encode_bf16_rows(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  return encode_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, cols, rows, cols * 2, 64, box_rows,
                   CU_TENSOR_MAP_SWIZZLE_128B);
}

// Packed 4-bit tiles: 128 rows x 8 words (32 bytes) per box, stored with the 32-byte
// swizzle (the 16-byte half c of row r lands at c ^ ((r >> 2) & 1)), so that the dequant
// threads, one or two per row, read their halves without bank conflicts.
bool encode_packed(CUtensorMap* m, const void* base, uint64_t words, uint64_t rows) {
  return encode_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, base, words, rows, words * 4, 8, GX_BM,
                   CU_TENSOR_MAP_SWIZZLE_32B);
}

}  // namespace

bool moe::encode_bf16_sw128(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  if (!get_encode()) {
    snprintf(g_detail, sizeof g_detail, "cuTensorMapEncodeTiled entry point unavailable");
    return false;
  }
  return encode_bf16_rows(m, base, cols, rows, box_rows);
}

namespace {

bool qmat_ok(const moe_qmat_t& q, moe_status_t* st) {
  if (!q.q || !q.scales || !q.biases) { *st = MOE_ERR_INVALID_ARG; return false; }
  if (!aligned(q.q, 16) || !aligned(q.scales, 16) || !aligned(q.biases, 16)) { *st = MOE_ERR_ALIGNMENT; return false; }
  return true;
}

bool ranges_overlap(const void* a, const void* b, size_t bytes) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + bytes && y < x + bytes;
}

moe_status_t cuda_fail(const char* what, cudaError_t e) {
  set_detail(what, e);
  return MOE_ERR_CUDA;
}

#define MOE_TRY(call, what)                       \
  do {                                            \
    const cudaError_t e_ = (call);                \
    if (e_ != cudaSuccess) return cuda_fail(what, e_); \
  } while (0)

moe_status_t route_prefill(moe_layer* L, const void* x, int T, int gather, cudaStream_t s) {
  const int nblk = (T + RT_BM - 1) / RT_BM;
  CUtensorMap tm_x;
  if (!encode_bf16_rows(&tm_x, x, HID, T, RT_BM)) return MOE_ERR_CUDA;
  RouteParams rp{static_cast<const __nv_bfloat16*>(x), T, L->w.router_bias, L->topk_idx, L->topk_w, L->hist, L->err,
                 wait_limit_ns()};
  // up to RC2_MAX_T tokens a token block's contraction is cut in K parts, one CTA of a
  // cluster each (four parts up to RC_MAX_T tokens, two above)
  MOE_TRY(timed(K_ROUTER, s, L->err,
                [&] {
                  return T <= RC2_MAX_T ? launch_router_cluster(tm_x, L->tm_wr, rp, s)
                                        : launch_router_prefill(tm_x, L->tm_wr, rp, s);
                }),
          "router launch");
  ScanParams sp{L->hist, nblk, T, L->base, L->counts, L->offsets, L->blocks};
  // up to SCAN_FUSE_NBLK router blocks the scatter derives its bases from the histograms
  // itself and one extra CTA of it writes the scan's tables: one launch (and one
  // dependent-launch wait) fewer
  const int fused = nblk <= SCAN_FUSE_NBLK ? 1 : 0;
  if (!fused) MOE_TRY(timed(K_SCAN, s, L->err, [&] { return launch_scan(sp, s); }), "scan launch");
  ScatterParams scp{L->topk_idx, L->topk_w, L->base, T, L->row_dst, L->slot_row, L->row_w,
                    static_cast<const __nv_bfloat16*>(x),
                    static_cast<const __nv_bfloat16*>(L->w.shared_gate_w), L->x_ilv, gather, L->err, fused, sp};
  MOE_TRY(timed(K_SCATTER, s, L->err, [&] { return launch_scatter(scp, nblk + fused, s); }), "scatter launch");
  return MOE_OK;
}

DecodeParams decode_params(moe_layer* L, const void* x, int T, void* out, int residual) {
  DecodeParams p;
  std::memset(&p, 0, sizeof p);
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.T = T;
  p.router_w = static_cast<const __nv_bfloat16*>(L->w.router_w);
  p.router_bias = L->w.router_bias;
  p.shared_gate_w = static_cast<const __nv_bfloat16*>(L->w.shared_gate_w);
  p.logits = L->dec_logits;
  p.counter = L->dec_counter;
  p.topk_idx = L->topk_idx;
  p.topk_w = L->topk_w;
  p.counts = L->counts;
  p.offsets = L->offsets;
  p.perm = L->row_dst;
  p.act_expert = L->dec_act_expert;
  p.act_w = L->dec_act_w;
  p.n_active = L->dec_n_active;
  auto Q = [](const moe_qmat_t& m, const uint32_t*& q, const uint16_t*& sc, const uint16_t*& bi) {
    q = static_cast<const uint32_t*>(m.q);
    sc = static_cast<const uint16_t*>(m.scales);
    bi = static_cast<const uint16_t*>(m.biases);
  };
  Q(L->w.gate, p.gq, p.gs, p.gb);
  Q(L->w.up, p.uq, p.us, p.ub);
  Q(L->w.down, p.dq, p.ds, p.db);
  Q(L->w.sh_gate, p.sgq, p.sgs, p.sgb);
  Q(L->w.sh_up, p.suq, p.sus, p.sub);
  Q(L->w.sh_down, p.sdq, p.sds, p.sdb);
  p.hw = L->dec_hw;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.residual = residual;
  p.err = L->err;
  return p;
}

DecLayer dec_layer(const moe_layer* L) {
  DecLayer d;
  std::memset(&d, 0, sizeof d);
  d.router_w = static_cast<const __nv_bfloat16*>(L->w.router_w);
  d.router_bias = L->w.router_bias;
  d.shared_gate_w = static_cast<const __nv_bfloat16*>(L->w.shared_gate_w);
  d.norm_w = static_cast<const __nv_bfloat16*>(L->w.norm_w);
  auto Q = [](const moe_qmat_t& m, const uint32_t*& q, const uint16_t*& sc, const uint16_t*& bi) {
    q = static_cast<const uint32_t*>(m.q);
    sc = static_cast<const uint16_t*>(m.scales);
    bi = static_cast<const uint16_t*>(m.biases);
  };
  Q(L->w.gate, d.gq, d.gs, d.gb);
  Q(L->w.up, d.uq, d.us, d.ub);
  Q(L->w.down, d.dq, d.ds, d.db);
  Q(L->w.sh_gate, d.sgq, d.sgs, d.sgb);
  Q(L->w.sh_up, d.suq, d.sus, d.sub);
  Q(L->w.sh_down, d.sdq, d.sds, d.sdb);
  d.err = L->err;
  return d;
}

// Decode forward (T <= 8) of n consecutive layers in one cooperative launch per
// DEC_MAX_LAYERS layers; the scratch (logits, h', barrier words) is the first layer's.
moe_status_t decode_forward(moe_layer* const* layers, int n, const void* x, int T, void* out, int residual,
                            cudaStream_t s) {
  static DecLayersParams p;   // large (about 9 KB): kept off the stack, filled under the lock
  static std::mutex m;
  std::lock_guard<std::mutex> lk(m);
  moe_layer* L0 = layers[0];
  for (int base = 0; base < n; base += DEC_MAX_LAYERS) {
    const int cnt = n - base < DEC_MAX_LAYERS ? n - base : DEC_MAX_LAYERS;
    p.x = static_cast<const __nv_bfloat16*>(base == 0 ? x : out);
    p.out = static_cast<__nv_bfloat16*>(out);
    p.T = T;
    p.n_layers = cnt;
    p.residual = residual;
    p.lt = L0->dec_lt;
    p.ht = L0->dec_ht;
    p.xt = L0->dec_xt;
    p.sync = L0->dec_sync;
    p.topk_idx = nullptr;
    p.topk_w = nullptr;
    p.wait_ns = wait_limit_ns();
    p.trace = decode_trace() ? L0->dec_trace : nullptr;
    for (int i = 0; i < cnt; ++i) p.layer[i] = dec_layer(layers[base + i]);
    MOE_TRY(timed(K_DEC_LAYERS, s, L0->err, [&] { return launch_decode_layers(p, s); }), "decode launch");
  }
  return MOE_OK;
}

// The layer's input to routing and experts: x itself, or its RMSNorm when the layer has one.
// The layer's input: x, or its RMSNorm in L->xn (computed here unless the previous
// stacked layer's combine already wrote it: xn_ready).
moe_status_t layer_input(moe_layer* L, const void* x, int T, cudaStream_t s, const void** xin, bool xn_ready) {
  *xin = x;
  if (!L->w.norm_w) return MOE_OK;
  if (xn_ready) {
    *xin = L->xn;
    return MOE_OK;
  }
  MOE_TRY(timed(K_NORM, s, L->err,
                [&] {
                  return launch_rmsnorm(static_cast<const __nv_bfloat16*>(x),
                                        static_cast<const __nv_bfloat16*>(L->w.norm_w), L->xn, T, s);
                }),
          "rmsnorm launch");
  *xin = L->xn;
  return MOE_OK;
}

// One prefill layer.  next: the following stacked layer, whose input RMSNorm (if it has
// one) the combine computes into next->xn; xn_ready: this layer's RMSNorm is already in
// L->xn.
moe_status_t forward_impl(moe_layer* L, const void* x_orig, int T, void* out, int residual, cudaStream_t s,
                          moe_layer* next = nullptr, bool xn_ready = false) {
  if (T <= DEC_MAX_T) return decode_forward(&L, 1, x_orig, T, out, residual, s);
  const void* x = nullptr;
  const moe_status_t sn = layer_input(L, x_orig, T, s, &x, xn_ready);
  if (sn != MOE_OK) return sn;
  // the scatter's copy of x and shared gate are already there when the previous layer's
  // combine wrote them with the normalised input
  const moe_status_t st = route_prefill(L, x, T, xn_ready && L->w.norm_w ? 0 : 1, s);
  if (st != MOE_OK) return st;
  auto U16 = [](const void* p) { return static_cast<const uint16_t*>(p); };
  const moe_weights_t& w = L->w;
  GateUpParams gp{L->blocks, L->offsets, L->counts,
                  U16(w.gate.scales), U16(w.gate.biases), U16(w.up.scales), U16(w.up.biases),
                  U16(w.sh_gate.scales), U16(w.sh_gate.biases), U16(w.sh_up.scales), U16(w.sh_up.biases),
                  L->h, T, L->err, pipe_trace() ? L->pipe : nullptr, L->x_ilv, L->row_dst, wait_limit_ns()};
  DownParams dp{L->blocks, L->offsets, L->counts, U16(w.down.scales), U16(w.down.biases),
                U16(w.sh_down.scales), U16(w.sh_down.biases), L->y, T, L->err,
                pipe_trace() ? L->pipe + 16 : nullptr, wait_limit_ns()};
  if (T <= GV_MAX_T) {
    // a few rows per expert: weight-streaming GEMVs instead of 128-row tcgen05 tiles
    MOE_TRY(timed(K_GATEUP, s, L->err,
                  [&] { return launch_gateup_gemv(gp, w.gate.q, w.up.q, w.sh_gate.q, w.sh_up.q, s); }),
            "gate/up launch");
    MOE_TRY(timed(K_DOWN, s, L->err, [&] { return launch_down_gemv(dp, L->h, w.down.q, w.sh_down.q, s); }),
            "down launch");
  } else {
    const int grid_gu = gemm_grid(T, GU_MBLK, L->num_sms), grid_dn = gemm_grid(T, DN_MBLK, L->num_sms);
    MOE_TRY(timed(K_GATEUP, s, L->err,
                  [&] { return launch_gateup(L->tm_qg, L->tm_qu, L->tm_sqg, L->tm_squ, L->tm_hs, gp, grid_gu, s); }),
            "gate/up launch");
    dp.small_apart = T <= DS_MAX_T ? 1 : 0;
    MOE_TRY(timed(K_DOWN, s, L->err,
                  [&] { return launch_down(L->tm_qd, L->tm_sqd, L->tm_h, L->tm_y, dp, grid_dn, s); }),
            "down launch");
    if (dp.small_apart) {
      // the small token blocks (at most one per expert), operands swapped
      const int grid_ds = L->num_sms < (NEXP + 1) * DS_PAIRS ? L->num_sms : (NEXP + 1) * DS_PAIRS;
      MOE_TRY(timed(K_DOWN_SWAP, s, L->err,
                    [&] { return launch_down_swap(L->tm_qd, L->tm_sqd, L->tm_h, dp, grid_ds, s); }),
              "down (small blocks) launch");
    }
  }
  MOE_TRY(timed(K_COMBINE, s, L->err,
                [&] {
                  NextLayerIn nx{};
                  if (next && next->w.norm_w)
                    nx = NextLayerIn{static_cast<const __nv_bfloat16*>(next->w.norm_w),
                                     static_cast<const __nv_bfloat16*>(next->w.shared_gate_w), next->xn,
                                     next->x_ilv, next->row_dst, next->row_w};
                  return launch_combine(L->y, L->slot_row, L->row_w, static_cast<const __nv_bfloat16*>(x_orig),
                                        static_cast<__nv_bfloat16*>(out), T, residual, nx, s);
                }),
          "combine launch");
  return MOE_OK;
}

moe_status_t check_call(moe_layer* L, const void* x, int T, const void* out) {
  if (!L || !x || !out) return MOE_ERR_INVALID_ARG;
  if (T < 1 || T > L->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16)) return MOE_ERR_ALIGNMENT;
  return MOE_OK;
}

}  // namespace

extern "C" {

size_t moe_workspace_bytes(const moe_config_t* cfg) {
  if (!cfg || !config_ok(cfg)) return 0;
  return carve(cfg->max_tokens, nullptr, nullptr);
}

moe_status_t moe_layer_create(const moe_config_t* cfg, const moe_weights_t* weights, void* workspace,
                              size_t workspace_bytes, moe_layer_t** out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || !weights) return MOE_ERR_INVALID_ARG;
  if (!config_ok(cfg)) return MOE_ERR_UNSUPPORTED;
  moe_status_t st = MOE_OK;
  const moe_qmat_t* mats[6] = {&weights->gate, &weights->up, &weights->down,
                               &weights->sh_gate, &weights->sh_up, &weights->sh_down};
  for (const moe_qmat_t* m : mats)
    if (!qmat_ok(*m, &st)) return st;
  if (!weights->router_w || !weights->shared_gate_w || !workspace) return MOE_ERR_INVALID_ARG;
  if (!aligned(weights->router_w, 16) || !aligned(weights->shared_gate_w, 16) ||
      (weights->router_bias && !aligned(weights->router_bias, 16)) ||
      (weights->norm_w && !aligned(weights->norm_w, 16)) || !aligned(workspace, 256))
    return MOE_ERR_ALIGNMENT;
  const size_t need = carve(cfg->max_tokens, nullptr, nullptr);
  if (workspace_bytes < need) return MOE_ERR_WORKSPACE;

  moe_layer* L = new (std::nothrow) moe_layer;
  if (!L) return MOE_ERR_CUDA;
  std::memset(L, 0, sizeof *L);
  L->cfg = *cfg;
  L->w = *weights;
  L->ws = static_cast<uint8_t*>(workspace);
  L->ws_bytes = workspace_bytes;
  carve(cfg->max_tokens, L->ws, L);

  auto fail = [&](moe_status_t s) { delete L; return s; };
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&L->num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(cuda_fail("device query", e));
  if (!schedules_fit(cfg->max_tokens, L->num_sms)) {
    snprintf(g_detail, sizeof g_detail, "max_tokens %d needs more tiles per CTA than the schedules hold on %d SMs",
             cfg->max_tokens, L->num_sms);
    return fail(MOE_ERR_UNSUPPORTED);
  }
  if (!get_encode()) {
    snprintf(g_detail, sizeof g_detail, "cuTensorMapEncodeTiled entry point unavailable");
    return fail(MOE_ERR_CUDA);
  }
  if ((e = set_router_attributes()) != cudaSuccess || (e = set_gemm_attributes()) != cudaSuccess)
    return fail(cuda_fail("kernel attributes", e));
  // workspace state shared by every layer bound to it: the error word, the decode
  // ticket and the fused decode kernel's tagged tables and epoch, which start at zero
  // (no tag is zero) -- nothing layer-specific may live in the workspace
  if ((e = cudaMemset(L->err, 0, 256)) != cudaSuccess || (e = cudaMemset(L->dec_counter, 0, 256)) != cudaSuccess ||
      (e = cudaMemset(L->pipe, 0, 32 * 8)) != cudaSuccess ||
      (e = cudaMemset(L->dec_sync, 0, 256)) != cudaSuccess ||
      (e = cudaMemset(L->dec_lt, 0, DEC_LT_WORDS * 8)) != cudaSuccess ||
      (e = cudaMemset(L->dec_ht, 0, DEC_HT_WORDS * 8)) != cudaSuccess ||
      (e = cudaMemset(L->dec_xt, 0, DEC_XT_WORDS * 8)) != cudaSuccess ||
      (e = cudaDeviceSynchronize()) != cudaSuccess)
    return fail(cuda_fail("workspace init", e));

  const int Tm = cfg->max_tokens;
  bool ok = encode_bf16_rows(&L->tm_wr, weights->router_w, HID, NEXP, NEXP) &&
            encode_packed(&L->tm_qg, weights->gate.q, HID / 8, static_cast<uint64_t>(NEXP) * INTER) &&
            encode_packed(&L->tm_qu, weights->up.q, HID / 8, static_cast<uint64_t>(NEXP) * INTER) &&
            encode_packed(&L->tm_sqg, weights->sh_gate.q, HID / 8, SH_INTER) &&
            encode_packed(&L->tm_squ, weights->sh_up.q, HID / 8, SH_INTER) &&
            encode_packed(&L->tm_qd, weights->down.q, INTER / 8, static_cast<uint64_t>(NEXP) * HID) &&
            encode_packed(&L->tm_sqd, weights->sh_down.q, SH_INTER / 8, HID) &&
            encode_bf16_rows(&L->tm_h, L->h, INTER, 9ull * Tm, GX_XBOX) &&
            // epilogue stores of 32 x 32 bf16 boxes from staging tiles written by stmatrix,
            // 64-byte swizzled (16-byte chunk c of staged row k at c ^ ((k >> 1) & 3)) so
            // that stmatrix's eight rows of a matrix fall in different banks
            encode_2d(&L->tm_hs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, L->h, INTER, 9ull * Tm, INTER * 2, 32, 32,
                      CU_TENSOR_MAP_SWIZZLE_64B) &&
            encode_2d(&L->tm_y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, L->y, HID, 9ull * Tm, HID * 2, 32, 32,
                      CU_TENSOR_MAP_SWIZZLE_64B);
  if (!ok) return fail(MOE_ERR_CUDA);
  *out = L;
  return MOE_OK;
}

moe_status_t moe_route(moe_layer_t* L, const void* x, int T, int32_t* topk_idx, float* topk_w, int32_t* counts,
                       int32_t* offsets, int32_t* perm, moe_stream_t stream) {
  if (!L || !x) return MOE_ERR_INVALID_ARG;
  if (T < 1 || T > L->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16)) return MOE_ERR_ALIGNMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const void* xin = nullptr;
  const moe_status_t sn = layer_input(L, x, T, s, &xin, false);
  if (sn != MOE_OK) return sn;
  x = xin;
  if (T <= DEC_MAX_T) {
    const DecodeParams p = decode_params(L, x, T, nullptr, 0);
    MOE_TRY(timed(K_DEC_ROUTER, s, L->err, [&] { return launch_decode_router(p, s); }), "decode router launch");
  } else {
    const moe_status_t st = route_prefill(L, x, T, 0, s);
    if (st != MOE_OK) return st;
  }
  const size_t slots = static_cast<size_t>(T) * TOPK;
  if (topk_idx) MOE_TRY(cudaMemcpyAsync(topk_idx, L->topk_idx, slots * 4, cudaMemcpyDeviceToDevice, s), "copy idx");
  if (topk_w) MOE_TRY(cudaMemcpyAsync(topk_w, L->topk_w, slots * 4, cudaMemcpyDeviceToDevice, s), "copy w");
  if (counts) MOE_TRY(cudaMemcpyAsync(counts, L->counts, NEXP * 4, cudaMemcpyDeviceToDevice, s), "copy counts");
  if (offsets)
    MOE_TRY(cudaMemcpyAsync(offsets, L->offsets, (NEXP + 1) * 4, cudaMemcpyDeviceToDevice, s), "copy offsets");
  if (perm) MOE_TRY(cudaMemcpyAsync(perm, L->row_dst, slots * 4, cudaMemcpyDeviceToDevice, s), "copy perm");
  return MOE_OK;
}

moe_status_t moe_forward(moe_layer_t* L, const void* x, int T, void* out, moe_stream_t stream) {
  const moe_status_t st = check_call(L, x, T, out);
  if (st != MOE_OK) return st;
  if (ranges_overlap(x, out, static_cast<size_t>(T) * HID * 2)) return MOE_ERR_INVALID_ARG;
  return forward_impl(L, x, T, out, 0, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_forward_residual(moe_layer_t* L, const void* x, int T, void* out, moe_stream_t stream) {
  const moe_status_t st = check_call(L, x, T, out);
  if (st != MOE_OK) return st;
  if (x != out && ranges_overlap(x, out, static_cast<size_t>(T) * HID * 2)) return MOE_ERR_INVALID_ARG;
  return forward_impl(L, x, T, out, 1, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_stack_forward(moe_layer_t* const* layers, int n_layers, void* x_io, int T, moe_stream_t stream) {
  if (!layers || n_layers < 1 || !x_io) return MOE_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l) {
    const moe_status_t st = check_call(layers[l], x_io, T, x_io);
    if (st != MOE_OK) return st;
  }
  if (T <= DEC_MAX_T) return decode_forward(layers, n_layers, x_io, T, x_io, 1, reinterpret_cast<cudaStream_t>(stream));
  // each layer's combine also normalises the next layer's input (no separate RMSNorm pass)
  for (int l = 0; l < n_layers; ++l) {
    moe_layer* next = l + 1 < n_layers ? layers[l + 1] : nullptr;
    const moe_status_t st = forward_impl(layers[l], x_io, T, x_io, 1, reinterpret_cast<cudaStream_t>(stream), next,
                                         l > 0);
    if (st != MOE_OK) return st;
  }
  return MOE_OK;
}

moe_status_t moe_stack_forward_host(moe_layer_t* const* layers, int n_layers, const void* x_host, int T,
                                    void* out_host, moe_stream_t stream) {
  if (!layers || n_layers < 1 || !x_host || !out_host || !layers[0]) return MOE_ERR_INVALID_ARG;
  moe_layer* L0 = layers[0];
  if (T < 1 || T > L0->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t bytes = static_cast<size_t>(T) * HID * 2;
  MOE_TRY(cudaMemcpyAsync(L0->x_io, x_host, bytes, cudaMemcpyHostToDevice, s), "copy in");
  const moe_status_t st = moe_stack_forward(layers, n_layers, L0->x_io, T, stream);
  if (st != MOE_OK) return st;
  MOE_TRY(cudaMemcpyAsync(out_host, L0->x_io, bytes, cudaMemcpyDeviceToHost, s), "copy out");
  return MOE_OK;
}

int moe_forward_launches(const moe_layer_t* L, int T) {
  if (!L || T < 1 || T > L->cfg.max_tokens) return 0;
  return T <= DEC_MAX_T ? 1
                        : 6 + (T > GV_MAX_T && T <= DS_MAX_T ? 1 : 0) + (L->w.norm_w ? 1 : 0) -
                              ((T + RT_BM - 1) / RT_BM <= SCAN_FUSE_NBLK ? 1 : 0);
}

int moe_stack_forward_launches(const moe_layer_t* const* layers, int n_layers, int T) {
  if (!layers || n_layers < 1) return 0;
  for (int l = 0; l < n_layers; ++l)
    if (!layers[l] || T < 1 || T > layers[l]->cfg.max_tokens) return 0;
  if (T <= DEC_MAX_T) return (n_layers + DEC_MAX_LAYERS - 1) / DEC_MAX_LAYERS;
  // layers after the first get their input RMSNorm from the previous layer's combine
  int n = 0;
  for (int l = 0; l < n_layers; ++l) n += moe_forward_launches(layers[l], T) - (l > 0 && layers[l]->w.norm_w ? 1 : 0);
  return n;
}

moe_status_t moe_layer_get_error(moe_layer_t* L) {
  if (!L) return MOE_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail("synchronize", e);
  unsigned int v = 0;
  if ((e = cudaMemcpy(&v, L->err, 4, cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail("read error word", e);
  if ((e = cudaMemset(L->err, 0, 4)) != cudaSuccess) return cuda_fail("clear error word", e);
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail("synchronize", e);
  if (v & ERRBIT_TIMEOUT) return MOE_ERR_TIMEOUT;
  if (v & ERRBIT_BOUNDS) return MOE_ERR_DEVICE_BOUNDS;
  return MOE_OK;
}

void moe_layer_destroy(moe_layer_t* L) { delete L; }

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported layer shape or quantisation";
    case MOE_ERR_ALIGNMENT: return "misaligned pointer";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_DEVICE_BOUNDS: return "device-side index out of range";
    case MOE_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

const char* moe_last_error_detail(void) { return g_detail; }

moe_status_t moe_decode_trace(moe_layer_t* L, unsigned long long* out, size_t n_words) {
  if (!L || !out) return MOE_ERR_INVALID_ARG;
  if (n_words > DEC_TRACE_WORDS) n_words = DEC_TRACE_WORDS;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(out, L->dec_trace, n_words * 8, cudaMemcpyDeviceToHost);
  return e == cudaSuccess ? MOE_OK : cuda_fail("decode trace", e);
}

void moe_set_wait_limit_ns(unsigned long long ns) { g_wait_ns.store(ns ? ns : WAIT_LIMIT_NS, std::memory_order_relaxed); }

moe_status_t moe_pipeline_counters(moe_layer_t* L, unsigned long long* out) {
  if (!L || !out) return MOE_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(out, L->pipe, 32 * 8, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(L->pipe, 0, 32 * 8);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  return e == cudaSuccess ? MOE_OK : cuda_fail("pipeline counters", e);
}

void moe_profiler_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof.m);
  g_prof.on = on != 0;
}

int moe_profiler_read(const char** names, double* total_ms, long long* launches, int max) {
  std::lock_guard<std::mutex> lk(g_prof.m);
  double tot[K_COUNT] = {0};
  long long cnt[K_COUNT] = {0};
  for (const ProfRec& r : g_prof.recs) {
    float ms = 0.0f;
    if (cudaEventSynchronize(r.b) == cudaSuccess && cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
      tot[r.id] += ms;
      cnt[r.id] += 1;
    }
    g_prof.pool.push_back(r.a);
    g_prof.pool.push_back(r.b);
  }
  g_prof.recs.clear();
  for (int i = 0; i < K_COUNT && i < max; ++i) {
    if (names) names[i] = kKernelNames[i];
    if (total_ms) total_ms[i] = tot[i];
    if (launches) launches[i] = cnt[i];
  }
  return K_COUNT;
}

}  // extern "C"
