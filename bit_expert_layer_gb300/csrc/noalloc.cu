// noalloc.cu -- moe_decode_forward_static: the decode forward (T <= 8 tokens) for
// callers that cannot allocate device memory.
//
// Who needs it: a host that embeds this library as a plug-in and owns every byte of
// device memory itself (it hands out no allocation hook and no workspace), and
// latency-critical decode loops that must never reach cudaMalloc, which can
// synchronise the whole device.  Such a caller cannot provide the workspace that
// moe_layer_create requires, so this entry point keeps the decode path's scratch in one
// fixed-size array in device memory that the library owns for the life of the process.
//
// The scratch is the file-scope array below.  On the host its name is only a stand-in
// symbol, not a device address, so before the first launch on a device this file asks
// the runtime for the array's device address (cudaGetSymbolAddress, once per device,
// with that device current) and passes that address to the kernels.
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "moe_layer.h"

namespace moe {

namespace {

// Layout of the static scratch for up to DEC_MAX_T tokens.
struct StaticLayout {
  size_t err, sync, lt, ht, xt, topk_idx, topk_w, total;
};

constexpr size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

constexpr StaticLayout make_layout() {
  StaticLayout L{};
  size_t o = 0;
  L.err = o;        o = align256(o + 4);
  L.sync = o;       o = align256(o + 16);
  L.lt = o;         o = align256(o + DEC_LT_WORDS * 8);
  L.ht = o;         o = align256(o + DEC_HT_WORDS * 8);
  L.xt = o;         o = align256(o + DEC_XT_WORDS * 8);
  L.topk_idx = o;   o = align256(o + DEC_MAX_T * TOPK * 4);
  L.topk_w = o;     o = align256(o + DEC_MAX_T * TOPK * 4);
  L.total = o;
  return L;
}

constexpr StaticLayout kLayout = make_layout();
constexpr size_t kStaticScratchBytes = 3u << 20;   // 3 MiB, held by every device that loads the library
static_assert(kLayout.total <= kStaticScratchBytes, "static scratch too small for the decode path");

}  // namespace

// The decode path's scratch.  Every call of moe_decode_forward_static on a device uses
// this same array, which keeps the last call's contents between calls.
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_addr_mutex;
unsigned char* g_addr[kMaxDevices] = {};

// The array's device address on the current device, looked up on the first call there.
cudaError_t scratch_address(unsigned char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_addr_mutex);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

bool ok16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) % 16) == 0; }

moe_status_t fail(const char* what, cudaError_t e) {
  set_error_detail(what, e);
  return MOE_ERR_CUDA;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_decode_forward_static(const moe_weights_t* w, const void* x, int T, void* out,
                                                  int residual, moe_stream_t stream) {
  if (!w || !x || !out) return MOE_ERR_INVALID_ARG;
  if (T < 1 || T > DEC_MAX_T) {
    char msg[160];
    snprintf(msg, sizeof msg, "moe_decode_forward_static: T=%d is outside 1..%d, the limit of its static scratch", T,
             DEC_MAX_T);
    set_error_detail(msg, cudaSuccess);
    fprintf(stderr, "%s\n", msg);
    return MOE_ERR_INVALID_ARG;
  }
  const moe_qmat_t* mats[6] = {&w->gate, &w->up, &w->down, &w->sh_gate, &w->sh_up, &w->sh_down};
  for (const moe_qmat_t* m : mats)
    if (!ok16(m->q) || !ok16(m->scales) || !ok16(m->biases)) return MOE_ERR_ALIGNMENT;
  if (!ok16(w->router_w) || !ok16(w->shared_gate_w) || !ok16(x) || !ok16(out) ||
      (w->router_bias && !ok16(w->router_bias)) || (w->norm_w && !ok16(w->norm_w)))
    return MOE_ERR_ALIGNMENT;
  const uintptr_t xa = reinterpret_cast<uintptr_t>(x), oa = reinterpret_cast<uintptr_t>(out);
  const size_t bytes = static_cast<size_t>(T) * HID * 2;
  if (x != out && xa < oa + bytes && oa < xa + bytes) return MOE_ERR_INVALID_ARG;
  if (x == out && !residual) return MOE_ERR_INVALID_ARG;

  unsigned char* base = nullptr;
  cudaError_t e = scratch_address(&base);
  if (e != cudaSuccess) return fail("moe_decode_forward_static: scratch address", e);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the array starts at zero when the library is loaded: the error word (which collects
  // the device errors of every call until moe_decode_static_get_error reads it), the
  // tagged tables and the epoch word; the kernel keeps the tables and the epoch valid

  static DecLayersParams p;   // about 9 KB: kept off the stack, filled under the lock
  static std::mutex m;
  std::lock_guard<std::mutex> lk(m);
  std::memset(&p, 0, sizeof p);
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.T = T;
  p.n_layers = 1;
  p.residual = residual ? 1 : 0;
  p.lt = reinterpret_cast<unsigned long long*>(base + kLayout.lt);
  p.ht = reinterpret_cast<unsigned long long*>(base + kLayout.ht);
  p.xt = reinterpret_cast<unsigned long long*>(base + kLayout.xt);
  p.sync = reinterpret_cast<unsigned int*>(base + kLayout.sync);
  p.topk_idx = reinterpret_cast<int*>(base + kLayout.topk_idx);
  p.topk_w = reinterpret_cast<float*>(base + kLayout.topk_w);
  p.wait_ns = wait_limit_ns();
  DecLayer& d = p.layer[0];
  d.router_w = static_cast<const __nv_bfloat16*>(w->router_w);
  d.router_bias = w->router_bias;
  d.shared_gate_w = static_cast<const __nv_bfloat16*>(w->shared_gate_w);
  d.norm_w = static_cast<const __nv_bfloat16*>(w->norm_w);
  auto Q = [](const moe_qmat_t& mq, const uint32_t*& q, const uint16_t*& sc, const uint16_t*& bi) {
    q = static_cast<const uint32_t*>(mq.q);
    sc = static_cast<const uint16_t*>(mq.scales);
    bi = static_cast<const uint16_t*>(mq.biases);
  };
  Q(w->gate, d.gq, d.gs, d.gb);
  Q(w->up, d.uq, d.us, d.ub);
  Q(w->down, d.dq, d.ds, d.db);
  Q(w->sh_gate, d.sgq, d.sgs, d.sgb);
  Q(w->sh_up, d.suq, d.sus, d.sub);
  Q(w->sh_down, d.sdq, d.sds, d.sdb);
  d.err = reinterpret_cast<unsigned int*>(base + kLayout.err);
  e = launch_decode_layers(p, s);
  if (e != cudaSuccess) return fail("moe_decode_forward_static: launch", e);
  return MOE_OK;
}

extern "C" moe_status_t moe_decode_static_get_error(void) {
  unsigned char* base = nullptr;
  cudaError_t e = scratch_address(&base);
  if (e != cudaSuccess) return fail("moe_decode_static_get_error: scratch address", e);
  unsigned int v = 0;
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) return fail("moe_decode_static_get_error: synchronize", e);
  if ((e = cudaMemcpy(&v, base + kLayout.err, 4, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return fail("moe_decode_static_get_error: read", e);
  if ((e = cudaMemset(base + kLayout.err, 0, 4)) != cudaSuccess) return fail("moe_decode_static_get_error: clear", e);
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) return fail("moe_decode_static_get_error: synchronize", e);
  if (v & ERRBIT_TIMEOUT) return MOE_ERR_TIMEOUT;
  if (v & ERRBIT_BOUNDS) return MOE_ERR_DEVICE_BOUNDS;
  return MOE_OK;
}
