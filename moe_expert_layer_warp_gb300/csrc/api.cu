// api.cu — the extern "C" entry points of libmoewarp.so declared in
// include/moe_warp.h: argument checks, scratch layout, kernel launches.
// Nothing here allocates device memory.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include <mutex>

#include "moe_warp.h"
#include "launch.h"

namespace {

// Device error word written by kernels (see common.cuh). One per device the
// library runs on; host code reaches it through cudaGetSymbolAddress.
__device__ unsigned int g_moe_err;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int num_sms = 0;
  unsigned int* err = nullptr;
};

DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;
thread_local char g_last_cuda_err[256] = "";

moe_status cuda_fail(cudaError_t e, const char* where) {
  snprintf(g_last_cuda_err, sizeof g_last_cuda_err, "%s: %s", where, cudaGetErrorString(e));
  return MOE_ECUDA;
}

moe_status device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return MOE_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_moe_err);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
    d.err = static_cast<unsigned int*>(p);
    d.ready = true;
  }
  *out = &d;
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status check_desc(const moe_layer_desc* d) {
  if (!d) return MOE_EINVAL;
  if (d->d <= 0 || d->inter <= 0 || d->n_experts <= 0 || d->top_k <= 0) return MOE_EINVAL;
  if (d->top_k > d->n_experts || d->n_experts > MOE_MAX_EXPERTS || d->top_k > MOE_MAX_TOPK)
    return MOE_EINVAL;
  if (d->n_shared < 0 || d->n_shared > MOE_MAX_SHARED) return MOE_EINVAL;
  if (d->wdtype != MOE_W_F32 && d->wdtype != MOE_W_BF16) return MOE_EINVAL;
  if (d->d % 64 != 0 || d->inter % 64 != 0) return MOE_EUNSUPPORTED;
  return MOE_OK;
}

moe_status check_n(const moe_layer_desc* d, int32_t n) {
  if (n < 1 || n > MOE_MAX_TOKENS || (int64_t)n * d->top_k > MOE_MAX_PAIRS) return MOE_EINVAL;
  return MOE_OK;
}

// Scratch layout for passes of up to n_max tokens (every region 256-byte
// aligned relative to the workspace base); hrows = n_max·k + s·n_max:
//   logits   [n_max][E] fp32          routing
//   h        [hrows][I] fp32          SwiGLU activations, CUDA-core groups
//   h16      [2][hrows][I] bf16       SwiGLU activations of tensor-core groups, hi and lo halves
//   xg       [n_max·k][d] fp32        x rows gathered in union order
//   xg16     [2][n_max·k][d] bf16     their hi and lo bf16 halves
//   x16      [2][n_max][d] bf16       hi and lo bf16 halves of x
//   x32      [n_max][d] fp32          a copy of x (CUDA-core kernel input)
//   sync     [kCcSyncInts] int32      CUDA-core kernel job counter, group counts
//   sync_mma [kMmaSyncInts] int32     tensor-core kernel job counter, group counts, piece counts
//   ydone    [64] int32                phase-1 units stored, for the combine fused into the kernel
//   part     [kMmaPartBytes]           tensor-core kernel partial sums of K pieces (bf16 layers)
struct WsLayout {
  size_t logits, h, h16, xg, xg16, x16, x32, sync, sync_mma, ydone, part, part_bytes, total;
};

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

WsLayout ws_layout(const moe_layer_desc* d, int32_t n_max) {
  WsLayout L;
  const size_t hrows = (size_t)n_max * d->top_k + (size_t)d->n_shared * n_max;
  const size_t pairs = (size_t)n_max * d->top_k;
  size_t off = 0;
  L.logits = off;
  off = align256(off + (size_t)n_max * d->n_experts * 4);
  L.h = off;
  off = align256(off + hrows * d->inter * 4);
  L.h16 = off;
  off = align256(off + 2 * hrows * d->inter * 2);
  L.xg = off;
  off = align256(off + pairs * d->d * 4);
  L.xg16 = off;
  off = align256(off + 2 * pairs * d->d * 2);
  L.x16 = off;
  off = align256(off + 2 * (size_t)n_max * d->d * 2);
  L.x32 = off;
  off = align256(off + (size_t)n_max * d->d * 4);
  L.sync = off;
  off = align256(off + (size_t)moe::kCcSyncInts * 4);
  L.sync_mma = off;
  off = align256(off + (size_t)moe::kMmaSyncInts * 4);
  L.ydone = off;
  off = align256(off + 64 * 4);
  L.part = off;
  L.part_bytes = d->wdtype == MOE_W_BF16 ? moe::kMmaPartBytes : 0;
  off = align256(off + L.part_bytes);
  L.total = off;
  return L;
}

// Which expert kernel a bf16 call runs on; the two never share a call (run
// side by side they slow each other). The tensor-core kernel streams each
// weight tile through shared memory into the tensor cores with no
// per-element instruction, so it keeps its rate however many tokens a group
// holds; but it works in 128-row tiles, a group's down tiles wait for all of
// its gate/up tiles, and with fewer tiles than SMs it must cut tiles along K
// and add the pieces across CTAs. The CUDA-core kernel works in 32- and
// 64-row tiles, so few groups still fill the GPU, but its arithmetic per
// weight byte grows with the tokens per group. Measured on GB300 with each
// kernel forced (DeepSeek-V2-Lite-, Mixtral- and DeepSeek-V3-shaped layers,
// per-slot pairs of one expert run side by side): one-token groups
// (per-slot) go faster on CUDA cores below ~400 tiles or 12 groups, and at
// any count when an expert spans 128 or more 128-row tiles (Mixtral: 1-15 %
// faster; V3, 72 tiles, is 9 % faster on the tensor cores); dedup groups,
// which hold several tokens, go faster on the tensor cores from ~350 tiles
// with 15 groups or more, or with 3 tokens or more per group, or in passes
// of more tokens than a CUDA-core sub-group holds (kCcSub): there a group
// of correlated tokens outgrows one sub-group, and its sub-groups each read
// the expert again (measured, Mixtral-shaped dedup at 5 tokens: 13 % slower
// on CUDA cores at rho = 0.9, 59 % at 0.99).
// The groups of a dedup call are known only on the device: the estimate
// takes half of min(E, n·k) distinct experts, which the union reaches at
// hidden-state correlations near 0.9; far from it the estimate can pick the
// slower kernel (measured: up to 6 % on the Mixtral-shaped calls at 5-6
// tokens and rho = 0). MOE_MMA_MIN_M in the environment (read once; for
// tuning) fixes instead the smallest group that runs on the tensor cores.
int mma_min_m(const moe_layer_desc* d, int engine, int32_t n) {
  static const int forced = [] {
    const char* e = getenv("MOE_MMA_MIN_M");
    const int x = e ? atoi(e) : 0;
    return x >= 1 ? x : 0;
  }();
  if (forced) return forced;
  const int tiles = (d->inter + 127) / 128 + (d->d + 127) / 128;  // per group
  const int pairs = n * d->top_k;
  const int shared = d->n_shared * ((n + moe::kMmaSub - 1) / moe::kMmaSub);
  bool mma;
  if (engine == 0) {
    const int groups = pairs + shared;
    mma = groups * tiles >= 400 && groups >= 12 && tiles < 128;
  } else {
    const int routed = std::max(1, std::min(d->n_experts, pairs) / 2);
    const int groups = routed + shared;
    mma = groups * tiles >= 350 && (groups >= 15 || pairs >= 3 * routed || n > moe::kCcSub);
  }
  return mma ? 1 : 0x7fffffff;
}

moe_status check_ws(const moe_layer_desc* d, int32_t n, const void* ws, size_t ws_bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_EINVAL;
  if (ws_bytes < ws_layout(d, n).total) return MOE_EINVAL;
  return MOE_OK;
}

moe_status check_weights(const moe_layer_desc* d, const moe_layer_weights* w) {
  if (!w) return MOE_EINVAL;
  if (!w->w_gate || !w->w_up || !w->w_down) return MOE_EINVAL;
  if (!aligned16(w->w_gate) || !aligned16(w->w_up) || !aligned16(w->w_down)) return MOE_EINVAL;
  if (d->n_shared > 0) {
    if (!w->ws_gate || !w->ws_up || !w->ws_down) return MOE_EINVAL;
    if (!aligned16(w->ws_gate) || !aligned16(w->ws_up) || !aligned16(w->ws_down))
      return MOE_EINVAL;
  }
  return MOE_OK;
}

#define MOE_TRY(expr)                  \
  do {                                 \
    moe_status _st = (expr);           \
    if (_st != MOE_OK) return _st;     \
  } while (0)

}  // namespace

extern "C" {

size_t moe_workspace_bytes(const moe_layer_desc* desc, int32_t n_max) {
  if (check_desc(desc) != MOE_OK || check_n(desc, n_max) != MOE_OK) return 0;
  return ws_layout(desc, n_max).total;
}

moe_status moe_gate(const moe_layer_desc* desc, const float* w_router, const float* x, int32_t n,
                    float* logits, void* stream) {
  MOE_TRY(check_desc(desc));
  MOE_TRY(check_n(desc, n));
  if (!w_router || !x || !logits) return MOE_EINVAL;
  if (!aligned16(w_router) || !aligned16(x) || (reinterpret_cast<uintptr_t>(logits) & 3u) != 0)
    return MOE_EINVAL;
  DeviceInfo* di;
  MOE_TRY(device_info(&di));
  cudaError_t e = moe::launch_gate(desc->d, desc->n_experts, n, x, w_router, logits,
                                   static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_gate launch");
}

moe_status moe_route(const moe_layer_desc* desc, const float* w_router, const float* x,
                     int32_t n, int32_t* topk_idx, float* topk_w, void* workspace,
                     size_t workspace_bytes, void* stream) {
  return moe_route_biased(desc, w_router, nullptr, 1, x, n, topk_idx, topk_w, workspace,
                          workspace_bytes, stream);
}

moe_status moe_route_biased(const moe_layer_desc* desc, const float* w_router, const float* bias,
                            int32_t bias_in_weights, const float* x, int32_t n,
                            int32_t* topk_idx, float* topk_w, void* workspace,
                            size_t workspace_bytes, void* stream) {
  MOE_TRY(check_desc(desc));
  if (bias_in_weights != 0 && bias_in_weights != 1) return MOE_EINVAL;
  if (bias && (reinterpret_cast<uintptr_t>(bias) & 3u) != 0) return MOE_EINVAL;
  MOE_TRY(check_n(desc, n));
  if (!w_router || !x || !topk_idx || !topk_w) return MOE_EINVAL;
  if (!aligned16(w_router) || !aligned16(x)) return MOE_EINVAL;
  MOE_TRY(check_ws(desc, n, workspace, workspace_bytes));
  DeviceInfo* di;
  MOE_TRY(device_info(&di));
  WsLayout L = ws_layout(desc, n);
  float* logits = reinterpret_cast<float*>(static_cast<char*>(workspace) + L.logits);
  cudaError_t e = moe::launch_route(desc->d, desc->n_experts, desc->top_k, n, x, w_router, bias,
                                    bias_in_weights, logits, topk_idx, topk_w,
                                    static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_route launch");
}

moe_status moe_build_union(const moe_layer_desc* desc, const int32_t* topk_idx, int32_t n,
                           const moe_union* u, void* stream) {
  MOE_TRY(check_desc(desc));
  MOE_TRY(check_n(desc, n));
  if (!topk_idx || !u || !u->union_ids || !u->union_count || !u->offsets || !u->pair_tok ||
      !u->pair_slot || !u->bytes)
    return MOE_EINVAL;
  if ((reinterpret_cast<uintptr_t>(u->bytes) & 7u) != 0) return MOE_EINVAL;
  DeviceInfo* di;
  MOE_TRY(device_info(&di));
  cudaError_t e = moe::launch_union(desc->d, desc->inter, desc->n_experts, desc->top_k,
                                    desc->n_shared, desc->wdtype == MOE_W_F32 ? 4 : 2, n,
                                    topk_idx, u->union_ids, u->union_count, u->offsets,
                                    u->pair_tok, u->pair_slot, u->bytes, di->err,
                                    static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_build_union launch");
}

}  // extern "C"

namespace {

moe_status check_route_union(const moe_layer_desc* desc, const float* w_router, const float* bias,
                             int32_t bias_in_weights, const float* x, int32_t n,
                             const int32_t* topk_idx, const float* topk_w, const moe_union* u,
                             const void* workspace, size_t workspace_bytes) {
  MOE_TRY(check_desc(desc));
  if (bias_in_weights != 0 && bias_in_weights != 1) return MOE_EINVAL;
  if (bias && (reinterpret_cast<uintptr_t>(bias) & 3u) != 0) return MOE_EINVAL;
  MOE_TRY(check_n(desc, n));
  if (!w_router || !x || !topk_idx || !topk_w) return MOE_EINVAL;
  if (!aligned16(w_router) || !aligned16(x)) return MOE_EINVAL;
  if (!u || !u->union_ids || !u->union_count || !u->offsets || !u->pair_tok || !u->pair_slot ||
      !u->bytes)
    return MOE_EINVAL;
  if ((reinterpret_cast<uintptr_t>(u->bytes) & 7u) != 0) return MOE_EINVAL;
  return check_ws(desc, n, workspace, workspace_bytes);
}

// Routing and union (arguments already checked); prep: null, or the pass's
// prep work done by the routing kernels.
moe_status launch_route_union(const moe_layer_desc* desc, const float* w_router, const float* bias,
                              int32_t bias_in_weights, const float* x, int32_t n,
                              int32_t* topk_idx, float* topk_w, const moe_union* u,
                              void* workspace, const moe::PassPrep* prep, void* stream) {
  WsLayout L = ws_layout(desc, n);
  float* logits = reinterpret_cast<float*>(static_cast<char*>(workspace) + L.logits);
  cudaError_t e = moe::launch_route_union(
      desc->d, desc->inter, desc->n_experts, desc->top_k, desc->n_shared,
      desc->wdtype == MOE_W_F32 ? 4 : 2, n, x, w_router, bias, bias_in_weights, logits, topk_idx,
      topk_w, u->union_ids, u->union_count, u->offsets, u->pair_tok, u->pair_slot, u->bytes, prep,
      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_route_union launch");
}

}  // namespace

extern "C" {

moe_status moe_route_union(const moe_layer_desc* desc, const float* w_router, const float* bias,
                           int32_t bias_in_weights, const float* x, int32_t n,
                           int32_t* topk_idx, float* topk_w, const moe_union* u, void* workspace,
                           size_t workspace_bytes, void* stream) {
  MOE_TRY(check_route_union(desc, w_router, bias, bias_in_weights, x, n, topk_idx, topk_w, u,
                            workspace, workspace_bytes));
  DeviceInfo* di;
  MOE_TRY(device_info(&di));
  return launch_route_union(desc, w_router, bias, bias_in_weights, x, n, topk_idx, topk_w, u,
                            workspace, nullptr, stream);
}

}  // extern "C"

namespace {

moe_status check_engine(const moe_layer_desc* desc, const moe_layer_weights* w, const float* x,
                        int32_t n, const float* topk_w, const void* workspace,
                        size_t workspace_bytes, const float* y_slot) {
  MOE_TRY(check_desc(desc));
  MOE_TRY(check_n(desc, n));
  MOE_TRY(check_weights(desc, w));
  if (!x || !topk_w || !y_slot || !aligned16(x)) return MOE_EINVAL;
  return check_ws(desc, n, workspace, workspace_bytes);
}

// The arguments of one expert-engine call (already checked); y non-null
// fuses the combine into the expert kernel's last phase.
moe::ExpertArgs expert_args(int engine, const moe_layer_desc* desc, const moe_layer_weights* w,
                            const float* x, int32_t n, const int32_t* topk_idx,
                            const moe_union* u, const float* topk_w, void* workspace,
                            float* y_slot, float* y, const DeviceInfo* di) {
  WsLayout L = ws_layout(desc, n);
  moe::ExpertArgs a;
  memset(&a, 0, sizeof a);
  a.d = desc->d;
  a.I = desc->inter;
  a.E = desc->n_experts;
  a.k = desc->top_k;
  a.s = desc->n_shared;
  a.n = n;
  a.wdtype = desc->wdtype;
  a.engine = engine;
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  if (u) {
    a.union_ids = u->union_ids;
    a.union_count = u->union_count;
    a.offsets = u->offsets;
    a.pair_tok = u->pair_tok;
    a.pair_slot = u->pair_slot;
  }
  a.x = x;
  a.w_gate = w->w_gate;
  a.w_up = w->w_up;
  a.w_down = w->w_down;
  a.ws_gate = w->ws_gate;
  a.ws_up = w->ws_up;
  a.ws_down = w->ws_down;
  a.h = reinterpret_cast<float*>(static_cast<char*>(workspace) + L.h);
  char* ws = static_cast<char*>(workspace);
  a.xg = reinterpret_cast<float*>(ws + L.xg);
  const size_t hrows = (size_t)n * desc->top_k + (size_t)desc->n_shared * n;
  a.h16 = reinterpret_cast<uint16_t*>(ws + L.h16);
  a.h16lo = a.h16 + hrows * desc->inter;
  a.xg16 = reinterpret_cast<uint16_t*>(ws + L.xg16);
  a.xg16lo = a.xg16 + (size_t)n * desc->top_k * desc->d;
  a.x16 = reinterpret_cast<uint16_t*>(ws + L.x16);
  a.x16lo = a.x16 + (size_t)n * desc->d;
  a.x32 = reinterpret_cast<float*>(ws + L.x32);
  a.sync = reinterpret_cast<int*>(ws + L.sync);
  a.sync_mma = reinterpret_cast<int*>(ws + L.sync_mma);
  a.part = reinterpret_cast<float*>(ws + L.part);
  a.part_bytes = L.part_bytes;
  // fp32 weights never go to the tensor cores (a tf32 product would miss the
  // fp32 tolerance), so every fp32 group stays on the CUDA-core kernel.
  a.mma_min_m = desc->wdtype == MOE_W_BF16 ? mma_min_m(desc, engine, n) : 0x7fffffff;
  a.y_slot = y_slot;
  a.y = y;
  a.ydone = reinterpret_cast<int*>(ws + L.ydone);
  // Measured on GB300 (V2-Lite): normal eviction of the weight lines speeds
  // per-slot calls of 5 and 9 tokens by 2-4 % and slows 1- and 2-token
  // calls and dedup calls, which repeat no expert, by 0.4-3 %.
  a.keep_weights = engine == 0 && n >= 3 ? 1 : 0;
  // Measured on GB300 (V2-Lite passes): prefetching the shared experts'
  // weights into L2 while the expert kernel waits for the routing makes dedup
  // passes 0.4-4.2 us shorter and one-token per-slot passes 0.5 us shorter;
  // per-slot calls on the tensor cores, which lean on L2 for their repeated
  // experts, were 0.9-1.0 us longer with it.
  a.prefetch_shared = engine == 1 || a.mma_min_m > n ? 1 : 0;
  a.err = di->err;
  return a;
}

// One expert-engine call with its own prep kernel.
moe_status run_engine(int engine, const moe_layer_desc* desc, const moe_layer_weights* w,
                      const float* x, int32_t n, const int32_t* topk_idx, const moe_union* u,
                      const float* topk_w, void* workspace, size_t workspace_bytes,
                      float* y_slot, void* stream) {
  MOE_TRY(check_engine(desc, w, x, n, topk_w, workspace, workspace_bytes, y_slot));
  DeviceInfo* di;
  MOE_TRY(device_info(&di));
  const moe::ExpertArgs a =
      expert_args(engine, desc, w, x, n, topk_idx, u, topk_w, workspace, y_slot, nullptr, di);
  cudaError_t e = moe::launch_expert_engine(a, di->num_sms, false, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "expert engine launch");
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_verify_perslot(const moe_layer_desc* desc, const moe_layer_weights* weights,
                              const float* x, int32_t n, const int32_t* topk_idx,
                              const float* topk_w, void* workspace, size_t workspace_bytes,
                              float* y_slot, void* stream) {
  if (!topk_idx) return MOE_EINVAL;
  return run_engine(0, desc, weights, x, n, topk_idx, nullptr, topk_w, workspace,
                    workspace_bytes, y_slot, stream);
}

moe_status moe_verify_dedup(const moe_layer_desc* desc, const moe_layer_weights* weights,
                            const float* x, int32_t n, const moe_union* u, const float* topk_w,
                            void* workspace, size_t workspace_bytes, float* y_slot,
                            void* stream) {
  if (!u || !u->union_ids || !u->union_count || !u->offsets || !u->pair_tok || !u->pair_slot)
    return MOE_EINVAL;
  return run_engine(1, desc, weights, x, n, nullptr, u, topk_w, workspace, workspace_bytes,
                    y_slot, stream);
}

// ------------------------------------------------ allocation-free variant --
// Scratch for moe_verify_dedup_noalloc: a fixed array in the library's own
// device memory, so that a caller who cannot allocate device memory still
// gets the dedup engine. Every GPU that loads the library holds this array
// until the process exits. Host code must not pass the symbol itself to a
// kernel: on the host, g_noalloc_scratch names a host-side stand-in, not the
// device array. Its device address is looked up per device below.
}  // extern "C"

namespace {
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocSlot {
  bool ready = false;
  void* ptr = nullptr;
};
NoAllocSlot g_noalloc[kMaxDevices];

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (with that device current) and cached.
moe_status noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return MOE_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  NoAllocSlot& s = g_noalloc[dev];
  if (!s.ready) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(g_noalloc_scratch)");
    s.ptr = p;
    s.ready = true;
  }
  *out = s.ptr;
  return MOE_OK;
}
}  // namespace

extern "C" {

size_t moe_noalloc_scratch_limit(void) { return kNoAllocScratchBytes; }

moe_status moe_verify_dedup_noalloc(const moe_layer_desc* desc, const moe_layer_weights* weights,
                                    const float* x, int32_t n, const moe_union* u,
                                    const float* topk_w, float* y_slot, void* stream) {
  // Every refusal below leaves its own reason; none is left over from an
  // earlier call.
  g_last_cuda_err[0] = '\0';
  auto refuse = [](moe_status st, const char* why) {
    snprintf(g_last_cuda_err, sizeof g_last_cuda_err, "moe_verify_dedup_noalloc: %s", why);
    return st;
  };
  moe_status st = check_desc(desc);
  if (st != MOE_OK) return refuse(st, "invalid or unsupported layer descriptor");
  if (check_n(desc, n) != MOE_OK) return refuse(MOE_EINVAL, "pass size n out of range");
  const size_t need = ws_layout(desc, n).total;
  if (need > kNoAllocScratchBytes) {
    snprintf(g_last_cuda_err, sizeof g_last_cuda_err,
             "moe_verify_dedup_noalloc: this pass needs %zu bytes of scratch, above the "
             "static maximum of %zu bytes; use moe_verify_dedup with a workspace",
             need, kNoAllocScratchBytes);
    return MOE_EINVAL;
  }
  if (check_weights(desc, weights) != MOE_OK)
    return refuse(MOE_EINVAL, "null or misaligned weight pointer");
  if (!x || !topk_w || !y_slot || !aligned16(x))
    return refuse(MOE_EINVAL, "null x, topk_w or y_slot, or x not 16-byte aligned");
  if (!u || !u->union_ids || !u->union_count || !u->offsets || !u->pair_tok || !u->pair_slot)
    return refuse(MOE_EINVAL, "null union pointer");
  void* scratch = nullptr;
  MOE_TRY(noalloc_scratch(&scratch));
  return moe_verify_dedup(desc, weights, x, n, u, topk_w, scratch, kNoAllocScratchBytes, y_slot,
                          stream);
}

moe_status moe_combine(const moe_layer_desc* desc, const float* y_slot, int32_t n, float* y,
                       void* stream) {
  MOE_TRY(check_desc(desc));
  MOE_TRY(check_n(desc, n));
  if (!y_slot || !y || !aligned16(y_slot) || !aligned16(y)) return MOE_EINVAL;
  cudaError_t e = moe::launch_combine(desc->d, desc->top_k + desc->n_shared, n, y_slot, y,
                                      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_combine launch");
}

// A whole pass: routing and union, one engine, and the combine either as a
// launch of its own (fused = false) or as the expert kernel's last phase.
// The routing kernels also do the expert call's prep work (PassPrep), so
// that the expert kernel follows them directly.
static moe_status verify_pass(bool fused, const moe_layer_desc* desc,
                              const moe_layer_weights* weights, const float* bias,
                              int32_t bias_in_weights, const float* x, int32_t n, int32_t engine,
                              int32_t* topk_idx, float* topk_w, const moe_union* u,
                              void* workspace, size_t workspace_bytes, float* y_slot, float* y,
                              void* stream) {
  if (!weights || !y_slot || !y || (engine != MOE_ENGINE_PERSLOT && engine != MOE_ENGINE_DEDUP))
    return MOE_EINVAL;
  if (!aligned16(y_slot) || !aligned16(y)) return MOE_EINVAL;
  MOE_TRY(check_route_union(desc, weights->w_router, bias, bias_in_weights, x, n, topk_idx, topk_w,
                            u, workspace, workspace_bytes));
  MOE_TRY(check_engine(desc, weights, x, n, topk_w, workspace, workspace_bytes, y_slot));
  DeviceInfo* di;
  MOE_TRY(device_info(&di));
  const int eng = engine == MOE_ENGINE_PERSLOT ? 0 : 1;
  const moe::ExpertArgs a =
      expert_args(eng, desc, weights, x, n, eng == 0 ? topk_idx : nullptr, eng == 1 ? u : nullptr,
                  topk_w, workspace, y_slot, fused ? y : nullptr, di);
  const bool bf16 = desc->wdtype == MOE_W_BF16;
  moe::PassPrep pp;
  memset(&pp, 0, sizeof pp);
  pp.x32 = a.x32;
  pp.x16 = bf16 ? a.x16 : nullptr;
  pp.x16lo = bf16 ? a.x16lo : nullptr;
  pp.sync_cc = a.sync;
  pp.sync_mma = a.sync_mma;
  pp.ydone = a.y ? a.ydone : nullptr;
  if (eng == 1) {
    pp.xg = a.xg;
    pp.xg16 = bf16 ? a.xg16 : nullptr;
    pp.xg16lo = bf16 ? a.xg16lo : nullptr;
    const int pairs = n * desc->top_k;
    pp.gather_rows = (pairs + di->num_sms - 1) / di->num_sms;
  }
  MOE_TRY(launch_route_union(desc, weights->w_router, bias, bias_in_weights, x, n, topk_idx, topk_w,
                             u, workspace, &pp, stream));
  cudaError_t e = moe::launch_expert_engine(a, di->num_sms, true, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "expert engine launch");
  return fused ? MOE_OK : moe_combine(desc, y_slot, n, y, stream);
}

moe_status moe_verify_pass(const moe_layer_desc* desc, const moe_layer_weights* weights,
                           const float* bias, int32_t bias_in_weights, const float* x, int32_t n,
                           int32_t engine, int32_t* topk_idx, float* topk_w, const moe_union* u,
                           void* workspace, size_t workspace_bytes, float* y_slot, float* y,
                           void* stream) {
  return verify_pass(false, desc, weights, bias, bias_in_weights, x, n, engine, topk_idx, topk_w,
                     u, workspace, workspace_bytes, y_slot, y, stream);
}

moe_status moe_verify_pass_fused(const moe_layer_desc* desc, const moe_layer_weights* weights,
                                 const float* bias, int32_t bias_in_weights, const float* x,
                                 int32_t n, int32_t engine, int32_t* topk_idx, float* topk_w,
                                 const moe_union* u, void* workspace, size_t workspace_bytes,
                                 float* y_slot, float* y, void* stream) {
  return verify_pass(true, desc, weights, bias, bias_in_weights, x, n, engine, topk_idx, topk_w,
                     u, workspace, workspace_bytes, y_slot, y, stream);
}

moe_status moe_diag_bounded_wait(int32_t limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return MOE_EINVAL;
  DeviceInfo* di;
  MOE_TRY(device_info(&di));
  cudaError_t e = moe::launch_diag_wait((unsigned long long)limit_us * 1000ull, di->err,
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_diag_bounded_wait launch");
}

moe_status moe_last_device_error(void* stream) {
  DeviceInfo* di;
  MOE_TRY(device_info(&di));
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_moe_err, sizeof word);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol");
  if (word != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_moe_err, &zero, sizeof zero);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol");
    snprintf(g_last_cuda_err, sizeof g_last_cuda_err, "device error word 0x%08x", word);
    return (word & 0xffu) == 3u ? MOE_ETIMEOUT : MOE_EDEVICE;
  }
  return MOE_OK;
}

const char* moe_status_str(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_EINVAL: return "MOE_EINVAL: invalid argument";
    case MOE_ECUDA: return "MOE_ECUDA: CUDA runtime error";
    case MOE_ETIMEOUT: return "MOE_ETIMEOUT: a bounded device wait expired";
    case MOE_EUNSUPPORTED: return "MOE_EUNSUPPORTED: shape not covered";
    case MOE_EDEVICE: return "MOE_EDEVICE: a device-side check failed";
  }
  return "unknown moe_status";
}

const char* moe_last_cuda_error_string(void) { return g_last_cuda_err; }

}  // extern "C"
