// launch.h — host-side launchers of the kernels behind the C ABI. Internal to
// libmoewarp.so: api.cu validates arguments, then calls these.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_warp.h"

namespace moe {

// Launches `kernel` on `stream` with programmatic stream serialization, so
// that it may start while the previous kernel in the stream finishes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Routing: gate GEMV with compensated fp32 dots (writes logits[n][E] into
// scratch), then warp-per-token top-k + softmax over the k kept scores;
// bias (nullable) [E] is added to the logits for the selection, and to the
// softmax's inputs too when bias_in_weights.
cudaError_t launch_route(int d, int E, int k, int n, const float* x, const float* w_router,
                         const float* bias, int bias_in_weights, float* logits, int32_t* topk_idx,
                         float* topk_w, cudaStream_t stream);

// The gate GEMV alone: logits[n][E] = x·W_gᵀ (compensated fp32 dots).
cudaError_t launch_gate(int d, int E, int n, const float* x, const float* w_router, float* logits,
                        cudaStream_t stream);

// Union of selected experts, pairs grouped by (expert, token), byte counts.
cudaError_t launch_union(int d, int I, int E, int k, int s, int wbytes, int n,
                         const int32_t* topk_idx, int32_t* union_ids, int32_t* union_count,
                         int32_t* offsets, int32_t* pair_tok, int32_t* pair_slot,
                         uint64_t* bytes, unsigned int* err, cudaStream_t stream);

// What the expert call's prep kernel does, done instead by the routing
// kernels of a whole pass (moe_verify_pass), so that the expert kernel
// directly follows the routing. The gate kernel zeroes the expert kernels'
// counters (and ydone, when not null) and writes x32 = x and, when x16 is
// not null, x's bf16 hi/lo halves (x16, x16lo); with xg not null the
// top-k/union kernel also gathers the dedup rows: xg[r] = x[pair_tok[r]]
// and their bf16 hi/lo halves (xg16, xg16lo), in union order.
struct PassPrep {
  float* x32;
  uint16_t* x16;
  uint16_t* x16lo;
  int* sync_cc;
  int* sync_mma;
  int* ydone;
  float* xg;
  uint16_t* xg16;
  uint16_t* xg16lo;
  int gather_rows;  // union rows gathered per top-k/union CTA (≥ 1 when xg is not null)
};

// Routing and union in two launches: the gate GEMV, then the top-k of every
// token and the union built from that selection (one CTA; or, when prep
// gathers dedup rows, one CTA per prep->gather_rows rows, each computing the
// same selection and union, CTA 0 writing them out). prep: null, or the
// pass's prep work (above).
cudaError_t launch_route_union(int d, int I, int E, int k, int s, int wbytes, int n,
                               const float* x, const float* w_router, const float* bias,
                               int bias_in_weights, float* logits, int32_t* topk_idx,
                               float* topk_w, int32_t* union_ids, int32_t* union_count,
                               int32_t* offsets, int32_t* pair_tok, int32_t* pair_slot,
                               uint64_t* bytes, const PassPrep* prep, cudaStream_t stream);

// Everything the expert kernels read. h is the SwiGLU activation scratch,
// one fp32 row of length I per (pair or shared-expert token) row.
struct ExpertArgs {
  int d, I, E, k, s, n;
  int wdtype;           // 0 fp32, 1 bf16
  int engine;           // 0 per-slot, 1 dedup
  const int32_t* topk_idx;
  const float* topk_w;
  const int32_t* union_ids;    // dedup only
  const int32_t* union_count;  // dedup only
  const int32_t* offsets;      // dedup only
  const int32_t* pair_tok;     // dedup only
  const int32_t* pair_slot;    // dedup only
  const float* x;
  const void* w_gate;
  const void* w_up;
  const void* w_down;
  const void* ws_gate;
  const void* ws_up;
  const void* ws_down;
  float* h;             // [n·k + s·n][I] fp32 scratch (CUDA-core groups)
  float* xg;            // [n·k][d] fp32 scratch: x rows gathered in union order (dedup)
  float* x32;           // [n][d] fp32 scratch: a copy of x, so that the CUDA-core kernel's
                        //   tensor maps point into the workspace only
  uint16_t* h16;        // [n·k + s·n][I] bf16 scratch (tensor-core groups): hi half of h
  uint16_t* h16lo;      //   and lo half: h = hi + lo to ~16 extra mantissa bits
  uint16_t* xg16;       // [n·k][d] bf16 scratch: hi half of xg
  uint16_t* xg16lo;     //   and lo half
  uint16_t* x16;        // [n][d] bf16 scratch: hi half of x
  uint16_t* x16lo;      //   and lo half
  int* sync;            // [kCcSyncInts] CUDA-core kernel's job counter and group counts
  int* sync_mma;        // [kMmaSyncInts] tensor-core kernel's job counter, group counts and
                        //   arrival counts of jobs cut along K
  float* part;          // [part_bytes] tensor-core kernel's partial sums of jobs cut along K
  size_t part_bytes;
  int mma_min_m;        // groups with at least this many tokens run on tensor cores
  int cc_waits_prep;    // 1: the CUDA-core kernel directly follows the prep kernel (or the
                        //   pass's top-k/union kernel), not the tensor-core kernel
  int keep_weights;     // 1: weight loads use normal L2 eviction (per-slot calls of 3+ tokens,
                        //   whose repeated experts L2 can serve), else evict-first
  float* y_slot;
  int prefetch_shared;  // 1: each CTA prefetches its share of the shared experts' weights into
                        //   L2 while it waits for the kernel before it
  float* y;             // [n][d] or null: the combine fused into the kernel's last phase
  int* ydone;           // [1] phase-1 units stored by the call's CTAs, when y is set
  unsigned int* err;
};

// The expert engine of one call: a prep kernel (counters zeroed, rows
// gathered and rounded for the tensor cores), the tensor-core kernel (bf16
// weights only) and the CUDA-core kernel. prepped: the routing kernels just
// before did the prep work (PassPrep), so no prep kernel runs.
cudaError_t launch_expert_engine(const ExpertArgs& a, int num_sms, bool prepped,
                                 cudaStream_t stream);

// Expert FFNs of the groups below mma_min_m tokens on CUDA cores in one
// persistent launch, weights streamed through a ring of shared-memory stages
// filled by the TMA engine: h = silu(Wg x)⊙(Wu x), then y_slot = w·(W_down h).
cudaError_t launch_expert_cc(const ExpertArgs& a, int num_sms, cudaStream_t stream);

// Tokens per plan entry of the CUDA-core and tensor-core kernels, and the
// ints of counter scratch each kernel uses: a job counter and one count per
// entry; the tensor-core kernel adds, per phase, kMmaCntInts arrival counts
// of the pieces of jobs cut along K (one per (entry, tile, quarter of rows)).
constexpr int kCcSub = 4;
constexpr int kMmaSub = 32;
constexpr int kMmaCntInts = 4096;
constexpr int kCcSyncInts = 1 + MOE_MAX_PAIRS + MOE_MAX_SHARED * ((MOE_MAX_TOKENS + kCcSub - 1) / kCcSub);
constexpr int kMmaEntries = MOE_MAX_PAIRS + MOE_MAX_SHARED * ((MOE_MAX_TOKENS + kMmaSub - 1) / kMmaSub);
constexpr int kMmaSyncInts = 1 + kMmaEntries + 2 * kMmaCntInts;
// Scratch for the partial sums of the tensor-core kernel's K pieces; it
// bounds how finely a phase is cut (more pieces need more partials).
constexpr size_t kMmaPartBytes = size_t(24) << 20;

// Tensor-core expert kernel (tcgen05 + TMEM) for groups of ≥ mma_min_m tokens.
cudaError_t launch_expert_mma(const ExpertArgs& a, int num_sms, cudaStream_t stream);

// Failure-detection self-test: a bounded mbarrier wait that expires.
cudaError_t launch_diag_wait(unsigned long long limit_ns, unsigned int* err, cudaStream_t stream);

// y[t] = Σ_j y_slot[t][j] over the k+s slots, in slot order.
cudaError_t launch_combine(int d, int slots, int n, const float* y_slot, float* y,
                           cudaStream_t stream);

}  // namespace moe
