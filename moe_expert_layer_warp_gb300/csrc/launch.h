// launch.h — host-side launchers of the kernels behind the C ABI. Internal to
// libmoewarp.so: api.cu validates arguments, then calls these.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Routing: gate GEMV with compensated fp32 dots (writes logits[n][E] into
// scratch), then warp-per-token top-k + softmax over the k kept logits.
cudaError_t launch_route(int d, int E, int k, int n, const float* x, const float* w_router,
                         float* logits, int32_t* topk_idx, float* topk_w, cudaStream_t stream);

// Union of selected experts, pairs grouped by (expert, token), byte counts.
cudaError_t launch_union(int d, int I, int E, int k, int s, int wbytes, int n,
                         const int32_t* topk_idx, int32_t* union_ids, int32_t* union_count,
                         int32_t* offsets, int32_t* pair_tok, int32_t* pair_slot,
                         uint64_t* bytes, unsigned int* err, cudaStream_t stream);

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
  float* h;             // [n·k + s·n][I] fp32 scratch
  float* xg;            // [n·k][d] fp32 scratch: x rows gathered in union order (dedup)
  int* sync;            // [kSyncInts] scratch: job counter and per-group counts (zeroed per call)
  float* y_slot;
  unsigned int* err;
};

// Expert FFNs over the pass on CUDA cores in one persistent launch, weights
// streamed through a ring of shared-memory stages filled by the TMA engine:
// h = silu(Wg x)⊙(Wu x), then y_slot = w · (W_down h).
cudaError_t launch_expert_engine(const ExpertArgs& a, int num_sms, cudaStream_t stream);

// Ints of scratch the engine's job counter and group counts occupy.
constexpr int kEngineSyncInts = 1 + 512 + 4 * 16;

// y[t] = Σ_j y_slot[t][j] over the k+s slots, in slot order.
cudaError_t launch_combine(int d, int slots, int n, const float* y_slot, float* y,
                           cudaStream_t stream);

}  // namespace moe
