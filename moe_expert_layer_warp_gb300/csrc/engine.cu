// engine.cu — one expert-engine call: the prep kernel and the launch order of
// the tensor-core and CUDA-core expert kernels.
#include <cuda_bf16.h>
#include <string.h>

#include "moe_warp.h"
#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

// Runs right before the expert kernels and lets them launch as soon as it
// starts (programmatic dependent launch); they wait for it before touching
// its outputs. The grid zeroes both kernels' job counters and group counts,
// and the fused combine's count when the call has one.
// Blocks [0, gather_rows): xg[r] = x[pair_tok[r]] (fp32) and its bf16 hi/lo
// halves (dedup, union order). Blocks [gather_rows, gather_rows + n): x32 =
// a copy of x and, for bf16 layers, the bf16 hi/lo halves of x.
// hi = bf16(v), lo = bf16(v − hi).
__global__ void __launch_bounds__(256)
    engine_prep_kernel(int d, int n, int gather_rows, int halves, const float* __restrict__ x,
                       const int32_t* __restrict__ pair_tok, float* __restrict__ xg,
                       uint16_t* __restrict__ xg16, uint16_t* __restrict__ xg16lo,
                       float* __restrict__ x32, uint16_t* __restrict__ x16,
                       uint16_t* __restrict__ x16lo, int* __restrict__ sync_cc,
                       int* __restrict__ sync_mma, int* __restrict__ ydone) {
  pdl_wait();     // the union (dedup) or routing that precedes it
  pdl_trigger();
  {  // counters, spread over the grid (int4 stores; every region is 256-byte aligned and
     // padded to 256 bytes)
    const int nt = gridDim.x * blockDim.x, t = blockIdx.x * blockDim.x + threadIdx.x;
    const int4 z = make_int4(0, 0, 0, 0);
    for (int i = t; i < (kCcSyncInts + 3) / 4; i += nt) reinterpret_cast<int4*>(sync_cc)[i] = z;
    for (int i = t; i < (kMmaSyncInts + 3) / 4; i += nt) reinterpret_cast<int4*>(sync_mma)[i] = z;
    if (t == 0 && ydone) *reinterpret_cast<int4*>(ydone) = z;
  }
  const int b = blockIdx.x;
  const float* src;
  float* dst32 = nullptr;
  uint16_t *hi, *lo;
  if (b < gather_rows) {
    src = x + (size_t)pair_tok[b] * d;
    dst32 = xg + (size_t)b * d;
    hi = xg16 + (size_t)b * d;
    lo = xg16lo + (size_t)b * d;
  } else if (b < gather_rows + n) {
    src = x + (size_t)(b - gather_rows) * d;
    dst32 = x32 + (size_t)(b - gather_rows) * d;
    hi = x16 + (size_t)(b - gather_rows) * d;
    lo = x16lo + (size_t)(b - gather_rows) * d;
    if (!halves) hi = lo = nullptr;
  } else {
    return;
  }
  for (int i = threadIdx.x; i < d / 4; i += blockDim.x) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(src) + i);
    reinterpret_cast<float4*>(dst32)[i] = v;
    if (hi) split_bf16x4(v, reinterpret_cast<uint2*>(hi) + i, reinterpret_cast<uint2*>(lo) + i);
  }
}

}  // namespace

cudaError_t launch_expert_engine(const ExpertArgs& a, int num_sms, bool prepped,
                                 cudaStream_t stream) {
  cudaError_t e = cudaSuccess;
  if (!prepped) {
    const int gather = a.engine == 1 ? a.n * a.k : 0;
    e = launch_pdl(engine_prep_kernel, dim3(max(gather + a.n, 4)), dim3(256), 0, stream, a.d, a.n,
                   gather, a.wdtype == 1 ? 1 : 0, a.x, a.pair_tok, a.xg, a.xg16, a.xg16lo, a.x32,
                   a.x16, a.x16lo, a.sync, a.sync_mma, a.y ? a.ydone : nullptr);
    if (e != cudaSuccess) return e;
  }
  // The tensor-core kernel runs only where a group can reach mma_min_m
  // tokens: a group never holds more than the pass's n tokens, and per-slot
  // routed groups hold one. The CUDA-core kernel runs unless every group
  // goes to the tensor cores (mma_min_m ≤ 1).
  const bool mma = a.wdtype == 1 && a.n >= a.mma_min_m &&
                   (a.engine == 1 || a.s > 0 || a.mma_min_m <= 1);
  const bool cc = !(mma && a.mma_min_m <= 1);
  ExpertArgs b = a;
  b.cc_waits_prep = mma ? 0 : 1;
  // The combine is fused into the expert kernel's last phase when one kernel
  // runs the whole call; a call split between the two kernels (only when
  // MOE_MMA_MIN_M forces it) combines in a launch of its own afterwards.
  const bool split = mma && cc;
  if (split) b.y = nullptr;
  if (mma) {
    e = launch_expert_mma(b, num_sms, stream);
    if (e != cudaSuccess || !cc) return e;
  }
  e = launch_expert_cc(b, num_sms, stream);
  if (e != cudaSuccess || !split || !a.y) return e;
  return launch_combine(a.d, a.k + a.s, a.n, a.y_slot, a.y, stream);
}

}  // namespace moe
