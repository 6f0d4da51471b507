// route_union.cu — routing (gate GEMV + top-k + softmax over the kept
// logits), the union of selected experts, and the weighted combine.
//
// Sources: "Deep Dive into Mixture of Experts: From 1991 to DeepSeek-V3",
// §2 (top-k gating sketch: logits = x·W_g, topk, softmax over the k kept
// logits, output = Σ weight·expert(x)) and §5 (shared experts added
// unweighted); "Speculative Decoding for Mixture-of-Experts Models: Expert
// Bytes, Kernel Bandwidth and the Best Draft Length", abstract (the union of
// selected experts is what a deduplicating engine reads once per pass).
#include <math.h>
#include <string.h>

#include "moe_warp.h"
#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

// ------------------------------------------------------------------ gate --
// One CTA per (expert, tile of kGateTokens tokens); its 8 warps split d into
// 8 contiguous ranges. The dot is accumulated with error-free
// transformations (TwoProd by FMA, Knuth's TwoSum) — the compensated dot of
// Ogita, Rump and Oishi (2005) — so the returned fp32 logit is the exact dot
// rounded once, up to a term of order u²·Σ|x_i·w_i|. That keeps the top-k
// selection identical to an exact computation except at near-ties far below
// fp32 resolution. Partial (sum, compensation) pairs are combined in a fixed
// order, so the result does not depend on scheduling.
constexpr int kGateWarps = 8;
constexpr int kGateTokens = 8;

// Prefetch of `bytes` (a multiple of 16) at a 16-byte aligned global
// address into L2 (no completion).
MOE_DEV void l2_prefetch_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

MOE_DEV void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

MOE_DEV void dot2_step(float a, float b, float& s, float& c) {
  const float p = __fmul_rn(a, b);
  const float ep = __fmaf_rn(a, b, -p);  // exact: a·b = p + ep
  float es;
  two_sum(s, p, s, es);                  // exact: s_old + p = s + es
  c = __fadd_rn(c, __fadd_rn(ep, es));
}

// (s, c) += (s2, c2) with the sums combined exactly
MOE_DEV void pair_add(float& s, float& c, float s2, float c2) {
  float sn, en;
  two_sum(s, s2, sn, en);
  c = __fadd_rn(__fadd_rn(c, c2), en);
  s = sn;
}

// The pass's prep work that needs only x (PassPrep), done by the gate: the
// expert kernels' counters are zeroed over the whole grid (int4 stores:
// every region is 256-byte aligned and padded to 256 bytes), and x32 = x and
// x's bf16 halves are written from the x values the dot products load, the
// CTAs of expert e writing the float4 columns c with c mod E = e (so that no
// SM stores much).
MOE_DEV void pass_prep_zero(const PassPrep& pp) {
  const int nt = gridDim.x * gridDim.y * blockDim.x;
  const int t = (blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x;
  const int4 z = make_int4(0, 0, 0, 0);
  for (int i = t; i < (kCcSyncInts + 3) / 4; i += nt) reinterpret_cast<int4*>(pp.sync_cc)[i] = z;
  for (int i = t; i < (kMmaSyncInts + 3) / 4; i += nt) reinterpret_cast<int4*>(pp.sync_mma)[i] = z;
  if (t == 0 && pp.ydone) *reinterpret_cast<int4*>(pp.ydone) = z;
}

__global__ void __launch_bounds__(kGateWarps * 32)
    gate_logits_kernel(int d, int E, int n, const float* __restrict__ x,
                       const float* __restrict__ wg, float* __restrict__ logits, PassPrep pp) {
  __shared__ float part[kGateWarps][kGateTokens][2];
  // W_g is constant: its row can move into L2 while the previous kernel
  // finishes (one prefetch per expert row)
  if (threadIdx.x == 0 && blockIdx.y == 0) l2_prefetch_bulk(wg + (size_t)blockIdx.x * d, d * 4);
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x;
  if (pp.x32) pass_prep_zero(pp);
  const bool write_x = pp.x32 != nullptr;
  const int t0 = blockIdx.y * kGateTokens;
  const int nt = min(kGateTokens, n - t0);
  const int chunk4 = (d / kGateWarps) >> 2;  // float4s per warp (d is a multiple of 64)
  const int base4 = warp * chunk4;
  float s[kGateTokens], c[kGateTokens];
#pragma unroll
  for (int t = 0; t < kGateTokens; ++t) s[t] = c[t] = 0.f;
  const float4* wrow = reinterpret_cast<const float4*>(wg + (size_t)e * d) + base4;
  const float4* xrow = reinterpret_cast<const float4*>(x + (size_t)t0 * d) + base4;
  const int d4 = d >> 2;
  for (int i = lane; i < chunk4; i += 32) {
    // every load of the step first, so that they are in flight together
    const float4 w = __ldg(wrow + i);
    float4 xv[kGateTokens];
#pragma unroll
    for (int t = 0; t < kGateTokens; ++t)
      xv[t] = t < nt ? __ldg(xrow + (size_t)t * d4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    if (write_x && (base4 + i) % E == e) {
#pragma unroll
      for (int t = 0; t < kGateTokens; ++t) {
        if (t < nt) {
          const size_t o = (size_t)(t0 + t) * d4 + base4 + i;
          reinterpret_cast<float4*>(pp.x32)[o] = xv[t];
          if (pp.x16)
            split_bf16x4(xv[t], reinterpret_cast<uint2*>(pp.x16) + o,
                         reinterpret_cast<uint2*>(pp.x16lo) + o);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kGateTokens; ++t) {
      if (t < nt) {
        dot2_step(w.x, xv[t].x, s[t], c[t]);
        dot2_step(w.y, xv[t].y, s[t], c[t]);
        dot2_step(w.z, xv[t].z, s[t], c[t]);
        dot2_step(w.w, xv[t].w, s[t], c[t]);
      }
    }
  }
  // Butterfly combine inside the warp; TwoSum is exact and commutative, so
  // every lane ends with the same pair.
#pragma unroll
  for (int t = 0; t < kGateTokens; ++t) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float so = __shfl_xor_sync(0xffffffffu, s[t], o);
      const float co = __shfl_xor_sync(0xffffffffu, c[t], o);
      pair_add(s[t], c[t], so, co);
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int t = 0; t < kGateTokens; ++t) {
      part[warp][t][0] = s[t];
      part[warp][t][1] = c[t];
    }
  }
  __syncthreads();
  if (threadIdx.x < nt) {
    const int t = threadIdx.x;
    float ss = part[0][t][0], cc = part[0][t][1];
    for (int w = 1; w < kGateWarps; ++w) pair_add(ss, cc, part[w][t][0], part[w][t][1]);
    logits[(size_t)(t0 + t) * E + e] = __fadd_rn(ss, cc);
  }
}

// ------------------------------------------------------------------ top-k --
// One warp per token. Expert e lives in lane e%32, register e/32. k rounds of
// warp argmax; the larger score wins, equal scores go to the lower index.
// The score is the logit, or fl(logit + bias[e]) with a routing bias
// ("Deep Dive into Mixture of Experts", §5, DeepSeek-style routing sketch);
// the softmax then runs over the kept biased scores (bias_in_weights) or the
// kept experts' unbiased logits.
constexpr int kTopkWarps = 8;
constexpr int kPerLane = MOE_MAX_EXPERTS / 32;

// One warp selects token t's k experts and writes them and their weights to
// topk_idx / topk_w (when not null); the selected indices also go to
// sel[t·k + j] when sel is not null. Each round
// takes the warp maximum of order-preserving integer keys of the remaining
// scores (redux.sync), then the lowest expert index holding that key, so
// the larger score wins and equal scores go to the lower index.
MOE_DEV uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u << 1) == 0u) u = 0u;  // -0 and +0 compare equal, so they get one key
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

MOE_DEV float key_score(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

MOE_DEV void topk_token(int t, int lane, int E, int k, const float* __restrict__ logits,
                        const float* __restrict__ bias, int bias_in_weights,
                        int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int* sel) {
  uint32_t key[kPerLane];
  uint32_t taken = 0;
#pragma unroll
  for (int r = 0; r < kPerLane; ++r) {
    const int e = lane + 32 * r;
    if (e < E) {
      const float v =
          bias ? __fadd_rn(logits[(size_t)t * E + e], bias[e]) : logits[(size_t)t * E + e];
      key[r] = score_key(v);
    } else {
      key[r] = 0u;
      taken |= 1u << r;
    }
  }
  float my_v = 0.f, v0 = 0.f;
  int my_e = 0;
  for (int j = 0; j < k; ++j) {
    // this lane's best remaining key (the lower register, so the lower
    // expert index, on equal keys); 0 when none remains
    uint32_t bk = 0u;
    int br = -1;
#pragma unroll
    for (int r = 0; r < kPerLane; ++r) {
      if (!((taken >> r) & 1u) && (br < 0 || key[r] > bk)) {
        bk = key[r];
        br = r;
      }
    }
    const uint32_t mk = __reduce_max_sync(0xffffffffu, br >= 0 ? bk : 0u);
    const uint32_t cand = (br >= 0 && bk == mk) ? (uint32_t)(lane + 32 * br) : 0xffffffffu;
    const int be = (int)__reduce_min_sync(0xffffffffu, cand);
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    const float bv = key_score(mk);
    if (j == 0) v0 = bv;
    if (lane == j) {
      my_v = bv;
      my_e = be;
    }
  }
  if (bias && !bias_in_weights) {
    // selection only: the softmax runs over the kept experts' own logits
    my_v = (lane < k) ? logits[(size_t)t * E + my_e] : -INFINITY;
    v0 = my_v;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v0 = fmaxf(v0, __shfl_xor_sync(0xffffffffu, v0, o));
  }
  const float ej = (lane < k) ? expf(my_v - v0) : 0.f;
  const float z = warp_sum(ej);
  if (lane < k) {
    if (topk_idx) {
      topk_idx[(size_t)t * k + lane] = my_e;
      topk_w[(size_t)t * k + lane] = ej / z;
    }
    if (sel) sel[t * k + lane] = my_e;
  }
}

__global__ void __launch_bounds__(kTopkWarps * 32)
    topk_kernel(int E, int k, int n, const float* __restrict__ logits,
                const float* __restrict__ bias, int bias_in_weights,
                int32_t* __restrict__ topk_idx, float* __restrict__ topk_w) {
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kTopkWarps + warp;
  if (t < n) topk_token(t, lane, E, k, logits, bias, bias_in_weights, topk_idx, topk_w, nullptr);
}

// ------------------------------------------------------------------ union --
// One CTA. Counting sort of the n·k (token, slot) pairs by expert; the rank of
// a pair inside its expert is the number of earlier pairs (token-major order)
// with the same expert, so the result is independent of scheduling.
constexpr int kUnionThreads = 512;
constexpr int kRouteUnionThreads = 1024;

struct UnionOut {
  int32_t* union_ids;
  int32_t* union_count;
  int32_t* offsets;
  int32_t* pair_tok;
  int32_t* pair_slot;
  uint64_t* bytes;
};

// The union from the pairs' experts sidx[0 .. n·k) in shared memory, with
// cnt[] zeroed; every thread of the CTA calls it. write: the CTA writes the
// union out; rtok (shared memory, or null): receives the token of each row
// of the union order.
MOE_DEV void union_body(int E, int k, int n, uint64_t expert_bytes, int s, const int* sidx,
                        int* cnt, int* start, const UnionOut& out, bool write, int* rtok) {
  int32_t* __restrict__ union_ids = out.union_ids;
  int32_t* __restrict__ offsets = out.offsets;
  const int P = n * k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __syncthreads();
  for (int p = tid; p < P; p += blockDim.x) atomicAdd(&cnt[sidx[p]], 1);
  __syncthreads();
  if (warp == 0) {
    // lane owns experts [8·lane, 8·lane+8)
    constexpr int per = MOE_MAX_EXPERTS / 32;
    int lc[per];
    int sc = 0, sp = 0;
#pragma unroll
    for (int r = 0; r < per; ++r) {
      const int e = lane * per + r;
      lc[r] = (e < E) ? cnt[e] : 0;
      sc += lc[r];
      sp += (lc[r] > 0);
    }
    int ic = sc, ip = sp;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int tc = __shfl_up_sync(0xffffffffu, ic, o);
      const int tp = __shfl_up_sync(0xffffffffu, ip, o);
      if (lane >= o) {
        ic += tc;
        ip += tp;
      }
    }
    int ec = ic - sc, ep = ip - sp;
#pragma unroll
    for (int r = 0; r < per; ++r) {
      const int e = lane * per + r;
      if (e < E) {
        start[e] = ec;
        if (lc[r] > 0) {
          if (write) {
            union_ids[ep] = e;
            offsets[ep] = ec;
          }
          ++ep;
        }
        ec += lc[r];
      }
    }
    if (lane == 31 && write) {
      offsets[ip] = ic;
      *out.union_count = ip;
      out.bytes[0] = (uint64_t)P * expert_bytes;
      out.bytes[1] = (uint64_t)ip * expert_bytes;
      out.bytes[2] = (uint64_t)s * expert_bytes;
    }
  }
  __syncthreads();
  for (int p = tid; p < P; p += blockDim.x) {
    const int e = sidx[p];
    int rank = 0;
    for (int q = 0; q < p; ++q) rank += (sidx[q] == e);
    const int row = start[e] + rank;
    if (write) {
      out.pair_tok[row] = p / k;
      out.pair_slot[row] = p - (p / k) * k;
    }
    if (rtok) rtok[row] = p / k;
  }
}

__global__ void __launch_bounds__(kUnionThreads)
    union_kernel(int E, int k, int n, uint64_t expert_bytes, int s,
                 const int32_t* __restrict__ topk_idx, UnionOut o, unsigned int* err) {
  __shared__ int sidx[MOE_MAX_PAIRS];
  __shared__ int cnt[MOE_MAX_EXPERTS];
  __shared__ int start[MOE_MAX_EXPERTS];
  pdl_wait();
  pdl_trigger();
  const int P = n * k;
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
  for (int p = tid; p < P; p += blockDim.x) {
    int v = topk_idx[p];
    if (v < 0 || v >= E) {
      report_error(err, ERR_CHECK, 0x101);
      v = 0;
    }
    sidx[p] = v;
  }
  union_body(E, k, n, expert_bytes, s, sidx, cnt, start, o, true, nullptr);
}

// Top-k and union: warp w selects tokens w, w + 32, …, into shared memory,
// then the CTA builds the union; the same selection and the same union as
// topk_kernel then union_kernel. CTA 0 writes them out (topk_idx / topk_w
// and the union). When pp.xg is not null (a whole dedup pass), every CTA
// computes the same selection and union from the same logits, and CTA c
// gathers union rows [c·R, (c+1)·R), R = pp.gather_rows: xg[r] =
// x[pair_tok[r]] and, when pp.xg16 is not null, its bf16 hi/lo halves (R is
// chosen so that the grid spans the SMs: one SM stores only a few rows fast).

__global__ void __launch_bounds__(kRouteUnionThreads)
    topk_union_kernel(int E, int k, int n, uint64_t expert_bytes, int s,
                      const float* __restrict__ logits, const float* __restrict__ bias,
                      int bias_in_weights, int32_t* __restrict__ topk_idx,
                      float* __restrict__ topk_w, UnionOut o, int d, const float* __restrict__ x,
                      PassPrep pp) {
  __shared__ int sidx[MOE_MAX_PAIRS];
  __shared__ int cnt[MOE_MAX_EXPERTS];
  __shared__ int start[MOE_MAX_EXPERTS];
  __shared__ int rtok[MOE_MAX_PAIRS];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool write = blockIdx.x == 0;
  for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
  for (int t = warp; t < n; t += blockDim.x >> 5)
    topk_token(t, lane, E, k, logits, bias, bias_in_weights, write ? topk_idx : nullptr,
               topk_w, sidx);
  union_body(E, k, n, expert_bytes, s, sidx, cnt, start, o, write, pp.xg ? rtok : nullptr);
  if (!pp.xg) return;
  __syncthreads();  // rtok complete
  const int P = n * k, d4 = d >> 2;
  const int r0 = blockIdx.x * pp.gather_rows, r1 = min(P, r0 + pp.gather_rows);
  const int items = (r1 - r0) * d4;
  // kBatch loads in flight per thread before their stores
  constexpr int kBatch = 4;
  for (int i0 = tid; i0 < items; i0 += kBatch * blockDim.x) {
    float4 v[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int i = i0 + b * blockDim.x;
      if (i < items) {
        const int r = r0 + i / d4, c = i - (i / d4) * d4;
        v[b] = __ldg(reinterpret_cast<const float4*>(x + (size_t)rtok[r] * d) + c);
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int i = i0 + b * blockDim.x;
      if (i < items) {
        const int r = r0 + i / d4, c = i - (i / d4) * d4;
        reinterpret_cast<float4*>(pp.xg + (size_t)r * d)[c] = v[b];
        if (pp.xg16)
          split_bf16x4(v[b], reinterpret_cast<uint2*>(pp.xg16 + (size_t)r * d) + c,
                       reinterpret_cast<uint2*>(pp.xg16lo + (size_t)r * d) + c);
      }
    }
  }
}

// ---------------------------------------------------------------- combine --
__global__ void __launch_bounds__(256)
    combine_kernel(int d, int slots, const float* __restrict__ y_slot, float* __restrict__ y) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.y;
  const int c4 = blockIdx.x * blockDim.x + threadIdx.x;
  if (c4 * 4 >= d) return;
  const float4* src = reinterpret_cast<const float4*>(y_slot + (size_t)t * slots * d) + c4;
  // every slot's load first, so that they are in flight together; then the
  // sum in slot order
  constexpr int kMaxSlots = MOE_MAX_TOPK + MOE_MAX_SHARED;
  float4 v[kMaxSlots];
#pragma unroll
  for (int j = 0; j < kMaxSlots; ++j)
    if (j < slots) v[j] = __ldg(src + (size_t)j * (d >> 2));
  float4 acc = v[0];
#pragma unroll
  for (int j = 1; j < kMaxSlots; ++j) {
    if (j < slots) {
      acc.x += v[j].x;
      acc.y += v[j].y;
      acc.z += v[j].z;
      acc.w += v[j].w;
    }
  }
  reinterpret_cast<float4*>(y + (size_t)t * d)[c4] = acc;
}

// ------------------------------------------------------------ diagnostic --
// Waits on an mbarrier that nothing arrives on, with the same bounded wait as
// the expert kernels but a short limit: it records ERR_TIMEOUT and returns.
__global__ void diag_wait_kernel(unsigned long long limit_ns, unsigned int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_for(&bar, 0, err, 0x900, limit_ns);
  __syncthreads();
}

}  // namespace

cudaError_t launch_diag_wait(unsigned long long limit_ns, unsigned int* err, cudaStream_t stream) {
  diag_wait_kernel<<<1, 32, 0, stream>>>(limit_ns, err);
  return cudaGetLastError();
}

cudaError_t launch_route(int d, int E, int k, int n, const float* x, const float* w_router,
                         const float* bias, int bias_in_weights, float* logits, int32_t* topk_idx,
                         float* topk_w, cudaStream_t stream) {
  dim3 g1(E, (n + kGateTokens - 1) / kGateTokens);
  PassPrep none;
  memset(&none, 0, sizeof none);
  cudaError_t e = launch_pdl(gate_logits_kernel, g1, dim3(kGateWarps * 32), 0, stream, d, E, n, x,
                             w_router, logits, none);
  if (e != cudaSuccess) return e;
  dim3 g2((n + kTopkWarps - 1) / kTopkWarps);
  return launch_pdl(topk_kernel, g2, dim3(kTopkWarps * 32), 0, stream, E, k, n,
                    static_cast<const float*>(logits), bias, bias_in_weights, topk_idx, topk_w);
}

cudaError_t launch_gate(int d, int E, int n, const float* x, const float* w_router, float* logits,
                        cudaStream_t stream) {
  dim3 g1(E, (n + kGateTokens - 1) / kGateTokens);
  PassPrep none;
  memset(&none, 0, sizeof none);
  return launch_pdl(gate_logits_kernel, g1, dim3(kGateWarps * 32), 0, stream, d, E, n, x,
                    w_router, logits, none);
}

cudaError_t launch_union(int d, int I, int E, int k, int s, int wbytes, int n,
                         const int32_t* topk_idx, int32_t* union_ids, int32_t* union_count,
                         int32_t* offsets, int32_t* pair_tok, int32_t* pair_slot,
                         uint64_t* bytes, unsigned int* err, cudaStream_t stream) {
  const uint64_t eb = 3ull * (uint64_t)d * (uint64_t)I * (uint64_t)wbytes;
  const UnionOut o{union_ids, union_count, offsets, pair_tok, pair_slot, bytes};
  return launch_pdl(union_kernel, dim3(1), dim3(kUnionThreads), 0, stream, E, k, n, eb, s,
                    topk_idx, o, err);
}

cudaError_t launch_route_union(int d, int I, int E, int k, int s, int wbytes, int n,
                               const float* x, const float* w_router, const float* bias,
                               int bias_in_weights, float* logits, int32_t* topk_idx,
                               float* topk_w, int32_t* union_ids, int32_t* union_count,
                               int32_t* offsets, int32_t* pair_tok, int32_t* pair_slot,
                               uint64_t* bytes, const PassPrep* prep, cudaStream_t stream) {
  PassPrep pp;
  memset(&pp, 0, sizeof pp);
  if (prep) pp = *prep;
  dim3 g1(E, (n + kGateTokens - 1) / kGateTokens);
  cudaError_t e = launch_pdl(gate_logits_kernel, g1, dim3(kGateWarps * 32), 0, stream, d, E, n, x,
                             w_router, logits, pp);
  if (e != cudaSuccess) return e;
  const uint64_t eb = 3ull * (uint64_t)d * (uint64_t)I * (uint64_t)wbytes;
  const UnionOut o{union_ids, union_count, offsets, pair_tok, pair_slot, bytes};
  const int ctas = pp.xg ? (n * k + pp.gather_rows - 1) / pp.gather_rows : 1;
  return launch_pdl(topk_union_kernel, dim3(ctas), dim3(kRouteUnionThreads), 0, stream, E, k, n,
                    eb, s, static_cast<const float*>(logits), bias, bias_in_weights, topk_idx,
                    topk_w, o, d, x, pp);
}

cudaError_t launch_combine(int d, int slots, int n, const float* y_slot, float* y,
                           cudaStream_t stream) {
  dim3 g((d / 4 + 255) / 256, n);
  return launch_pdl(combine_kernel, g, dim3(256), 0, stream, d, slots, y_slot, y);
}

}  // namespace moe
