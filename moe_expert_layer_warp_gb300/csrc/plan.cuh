// plan.cuh — the group table both expert kernels build at start-up.
//
// A "group" is one expert applied to a set of tokens whose activation rows
// are consecutive rows of the h scratch:
//   per-slot: one group per (token, slot) pair, rows in pair order t·k + j
//             (the pairs that chose the same expert are sibling entries, so
//             that their jobs run side by side; each still reads the expert);
//   dedup:    one group per union expert, rows in the union's (expert, token)
//             order (moe_build_union's offsets);
//   both:     each shared expert over all n tokens, rows n·k + i·n + t.
// Groups with at least `mma_min_m` tokens belong to the tensor-core kernel,
// the others to the CUDA-core kernel. Each kernel splits its groups into
// sub-groups of at most SUB tokens (one plan entry each), the shared experts'
// entries first. Sibling sub-groups of one group take consecutive jobs tile
// by tile (job_entry), so their CTAs read each weight tile at nearly the same
// time and L2 serves the repeats.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace moe {

struct Entry {
  int src;         // routed expert id (>= 0), or -(i+1) for shared expert i
  int row0;        // first activation row (in h)
  int arow;        // first row of the phase-0 input box (x row or gathered-x row); phase 1
                   //   reads h at row0
  uint16_t first;  // first entry of this group's sub-groups
  uint8_t m;       // tokens of this sub-group (≤ 32)
  uint8_t q;       // number of sibling entries of this group (≤ 255)
};
static_assert(sizeof(Entry) == 16, "plan entry");
static_assert(MOE_MAX_TOKENS * (MOE_MAX_TOPK + MOE_MAX_SHARED) <= 65536, "slot rows fit 16 bits");
static_assert((MOE_MAX_TOKENS + kCcSub - 1) / kCcSub <= 255 && kMmaSub <= 255, "sub-groups fit 8 bits");

MOE_DEV Entry make_entry(int src, int row0, int m, int arow, int first, int q) {
  Entry e;
  e.src = src;
  e.row0 = row0;
  e.arow = arow;
  e.first = (uint16_t)first;
  e.m = (uint8_t)m;
  e.q = (uint8_t)q;
  return e;
}

// Job jj of a phase with T tiles per entry: the jobs of a group's q sub-groups
// are the q·T consecutive jobs from first·T, ordered tile-major.
MOE_DEV void job_entry(const Entry* plan, int jj, int T, int* entry, int* tile) {
  const Entry& eg = plan[jj / T];
  const int local = jj - eg.first * T;
  *entry = eg.first + local % eg.q;
  *tile = local / eg.q;
}

// Job jj of a phase whose (entry, tile) pairs are each cut into S pieces
// along K: the jobs of a group's q sub-groups are the q·T·S consecutive jobs
// from first·T·S, ordered tile, then piece, then sub-group, so that the
// sub-groups that read the same weights take consecutive jobs.
MOE_DEV void job_decode(const Entry* plan, int jj, int T, int S, int* entry, int* tile,
                        int* piece) {
  const int TS = T * S;
  const Entry& eg = plan[jj / TS];
  const int local = jj - eg.first * TS;
  *entry = eg.first + local % eg.q;
  const int rest = local / eg.q;
  *tile = rest / S;
  *piece = rest - (rest / S) * S;
}

// Exclusive prefix sum over the block (one value per thread). Returns the
// thread's offset; *total receives the sum. Uses scratch[0..warps].
MOE_DEV int block_exclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) scratch[warp] = inc;
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the warp totals (nwarps ≤ 32)
    const int c = lane < nwarps ? scratch[lane] : 0;
    int run = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, run, o);
      if (lane >= o) run += t;
    }
    if (lane < nwarps) scratch[lane] = run - c;
    if (lane == 31) scratch[nwarps] = run;
  }
  __syncthreads();
  const int r = scratch[warp] + inc - v;
  *total = scratch[nwarps];
  __syncthreads();
  return r;
}

// Builds this kernel's entries and the per-row output maps (slot row,
// combine weight) in shared memory; returns the number of entries.
// MMA_SIDE selects groups with m ≥ a.mma_min_m, else the others.
// Needs blockDim.x ≥ MOE_MAX_EXPERTS (one thread per union expert),
// 2·blockDim.x ≥ MOE_MAX_PAIRS (a thread loads at most two pairs) and room
// for 2·MOE_MAX_EXPERTS ints in row_w (the per-slot sort's scratch).
template <int SUB, bool MMA_SIDE>
MOE_DEV int build_plan(const ExpertArgs& a, Entry* plan, uint16_t* row_out, float* row_w,
                       int* scratch) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int P = a.n * a.k, S = a.k + a.s;
  auto mine = [&](int m) { return (m >= a.mma_min_m) == MMA_SIDE; };
  // the shared experts' entries come first: their jobs are the first handed
  // out, while their weights are still in L2 when the call prefetched them
  const int per = mine(a.n) ? (a.n + SUB - 1) / SUB : 0;
  const int Sh = a.s * per;
  int nr = 0;
  if (a.engine == 0) {
    // every global load first, so that one round trip serves them (a thread
    // holds at most two pairs)
    float wreg[2] = {0.f, 0.f};
    int ereg[2] = {0, 0};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int p = tid + i * nt;
      if (p < P) {
        wreg[i] = a.topk_w[p];
        ereg[i] = a.topk_idx[p];
      }
    }
    if (mine(1)) {
      // One entry per (token, slot) pair — every slot still streams its own
      // expert's weights — but the pairs that chose the same expert are
      // siblings of one group, so their jobs run tile by tile side by side
      // and L2 serves the repeated reads at the same moment. Entries in
      // (expert, pair) order: a stable counting sort with row_w and row_out
      // as its scratch (both rewritten below). The order must not depend on
      // scheduling: every CTA builds the same plan, and a job number names
      // the same entry in all of them. An expert id outside [0, E) is
      // recorded as an error and read as expert 0.
      int* cnt = reinterpret_cast<int*>(row_w);
      int* start = cnt + MOE_MAX_EXPERTS;
      uint16_t* eid = row_out;
      for (int e = tid; e < a.E; e += nt) cnt[e] = 0;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int p = tid + i * nt;
        if (p < P) {
          int e = ereg[i];
          if (e < 0 || e >= a.E) {
            report_error(a.err, ERR_CHECK, 0x231);
            e = 0;
          }
          eid[p] = (uint16_t)e;
        }
      }
      __syncthreads();
      for (int p = tid; p < P; p += nt) atomicAdd(&cnt[eid[p]], 1);
      __syncthreads();
      int total;
      const int off = block_exclusive_scan(tid < a.E ? cnt[tid] : 0, scratch, &total);
      if (tid < a.E) start[tid] = off;
      __syncthreads();
      for (int p = tid; p < P; p += nt) {
        const int e = eid[p];
        int rank = 0;
        for (int q = 0; q < p; ++q) rank += (eid[q] == e);
        plan[Sh + start[e] + rank] = make_entry(e, p, 1, p / a.k, Sh + start[e], cnt[e]);
      }
      __syncthreads();
      nr = P;
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int p = tid + i * nt;
      if (p < P) {
        const int t = p / a.k, j = p - t * a.k;
        row_out[p] = (uint16_t)(t * S + j);
        row_w[p] = wreg[i];
      }
    }
  } else {
    // every load that needs no other first, so that one round trip serves
    // them: the union's count, expert tid's entry (read for every tid < E;
    // the arrays hold E and E + 1 ints), and rows tid, tid + nt's pairs
    int U = *a.union_count;
    int m = 0, e = 0, r0 = 0;
    if (tid < a.E) {
      r0 = a.offsets[tid];
      m = a.offsets[tid + 1] - r0;
      e = a.union_ids[tid];
    }
    int ptok[2] = {0, 0}, pslot[2] = {0, 0};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = tid + i * nt;
      if (r < P) {
        ptok[i] = a.pair_tok[r];
        pslot[i] = a.pair_slot[r];
      }
    }
    if (U < 0 || U > a.E) {  // not a union of this layer: run nothing, flag it
      if (tid == 0) report_error(a.err, ERR_CHECK, 0x230);
      U = 0;
    }
    if (tid >= U) m = e = r0 = 0;
    const int nsub = (m > 0 && mine(m)) ? (m + SUB - 1) / SUB : 0;
    const int pos = block_exclusive_scan(nsub, scratch, &nr);
    for (int q = 0; q < nsub; ++q) {
      const int rr = r0 + q * SUB;
      plan[Sh + pos + q] = make_entry(e, rr, min(SUB, m - q * SUB), rr, Sh + pos, nsub);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = tid + i * nt;
      if (r < P) {
        int t = ptok[i], j = pslot[i];
        if (t < 0 || t >= a.n || j < 0 || j >= a.k) {  // not a pair of this pass: flag it
          report_error(a.err, ERR_CHECK, 0x232);
          t = j = 0;
        }
        row_out[r] = (uint16_t)(t * S + j);
        row_w[r] = a.topk_w[t * a.k + j];
      }
    }
  }
  for (int q = tid; q < Sh; q += nt) {
    const int i = q / per, c = q - (q / per) * per;
    const int rr = P + i * a.n + c * SUB;
    plan[q] = make_entry(-(i + 1), rr, min(SUB, a.n - c * SUB), c * SUB, i * per, per);
  }
  for (int r = tid; r < a.s * a.n; r += nt) {
    const int i = r / a.n, t = r - (r / a.n) * a.n;
    row_out[P + r] = (uint16_t)(t * S + a.k + i);
    row_w[P + r] = 1.f;
  }
  return Sh + nr;
}

// Upper bound of a kernel's entries for sub-groups of SUB tokens.
constexpr int max_entries(int sub) {
  return MOE_MAX_PAIRS + MOE_MAX_SHARED * ((MOE_MAX_TOKENS + sub - 1) / sub);
}

// This CTA's share of an L2 prefetch of the shared experts' weights (they
// do not depend on the routing), issued by one thread while the CTA waits for
// the kernel before it: gridDim.x slices of each of W_gate, W_up and W_down,
// in bulk prefetches of at most 32 KB (16-byte aligned, sizes multiples of
// 16: the arrays are 16-byte aligned and d is a multiple of 64).
MOE_DEV void shared_l2_prefetch(const ExpertArgs& a) {
  if (a.s <= 0) return;
  const size_t bytes = (size_t)a.s * a.I * a.d * (a.wdtype == 1 ? 2 : 4);
  const char* arr[3] = {static_cast<const char*>(a.ws_gate), static_cast<const char*>(a.ws_up),
                        static_cast<const char*>(a.ws_down)};
  const size_t chunk = ((bytes / gridDim.x) + 15) & ~size_t(15);
  for (int j = 0; j < 3; ++j) {
    const size_t end = min(bytes, (size_t)(blockIdx.x + 1) * chunk);
    for (size_t off = (size_t)blockIdx.x * chunk; off < end; off += 32768) {
      const uint32_t sz = (uint32_t)min((size_t)32768, end - off);
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(arr[j] + off), "r"(sz)
                   : "memory");
    }
  }
}

MOE_DEV int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

MOE_DEV int atom_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

MOE_DEV void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

MOE_DEV void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Bounded wait until *p ≥ target (acquire). False on timeout (recorded).
MOE_DEV bool wait_count(const int* p, int target, unsigned int* err, unsigned int site) {
  const unsigned long long t0 = global_ns();
  unsigned int it = 0;
  while (ld_acquire(p) < target) {
    if ((++it & 255u) == 0 && global_ns() - t0 > kWaitLimitNs) {
      report_error(err, ERR_TIMEOUT, site);
      return false;
    }
  }
  return true;
}

// The weighted combine fused into the expert kernel as its last phase
// ("Deep Dive into Mixture of Experts", §2 and §5 sketches: the layer output
// is the weighted sum of the selected experts plus the shared experts). Every
// CTA of the kernel calls it once, with all its threads, after the CTA's last
// job: *mine (shared memory) counts the phase-1 units (row quarters or warp
// rows) the CTA stored, `target` the units the whole call stores. The CTA publishes
// its count with one GPU-scope release (its threads' slot stores are ordered
// before it by the barrier), waits (bounded, acquire) until the call's count
// reaches the target, then sums its share of the [n][d/4] float4 columns:
// y[t] = Σ_j y_slot[t][j] in slot order j = 0, 1, …, the same additions in
// the same order as moe_combine, so y is bitwise what a separate combine
// gives. A CTA that never ran a job adds nothing to the count, so nothing
// here needs the grid to be resident at once. `flag` is one int of shared
// memory; bar_sync() synchronises the calling threads (all of which call
// this). Returns false if the CTA had stopped on an error (`abort`) or the
// wait expired (recorded).
template <typename Bar>
MOE_DEV bool tail_combine(const ExpertArgs& a, const int* mine, int target,
                          const volatile int* abort, int* flag, int tid, int nthreads,
                          Bar bar_sync) {
  bar_sync();  // every calling thread's slot stores and counts before thread 0's release
  if (tid == 0) {
    // a CTA that stopped on an error publishes nothing (the others' waits
    // then expire and report it too)
    int ok = 0;
    if (*abort == 0) {
      red_release_add(a.ydone, *reinterpret_cast<const volatile int*>(mine));
      ok = wait_count(a.ydone, target, a.err, 0x500) ? 1 : 0;
    }
    *reinterpret_cast<volatile int*>(flag) = ok;
  }
  bar_sync();
  if (*reinterpret_cast<volatile int*>(flag) == 0) return false;
  const int S = a.k + a.s, d4 = a.d >> 2;
  const int items = a.n * d4;
  // The slots' loads go out kChunk at a time, so that one L2 round trip
  // serves up to kChunk slots; the additions stay in slot order.
  constexpr int kChunk = 8;
  for (int i = blockIdx.x * nthreads + tid; i < items; i += gridDim.x * nthreads) {
    const int t = i / d4, c4 = i - t * d4;
    const float4* src = reinterpret_cast<const float4*>(a.y_slot + (size_t)t * S * a.d) + c4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j0 = 0; j0 < S; j0 += kChunk) {
      float4 v[kChunk];
#pragma unroll
      for (int j = 0; j < kChunk; ++j)
        if (j0 + j < S) v[j] = __ldcg(src + (size_t)(j0 + j) * d4);
#pragma unroll
      for (int j = 0; j < kChunk; ++j) {
        if (j0 + j == 0) {
          acc = v[0];
        } else if (j0 + j < S) {
          acc.x = __fadd_rn(acc.x, v[j].x);
          acc.y = __fadd_rn(acc.y, v[j].y);
          acc.z = __fadd_rn(acc.z, v[j].z);
          acc.w = __fadd_rn(acc.w, v[j].w);
        }
      }
    }
    reinterpret_cast<float4*>(a.y + (size_t)t * a.d)[c4] = acc;
  }
  return true;
}

}  // namespace moe
