// expert_stream.cu — the expert FFNs of one verification pass on CUDA cores,
// with each expert's weights streamed from HBM by tensor-map TMA into a ring
// of shared-memory stages, one persistent CTA per SM.
//
// Sources: "Speculative Decoding for Mixture-of-Experts Models: Expert Bytes,
// Kernel Bandwidth and the Best Draft Length", abstract — the per-slot engine
// reads a selected expert once per token, the deduplicating engine reads each
// selected expert once per pass for all tokens that chose it; "Deep Dive into
// Mixture of Experts: From 1991 to DeepSeek-V3", §2 (weighted sum of the
// selected experts) and §5 (shared experts, unweighted). Each expert is
// W_down(silu(W_gate x) ⊙ W_up x).
//
// Work decomposition. A "group" is one expert applied to a set of tokens
// whose activation rows are consecutive rows of h (one fp32 row of I per
// token), split into sub-groups of at most kMaxM = 4 tokens:
//   per-slot: one group per (token, slot) pair, rows in pair order t·k + j;
//   dedup:    one group per union expert, rows in the union's (expert, token)
//             order;
//   both:     each shared expert over all n tokens, rows n·k + i·n + t.
// Phase 0 computes h = silu(W_gate x) ⊙ (W_up x) in tiles of 32 rows of I;
// phase 1 computes y_slot = w · (W_down h) in tiles of 64 rows of d. A job is
// (sub-group, tile); CTA b's first job is job b, after which the producer
// thread of each CTA takes the next job from a global counter. The
// sub-groups of one group take consecutive jobs tile by tile, so that L2
// serves their repeated weight tiles.
//
// A stage holds 32 KB of weights — 32 rows of W_gate and the same 32 rows of
// W_up, or 64 rows of W_down, × K_s = 256 bf16 / 128 fp32 columns — and the
// sub-group's input rows for those columns (1 or 4 rows of x, of x gathered
// per union expert, or of h). The weights arrive as ONE tensor-map box where
// possible: W_gate and W_up are read through one map whose outermost
// dimension steps from one matrix to the other, so a phase-0 stage is a
// single [2][32][K_s] box. An SM's TMA stream completes boxes at a roughly
// fixed rate whatever their size, so fewer, larger boxes per stage raise
// what one SM can pull from HBM (about 30 GB/s with two 8 KB boxes and an
// input box per stage, about 65 GB/s with one 32 KB box and an input box;
// the GPU-wide share of an SM is about 45 GB/s). Each of the 16 consumer
// warps owns 4 weight rows: lane l holds 16 bytes of each and the same
// columns of every token, so every weight byte is read from shared memory
// once and used for all tokens of the sub-group. Columns beyond K arrive
// zero-filled from the TMA and contribute nothing. A publisher warp makes
// finished phase-0 tiles visible to other CTAs' phase-1 jobs. When the call
// fuses the combine, the consumer warps count the phase-1 rows they stored
// and, after the CTA's last job, take part in the kernel's last phase
// (tail_combine): once the whole call's rows are stored, they sum their
// share of y over the slots in slot order.
#include <math.h>

#include "moe_warp.h"
#include "common.cuh"
#include "launch.h"
#include "plan.cuh"
#include "tmap.h"

namespace moe {
namespace {

constexpr int kConsumerWarps = 16;
constexpr int kThreads = (kConsumerWarps + 2) * 32;  // + producer warp + publisher warp
constexpr int kPubSlots = 8;                         // ring of finished phase-0 jobs
constexpr int kRowChunks = 64;                       // weight rows per stage
constexpr int kChunkBytes = 512;                     // bytes of one weight row per stage
constexpr int kMaxM = kCcSub;
constexpr int kStages = 5;
constexpr int kMaxRows = MOE_MAX_PAIRS + MOE_MAX_SHARED * MOE_MAX_TOKENS;
constexpr int kMaxEntries = max_entries(kMaxM);
constexpr int kRowsPhase0 = 32;  // rows of I per phase-0 tile (gate and up)
constexpr int kRowsPhase1 = 64;  // rows of d per phase-1 tile
static_assert(2 * kRowsPhase0 == kRowChunks && kRowsPhase1 == kRowChunks, "stage rows");
static_assert(kRowChunks == 4 * kConsumerWarps, "four weight rows per consumer warp");
static_assert(1 + kMaxEntries == kCcSyncInts, "engine scratch size");

// Tensor maps of one launch. w0/w1/w2: routed experts' W_gate, W_up, W_down
// ([E][rows][K]); sw0/sw1/sw2: the shared experts'. gu/sgu: W_gate and W_up
// as one [2][E][I][K] tensor (the outer stride is the distance between the
// two arrays) when that distance is expressible (pair/spair); up_first when
// W_up lies below W_gate. a1/aM: phase-0 input rows of routed groups (x, or
// x gathered in union order) with a box of 1 or kMaxM rows; s1/sM: phase-0
// input rows of shared-expert groups (x); h1/hM: phase-1 input rows (h).
struct Maps {
  CUtensorMap w0, w1, w2, sw0, sw1, sw2, a1, aM, s1, sM, h1, hM, gu, sgu;
  int pair, spair, up_first, sup_first;
};

struct Params {
  Maps maps;
  ExpertArgs a;
};

template <int WB>
struct Layout {
  static constexpr int EPL = 16 / WB;           // weight elements per lane per chunk
  static constexpr int KS = 32 * EPL;           // K columns per stage
  static constexpr int kWBytes = kRowChunks * kChunkBytes;
  static constexpr int kXBytes = kMaxM * KS * 4;
  static constexpr int kStageBytes = kWBytes + kXBytes;
  static constexpr int kOffBar = kStages * kStageBytes;
  static constexpr int kOffPlan = kOffBar + (2 * kStages + 2 * kPubSlots) * 8;
  static constexpr int kOffRowOut = kOffPlan + kMaxEntries * (int)sizeof(Entry);
  static constexpr int kOffRowW = kOffRowOut + kMaxRows * 2;
  static constexpr int kOffMisc = kOffRowW + kMaxRows * 4;
  static constexpr int kBytes = kOffMisc + 96 * 4;
};

// Columns a lane owns inside a stage, chosen so that its shared-memory reads
// are conflict-free: bf16 stages (256 columns) give lane l the runs
// [4l, 4l+4) and [128+4l, 128+4l+4) — two 8-byte weight reads and two 16-byte
// input reads; fp32 stages (128 columns) give it [4l, 4l+4). Values are
// handled as float2 pairs for the packed fp32x2 FMA.
template <int WB>
struct LaneMap;

template <>
struct LaneMap<2> {
  static constexpr int NP = 4;  // float2 pairs per lane per row
  static MOE_DEV void load_w(const unsigned char* row, int lane, float2 (&w)[NP]) {
    const uint2 u = *reinterpret_cast<const uint2*>(row + lane * 8);
    const uint2 v = *reinterpret_cast<const uint2*>(row + 256 + lane * 8);
    w[0] = make_float2(bf16lo(u.x), bf16hi(u.x));
    w[1] = make_float2(bf16lo(u.y), bf16hi(u.y));
    w[2] = make_float2(bf16lo(v.x), bf16hi(v.x));
    w[3] = make_float2(bf16lo(v.y), bf16hi(v.y));
  }
  static MOE_DEV void load_x(const float* row, int lane, float2 (&x)[NP]) {
    const float4 u = *reinterpret_cast<const float4*>(row + lane * 4);
    const float4 v = *reinterpret_cast<const float4*>(row + 128 + lane * 4);
    x[0] = make_float2(u.x, u.y);
    x[1] = make_float2(u.z, u.w);
    x[2] = make_float2(v.x, v.y);
    x[3] = make_float2(v.z, v.w);
  }
};

template <>
struct LaneMap<4> {
  static constexpr int NP = 2;
  static MOE_DEV void load_w(const unsigned char* row, int lane, float2 (&w)[NP]) {
    const float4 u = *reinterpret_cast<const float4*>(row + lane * 16);
    w[0] = make_float2(u.x, u.y);
    w[1] = make_float2(u.z, u.w);
  }
  static MOE_DEV void load_x(const float* row, int lane, float2 (&x)[NP]) {
    const float4 u = *reinterpret_cast<const float4*>(row + lane * 4);
    x[0] = make_float2(u.x, u.y);
    x[1] = make_float2(u.z, u.w);
  }
};

static_assert(MOE_MAX_EXPERTS <= kThreads && MOE_MAX_PAIRS <= 2 * kThreads,
              "build_plan: one thread per expert, two pairs per thread");
static_assert(kMaxRows >= 2 * MOE_MAX_EXPERTS, "build_plan: row_w holds its sort scratch");

// One launch runs both phases. Jobs 0 .. J0-1 are phase-0 jobs (group-major),
// jobs J0 .. J0+J1-1 phase-1 jobs (group-major); the producer thread of each
// CTA takes the next job from a global counter, so every job taken belongs to
// a resident CTA. A phase-1 job may load its group's h rows only once all
// phase-0 tiles of that group are written: consumer warps count them in
// done0[group]; the producer waits for the count (bounded) before issuing
// the h box, while the job's weight boxes are already in flight.
template <int WB>
__global__ void __launch_bounds__(kThreads, 1) expert_engine_kernel(const __grid_constant__ Params prm) {
  using L = Layout<WB>;
  constexpr int KS = L::KS;
  const ExpertArgs& a = prm.a;
  extern __shared__ __align__(1024) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* empty = full + kStages;
  uint64_t* pub_full = empty + kStages;    // consumer warps → publisher: a phase-0 job's h is stored
  uint64_t* pub_empty = pub_full + kPubSlots;
  Entry* plan = reinterpret_cast<Entry*>(smem + L::kOffPlan);
  uint16_t* row_out = reinterpret_cast<uint16_t*>(smem + L::kOffRowOut);
  float* row_w = reinterpret_cast<float*>(smem + L::kOffRowW);
  int* misc = reinterpret_cast<int*>(smem + L::kOffMisc);  // [0..31] scan scratch
  volatile int* stage_job = misc + 32;                     // [kStages]
  volatile int* abort_flag = misc + 48;
  volatile int* pub_entry = misc + 52;                     // [kPubSlots]
  int* tail_flag = misc + 64;                              // fused combine: the wait's outcome
  int* ph1_done = misc + 65;                               // phase-1 warp rows stored by this CTA
  int* tail_target = misc + 66;                            // ... and by the whole call

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    for (int i = 0; i < kPubSlots; ++i) {
      mbar_init(&pub_full[i], kConsumerWarps);
      mbar_init(&pub_empty[i], 1);
    }
    *ph1_done = 0;
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == (kConsumerWarps + 1) * 32 && a.prefetch_shared) shared_l2_prefetch(a);
  if (threadIdx.x == kConsumerWarps * 32) {
    prefetch_tmap(prm.maps.pair ? &prm.maps.gu : &prm.maps.w0);
    prefetch_tmap(&prm.maps.w2);
    prefetch_tmap(&prm.maps.a1);
  }
  // The kernel before this one — the prep kernel, or the top-k/union kernel
  // of a whole pass — must be complete: it wrote the routing, the union and
  // the rows this kernel reads, and zeroed its counters. When this kernel
  // follows the tensor-core kernel, that kernel released it only after its
  // own wait, so this kernel starts at once and waits for the tensor-core
  // kernel only before it exits (below).
  if (a.cc_waits_prep) pdl_wait();
  pdl_trigger();
  const int n_groups = build_plan<kMaxM, false>(a, plan, row_out, row_w, misc);
  __syncthreads();

  const int T0 = a.I / kRowsPhase0, T1 = a.d / kRowsPhase1;
  const int J0 = n_groups * T0, J = J0 + n_groups * T1;
  const int nks0 = (a.d + KS - 1) / KS, nks1 = (a.I + KS - 1) / KS;
  int* job_counter = a.sync;
  int* done0 = a.sync + 1;
  const int done_target = T0;  // one publication per phase-0 tile
  // every (entry, phase-1 tile) stores sixteen warp rows of four; kept in
  // shared memory, so that the consumer loop holds no register for it
  if (threadIdx.x == 0) *tail_target = n_groups * T1 * kConsumerWarps;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------ producer thread --
    if (lane == 0) {
      const uint64_t pol_w = weight_policy(a.keep_weights);
      const uint64_t pol_x = l2_evict_last_policy();
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      // the first job is blockIdx.x; the counter hands
      // out jobs gridDim.x, gridDim.x + 1, … after it
      for (bool first = true; ok; first = false) {
        int job = first ? min((int)blockIdx.x, J) : atomicAdd(job_counter, 1) + (int)gridDim.x;
        if (job >= J) {
          // end marker for the consumers
          if (!mbar_wait(&empty[stage], phase ^ 1u, a.err, 0x201)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          stage_job[stage] = -1;
          mbar_arrive(&full[stage]);
          break;
        }
        const int ph = job < J0 ? 0 : 1;
        const int jj = ph == 0 ? job : job - J0;
        int g, tile;
        job_entry(plan, jj, ph == 0 ? T0 : T1, &g, &tile);
        const Entry en = plan[g];
        const bool shared_expert = en.src < 0;
        const int ecoord = shared_expert ? -en.src - 1 : en.src;
        const CUtensorMap *m0, *m1 = nullptr, *mx;
        if (ph == 0) {
          m0 = shared_expert ? &prm.maps.sw0 : &prm.maps.w0;
          m1 = shared_expert ? &prm.maps.sw1 : &prm.maps.w1;
          mx = shared_expert ? (en.m == 1 ? &prm.maps.s1 : &prm.maps.sM)
                             : (en.m == 1 ? &prm.maps.a1 : &prm.maps.aM);
        } else {
          m0 = shared_expert ? &prm.maps.sw2 : &prm.maps.w2;
          mx = en.m == 1 ? &prm.maps.h1 : &prm.maps.hM;
        }
        const int arow = ph == 0 ? en.arow : en.row0;
        const uint32_t xbytes = (en.m == 1 ? 1 : kMaxM) * KS * 4;
        const int nks = ph == 0 ? nks0 : nks1;
        for (int ks = 0; ks < nks; ++ks) {
          if (*abort_flag) {
            ok = false;
            break;
          }
          if (!mbar_wait(&empty[stage], phase ^ 1u, a.err, 0x200)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          unsigned char* st = smem + stage * L::kStageBytes;
          if (ks == 0) stage_job[stage] = job;
          mbar_arrive_expect_tx(&full[stage], kRowChunks * kChunkBytes + xbytes);
          const int k0 = ks * KS;
          if (ph == 0) {
            if (shared_expert ? prm.maps.spair : prm.maps.pair) {
              tma_load_4d(st, shared_expert ? &prm.maps.sgu : &prm.maps.gu, k0, tile * kRowsPhase0,
                          ecoord, 0, &full[stage], pol_w);
            } else {
              tma_load_3d(st, m0, k0, tile * kRowsPhase0, ecoord, &full[stage], pol_w);
              tma_load_3d(st + kRowsPhase0 * kChunkBytes, m1, k0, tile * kRowsPhase0, ecoord,
                          &full[stage], pol_w);
            }
          } else {
            tma_load_3d(st, m0, k0, tile * kRowsPhase1, ecoord, &full[stage], pol_w);
            if (ks == 0) {
              // the group's h rows must be complete before they are read
              const unsigned long long t0 = global_ns();
              unsigned int it = 0;
              while (ld_acquire(done0 + g) < done_target) {
                if ((++it & 255u) == 0 && global_ns() - t0 > kWaitLimitNs) {
                  report_error(a.err, ERR_TIMEOUT, 0x240);
                  *abort_flag = 1;
                  ok = false;
                  break;
                }
              }
              fence_proxy_async_global();
            }
          }
          // On a failed dependency wait the box is still issued (it reads
          // valid memory) so that the stage completes and nothing is left
          // in flight; the abort flag stops everything after it.
          tma_load_2d(st + L::kWBytes, mx, k0, arow, &full[stage], pol_x);
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Give copies already issued a bounded chance to land before the CTA
        // exits, so that none writes into shared memory after it is released.
        const int outstanding = min(issued, kStages);
        for (int i = 1; i <= outstanding; ++i) {
          const int idx = issued - i;
          mbar_wait(&full[idx % kStages], (uint32_t)((idx / kStages) & 1), a.err, 0x210);
        }
      }
    }
    // Every path out of this kernel passes here: the grid cannot complete
    // before the tensor-core kernel it overlaps has completed.
    if (!a.cc_waits_prep) pdl_wait();
    return;
  }

  if (warp == kConsumerWarps + 1) {
    // ---------------------------------------------------- publisher thread --
    // Publishes each finished phase-0 job to the group's phase-1 jobs in other
    // CTAs with a GPU-scope release, so that the consumer warps only ever pay
    // a CTA-scope arrive. The consumers' h stores are ordered before their
    // arrive (release, CTA scope); this thread's wait acquires them and its
    // release reduction makes them visible GPU-wide before the count.
    if (lane == 0) {
      for (int pn = 0;; ++pn) {
        const int ps = pn % kPubSlots;
        if (!mbar_wait(&pub_full[ps], (uint32_t)((pn / kPubSlots) & 1), a.err, 0x251)) break;
        const int e = pub_entry[ps];
        if (e < 0) break;
        red_release_add(done0 + e, 1);
        mbar_arrive(&pub_empty[ps]);
      }
    }
    return;
  }


  // --------------------------------------------------------- consumer warps --
  // Warp w owns four weight rows of every stage: in phase 0 gate rows 2w and
  // 2w+1 and the same up rows of the 32-row tile (so h for those rows is
  // finished inside the warp), in phase 1 rows 4w .. 4w+3 of the 64-row tile.
  using LM = LaneMap<WB>;
  constexpr int NP = LM::NP;
  int stage = 0;
  uint32_t phase = 0;
  int pub_n = 0;  // phase-0 jobs handed to the publisher so far
  // Every exit below is taken by the whole warp, and every path leads to the
  // consumers' last phase (consumers_done), where all 16 consumer warps meet.
  for (;;) {
    if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], phase, a.err, 0x220))) {
      *abort_flag = 1;
      goto consumers_done;
    }
    if (__any_sync(0xffffffffu, *abort_flag != 0)) goto consumers_done;
    const int job = stage_job[stage];
    if (job < 0) {
      // end marker for the publisher
      if (lane == 0) {
        const int ps = pub_n % kPubSlots;
        if (mbar_wait(&pub_empty[ps], (uint32_t)(((pub_n / kPubSlots) & 1) ^ 1), a.err, 0x252)) {
          if (warp == 0) pub_entry[ps] = -1;
          mbar_arrive(&pub_full[ps]);
        }
      }
      break;
    }
    const int ph = job < J0 ? 0 : 1;
    const int jj = ph == 0 ? job : job - J0;
    int g, tile;
    job_entry(plan, jj, ph == 0 ? T0 : T1, &g, &tile);
    const Entry en = plan[g];
    const int m = en.m;
    const int nks = ph == 0 ? nks0 : nks1;
    // stage rows of this warp: phase 0 gate 2w, gate 2w+1, up 2w, up 2w+1
    // (the box holds one matrix's 32 rows, then the other's); phase 1 4w..4w+3
    int wrow[4];
    if (ph == 0) {
      const int gate0 = (en.src < 0 ? prm.maps.sup_first : prm.maps.up_first) ? kRowsPhase0 : 0;
      const int up0 = kRowsPhase0 - gate0;
      wrow[0] = gate0 + 2 * warp;
      wrow[1] = gate0 + 2 * warp + 1;
      wrow[2] = up0 + 2 * warp;
      wrow[3] = up0 + 2 * warp + 1;
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) wrow[q] = 4 * warp + q;
    }
    float2 acc[4][kMaxM];
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int t = 0; t < kMaxM; ++t) acc[q][t] = make_float2(0.f, 0.f);
    for (int ks = 0; ks < nks; ++ks) {
      if (ks > 0 && !__all_sync(0xffffffffu, mbar_wait(&full[stage], phase, a.err, 0x221))) {
        *abort_flag = 1;
        goto consumers_done;
      }
      const unsigned char* st = smem + stage * L::kStageBytes;
      const float* sx = reinterpret_cast<const float*>(st + L::kWBytes);
      float2 wv[4][NP];
#pragma unroll
      for (int q = 0; q < 4; ++q) LM::load_w(st + wrow[q] * kChunkBytes, lane, wv[q]);
#pragma unroll
      for (int t = 0; t < kMaxM; ++t) {
        if (t < m) {
          float2 xv[NP];
          LM::load_x(sx + t * KS, lane, xv);
#pragma unroll
          for (int p = 0; p < NP; ++p)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[q][t] = __ffma2_rn(wv[q][p], xv[p], acc[q][t]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    float r[4][kMaxM];
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int t = 0; t < kMaxM; ++t)
        r[q][t] = (t < m) ? warp_sum(acc[q][t].x + acc[q][t].y) : 0.f;
    if (lane == 0) {
      if (ph == 0) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int row = tile * kRowsPhase0 + 2 * warp + j;
#pragma unroll
          for (int t = 0; t < kMaxM; ++t)
            if (t < m) a.h[(size_t)(en.row0 + t) * a.I + row] = silu(r[j][t]) * r[2 + j][t];
        }
        // hand the finished job to the publisher thread (see above)
        const int ps = pub_n % kPubSlots;
        if (!mbar_wait(&pub_empty[ps], (uint32_t)(((pub_n / kPubSlots) & 1) ^ 1), a.err, 0x250)) {
          *abort_flag = 1;
        } else {
          pub_entry[ps] = g;
          mbar_arrive(&pub_full[ps]);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int row = tile * kRowsPhase1 + 4 * warp + q;
#pragma unroll
          for (int t = 0; t < kMaxM; ++t) {
            if (t < m) {
              const int rr = en.row0 + t;
              a.y_slot[(size_t)row_out[rr] * a.d + row] = row_w[rr] * r[q][t];
            }
          }
        }
        atomicAdd(ph1_done, 1);  // this warp's rows of the tile (fused combine)
      }
    }
    if (ph == 0) ++pub_n;
  }
consumers_done:
  // The combine fused as the last phase: every (entry, phase-1 tile) stores
  // sixteen warp rows of four (one per consumer warp). The producer and
  // publisher warps have left; the consumers synchronise on barrier 1.
  if (a.y)
    tail_combine(a, ph1_done, *tail_target, abort_flag, tail_flag, (int)threadIdx.x,
                 kConsumerWarps * 32,
                 [] { asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory"); });
}

// ------------------------------------------------------------------ host --
bool weight_map(CUtensorMap* m, const void* p, int WB, int n_mat, int rows, int K, int box_rows) {
  const int ks = WB == 2 ? 256 : 128;
  const uint64_t dims[3] = {(uint64_t)K, (uint64_t)rows, (uint64_t)n_mat};
  const uint64_t strides[2] = {(uint64_t)K * WB, (uint64_t)rows * K * WB};
  const uint32_t box[3] = {(uint32_t)ks, (uint32_t)box_rows, 1};
  return make_tmap(m, p, WB == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                   3, dims, strides, box);
}

// W_gate and W_up of n_mat experts as one 4-D tensor [2][n_mat][rows][K]
// whose outer stride is the byte distance between the two arrays (based at
// the lower one: up_first when that is W_up), so that one box carries the
// same rows of both. Needs the distance to be a non-zero multiple of 16
// bytes below 2^40 (the tensor map's stride limit); otherwise returns false
// and the kernel loads the two matrices as separate boxes.
bool pair_map(CUtensorMap* m, int* up_first, const void* gate, const void* up, int WB, int n_mat,
              int rows, int K) {
  const int ks = WB == 2 ? 256 : 128;
  const uintptr_t pg = reinterpret_cast<uintptr_t>(gate), pu = reinterpret_cast<uintptr_t>(up);
  const uint64_t delta = pu > pg ? pu - pg : pg - pu;
  const uint64_t mat = (uint64_t)rows * K * WB;
  if (delta == 0 || delta % 16 != 0 || delta >= (1ull << 40)) return false;
  *up_first = pu < pg ? 1 : 0;
  const uint64_t dims[4] = {(uint64_t)K, (uint64_t)rows, (uint64_t)n_mat, 2};
  const uint64_t strides[3] = {(uint64_t)K * WB, mat, delta};
  const uint32_t box[4] = {(uint32_t)ks, (uint32_t)kRowsPhase0, 1, 2};
  return make_tmap(m, reinterpret_cast<const void*>(pu < pg ? pu : pg),
                   WB == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                   dims, strides, box);
}

bool act_map(CUtensorMap* m, const float* p, int rows, int K, int ks, int box_rows) {
  const uint64_t dims[2] = {(uint64_t)K, (uint64_t)rows};
  const uint64_t strides[1] = {(uint64_t)K * 4};
  const uint32_t box[2] = {(uint32_t)ks, (uint32_t)box_rows};
  return make_tmap(m, p, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, dims, strides, box);
}

// Every tensor map of one launch.
template <int WB>
bool build_maps(const ExpertArgs& a, Maps* M) {
  memset(M, 0, sizeof *M);
  constexpr int ks = Layout<WB>::KS;
  const int P = a.n * a.k;
  const int hrows = P + a.s * a.n;
  bool ok = true;
  ok &= weight_map(&M->w0, a.w_gate, WB, a.E, a.I, a.d, kRowsPhase0);
  ok &= weight_map(&M->w1, a.w_up, WB, a.E, a.I, a.d, kRowsPhase0);
  ok &= weight_map(&M->w2, a.w_down, WB, a.E, a.d, a.I, kRowsPhase1);
  M->pair = pair_map(&M->gu, &M->up_first, a.w_gate, a.w_up, WB, a.E, a.I, a.d) ? 1 : 0;
  if (!M->pair) M->up_first = 0;
  if (a.s > 0) {
    ok &= weight_map(&M->sw0, a.ws_gate, WB, a.s, a.I, a.d, kRowsPhase0);
    ok &= weight_map(&M->sw1, a.ws_up, WB, a.s, a.I, a.d, kRowsPhase0);
    ok &= weight_map(&M->sw2, a.ws_down, WB, a.s, a.d, a.I, kRowsPhase1);
    M->spair = pair_map(&M->sgu, &M->sup_first, a.ws_gate, a.ws_up, WB, a.s, a.I, a.d) ? 1 : 0;
    if (!M->spair) M->sup_first = 0;
  }
  const float* xa = a.engine == 0 ? a.x32 : a.xg;
  const int xa_rows = a.engine == 0 ? a.n : P;
  ok &= act_map(&M->a1, xa, xa_rows, a.d, ks, 1);
  ok &= act_map(&M->aM, xa, xa_rows, a.d, ks, kMaxM);
  ok &= act_map(&M->s1, a.x32, a.n, a.d, ks, 1);
  ok &= act_map(&M->sM, a.x32, a.n, a.d, ks, kMaxM);
  ok &= act_map(&M->h1, a.h, hrows, a.I, ks, 1);
  ok &= act_map(&M->hM, a.h, hrows, a.I, ks, kMaxM);
  return ok;
}

template <int WB>
cudaError_t launch_engine(const ExpertArgs& a, int num_sms, cudaStream_t stream) {
  auto kern = expert_engine_kernel<WB>;
  constexpr int bytes = Layout<WB>::kBytes;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  Params prm;
  memset(&prm, 0, sizeof prm);
  prm.a = a;
  // Everything the tensor maps depend on; an earlier call with the same key
  // reuses its maps.
  struct Key {
    const void* p[9];
    int v[8];
  } key;
  memset(&key, 0, sizeof key);
  const void* kp[9] = {a.w_gate, a.w_up, a.w_down, a.ws_gate, a.ws_up, a.ws_down, a.x32, a.xg, a.h};
  memcpy(key.p, kp, sizeof kp);
  const int kv[8] = {a.d, a.I, a.E, a.k, a.s, a.n, a.engine, dev};
  memcpy(key.v, kv, sizeof kv);
  static RecentCache<Key, Maps> cache;
  if (!cache.get(key, &prm.maps)) {
    if (!build_maps<WB>(a, &prm.maps)) return cudaErrorInvalidValue;
    cache.put(key, prm.maps);
  }
  // Programmatic dependent launch: the engine's prologue overlaps the prep
  // kernel; its griddepcontrol.wait orders every use of the prep's outputs.
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, prm);
}

}  // namespace

cudaError_t launch_expert_cc(const ExpertArgs& a, int num_sms, cudaStream_t stream) {
  return a.wdtype == 1 ? launch_engine<2>(a, num_sms, stream) : launch_engine<4>(a, num_sms, stream);
}

}  // namespace moe
