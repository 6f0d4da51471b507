// expert_mma.cu — the expert FFNs of a verification pass on the
// 5th-generation tensor cores (tcgen05.mma, accumulators in TMEM), every
// weight tile streamed from HBM by TMA once per group.
//
// Sources: "Speculative Decoding for Mixture-of-Experts Models: Expert Bytes,
// Kernel Bandwidth and the Best Draft Length", abstract — the per-slot engine
// reads a selected expert once per token, the deduplicating engine reads it
// once per pass for all the tokens that chose it; "Deep Dive into Mixture of
// Experts: From 1991 to DeepSeek-V3", §2 and §5 (weighted routed experts,
// unweighted shared experts). Each expert is W_down(silu(W_gate x) ⊙ W_up x).
//
// A group's FFN is a contraction over its tokens
//   H[tokens][I] = silu(X·W_gateᵀ) ⊙ (X·W_upᵀ),   Y[tokens][d] = H·W_downᵀ,
// computed as D = W·Xᵀ with the weights as the A operand (M = 128 weight rows
// per tile) and the group's tokens as B, fp32 accumulation. With one to a few
// tokens the tensor cores idle most of the time; what matters is that the
// weights flow from HBM to shared memory to the tensor core with no
// per-element instruction. The weights are bf16 exactly; each fp32
// activation is split as hi + lo, both bf16 (hi = bf16(v), lo = bf16(v − hi)),
// so activations keep ~16 more mantissa bits than one bf16 rounding. The two
// halves are separate columns of one B tile — rows [0, h) the tokens' hi
// halves, rows [h, 2h) their lo halves, h = 8, 16 or 32 ≥ the group's tokens,
// N = 2h — so one MMA per K-step covers both, and the epilogue adds column t
// and column h + t. Phase 0 stacks 64 rows of W_gate over the same 64 rows
// of W_up as one 128-row A tile, so one accumulator holds both products
// (TMEM lanes 0-63 and 64-127) and a phase-0 job covers 64 rows of I — half
// the bytes of a 128-row gate tile plus a 128-row up tile, which halves the
// grain of the work a call is dealt in without cutting K. The epilogue
// warps of the up half hand their values to the gate half through shared
// memory, which writes h as its hi/lo halves. Phase 1 (down) writes the
// weighted slot outputs. When the call fuses the combine, every CTA counts
// the row quarters it stored and, after its last job, takes part in the
// kernel's last phase (tail_combine): once the whole call's quarters are
// stored, it sums its share of y over the slots in slot order. Every stage carries two 64-column K-steps; the
// ring holds as many stages as fit for the call's largest token tile (5 for
// h ≤ 16, 4 for h = 32), which matters most for per-slot calls, about half
// of whose weight reads hit L2 and half miss to DRAM.
//
// Jobs. A job is (entry, tile, piece of K). When a phase has fewer
// tiles than CTAs, each tile is cut into S ≤ 8 pieces along K so that every
// SM streams. Every piece stores its fp32 partial sums and counts
// itself per 32-row quarter with a release reduction (nothing waits for
// it); the CTA that runs a tile's last piece hands each quarter to one of its
// four finisher warps, which waits (bounded) until all pieces of the quarter
// are counted, adds them in piece order — a fixed order, so results are
// reproducible — and finishes the quarter off the tensor pipeline's path.
// A phase-1 job loads its group's h only after every phase-0 tile of the
// group is stored (a count in scratch, bounded acquire wait).
//
// Warp roles (one CTA per SM, persistent, jobs from a global counter):
//   warp 0    TMA producer (one thread),
//   warp 1    TMEM owner and MMA issuer (one thread), two accumulator slots,
//   warps 2-5 epilogue: TMEM → registers → partials / SwiGLU / weighting → global,
//   warp 6    publisher of phase-0 tiles finished by the epilogue (GPU-scope release),
//   warp 7    only helps build the group table,
//   warps 8-11 finishers of tiles cut into pieces (warp 8+q: rows 32q..32q+31).
#include <cuda_bf16.h>
#include <math.h>

#include "moe_warp.h"
#include "common.cuh"
#include "launch.h"
#include "plan.cuh"
#include "tcgen05.cuh"
#include "tmap.h"

namespace moe {
namespace {

constexpr int kM = 128;                             // A rows per tile (MMA M)
constexpr int kH0 = 64;                             // rows of I per phase-0 tile (gate and up)
constexpr int kSub = kMmaSub;                       // tokens per entry (≤ MMA N)
constexpr int kMaxStages = 5;
constexpr int kThreads = 384;
constexpr int kTileBytes = kM * 128;                // [128 rows][64 bf16]
constexpr int kBStepBytes = 2 * kSub * 128;         // one K-step of tokens: [2h ≤ 64 rows][64 bf16]
// A stage holds the weight tiles of two K-steps, then their token tiles
// (2 K-steps × [hi | lo] × h rows × 128 bytes). The ring's stage count is set
// per launch from the largest h of the call: 5 stages for h ≤ 16, 4 for 32.
constexpr int kRingBytes = 5 * (2 * kTileBytes + 2 * 2 * 16 * 128);
static_assert(4 * (2 * kTileBytes + 2 * kBStepBytes) <= kRingBytes, "four stages at h = 32");
constexpr int kMaxEntries = max_entries(kSub);
constexpr int kMaxRows = MOE_MAX_PAIRS + MOE_MAX_SHARED * MOE_MAX_TOKENS;
constexpr int kSlotCols = 128;                      // TMEM columns per accumulator slot (gate, up)
constexpr int kTmemCols = 2 * kSlotCols;
constexpr int kJobsPerCta = 1;                      // tiles are cut only while a phase has fewer than one per CTA
constexpr int kMaxPieces = 8;
static_assert(kMaxEntries == kMmaEntries, "tensor-core kernel entry count");
static_assert(kSub == 32, "the epilogue and the TMEM slots assume at most 32 tokens");

constexpr int kOffBar = kRingBytes;
constexpr int kPubSlots = 8;                        // ring of finished phase-0 jobs
constexpr int kFinSlots = 16;                       // per finisher: ring of quarters to finish
constexpr int kNumBars = 2 * kMaxStages + 4 + 1 + 2 * kPubSlots + 2 * 4 * kFinSlots + 2;
constexpr int kOffPlan = kOffBar + kNumBars * 8;
constexpr int kOffRowOut = kOffPlan + kMaxEntries * (int)sizeof(Entry);
constexpr int kOffRowW = kOffRowOut + kMaxRows * 2;
constexpr int kOffMisc = kOffRowW + kMaxRows * 4;
constexpr int kOffXch = kOffMisc + 160 * 4;         // [kH0 rows][kSub tokens] fp32: up → gate half
constexpr int kSmemBytes = kOffXch + kH0 * kSub * 4 + 1024;  // + slack to align the base to 1024
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

// Token tensors read as B, for h = 8, 16, 32 rows: routed-group inputs (x
// gathered in union order, or x for per-slot), shared-expert inputs (x),
// phase-1 inputs (h). Each is stored as its hi half then its lo half
// ([2][rows][K] bf16), so one box [2][h][64] brings both halves of a
// K-step — the B tile's rows [0, h) and [h, 2h) — and the h box spans
// two K-steps ([2 K-steps][2][h][64]).
enum { kXA, kXS, kHH, kNumB };

// Weight maps (bf16, 128-byte swizzle, 64-column K-steps). gu/sgu: W_gate
// and W_up as one [K/64][2][E][I][64] tensor (the pair stride is the
// distance between the two arrays, pair/spair set when expressible;
// up_first when W_up lies below W_gate), so one box carries the stacked
// 64 + 64-row A tiles of both K-steps of a phase-0 stage; wg/wu/swg/swu load
// 64-row tiles one K-step at a time otherwise. wd/swd: W_down viewed as
// [K/64][E][rows][64] (a 128-byte stride between 64-column K-steps), so one
// box carries the two K-steps of a phase-1 stage. An SM's TMA stream
// completes boxes at a roughly fixed rate, so fewer boxes per stage raise
// what one SM can pull from HBM.
struct Maps {
  CUtensorMap wg, wu, wd, swg, swu, swd, gu, sgu;
  CUtensorMap b[3][kNumB];                // [h = 8, 16, 32][tensor]
  int pair, spair, up_first, sup_first;
};

// Rows h of a group's B tile half for m tokens, and its index in Maps::b.
MOE_DEV int b_rows(int m) { return m <= 8 ? 8 : (m <= 16 ? 16 : 32); }
MOE_DEV int b_index(int h) { return h == 8 ? 0 : (h == 16 ? 1 : 2); }

struct Params {
  Maps maps;
  ExpertArgs a;
};

// How one phase is cut: T tiles per entry, nks K-steps per tile, S pieces of
// kc K-steps (the last may be shorter).
struct Cut {
  int T, nks, S, kc;
};

// Pieces per tile for `tiles` (entry, tile) pairs: enough for kJobsPerCta
// jobs per CTA, at most one per K-step, within the partial-sum scratch and
// the arrival counts; then every piece non-empty.
MOE_DEV Cut make_cut(int T, int nks, int tiles, int target, size_t budget, size_t slab_bytes) {
  Cut c{T, nks, 1, nks};
  if (tiles <= 0 || tiles >= target || 4 * tiles > kMmaCntInts) return c;
  int S = min(min((target + tiles - 1) / tiles, nks), kMaxPieces);
  while (S > 1 && (size_t)tiles * S * slab_bytes > budget) --S;
  if (S <= 1) return c;
  c.kc = (nks + S - 1) / S;
  c.S = (nks + c.kc - 1) / c.kc;
  return c;
}

MOE_DEV uint16_t to_bf16(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }

static_assert(MOE_MAX_EXPERTS <= kThreads && MOE_MAX_PAIRS <= 2 * kThreads,
              "build_plan: one thread per expert, two pairs per thread");
static_assert(kMaxRows >= 2 * MOE_MAX_EXPERTS, "build_plan: row_w holds its sort scratch");

__global__ void __launch_bounds__(kThreads, 1) expert_mma_kernel(const __grid_constant__ Params prm) {
  const ExpertArgs& a = prm.a;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* empty = full + kMaxStages;
  uint64_t* tfull = empty + kMaxStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* pub_full = drain + 1;  // epilogue warps → publisher: a phase-0 job's quarters
  uint64_t* pub_empty = pub_full + kPubSlots;
  uint64_t* fin_full = pub_empty + kPubSlots;  // [4][kFinSlots] epilogue warp q → finisher q
  uint64_t* fin_empty = fin_full + 4 * kFinSlots;
  uint64_t* xfull = fin_empty + 4 * kFinSlots;  // up-half epilogue warps → gate half
  uint64_t* xempty = xfull + 1;
  float* xch = reinterpret_cast<float*>(smem + kOffXch);
  Entry* plan = reinterpret_cast<Entry*>(smem + kOffPlan);
  uint16_t* row_out = reinterpret_cast<uint16_t*>(smem + kOffRowOut);
  float* row_w = reinterpret_cast<float*>(smem + kOffRowW);
  int* misc = reinterpret_cast<int*>(smem + kOffMisc);  // [0..15] scan scratch
  volatile int* stage_job = misc + 16;                  // [kMaxStages]
  volatile int* acc_job = misc + 24;                    // [2]
  uint32_t* tmem_base = reinterpret_cast<uint32_t*>(misc + 28);
  volatile int* abort_flag = misc + 32;
  volatile int* pub_entry = misc + 36;                  // [kPubSlots]
  int* pub_cnt = misc + 44;                             // [kPubSlots] quarters finished
  int* max_m = misc + 52;
  volatile int* fin_job = misc + 64;                    // [4][kFinSlots]
  int* tail_flag = misc + 128;                          // fused combine: the wait's outcome
  int* ph1_done = misc + 129;                           // phase-1 row quarters stored by this CTA

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4);
    }
    mbar_init(drain, 1);
    for (int i = 0; i < kPubSlots; ++i) {
      mbar_init(&pub_full[i], 4);
      mbar_init(&pub_empty[i], 1);
      pub_cnt[i] = 0;
    }
    for (int i = 0; i < 4 * kFinSlots; ++i) {
      mbar_init(&fin_full[i], 1);
      mbar_init(&fin_empty[i], 1);
    }
    mbar_init(xfull, 2);
    mbar_init(xempty, 2);
    *ph1_done = 0;
    *abort_flag = 0;
    *max_m = 0;
    fence_mbar_init();
  }
  if (warp == 1) umma::tmem_alloc(tmem_base, kTmemCols);
  if (threadIdx.x == 32 * 3 && a.prefetch_shared) shared_l2_prefetch(a);
  if (threadIdx.x == 32 * 2) {
    prefetch_tmap(prm.maps.pair ? &prm.maps.gu : &prm.maps.wg);
    prefetch_tmap(&prm.maps.wd);
    prefetch_tmap(&prm.maps.b[0][kXA]);
    prefetch_tmap(&prm.maps.b[0][kHH]);
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  // The kernel before this one — the prep kernel, or the top-k/union kernel
  // of a whole pass — has written the routing, the union and the rows this
  // kernel reads, and zeroed its counters.
  pdl_wait();
  // The CUDA-core kernel, if it runs, may start now on SMs this kernel leaves
  // free: it needs nothing from this kernel, and its inputs are complete.
  pdl_trigger();
  const int n_groups = build_plan<kSub, true>(a, plan, row_out, row_w, misc);
  __syncthreads();
  for (int i = threadIdx.x; i < n_groups; i += blockDim.x) atomicMax(max_m, plan[i].m);
  __syncthreads();
  const uint32_t tmem = *tmem_base;

  // Partial sums: slabs of [npad tokens][128 A rows] fp32 (phase 0: 64 gate
  // rows over 64 up rows).
  const int npad = *max_m <= 16 ? 16 : 32;
  // the ring: stages sized for the call's largest token tile
  const int stage_bytes = 2 * kTileBytes + 4 * b_rows(*max_m) * 128;
  const int n_stages = min(kMaxStages, kRingBytes / stage_bytes);
  const size_t slab0 = (size_t)npad * kM, slab1 = (size_t)npad * kM;  // floats
  const size_t budget0 = a.part_bytes / 2, budget1 = a.part_bytes - budget0;
  float* part0 = a.part;
  float* part1 = a.part + budget0 / 4;
  const int target = kJobsPerCta * (int)gridDim.x;
  const Cut c0 = make_cut(a.I / kH0, (a.d + 127) / 128, n_groups * (a.I / kH0), target, budget0,
                          slab0 * 4);
  const Cut c1 = make_cut((a.d + kM - 1) / kM, (a.I + 127) / 128,
                          n_groups * ((a.d + kM - 1) / kM), target, budget1, slab1 * 4);
  const int J0 = n_groups * c0.T * c0.S, J = J0 + n_groups * c1.T * c1.S;
  int* job_counter = a.sync_mma;
  int* done0 = a.sync_mma + 1;
  int* cnt0 = a.sync_mma + 1 + kMmaEntries;
  int* cnt1 = cnt0 + kMmaCntInts;
  const int done_target = 4 * c0.T;  // four per phase-0 tile (one per quarter, or 4 at once)

  auto decode = [&](int job, int* ph, int* g, int* tile, int* piece) {
    *ph = job < J0 ? 0 : 1;
    const Cut& c = *ph == 0 ? c0 : c1;
    job_decode(plan, *ph == 0 ? job : job - J0, c.T, c.S, g, tile, piece);
  };

  if (warp == 0) {
    // ------------------------------------------------------ producer thread --
    if (lane == 0) {
      const uint64_t pol_w = weight_policy(a.keep_weights);
      const uint64_t pol_x = l2_evict_last_policy();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      while (ok) {
        const int job = atomicAdd(job_counter, 1);
        if (job >= J) {
          if (mbar_wait(&empty[stage], phase ^ 1u, a.err, 0x301)) {
            stage_job[stage] = -1;
            mbar_arrive(&full[stage]);
          } else {
            *abort_flag = 1;
          }
          break;
        }
        int ph, g, tile, piece;
        decode(job, &ph, &g, &tile, &piece);
        const Entry en = plan[g];
        const bool sh = en.src < 0;
        const int ec = sh ? -en.src - 1 : en.src;
        const int hb = b_rows(en.m);
        const CUtensorMap* bm = prm.maps.b[b_index(hb)];
        const uint32_t bbytes = hb * 128;  // one half (hi or lo) of one K-step
        const Cut& c = ph == 0 ? c0 : c1;
        const int ks_end = min(c.nks, (piece + 1) * c.kc);
        for (int ks = piece * c.kc; ks < ks_end && ok; ++ks) {
          if (*abort_flag || !mbar_wait(&empty[stage], phase ^ 1u, a.err, 0x300)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          unsigned char* st = smem + stage * stage_bytes;
          unsigned char* bt = st + 2 * kTileBytes;
          if (ks == piece * c.kc) stage_job[stage] = job;
          if (ph == 0) {
            // A: [K-step][64 rows of the lower array][64 rows of the other]
            mbar_arrive_expect_tx(&full[stage], 2 * kTileBytes + 4 * bbytes);
            if (sh ? prm.maps.spair : prm.maps.pair) {
              tma_load_5d(st, sh ? &prm.maps.sgu : &prm.maps.gu, 0, tile * kH0, ec, 0, 2 * ks,
                          &full[stage], pol_w);
            } else {
              const CUtensorMap* wg = sh ? &prm.maps.swg : &prm.maps.wg;
              const CUtensorMap* wu = sh ? &prm.maps.swu : &prm.maps.wu;
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const int k0 = (2 * ks + j) * 64;
                tma_load_3d(st + j * kTileBytes, wg, k0, tile * kH0, ec, &full[stage], pol_w);
                tma_load_3d(st + j * kTileBytes + kTileBytes / 2, wu, k0, tile * kH0, ec,
                            &full[stage], pol_w);
              }
            }
            tma_load_4d(bt, &bm[sh ? kXS : kXA], 0, en.arow, 0, 2 * ks, &full[stage], pol_x);
          } else {
            mbar_arrive_expect_tx(&full[stage], 2 * kTileBytes + 4 * bbytes);
            tma_load_4d(st, sh ? &prm.maps.swd : &prm.maps.wd, 0, tile * kM, ec, 2 * ks,
                        &full[stage], pol_w);
            if (ks == piece * c.kc) {
              // the group's h rows must all be stored before they are read
              if (!wait_count(done0 + g, done_target, a.err, 0x340)) *abort_flag = 1;
              fence_proxy_async_global();
            }
            tma_load_4d(bt, &bm[kHH], 0, en.row0, 0, 2 * ks, &full[stage], pol_x);
          }
          if (++stage == n_stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issue thread --
    if (lane == 0) {
      int stage = 0, slot = 0;
      uint32_t phase = 0, sphase = 0;
      bool issued_any = false;
      for (;;) {
        if (*abort_flag || !mbar_wait(&full[stage], phase, a.err, 0x320)) {
          *abort_flag = 1;
          break;
        }
        const int job = stage_job[stage];
        if (!mbar_wait(&tempty[slot], sphase ^ 1u, a.err, 0x321)) {
          *abort_flag = 1;
          break;
        }
        umma::fence_after_sync();
        acc_job[slot] = job;
        if (job < 0) {
          __threadfence_block();
          mbar_arrive(&tfull[slot]);
          break;
        }
        int ph, g, tile, piece;
        decode(job, &ph, &g, &tile, &piece);
        const int m = plan[g].m;
        const uint32_t idesc = umma::idesc_bf16(kM, 2 * b_rows(m));
        const uint32_t dacc = tmem + slot * kSlotCols;
        const Cut& c = ph == 0 ? c0 : c1;
        const int ks0 = piece * c.kc, ks_end = min(c.nks, ks0 + c.kc);
        bool ok = true;
        for (int ks = ks0; ks < ks_end; ++ks) {
          if (ks > ks0 && !mbar_wait(&full[stage], phase, a.err, 0x322)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          // the stage's two K-steps: A tiles at st and st + kTileBytes, the
          // tokens' [hi | lo] rows at bt and bt + 2h·128 bytes
          const uint32_t st = smem_addr(smem + stage * stage_bytes);
          const uint64_t a0 = umma::desc_sw128(st);
          const uint64_t a1 = umma::desc_sw128(st + kTileBytes);
          const uint32_t bt = st + 2 * kTileBytes;
          const uint64_t b0 = umma::desc_sw128(bt);                   // K-step 0: hi | lo rows
          const bool first = ks == ks0;
          const uint64_t b1 = umma::desc_sw128(bt + 2 * b_rows(m) * 128);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            umma::mma_bf16(dacc, a0 + 2 * j, b0 + 2 * j, idesc, (!first || j != 0) ? 1u : 0u);
#pragma unroll
          for (int j = 0; j < 4; ++j) umma::mma_bf16(dacc, a1 + 2 * j, b1 + 2 * j, idesc, 1u);
          issued_any = true;
          umma::commit(&empty[stage]);  // frees the stage once these MMAs have read it
          if (++stage == n_stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma::commit(&tfull[slot]);     // accumulator ready once all MMAs are done
        if (++slot == 2) {
          slot = 0;
          sphase ^= 1u;
        }
      }
      // Every MMA issued by this thread has finished before TMEM is released.
      if (issued_any) {
        umma::commit(drain);
        mbar_wait(drain, 0, a.err, 0x323);
      }
    }
  } else if (warp >= 2 && warp < 6) {
    // ----------------------------------------------------------- epilogue --
    // Warp w handles rows 32·(w mod 4) .. +31 of every tile (its TMEM lanes).
    const int quad = warp & 3;
    const int r_in = quad * 32 + lane;
    int slot = 0;
    uint32_t sphase = 0;
    int pub_n = 0;  // phase-0 jobs handed to the publisher so far
    int fin_n = 0;  // quarters handed to finisher `quad` so far (lane 0)
    int x_n = 0;    // phase-0 tiles passed through xch so far
    uint64_t* my_fin_full = fin_full + quad * kFinSlots;
    uint64_t* my_fin_empty = fin_empty + quad * kFinSlots;
    volatile int* my_fin_job = fin_job + quad * kFinSlots;
    for (;;) {
      if (!mbar_wait(&tfull[slot], sphase, a.err, 0x330)) {
        *abort_flag = 1;
        break;
      }
      umma::fence_after_sync();
      const int job = acc_job[slot];
      if (job < 0) {
        // end marker for the publisher
        if (lane == 0) {
          const int ps = pub_n % kPubSlots;
          if (mbar_wait(&pub_empty[ps], (uint32_t)(((pub_n / kPubSlots) & 1) ^ 1), a.err, 0x352)) {
            if (warp == 2) pub_entry[ps] = -1;
            mbar_arrive(&pub_full[ps]);
          }
          {  // and for this quarter's finisher
            const int fs = fin_n % kFinSlots;
            if (mbar_wait(&my_fin_empty[fs], (uint32_t)(((fin_n / kFinSlots) & 1) ^ 1), a.err, 0x353)) {
              my_fin_job[fs] = -1;
              mbar_arrive(&my_fin_full[fs]);
            }
          }
        }
        break;
      }
      int ph, g, tile, piece;
      decode(job, &ph, &g, &tile, &piece);
      const Entry en = plan[g];
      const int m = en.m;
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + slot * kSlotCols;
      // Token c's sum is column c (hi half) plus column hb + c (lo half).
      const int hb = b_rows(m);
      // this warp's 32 rows of the tile: phase 0 gate or up rows (the half
      // holding rows 64·up_first .. +63 is the gate), phase 1 down rows
      uint32_t gr[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) gr[c] = 0u;
      {
        uint32_t t0[16], t1[16];
        if (hb == 8) {
          umma::ld_x16(taddr, t0);
          umma::wait_ld();
#pragma unroll
          for (int c = 0; c < 8; ++c)
            gr[c] = __float_as_uint(__uint_as_float(t0[c]) + __uint_as_float(t0[8 + c]));
        } else {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            if (half * 16 < hb) {
              umma::ld_x16(taddr + 16 * half, t0);
              umma::ld_x16(taddr + hb + 16 * half, t1);
              umma::wait_ld();
#pragma unroll
              for (int c = 0; c < 16; ++c)
                gr[16 * half + c] = __float_as_uint(__uint_as_float(t0[c]) + __uint_as_float(t1[c]));
            }
          }
        }
      }
      umma::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[slot]);  // accumulator slot free again
      float* gv = reinterpret_cast<float*>(gr);
      const Cut& cut = ph == 0 ? c0 : c1;
      if (cut.S > 1) {
        // A piece: store the partial sums of the warp's 32 rows and count
        // them (release, no wait). The CTA that runs the tile's last piece
        // hands each quarter to that quarter's finisher warp.
        const size_t sfl = ph == 0 ? slab0 : slab1;
        float* mine = (ph == 0 ? part0 : part1) +
                      ((size_t)(g * cut.T + tile) * cut.S + piece) * sfl;
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (c < m) mine[c * kM + r_in] = gv[c];
        __syncwarp();  // the warp's partials before lane 0's release
        if (lane == 0) red_release_add((ph == 0 ? cnt0 : cnt1) + (g * cut.T + tile) * 4 + quad, 1);
        if (lane == 0 && piece == cut.S - 1) {
          const int fs = fin_n % kFinSlots;
          if (!mbar_wait(&my_fin_empty[fs], (uint32_t)(((fin_n / kFinSlots) & 1) ^ 1), a.err, 0x354)) {
            *abort_flag = 1;
          } else {
            my_fin_job[fs] = job;
            mbar_arrive(&my_fin_full[fs]);
          }
          ++fin_n;
        }
        if (++slot == 2) {
          slot = 0;
          sphase ^= 1u;
        }
        continue;
      }
      // One piece: the epilogue finishes the tile's quarter itself.
      const int row = tile * kM + r_in;
      if (ph == 0) {
        // the up half hands its sums to the gate half (bounded waits on
        // two mbarriers; xch holds one tile's up rows at a time)
        const int upf = en.src < 0 ? prm.maps.sup_first : prm.maps.up_first;
        const int hrow = r_in & (kH0 - 1);
        const bool up_half = (quad >> 1) != upf;
        int xok = 1;  // lane 0 waits, the warp follows its result
        if (lane == 0)
          xok = up_half ? mbar_wait(xempty, (uint32_t)((x_n & 1) ^ 1), a.err, 0x356)
                        : mbar_wait(xfull, (uint32_t)(x_n & 1), a.err, 0x357);
        xok = __shfl_sync(0xffffffffu, xok, 0);
        __syncwarp();  // lane 0's acquire before every lane's accesses
        if (up_half) {
          if (xok) {
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (c < m) xch[hrow * kSub + c] = gv[c];
          }
          __syncwarp();
          if (xok && lane == 0) mbar_arrive(xfull);
        } else {
          const int irow = tile * kH0 + hrow;
          if (xok && irow < a.I) {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              if (c < m) {
                const float hv = silu(gv[c]) * xch[hrow * kSub + c];
                const uint16_t hi = to_bf16(hv);
                const size_t at = (size_t)(en.row0 + c) * a.I + irow;
                a.h16[at] = hi;
                a.h16lo[at] = to_bf16(hv - __uint_as_float((uint32_t)hi << 16));
              }
            }
          }
          __syncwarp();
          if (xok && lane == 0) mbar_arrive(xempty);
        }
        ++x_n;
        if (!xok) {
          *abort_flag = 1;
          break;
        }
        // Hand the quarter to the publisher thread: __syncwarp orders the
        // warp's h stores before lane 0's arrive (release, CTA scope).
        __syncwarp();
        if (lane == 0) {
          const int ps = pub_n % kPubSlots;
          if (!mbar_wait(&pub_empty[ps], (uint32_t)(((pub_n / kPubSlots) & 1) ^ 1), a.err, 0x350)) {
            *abort_flag = 1;
          } else {
            atomicAdd(&pub_cnt[ps], 1);
            if (warp == 2) pub_entry[ps] = g;
            mbar_arrive(&pub_full[ps]);
          }
        }
        ++pub_n;
      } else {
        if (tile * kM + quad * 32 < a.d) {  // warp-uniform: d is a multiple of 32
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if (c < m) {
              const int rr = en.row0 + c;
              a.y_slot[(size_t)row_out[rr] * a.d + row] = row_w[rr] * gv[c];
            }
          }
        }
        if (lane == 0) atomicAdd(ph1_done, 1);  // one row quarter stored (fused combine)
      }
      if (++slot == 2) {
        slot = 0;
        sphase ^= 1u;
      }
    }
  } else if (warp == 6) {
    // ---------------------------------------------------- publisher thread --
    // Publishes each phase-0 job's finished quarters to the group's phase-1
    // jobs with a GPU-scope release, so that the epilogue warps only pay a
    // CTA-scope arrive; this thread's wait acquires their h stores and its
    // release reduction makes them visible GPU-wide before the count.
    if (lane == 0) {
      for (int pn = 0;; ++pn) {
        const int ps = pn % kPubSlots;
        if (!mbar_wait(&pub_full[ps], (uint32_t)((pn / kPubSlots) & 1), a.err, 0x351)) break;
        const int e = pub_entry[ps];
        if (e < 0) break;
        const int q = pub_cnt[ps];
        pub_cnt[ps] = 0;
        if (q > 0) red_release_add(done0 + e, q);
        mbar_arrive(&pub_empty[ps]);
      }
    }
  } else if (warp >= 8) {
    // ---------------------------------------------------- finisher warps --
    // Finisher q, for each quarter q of a tile whose last piece ran here:
    // wait (bounded) until the S pieces of the quarter are counted, add the
    // pieces in piece order (lane l: row 32q + l; four tokens per round of
    // loads), finish the rows and, in phase 0, publish the quarter to the
    // group's phase-1 jobs. In phase 0 the finisher of a gate quarter also
    // waits for and adds the up rows 64 apart (quarter q ^ 2); the finisher
    // of an up quarter only publishes.
    const int q = warp - 8;
    const int row_in = q * 32 + lane;
    uint64_t* my_full = fin_full + q * kFinSlots;
    uint64_t* my_empty = fin_empty + q * kFinSlots;
    volatile int* my_job = fin_job + q * kFinSlots;
    for (int fn = 0;; ++fn) {
      const int fs = fn % kFinSlots;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&my_full[fs], (uint32_t)((fn / kFinSlots) & 1), a.err, 0x360);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      __syncwarp();
      if (!ok) break;
      const int job = my_job[fs];
      if (job < 0) break;
      int ph, g, tile, piece;
      decode(job, &ph, &g, &tile, &piece);
      const Cut& cut = ph == 0 ? c0 : c1;
      const Entry en = plan[g];
      const int upf = en.src < 0 ? prm.maps.sup_first : prm.maps.up_first;
      const bool up_q = ph == 0 && (q >> 1) != upf;
      if (lane == 0 && !up_q) {
        const int* cnt = (ph == 0 ? cnt0 : cnt1) + (g * cut.T + tile) * 4;
        ok = wait_count(cnt + q, cut.S, a.err, 0x361) &&
             (ph != 0 || wait_count(cnt + (q ^ 2), cut.S, a.err, 0x362));
        if (!ok) *abort_flag = 1;
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      __syncwarp();  // lane 0's acquire before every lane's reads
      const int m = en.m;
      const size_t sfl = ph == 0 ? slab0 : slab1;
      const float* base = (ph == 0 ? part0 : part1) + (size_t)(g * cut.T + tile) * cut.S * sfl;
      const int row = ph == 0 ? tile * kH0 + (row_in & (kH0 - 1)) : tile * kM + row_in;
      for (int cb = 0; ok && !up_q && cb < m; cb += 4) {
        float sg[4], su[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) sg[u] = su[u] = 0.f;
#pragma unroll
        for (int p = 0; p < kMaxPieces; ++p) {
          if (p < cut.S) {
            const float* src = base + (size_t)p * sfl;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if (cb + u < m) {
                sg[u] += __ldcg(src + (cb + u) * kM + row_in);
                if (ph == 0) su[u] += __ldcg(src + (cb + u) * kM + (row_in ^ kH0));
              }
            }
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = cb + u;
          if (c < m) {
            if (ph == 0) {
              if (row < a.I) {
                const float hv = silu(sg[u]) * su[u];
                const uint16_t hi = to_bf16(hv);
                const size_t at = (size_t)(en.row0 + c) * a.I + row;
                a.h16[at] = hi;
                a.h16lo[at] = to_bf16(hv - __uint_as_float((uint32_t)hi << 16));
              }
            } else if (row < a.d) {
              const int rr = en.row0 + c;
              a.y_slot[(size_t)row_out[rr] * a.d + row] = row_w[rr] * sg[u];
            }
          }
        }
      }
      if (ph == 1 && ok && lane == 0) atomicAdd(ph1_done, 1);  // one row quarter (fused combine)
      __syncwarp();  // every lane's stores before lane 0's release
      if (lane == 0) {
        if (ph == 0 && ok) red_release_add(done0 + g, 1);
        mbar_arrive(&my_empty[fs]);
      }
    }
  }
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    umma::fence_after_sync();
    umma::tmem_dealloc(tmem, kTmemCols);
  }
  // The combine fused as the last phase: every (entry, phase-1 tile) stores
  // four row quarters, through the epilogue or the finishers.
  if (a.y)
    tail_combine(a, ph1_done, n_groups * c1.T * 4, abort_flag, tail_flag, (int)threadIdx.x,
                 kThreads, [] { __syncthreads(); });
}

// W_gate or W_up [n_mat][rows][K] in 64-row boxes of one K-step.
bool w_map(CUtensorMap* m, const void* p, int n_mat, int rows, int K) {
  const uint64_t dims[3] = {(uint64_t)K, (uint64_t)rows, (uint64_t)n_mat};
  const uint64_t strides[2] = {(uint64_t)K * 2, (uint64_t)rows * K * 2};
  const uint32_t box[3] = {64, (uint32_t)kH0, 1};
  return make_tmap(m, p, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
}

// W_gate and W_up as one [K/64][2][n_mat][rows][64] tensor based at the
// lower of the two arrays: a box [2 K-steps][2][64 rows][64] is the stage's
// two stacked A tiles. False (load them separately) unless their distance is
// a non-zero multiple of 16 bytes below 2^40, the tensor map's stride limit.
bool pair_map(CUtensorMap* m, int* up_first, const void* gate, const void* up, int n_mat,
              int rows, int K) {
  const uintptr_t pg = reinterpret_cast<uintptr_t>(gate), pu = reinterpret_cast<uintptr_t>(up);
  const uint64_t delta = pu > pg ? pu - pg : pg - pu;
  if (delta == 0 || delta % 16 != 0 || delta >= (1ull << 40)) return false;
  *up_first = pu < pg ? 1 : 0;
  const uint64_t dims[5] = {64, (uint64_t)rows, (uint64_t)n_mat, 2, (uint64_t)(K / 64)};
  const uint64_t strides[4] = {(uint64_t)K * 2, (uint64_t)rows * K * 2, delta, 128};
  const uint32_t box[5] = {64, (uint32_t)kH0, 1, 2, 2};
  return make_tmap(m, reinterpret_cast<const void*>(pu < pg ? pu : pg),
                   CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
}

// W_down [n_mat][rows][K] viewed as [K/64][n_mat][rows][64]: a box of two
// 64-column K-steps lands as two consecutive 128-row tiles.
bool down_map(CUtensorMap* m, const void* p, int n_mat, int rows, int K) {
  const uint64_t dims[4] = {64, (uint64_t)rows, (uint64_t)n_mat, (uint64_t)(K / 64)};
  const uint64_t strides[3] = {(uint64_t)K * 2, (uint64_t)rows * K * 2, 128};
  const uint32_t box[4] = {64, (uint32_t)kM, 1, 2};
  return make_tmap(m, p, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
}

// Token rows [2 (hi, lo)][rows][K] bf16 viewed as [K/64][2][rows][64]: a box
// [2 K-steps][2][box_rows][64] is the B tiles of a stage's two K-steps (the
// K-step dimension outermost, 128 bytes apart).
bool b_map(CUtensorMap* m, const void* p, int rows, int K, int box_rows) {
  const uint64_t dims[4] = {64, (uint64_t)rows, 2, (uint64_t)(K / 64)};
  const uint64_t strides[3] = {(uint64_t)K * 2, (uint64_t)rows * K * 2, 128};
  const uint32_t box[4] = {64, (uint32_t)box_rows, 2, 2};
  return make_tmap(m, p, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
}

// Every tensor map of one launch.
bool build_maps(const ExpertArgs& a, Maps* M) {
  memset(M, 0, sizeof *M);
  const int P = a.n * a.k;
  const int hrows = P + a.s * a.n;
  bool ok = true;
  ok &= w_map(&M->wg, a.w_gate, a.E, a.I, a.d);
  ok &= w_map(&M->wu, a.w_up, a.E, a.I, a.d);
  ok &= down_map(&M->wd, a.w_down, a.E, a.d, a.I);
  M->pair = pair_map(&M->gu, &M->up_first, a.w_gate, a.w_up, a.E, a.I, a.d) ? 1 : 0;
  if (!M->pair) M->up_first = 0;
  if (a.s > 0) {
    ok &= w_map(&M->swg, a.ws_gate, a.s, a.I, a.d);
    ok &= w_map(&M->swu, a.ws_up, a.s, a.I, a.d);
    ok &= down_map(&M->swd, a.ws_down, a.s, a.d, a.I);
    M->spair = pair_map(&M->sgu, &M->sup_first, a.ws_gate, a.ws_up, a.s, a.I, a.d) ? 1 : 0;
    if (!M->spair) M->sup_first = 0;
  }
  // Phase-0 token rows: x gathered in union order (dedup) or x itself
  // (per-slot: an entry's row is its token); shared experts read x. The lo
  // halves follow the hi halves: xg16lo = xg16 + P·d, x16lo = x16 + n·d,
  // h16lo = h16 + hrows·I.
  const uint16_t* xa = a.engine == 1 ? a.xg16 : a.x16;
  const int xa_rows = a.engine == 1 ? P : a.n;
  if (a.xg16lo != a.xg16 + (size_t)P * a.d || a.x16lo != a.x16 + (size_t)a.n * a.d ||
      a.h16lo != a.h16 + (size_t)hrows * a.I)
    return false;
  for (int si = 0; si < 3; ++si) {
    const int br = 8 << si;
    CUtensorMap* B = M->b[si];
    ok &= b_map(&B[kXA], xa, xa_rows, a.d, br);
    ok &= b_map(&B[kXS], a.x16, a.n, a.d, br);
    ok &= b_map(&B[kHH], a.h16, hrows, a.I, br);
  }
  return ok;
}

}  // namespace

cudaError_t launch_expert_mma(const ExpertArgs& a, int num_sms, cudaStream_t stream) {
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(expert_mma_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  Params prm;
  memset(&prm, 0, sizeof prm);
  prm.a = a;
  // Everything the tensor maps depend on; a recent call with the same key
  // reuses its maps.
  struct Key {
    const void* p[13];
    int v[8];
  } key;
  memset(&key, 0, sizeof key);
  const void* kp[13] = {a.w_gate, a.w_up, a.w_down, a.ws_gate, a.ws_up, a.ws_down, a.xg16,
                        a.xg16lo, a.x16, a.x16lo, a.h16, a.h16lo, nullptr};
  memcpy(key.p, kp, sizeof kp);
  const int kv[8] = {a.d, a.I, a.E, a.k, a.s, a.n, a.engine, dev};
  memcpy(key.v, kv, sizeof kv);
  static RecentCache<Key, Maps> cache;
  if (!cache.get(key, &prm.maps)) {
    if (!build_maps(a, &prm.maps)) return cudaErrorInvalidValue;
    cache.put(key, prm.maps);
  }
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, expert_mma_kernel, prm);
}

}  // namespace moe
