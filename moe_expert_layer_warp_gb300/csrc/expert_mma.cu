// expert_mma.cu — the expert FFNs of groups that many tokens share, on the
// 5th-generation tensor cores (tcgen05.mma, accumulators in TMEM), weights
// streamed from HBM by TMA once per group.
//
// Sources: "Speculative Decoding for Mixture-of-Experts Models: Expert Bytes,
// Kernel Bandwidth and the Best Draft Length", abstract — the deduplicating
// engine reads each selected expert once per pass for all the tokens that
// chose it; "Deep Dive into Mixture of Experts: From 1991 to DeepSeek-V3", §2
// and §5 (weighted routed experts, unweighted shared experts). Each expert is
// W_down(silu(W_gate x) ⊙ W_up x).
//
// Once a group holds several tokens, its FFN is a dense contraction
//   H[tokens][I] = silu(X·W_gateᵀ) ⊙ (X·W_upᵀ),   Y[tokens][d] = H·W_downᵀ,
// computed here as D = W·Xᵀ with the weights as the A operand (M = 128 weight
// rows per tile) and the group's tokens as B (N = 16 or 32, sub-groups of at
// most 32 tokens), fp32 accumulation. The weights are bf16 exactly; each fp32
// activation is split as hi + lo, both bf16 (hi = bf16(v), lo = bf16(v − hi)),
// and both halves are multiplied into the same accumulator, so activations
// keep ~16 more mantissa bits than a single bf16 rounding would. Phase 0
// (gate and up, a 64-column K-step per stage, two accumulators) writes h as
// its hi/lo halves; phase 1 (down, two K-steps per stage) writes the weighted
// slot outputs. A phase-1
// job loads its group's h only after every phase-0 tile of the group is
// stored (counted in scratch, bounded acquire wait).
//
// Warp roles (one CTA per SM, persistent, jobs from a global counter):
//   warp 0    TMA producer (one thread),
//   warp 1    TMEM owner and MMA issuer (one thread), two accumulator slots,
//   warps 2-5 epilogue: TMEM → registers → SwiGLU or weighting → global,
//   warps 6-7 only help build the group table.
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

constexpr int kM = 128;                             // weight rows per tile
constexpr int kSub = kMmaSub;                       // tokens per entry (≤ MMA N)
constexpr int kStages = 4;
constexpr int kThreads = 256;
constexpr int kTileBytes = kM * 128;                // [128 rows][64 bf16]
constexpr int kBTileBytes = kSub * 128;             // [32 rows][64 bf16]
// stage: two weight tiles, then up to four token tiles (hi/lo × one or two K-steps)
constexpr int kStageBytes = 2 * kTileBytes + 4 * kBTileBytes;
constexpr int kMaxEntries = max_entries(kSub);
constexpr int kMaxRows = MOE_MAX_PAIRS + MOE_MAX_SHARED * MOE_MAX_TOKENS;
constexpr int kSlotCols = 64;                       // TMEM columns per accumulator slot
constexpr int kTmemCols = 2 * kSlotCols;
static_assert(1 + kMaxEntries == kMmaSyncInts, "tensor-core kernel scratch size");
static_assert(kSub == 32, "the epilogue and the TMEM slots assume at most 32 tokens");

constexpr int kOffBar = kStages * kStageBytes;
constexpr int kPubSlots = 8;                        // ring of finished phase-0 jobs
constexpr int kNumBars = 2 * kStages + 4 + 1 + 2 * kPubSlots;  // full, empty, tfull, tempty, drain, pub
constexpr int kOffPlan = kOffBar + kNumBars * 8;
constexpr int kOffRowOut = kOffPlan + kMaxEntries * (int)sizeof(Entry);
constexpr int kOffRowW = kOffRowOut + kMaxRows * 4;
constexpr int kOffMisc = kOffRowW + kMaxRows * 4;
constexpr int kSmemBytes = kOffMisc + 64 * 4 + 1024;  // + slack to align the base to 1024

struct Maps {
  CUtensorMap wg, wu, wd, swg, swu, swd;  // [E or s][rows][K] bf16, box 64 × 128 × 1
  CUtensorMap xa, xs, h;                  // hi halves [rows][K] bf16, box 64 × 32
  CUtensorMap xa_lo, xs_lo, h_lo;         // lo halves, same shapes
};

struct Params {
  Maps maps;
  ExpertArgs a;
};

MOE_DEV uint16_t to_bf16(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }

__global__ void __launch_bounds__(kThreads, 1) expert_mma_kernel(const __grid_constant__ Params prm) {
  const ExpertArgs& a = prm.a;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* pub_full = drain + 1;  // epilogue warps → publisher: a phase-0 job's h is stored
  uint64_t* pub_empty = pub_full + kPubSlots;
  Entry* plan = reinterpret_cast<Entry*>(smem + kOffPlan);
  int* row_out = reinterpret_cast<int*>(smem + kOffRowOut);
  float* row_w = reinterpret_cast<float*>(smem + kOffRowW);
  int* misc = reinterpret_cast<int*>(smem + kOffMisc);  // [0..15] scan scratch
  volatile int* stage_job = misc + 16;                  // [kStages]
  volatile int* acc_job = misc + 24;                    // [2]
  uint32_t* tmem_base = reinterpret_cast<uint32_t*>(misc + 28);
  volatile int* abort_flag = misc + 32;
  volatile int* pub_entry = misc + 36;                  // [kPubSlots]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
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
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) umma::tmem_alloc(tmem_base, kTmemCols);
  if (threadIdx.x == 32 * 2) {
    prefetch_tmap(&prm.maps.wg);
    prefetch_tmap(&prm.maps.wu);
    prefetch_tmap(&prm.maps.wd);
    prefetch_tmap(&prm.maps.xa);
    prefetch_tmap(&prm.maps.h);
  }
  const int n_groups = build_plan<kSub, true>(a, plan, row_out, row_w, misc);
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  pdl_wait();     // prep kernel's outputs
  // The CUDA-core kernel may start now, on SMs this kernel leaves free: it
  // needs nothing from this kernel, and the prep kernel is complete.
  pdl_trigger();
  const uint32_t tmem = *tmem_base;

  const int T0 = (a.I + kM - 1) / kM, T1 = (a.d + kM - 1) / kM;
  const int J0 = n_groups * T0, J = J0 + n_groups * T1;
  const int nks0 = a.d / 64, nks1 = (a.I + 127) / 128;
  int* job_counter = a.sync_mma;
  int* done0 = a.sync_mma + 1;
  const int done_target = T0;  // one publication per phase-0 tile

  if (warp == 0) {
    // ------------------------------------------------------ producer thread --
    if (lane == 0) {
      const uint64_t pol_w = l2_evict_first_policy();
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
        const int ph = job < J0 ? 0 : 1;
        const int jj = ph == 0 ? job : job - J0;
        int g, tile;
        job_entry(plan, jj, ph == 0 ? T0 : T1, &g, &tile);
        const Entry en = plan[g];
        const bool sh = en.src < 0;
        const int ec = sh ? -en.src - 1 : en.src;
        const int nks = ph == 0 ? nks0 : nks1;
        for (int ks = 0; ks < nks && ok; ++ks) {
          if (*abort_flag || !mbar_wait(&empty[stage], phase ^ 1u, a.err, 0x300)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          unsigned char* st = smem + stage * kStageBytes;
          unsigned char* bt = st + 2 * kTileBytes;
          if (ks == 0) stage_job[stage] = job;
          if (ph == 0) {
            const int k0 = ks * 64;
            mbar_arrive_expect_tx(&full[stage], 2 * kTileBytes + 2 * kBTileBytes);
            tma_load_3d(st, sh ? &prm.maps.swg : &prm.maps.wg, k0, tile * kM, ec, &full[stage], pol_w);
            tma_load_3d(st + kTileBytes, sh ? &prm.maps.swu : &prm.maps.wu, k0, tile * kM, ec,
                        &full[stage], pol_w);
            tma_load_2d(bt, sh ? &prm.maps.xs : &prm.maps.xa, k0, en.arow, &full[stage], pol_x);
            tma_load_2d(bt + kBTileBytes, sh ? &prm.maps.xs_lo : &prm.maps.xa_lo, k0, en.arow,
                        &full[stage], pol_x);
          } else {
            const int k0 = ks * 128;
            const CUtensorMap* wd = sh ? &prm.maps.swd : &prm.maps.wd;
            mbar_arrive_expect_tx(&full[stage], 2 * kTileBytes + 4 * kBTileBytes);
            tma_load_3d(st, wd, k0, tile * kM, ec, &full[stage], pol_w);
            tma_load_3d(st + kTileBytes, wd, k0 + 64, tile * kM, ec, &full[stage], pol_w);
            if (ks == 0) {
              // the group's h rows must all be stored before they are read
              if (!wait_count(done0 + g, done_target, a.err, 0x340)) *abort_flag = 1;
              fence_proxy_async_global();
            }
            tma_load_2d(bt, &prm.maps.h, k0, en.row0, &full[stage], pol_x);
            tma_load_2d(bt + kBTileBytes, &prm.maps.h_lo, k0, en.row0, &full[stage], pol_x);
            tma_load_2d(bt + 2 * kBTileBytes, &prm.maps.h, k0 + 64, en.row0, &full[stage], pol_x);
            tma_load_2d(bt + 3 * kBTileBytes, &prm.maps.h_lo, k0 + 64, en.row0, &full[stage],
                        pol_x);
          }
          if (++stage == kStages) {
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
        const int ph = job < J0 ? 0 : 1;
        const int jj = ph == 0 ? job : job - J0;
        int g, tile_unused;
        job_entry(plan, jj, ph == 0 ? T0 : T1, &g, &tile_unused);
        const int m = plan[g].m;
        const uint32_t idesc = umma::idesc_bf16(kM, m <= 16 ? 16 : 32);
        const uint32_t dacc = tmem + slot * kSlotCols;
        const int nks = ph == 0 ? nks0 : nks1;
        bool ok = true;
        for (int ks = 0; ks < nks; ++ks) {
          if (ks > 0 && !mbar_wait(&full[stage], phase, a.err, 0x322)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          const uint32_t st = smem_addr(smem + stage * kStageBytes);
          const uint64_t a0 = umma::desc_sw128(st);
          const uint64_t a1 = umma::desc_sw128(st + kTileBytes);
          const uint32_t bt = st + 2 * kTileBytes;
          const uint64_t b0 = umma::desc_sw128(bt);                   // hi, K-step 0
          const uint64_t b0l = umma::desc_sw128(bt + kBTileBytes);    // lo, K-step 0
          if (ph == 0) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t acc = (ks | j) != 0;
              umma::mma_bf16(dacc, a0 + 2 * j, b0 + 2 * j, idesc, acc);        // gate · x_hi
              umma::mma_bf16(dacc, a0 + 2 * j, b0l + 2 * j, idesc, 1u);        // gate · x_lo
              umma::mma_bf16(dacc + 32, a1 + 2 * j, b0 + 2 * j, idesc, acc);   // up · x_hi
              umma::mma_bf16(dacc + 32, a1 + 2 * j, b0l + 2 * j, idesc, 1u);   // up · x_lo
            }
          } else {
            const uint64_t b1 = umma::desc_sw128(bt + 2 * kBTileBytes);   // hi, K-step 1
            const uint64_t b1l = umma::desc_sw128(bt + 3 * kBTileBytes);  // lo, K-step 1
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              umma::mma_bf16(dacc, a0 + 2 * j, b0 + 2 * j, idesc, (ks | j) != 0);
              umma::mma_bf16(dacc, a0 + 2 * j, b0l + 2 * j, idesc, 1u);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              umma::mma_bf16(dacc, a1 + 2 * j, b1 + 2 * j, idesc, 1u);
              umma::mma_bf16(dacc, a1 + 2 * j, b1l + 2 * j, idesc, 1u);
            }
          }
          issued_any = true;
          umma::commit(&empty[stage]);  // frees the stage once these MMAs have read it
          if (++stage == kStages) {
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
    const int quad = warp & 3;
    const int r_in = quad * 32 + lane;
    int slot = 0;
    uint32_t sphase = 0;
    int pub_n = 0;  // phase-0 jobs handed to the publisher so far
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
        }
        break;
      }
      const int ph = job < J0 ? 0 : 1;
      const int jj = ph == 0 ? job : job - J0;
      int g, tile;
      job_entry(plan, jj, ph == 0 ? T0 : T1, &g, &tile);
      const Entry en = plan[g];
      const int m = en.m;
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + slot * kSlotCols;
      uint32_t v0[16], v1[16], u0[16], u1[16];
      umma::ld_x16(taddr, v0);
      if (m > 16) umma::ld_x16(taddr + 16, v1);
      if (ph == 0) {
        umma::ld_x16(taddr + 32, u0);
        if (m > 16) umma::ld_x16(taddr + 48, u1);
      }
      umma::wait_ld();
      umma::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[slot]);  // accumulator slot free again
      const int row = tile * kM + r_in;
      if (ph == 0) {
        if (row < a.I) {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if (c < m) {
              const float gv = __uint_as_float(c < 16 ? v0[c & 15] : v1[c & 15]);
              const float uv = __uint_as_float(c < 16 ? u0[c & 15] : u1[c & 15]);
              const float hv = silu(gv) * uv;
              const uint16_t hi = to_bf16(hv);
              const size_t at = (size_t)(en.row0 + c) * a.I + row;
              a.h16[at] = hi;
              a.h16lo[at] = to_bf16(hv - __uint_as_float((uint32_t)hi << 16));
            }
          }
        }
        // hand the finished job to the publisher thread: __syncwarp orders the
        // warp's h stores before lane 0's arrive (release, CTA scope)
        __syncwarp();
        if (lane == 0) {
          const int ps = pub_n % kPubSlots;
          if (!mbar_wait(&pub_empty[ps], (uint32_t)(((pub_n / kPubSlots) & 1) ^ 1), a.err, 0x350)) {
            *abort_flag = 1;
          } else {
            if (warp == 2) pub_entry[ps] = g;
            mbar_arrive(&pub_full[ps]);
          }
        }
        ++pub_n;
      } else if (row < a.d) {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (c < m) {
            const int rr = en.row0 + c;
            const float yv = __uint_as_float(c < 16 ? v0[c & 15] : v1[c & 15]);
            a.y_slot[(size_t)row_out[rr] * a.d + row] = row_w[rr] * yv;
          }
        }
      }
      if (++slot == 2) {
        slot = 0;
        sphase ^= 1u;
      }
    }
  } else if (warp == 6) {
    // ---------------------------------------------------- publisher thread --
    // Publishes each finished phase-0 job to the group's phase-1 jobs with a
    // GPU-scope release, so that the epilogue warps only pay a CTA-scope
    // arrive; this thread's wait acquires their h stores and its release
    // reduction makes them visible GPU-wide before the count.
    if (lane == 0) {
      for (int pn = 0;; ++pn) {
        const int ps = pn % kPubSlots;
        if (!mbar_wait(&pub_full[ps], (uint32_t)((pn / kPubSlots) & 1), a.err, 0x351)) break;
        const int e = pub_entry[ps];
        if (e < 0) break;
        red_release_add(done0 + e, 1);
        mbar_arrive(&pub_empty[ps]);
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
}

bool w_map(CUtensorMap* m, const void* p, int n_mat, int rows, int K) {
  const uint64_t dims[3] = {(uint64_t)K, (uint64_t)rows, (uint64_t)n_mat};
  const uint64_t strides[2] = {(uint64_t)K * 2, (uint64_t)rows * K * 2};
  const uint32_t box[3] = {64, (uint32_t)kM, 1};
  return make_tmap(m, p, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
}

bool b_map(CUtensorMap* m, const void* p, int rows, int K) {
  const uint64_t dims[2] = {(uint64_t)K, (uint64_t)rows};
  const uint64_t strides[1] = {(uint64_t)K * 2};
  const uint32_t box[2] = {64, (uint32_t)kSub};
  return make_tmap(m, p, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
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
  const int P = a.n * a.k;
  const int hrows = P + a.s * a.n;
  bool ok = true;
  ok &= w_map(&prm.maps.wg, a.w_gate, a.E, a.I, a.d);
  ok &= w_map(&prm.maps.wu, a.w_up, a.E, a.I, a.d);
  ok &= w_map(&prm.maps.wd, a.w_down, a.E, a.d, a.I);
  if (a.s > 0) {
    ok &= w_map(&prm.maps.swg, a.ws_gate, a.s, a.I, a.d);
    ok &= w_map(&prm.maps.swu, a.ws_up, a.s, a.I, a.d);
    ok &= w_map(&prm.maps.swd, a.ws_down, a.s, a.d, a.I);
  }
  if (a.engine == 1) {
    ok &= b_map(&prm.maps.xa, a.xg16, P, a.d);
    ok &= b_map(&prm.maps.xa_lo, a.xg16lo, P, a.d);
  } else {  // per-slot routed groups (one token each) never run here
    prm.maps.xa = prm.maps.xa_lo = prm.maps.wg;
  }
  ok &= b_map(&prm.maps.xs, a.x16, a.n, a.d);
  ok &= b_map(&prm.maps.xs_lo, a.x16lo, a.n, a.d);
  ok &= b_map(&prm.maps.h, a.h16, hrows, a.I);
  ok &= b_map(&prm.maps.h_lo, a.h16lo, hrows, a.I);
  if (!ok) return cudaErrorInvalidValue;
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
