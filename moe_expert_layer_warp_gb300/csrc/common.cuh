// common.cuh — device helpers shared by the kernels of libmoewarp.so:
// mbarrier and bulk-copy (TMA engine) wrappers in inline PTX for sm_103a,
// bounded waits that report to the library's device error word, and the
// kernel parameter blocks.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define MOE_DEV __device__ __forceinline__

namespace moe {

// ---------------------------------------------------------------- errors --
// Error word written by kernels (first writer wins):
//   bits 0..7  code (ERR_TIMEOUT, ERR_CHECK), bits 8..31 site id.
enum : unsigned int { ERR_TIMEOUT = 3u, ERR_CHECK = 5u };

MOE_DEV void report_error(unsigned int* err, unsigned int code, unsigned int site) {
  if (err) atomicCAS(err, 0u, (code & 0xffu) | (site << 8));
}

// A bounded wait gives up after this long (ns of %globaltimer). Kernels here
// finish in milliseconds; a wait this long means a lost copy or a logic error.
constexpr unsigned long long kWaitLimitNs = 400ull * 1000ull * 1000ull;
constexpr unsigned int kWaitLimitIters = 1u << 30;

MOE_DEV unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// -------------------------------------------------------------- mbarrier --
MOE_DEV uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

MOE_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

MOE_DEV void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

MOE_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

MOE_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

MOE_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits until the phase with the given parity has completed. Returns false
// (and records ERR_TIMEOUT at `site`) if it did not complete within limit_ns.
MOE_DEV bool mbar_wait_for(uint64_t* bar, uint32_t parity, unsigned int* err, unsigned int site,
                           unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (unsigned int i = 0; i < kWaitLimitIters; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 63u && global_ns() - t0 > limit_ns) break;
  }
  report_error(err, ERR_TIMEOUT, site);
  return false;
}

MOE_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned int* err, unsigned int site) {
  return mbar_wait_for(bar, parity, err, site, kWaitLimitNs);
}

// ----------------------------------------------------------- bulk copies --
// L2 policy for weights that are streamed once per pass: evict first, so the
// small activations that every CTA re-reads stay resident.
MOE_DEV uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

MOE_DEV uint64_t l2_evict_normal_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Weight loads: a per-slot call of several tokens reads an expert once per
// slot that chose it, and L2 serves the repeats only if the lines stay
// (normal eviction); otherwise every weight is read once, so its lines go
// first and the activations and routing data stay.
MOE_DEV uint64_t weight_policy(int keep_weights) {
  return keep_weights ? l2_evict_normal_policy() : l2_evict_first_policy();
}

MOE_DEV uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Global -> shared bulk copy on the TMA engine, completing `bytes` of
// transaction count on `bar`. dst/src 16-byte aligned, bytes a multiple of 16.
MOE_DEV void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                      uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Tensor-map (tiled) TMA loads: one instruction moves a whole box; the box's
// bytes (out-of-bounds parts zero-filled) complete on `bar`. Coordinates are
// innermost first.
MOE_DEV void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar,
                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

MOE_DEV void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar)),
      "l"(policy)
      : "memory");
}

MOE_DEV void tma_load_4d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_addr(bar)),
      "l"(policy)
      : "memory");
}

MOE_DEV void tma_load_5d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3, int c4,
                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
      "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

MOE_DEV void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------- programmatic dependent launch --
// Every kernel of a pass is launched with programmatic stream serialization.
// pdl_wait() blocks until the previous kernel in the stream has completed and
// its writes are visible; pdl_trigger() lets the next kernel be scheduled.
// Each kernel calls pdl_wait() before it exits, so completion stays ordered
// along the stream even where kernels overlap.
MOE_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MOE_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------- small utils --
MOE_DEV float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
MOE_DEV float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

MOE_DEV uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // round to nearest even
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Four fp32 values as bf16 hi/lo halves: hi = bf16(v), lo = bf16(v − hi),
// so hi + lo holds v to about 16 more mantissa bits than hi alone.
MOE_DEV void split_bf16x4(float4 v, uint2* hi, uint2* lo) {
  const uint2 h = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
  *hi = h;
  *lo = make_uint2(pack_bf16x2(v.x - bf16lo(h.x), v.y - bf16hi(h.x)),
                   pack_bf16x2(v.z - bf16lo(h.y), v.w - bf16hi(h.y)));
}

MOE_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

MOE_DEV float silu(float z) { return z / (1.0f + expf(-z)); }

}  // namespace moe
