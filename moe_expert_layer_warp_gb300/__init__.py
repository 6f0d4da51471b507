"""GB300-native mixture-of-experts layer over one speculative-decoding
verification pass: gate + top-k routing, union of selected experts, per-slot
and deduplicating expert engines, weighted combine, all in hand-written CUDA
for sm_103a behind the C ABI declared in include/moe_warp.h.

Submodules:
  api        thin ctypes binding of libmoewarp.so (same names as the C ABI)
  layer      a convenience wrapper running one pass through the C ABI
  stepmodel  host step-time model (effective bandwidths, u(n), r(n),
             crossover, best draft length)
  configs    the workload shapes
  synth      seeded synthetic weights and hidden states

The CUDA library is loaded on first use of ``api``; importing this package
does not load it, and every call fails loudly if it is missing.
"""
__all__ = ["api", "layer", "stepmodel", "configs", "synth"]
