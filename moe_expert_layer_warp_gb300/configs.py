"""The layer shapes and pass structures this library is exercised on.

Shapes follow the models the sources name for the method ("Speculative
Decoding for Mixture-of-Experts Models: Expert Bytes, Kernel Bandwidth and the
Best Draft Length", abstract: DeepSeek-V2-Lite; "Deep Dive into Mixture of
Experts: From 1991 to DeepSeek-V3", §4 Mixtral 8x7B and §5 DeepSeek-V3). Only
the shapes are used: the weights are synthetic (see synth.py).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Tuple

W_F32 = 0
W_BF16 = 1


@dataclass(frozen=True)
class LayerShape:
    d: int          # model dimension
    n_experts: int  # E routed experts
    top_k: int      # k
    inter: int      # I, SwiGLU intermediate
    n_shared: int   # s always-on experts
    wdtype: int     # W_F32 or W_BF16

    @property
    def wbytes(self) -> int:
        return 4 if self.wdtype == W_F32 else 2

    @property
    def expert_bytes(self) -> int:
        """E_b = 3·d·I·bytes(weight): W_gate, W_up and W_down of one expert."""
        return 3 * self.d * self.inter * self.wbytes


@dataclass(frozen=True)
class Workload:
    name: str
    shape: LayerShape
    pass_sizes: Tuple[int, ...]      # tokens per stream; a pass holds streams × n tokens
    rhos: Tuple[float, ...]          # AR(1) correlation of the hidden states
    weight_seed: int
    x_seed_base: int
    layers: int = 1                  # >1: a stack of independent layers
    streams: int = 1                 # independent AR(1) streams per pass
    passes: int = 1                  # independent passes per (n, rho)
    notes: str = field(default="", compare=False)


TINY = Workload(
    name="tiny-fp32", shape=LayerShape(256, 8, 2, 512, 0, W_F32), pass_sizes=(4,), rhos=(0.9,),
    weight_seed=0, x_seed_base=0,
    notes="d=256, 8 experts top-2, SwiGLU I=512, fp32 weights, n=4, AR(1) rho=0.9, seed 0")

V2_LITE = Workload(
    name="deepseek-v2-lite-layer", shape=LayerShape(2048, 64, 6, 1408, 2, W_BF16),
    pass_sizes=tuple(range(1, 10)), rhos=(0.9,), weight_seed=1, x_seed_base=100, passes=32,
    notes="d=2048, 64 routed top-6 + 2 shared, I=1408, bf16 weights, n=1..9, rho=0.9")

MIXTRAL = Workload(
    name="mixtral-8x7b-layer", shape=LayerShape(4096, 8, 2, 14336, 0, W_BF16),
    pass_sizes=tuple(range(1, 17)), rhos=(0.0, 0.5, 0.9), weight_seed=2, x_seed_base=200,
    passes=16, notes="d=4096, 8 experts top-2, I=14336, bf16 (352 MB per expert), n=1..16")

V2_LITE_STACK = Workload(
    name="deepseek-v2-lite-26-layer-stack", shape=LayerShape(2048, 64, 6, 1408, 2, W_BF16),
    pass_sizes=tuple(range(1, 10)), rhos=(0.0, 0.5, 0.9, 0.99), weight_seed=1000,
    x_seed_base=300, layers=26, passes=16,
    notes="26 independent V2-Lite-shaped layers (~30 GB bf16), each fed the same pass")

V3 = Workload(
    name="deepseek-v3-layer", shape=LayerShape(7168, 256, 8, 2048, 1, W_BF16),
    pass_sizes=(16,), rhos=(0.9,), weight_seed=3, x_seed_base=400, streams=4, passes=8,
    notes="d=7168, 256 routed top-8 + 1 shared, I=2048, bf16 (~22.6 GB); 4 AR(1) streams "
          "x 16 tokens = 64 tokens per pass")

ALL = (TINY, V2_LITE, MIXTRAL, V2_LITE_STACK, V3)
BY_NAME = {w.name: w for w in ALL}
