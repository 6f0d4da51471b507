"""Seeded synthetic inputs: layer weights and verification-pass hidden states.

This module holds none of the layer's arithmetic. It only draws random
numbers, so that the CUDA path and the CPU oracle can be fed the same inputs.

Recipe (the same for every workload):
  - router W_g [E][d]: numpy PCG64 ``default_rng([seed, 1])`` standard normal
    × 1/sqrt(d), stored as float32.
  - expert matrices: torch generator on the target device seeded with
    ``seed * 1_000_003 + m`` (m = 0 gate, 1 up, 2 down, 3/4/5 for the shared
    experts' gate/up/down), standard normal × 1/sqrt(fan_in) with fan_in = d
    for W_gate and W_up and I for W_down, drawn one expert at a time as
    float32 and rounded to bfloat16 (round to nearest even) for bf16 layers.
  - hidden states: each stream is an AR(1) sequence x_0 = e_0,
    x_t = rho·x_{t-1} + sqrt(1-rho²)·e_t, e_t ~ N(0, I_d) drawn by numpy
    PCG64 ``default_rng(seed)``, float64 recursion then rounded to float32.
    Streams of one pass are concatenated stream-major.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np
import torch

from .configs import W_BF16, W_F32, LayerShape


@dataclass
class LayerWeights:
    shape: LayerShape
    w_router: torch.Tensor            # [E][d] float32
    w_gate: torch.Tensor              # [E][I][d]
    w_up: torch.Tensor                # [E][I][d]
    w_down: torch.Tensor              # [E][d][I]
    ws_gate: Optional[torch.Tensor]   # [s][I][d] or None
    ws_up: Optional[torch.Tensor]
    ws_down: Optional[torch.Tensor]

    @property
    def device(self):
        return self.w_gate.device


def _wtorch_dtype(wdtype: int):
    return torch.float32 if wdtype == W_F32 else torch.bfloat16


def _fill(out: torch.Tensor, seed: int, fan_in: int):
    g = torch.Generator(device=out.device)
    g.manual_seed(seed)
    std = 1.0 / math.sqrt(fan_in)
    for e in range(out.shape[0]):
        r = torch.randn(out.shape[1:], generator=g, device=out.device, dtype=torch.float32)
        r.mul_(std)
        out[e].copy_(r)   # float32 -> bfloat16 copy rounds to nearest even
        del r


def make_layer(shape: LayerShape, seed: int, device="cpu") -> LayerWeights:
    E, d, I, s = shape.n_experts, shape.d, shape.inter, shape.n_shared
    rng = np.random.default_rng([seed, 1])
    wr = (rng.standard_normal((E, d)) * (1.0 / math.sqrt(d))).astype(np.float32)
    dt = _wtorch_dtype(shape.wdtype)
    dev = torch.device(device)
    w_gate = torch.empty((E, I, d), dtype=dt, device=dev)
    w_up = torch.empty((E, I, d), dtype=dt, device=dev)
    w_down = torch.empty((E, d, I), dtype=dt, device=dev)
    base = seed * 1_000_003
    _fill(w_gate, base + 0, d)
    _fill(w_up, base + 1, d)
    _fill(w_down, base + 2, I)
    ws = (None, None, None)
    if s > 0:
        ws_gate = torch.empty((s, I, d), dtype=dt, device=dev)
        ws_up = torch.empty((s, I, d), dtype=dt, device=dev)
        ws_down = torch.empty((s, d, I), dtype=dt, device=dev)
        _fill(ws_gate, base + 3, d)
        _fill(ws_up, base + 4, d)
        _fill(ws_down, base + 5, I)
        ws = (ws_gate, ws_up, ws_down)
    return LayerWeights(shape, torch.from_numpy(wr).to(dev), w_gate, w_up, w_down, *ws)


def ar1_stream(d: int, n: int, rho: float, seed: int) -> np.ndarray:
    """n consecutive hidden states of one AR(1) stream, float32 [n][d]."""
    rng = np.random.default_rng(seed)
    eps = rng.standard_normal((n, d))
    x = np.empty((n, d), np.float64)
    x[0] = eps[0]
    c = math.sqrt(max(0.0, 1.0 - rho * rho))
    for t in range(1, n):
        x[t] = rho * x[t - 1] + c * eps[t]
    return x.astype(np.float32)


def make_pass(d: int, n_per_stream: int, rho: float, seeds: Sequence[int]) -> np.ndarray:
    """One verification pass: len(seeds) independent streams of n_per_stream
    tokens each, concatenated stream-major. float32 [streams*n_per_stream][d]."""
    return np.concatenate([ar1_stream(d, n_per_stream, rho, s) for s in seeds], axis=0)


def weights_numpy(t: Optional[torch.Tensor]) -> Optional[np.ndarray]:
    """A host copy of a weight tensor in the form the oracle takes: float32,
    or uint16 bit patterns for bfloat16."""
    if t is None:
        return None
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()
