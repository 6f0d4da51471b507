"""Runs verification passes of one MoE layer through the C ABI.

``PassRunner`` owns the device buffers a pass needs (workspace, routing,
union, slot outputs, output) for passes of up to ``n_max`` tokens and calls
the library's entry points in order: moe_route → moe_build_union →
moe_verify_perslot or moe_verify_dedup → moe_combine. Buffers are allocated
once, through torch, at construction.
"""
from __future__ import annotations

import torch

from . import api
from .synth import LayerWeights

PERSLOT = "perslot"
DEDUP = "dedup"


class PassRunner:
    def __init__(self, weights: LayerWeights, n_max: int):
        sh = weights.shape
        self.shape = sh
        self.weights = weights
        self.n_max = n_max
        self.desc = api.make_desc(sh)
        self.wc = api.make_weights(weights)
        dev = weights.device
        if dev.type != "cuda":
            raise ValueError("weights must live on a CUDA device")
        k, E, d, s = sh.top_k, sh.n_experts, sh.d, sh.n_shared
        nbytes = api.moe_workspace_bytes(self.desc, n_max)
        if nbytes == 0:
            raise ValueError("invalid layer shape or n_max for this library: %r, %d" % (sh, n_max))
        i32 = dict(dtype=torch.int32, device=dev)
        f32 = dict(dtype=torch.float32, device=dev)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.topk_idx = torch.empty(n_max * k, **i32)
        self.topk_w = torch.empty(n_max * k, **f32)
        self.union_ids = torch.empty(E, **i32)
        self.union_count = torch.empty(1, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.pair_tok = torch.empty(n_max * k, **i32)
        self.pair_slot = torch.empty(n_max * k, **i32)
        self.bytes = torch.empty(3, dtype=torch.int64, device=dev)
        self.u = api.UnionC(*(api._ptr(t) for t in (self.union_ids, self.union_count,
                                                     self.offsets, self.pair_tok,
                                                     self.pair_slot, self.bytes)))
        self.y_slot = torch.empty(n_max * (k + s) * d, **f32)
        self.y = torch.empty(n_max * d, **f32)

    # -- single steps ---------------------------------------------------------
    def route(self, x: torch.Tensor, stream=None):
        n = x.shape[0]
        api.moe_route(self.desc, self.weights.w_router, x, n, self.topk_idx, self.topk_w,
                      self.workspace, stream)

    def build_union(self, n: int, stream=None):
        api.moe_build_union(self.desc, self.topk_idx, n, self.u, stream)

    def experts(self, x: torch.Tensor, engine: str, stream=None):
        n = x.shape[0]
        if engine == PERSLOT:
            api.moe_verify_perslot(self.desc, self.wc, x, n, self.topk_idx, self.topk_w,
                                   self.workspace, self.y_slot, stream)
        elif engine == DEDUP:
            api.moe_verify_dedup(self.desc, self.wc, x, n, self.u, self.topk_w, self.workspace,
                                 self.y_slot, stream)
        else:
            raise ValueError("engine must be %r or %r" % (PERSLOT, DEDUP))

    def combine(self, n: int, stream=None):
        api.moe_combine(self.desc, self.y_slot, n, self.y, stream)

    # -- a whole pass ---------------------------------------------------------
    def forward(self, x: torch.Tensor, engine: str = DEDUP, stream=None) -> torch.Tensor:
        """y [n][d] for the pass x [n][d] (fp32, on the layer's device)."""
        n = x.shape[0]
        if x.dtype != torch.float32 or x.shape[1] != self.shape.d or n > self.n_max:
            raise ValueError("x must be float32 [n<=%d][%d]" % (self.n_max, self.shape.d))
        self.route(x, stream)
        self.build_union(n, stream)
        self.experts(x, engine, stream)
        self.combine(n, stream)
        return self.y[: n * self.shape.d].view(n, self.shape.d)

    # -- views ---------------------------------------------------------------
    def routing(self, n: int):
        k = self.shape.top_k
        return (self.topk_idx[: n * k].view(n, k), self.topk_w[: n * k].view(n, k))

    def union(self, n: int):
        k = self.shape.top_k
        c = int(self.union_count.item())
        return {"union_ids": self.union_ids[:c], "count": c, "offsets": self.offsets[: c + 1],
                "pair_tok": self.pair_tok[: n * k], "pair_slot": self.pair_slot[: n * k],
                "bytes": self.bytes}

    def slots(self, n: int) -> torch.Tensor:
        sh = self.shape
        return self.y_slot[: n * (sh.top_k + sh.n_shared) * sh.d].view(
            n, sh.top_k + sh.n_shared, sh.d)
