"""Runs verification passes of one MoE layer through the C ABI.

``PassRunner`` owns the device buffers a pass needs (workspace, routing,
union, slot outputs, output) for passes of up to ``n_max`` tokens and calls
the library's entry points: forward() makes one moe_verify_pass call
(moe_route_union → moe_verify_perslot or moe_verify_dedup → moe_combine), or
one moe_verify_pass_fused call (the combine inside the expert kernel);
gate(), route(), build_union(), route_union(), experts() and combine() make
the single calls. Buffers are allocated
once, through torch, at construction, and so are the C arguments that point
at them: a call only marshals x and the stream.
"""
from __future__ import annotations

import ctypes

import torch

from . import api
from .synth import LayerWeights

PERSLOT = "perslot"
DEDUP = "dedup"


class PassRunner:
    def __init__(self, weights: LayerWeights, n_max: int, bias: torch.Tensor = None,
                 bias_in_weights: bool = True):
        """bias: optional per-expert routing bias [E] fp32 on the layer's
        device (DeepSeek-style routing); bias_in_weights: whether the kept
        experts' softmax includes it (see moe_route_biased)."""
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
        self.logits = torch.empty(n_max * E, **f32)
        self.y_slot = torch.empty(n_max * (k + s) * d, **f32)
        self.y = torch.empty(n_max * d, **f32)
        # C arguments fixed for the runner's lifetime
        V = ctypes.c_void_p
        self._lib = api.load()
        self._desc = ctypes.byref(self.desc)
        self._wref = ctypes.byref(self.wc)
        self._uref = ctypes.byref(self.u)
        self._ws = V(self.workspace.data_ptr())
        self._ws_bytes = nbytes
        self._router = V(weights.w_router.data_ptr())
        self._idx = V(self.topk_idx.data_ptr())
        self._tw = V(self.topk_w.data_ptr())
        self._logits = V(self.logits.data_ptr())
        self._yslot = V(self.y_slot.data_ptr())
        self._y = V(self.y.data_ptr())
        self.bias = None
        if bias is not None:
            if (bias.dtype != torch.float32 or bias.numel() != E or bias.device != dev or
                    not bias.is_contiguous()):
                raise ValueError("bias must be a contiguous float32 [%d] tensor on %s" % (E, dev))
            self.bias = bias
        self._bias = V(bias.data_ptr()) if bias is not None else None
        self._bias_w = 1 if bias_in_weights else 0

    def _x(self, x: torch.Tensor) -> ctypes.c_void_p:
        n = x.shape[0]
        if (x.dtype != torch.float32 or x.dim() != 2 or x.shape[1] != self.shape.d or
                n > self.n_max or n < 1 or x.device != self.weights.device or
                not x.is_contiguous()):
            raise ValueError("x must be a contiguous float32 [1..%d][%d] tensor on %s"
                             % (self.n_max, self.shape.d, self.weights.device))
        return ctypes.c_void_p(x.data_ptr())

    # -- single steps ---------------------------------------------------------
    def gate(self, x: torch.Tensor, stream=None, _xp=None):
        """The gate GEMV alone: self.logits[:n·E] = x·W_gᵀ."""
        xp = _xp or self._x(x)
        api._check(self._lib.moe_gate(self._desc, self._router, xp, x.shape[0], self._logits,
                                      api._stream(stream)), "moe_gate")

    def route(self, x: torch.Tensor, stream=None, _xp=None):
        xp = _xp or self._x(x)
        if self._bias is None:
            api._check(self._lib.moe_route(self._desc, self._router, xp, x.shape[0], self._idx,
                                           self._tw, self._ws, self._ws_bytes,
                                           api._stream(stream)), "moe_route")
        else:
            api._check(self._lib.moe_route_biased(self._desc, self._router, self._bias,
                                                  self._bias_w, xp, x.shape[0], self._idx,
                                                  self._tw, self._ws, self._ws_bytes,
                                                  api._stream(stream)), "moe_route_biased")

    def build_union(self, n: int, stream=None):
        api._check(self._lib.moe_build_union(self._desc, self._idx, n, self._uref,
                                             api._stream(stream)), "moe_build_union")

    def route_union(self, x: torch.Tensor, stream=None, _xp=None):
        """route() then build_union() in one library call (same results)."""
        xp = _xp or self._x(x)
        api._check(self._lib.moe_route_union(self._desc, self._router, self._bias, self._bias_w,
                                             xp, x.shape[0], self._idx, self._tw, self._uref,
                                             self._ws, self._ws_bytes, api._stream(stream)),
                   "moe_route_union")

    def experts(self, x: torch.Tensor, engine: str, stream=None, _xp=None):
        xp = _xp or self._x(x)
        n = x.shape[0]
        st = api._stream(stream)
        if engine == PERSLOT:
            api._check(self._lib.moe_verify_perslot(self._desc, self._wref, xp, n, self._idx,
                                                    self._tw, self._ws, self._ws_bytes,
                                                    self._yslot, st), "moe_verify_perslot")
        elif engine == DEDUP:
            api._check(self._lib.moe_verify_dedup(self._desc, self._wref, xp, n, self._uref,
                                                  self._tw, self._ws, self._ws_bytes,
                                                  self._yslot, st), "moe_verify_dedup")
        else:
            raise ValueError("engine must be %r or %r" % (PERSLOT, DEDUP))

    def combine(self, n: int, stream=None, out: torch.Tensor = None):
        y = self._y
        if out is not None:
            if (out.dtype != torch.float32 or out.numel() != n * self.shape.d or
                    out.device != self.weights.device or not out.is_contiguous()):
                raise ValueError("out must be a contiguous float32 [%d][%d] tensor on %s"
                                 % (n, self.shape.d, self.weights.device))
            y = ctypes.c_void_p(out.data_ptr())
        api._check(self._lib.moe_combine(self._desc, self._yslot, n, y, api._stream(stream)),
                   "moe_combine")

    # -- a whole pass ---------------------------------------------------------
    def forward(self, x: torch.Tensor, engine: str = DEDUP, stream=None,
                out: torch.Tensor = None, fused: bool = False) -> torch.Tensor:
        """y [n][d] for the pass x [n][d] (fp32, on the layer's device),
        written to `out` if given (a contiguous fp32 [n][d] device tensor),
        else to the runner's own buffer (overwritten by its next pass).
        fused: moe_verify_pass_fused (the combine as the expert kernel's last
        phase) instead of moe_verify_pass; the same results bit for bit."""
        xp = self._x(x)
        if engine not in (PERSLOT, DEDUP):
            raise ValueError("engine must be %r or %r" % (PERSLOT, DEDUP))
        n = x.shape[0]
        y = self._y
        if out is not None:
            if (out.dtype != torch.float32 or out.numel() != n * self.shape.d or
                    out.device != self.weights.device or not out.is_contiguous()):
                raise ValueError("out must be a contiguous float32 [%d][%d] tensor on %s"
                                 % (n, self.shape.d, self.weights.device))
            y = ctypes.c_void_p(out.data_ptr())
        eng = api.MOE_ENGINE_PERSLOT if engine == PERSLOT else api.MOE_ENGINE_DEDUP
        f = self._lib.moe_verify_pass_fused if fused else self._lib.moe_verify_pass
        api._check(f(self._desc, self._wref, self._bias, self._bias_w, xp, n, eng, self._idx,
                     self._tw, self._uref, self._ws, self._ws_bytes, self._yslot, y,
                     api._stream(stream)),
                   "moe_verify_pass_fused" if fused else "moe_verify_pass")
        return out if out is not None else self.y[: n * self.shape.d].view(n, self.shape.d)

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
