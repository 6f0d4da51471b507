"""Thin ctypes binding of libmoewarp.so — the same entry points as the C ABI
in include/moe_warp.h, taking torch CUDA tensors for the device pointers.

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels. If the library has not been built, or no CUDA device is present,
every call raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from .configs import LayerShape

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoewarp.so")

MOE_OK, MOE_EINVAL, MOE_ECUDA, MOE_ETIMEOUT, MOE_EUNSUPPORTED, MOE_EDEVICE = range(6)
MOE_MAX_TOKENS, MOE_MAX_PAIRS, MOE_MAX_EXPERTS, MOE_MAX_TOPK, MOE_MAX_SHARED = 128, 512, 256, 16, 4

EXPORTED = ("moe_workspace_bytes", "moe_route", "moe_build_union", "moe_verify_perslot",
            "moe_verify_dedup", "moe_combine", "moe_last_device_error", "moe_status_str",
            "moe_last_cuda_error_string", "moe_verify_dedup_noalloc", "moe_noalloc_scratch_limit",
            "moe_diag_bounded_wait", "moe_route_biased", "moe_route_union", "moe_verify_pass",
            "moe_verify_pass_fused", "moe_gate")


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__("%s failed: %s%s" % (where, status_str(status) if _lib else status,
                                              (" (" + detail + ")") if detail else ""))


class LayerDesc(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("inter", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("wdtype", ctypes.c_int32)]


class LayerWeightsC(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in
                ("w_router", "w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down")]


class UnionC(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in
                ("union_ids", "union_count", "offsets", "pair_tok", "pair_slot", "bytes")]


_lib = None


def load(path: str = LIB_PATH):
    """Loads libmoewarp.so and declares its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("libmoewarp.so is not built (expected at %s); run "
                           "__graft_entry__.build() or python -m "
                           "moe_expert_layer_warp_gb300.build" % path)
    lib = ctypes.CDLL(path)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    D = ctypes.POINTER(LayerDesc)
    W = ctypes.POINTER(LayerWeightsC)
    U = ctypes.POINTER(UnionC)
    lib.moe_workspace_bytes.argtypes = [D, I32]
    lib.moe_workspace_bytes.restype = SZ
    lib.moe_gate.argtypes = [D, P, P, I32, P, P]
    lib.moe_route.argtypes = [D, P, P, I32, P, P, P, SZ, P]
    lib.moe_route_biased.argtypes = [D, P, P, I32, P, I32, P, P, P, SZ, P]
    lib.moe_build_union.argtypes = [D, P, I32, U, P]
    lib.moe_route_union.argtypes = [D, P, P, I32, P, I32, P, P, U, P, SZ, P]
    lib.moe_verify_pass.argtypes = [D, W, P, I32, P, I32, I32, P, P, U, P, SZ, P, P, P]
    lib.moe_verify_pass_fused.argtypes = [D, W, P, I32, P, I32, I32, P, P, U, P, SZ, P, P, P]
    lib.moe_verify_perslot.argtypes = [D, W, P, I32, P, P, P, SZ, P, P]
    lib.moe_verify_dedup.argtypes = [D, W, P, I32, U, P, P, SZ, P, P]
    lib.moe_combine.argtypes = [D, P, I32, P, P]
    lib.moe_verify_dedup_noalloc.argtypes = [D, W, P, I32, U, P, P, P]
    lib.moe_noalloc_scratch_limit.argtypes = []
    lib.moe_noalloc_scratch_limit.restype = SZ
    lib.moe_last_device_error.argtypes = [P]
    lib.moe_diag_bounded_wait.argtypes = [I32, P]
    lib.moe_status_str.argtypes = [ctypes.c_int]
    lib.moe_status_str.restype = ctypes.c_char_p
    lib.moe_last_cuda_error_string.argtypes = []
    lib.moe_last_cuda_error_string.restype = ctypes.c_char_p
    for f in ("moe_route", "moe_build_union", "moe_verify_perslot", "moe_verify_dedup",
              "moe_combine", "moe_last_device_error", "moe_verify_dedup_noalloc",
              "moe_diag_bounded_wait", "moe_route_biased", "moe_route_union", "moe_verify_pass",
              "moe_verify_pass_fused", "moe_gate"):
        getattr(lib, f).restype = ctypes.c_int
    _lib = lib
    return lib


def status_str(status: int) -> str:
    return load().moe_status_str(status).decode()


def _check(status: int, where: str):
    if status != MOE_OK:
        detail = load().moe_last_cuda_error_string().decode()
        raise MoeError(status, where, detail)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor, got one on %s" % t.device)
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if isinstance(stream, ctypes.c_void_p):
        return stream
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_desc(shape: LayerShape) -> LayerDesc:
    return LayerDesc(shape.d, shape.n_experts, shape.top_k, shape.inter, shape.n_shared,
                     shape.wdtype)


def make_weights(w) -> LayerWeightsC:
    """From a synth.LayerWeights on a CUDA device."""
    return LayerWeightsC(_ptr(w.w_router), _ptr(w.w_gate), _ptr(w.w_up), _ptr(w.w_down),
                         _ptr(w.ws_gate), _ptr(w.ws_up), _ptr(w.ws_down))


def moe_workspace_bytes(desc: LayerDesc, n_max: int) -> int:
    return int(load().moe_workspace_bytes(ctypes.byref(desc), n_max))


def moe_gate(desc, w_router, x, n, logits, stream=None):
    _check(load().moe_gate(ctypes.byref(desc), _ptr(w_router), _ptr(x), n, _ptr(logits),
                           _stream(stream)), "moe_gate")


def moe_route(desc, w_router, x, n, topk_idx, topk_w, workspace, stream=None):
    _check(load().moe_route(ctypes.byref(desc), _ptr(w_router), _ptr(x), n, _ptr(topk_idx),
                            _ptr(topk_w), _ptr(workspace), workspace.numel() *
                            workspace.element_size(), _stream(stream)), "moe_route")


def moe_route_biased(desc, w_router, bias, bias_in_weights, x, n, topk_idx, topk_w, workspace,
                     stream=None):
    _check(load().moe_route_biased(ctypes.byref(desc), _ptr(w_router), _ptr(bias),
                                   1 if bias_in_weights else 0, _ptr(x), n, _ptr(topk_idx),
                                   _ptr(topk_w), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_route_biased")


def moe_build_union(desc, topk_idx, n, u: UnionC, stream=None):
    _check(load().moe_build_union(ctypes.byref(desc), _ptr(topk_idx), n, ctypes.byref(u),
                                  _stream(stream)), "moe_build_union")


def moe_route_union(desc, w_router, bias, bias_in_weights, x, n, topk_idx, topk_w, u: UnionC,
                    workspace, stream=None):
    _check(load().moe_route_union(ctypes.byref(desc), _ptr(w_router), _ptr(bias),
                                  1 if bias_in_weights else 0, _ptr(x), n, _ptr(topk_idx),
                                  _ptr(topk_w), ctypes.byref(u), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_route_union")


MOE_ENGINE_PERSLOT, MOE_ENGINE_DEDUP = 0, 1


def moe_verify_pass(desc, weights: LayerWeightsC, bias, bias_in_weights, x, n, engine, topk_idx,
                    topk_w, u: UnionC, workspace, y_slot, y, stream=None):
    _check(load().moe_verify_pass(ctypes.byref(desc), ctypes.byref(weights), _ptr(bias),
                                  1 if bias_in_weights else 0, _ptr(x), n, engine,
                                  _ptr(topk_idx), _ptr(topk_w), ctypes.byref(u), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _ptr(y_slot),
                                  _ptr(y), _stream(stream)), "moe_verify_pass")


def moe_verify_pass_fused(desc, weights: LayerWeightsC, bias, bias_in_weights, x, n, engine,
                          topk_idx, topk_w, u: UnionC, workspace, y_slot, y, stream=None):
    _check(load().moe_verify_pass_fused(ctypes.byref(desc), ctypes.byref(weights), _ptr(bias),
                                        1 if bias_in_weights else 0, _ptr(x), n, engine,
                                        _ptr(topk_idx), _ptr(topk_w), ctypes.byref(u),
                                        _ptr(workspace),
                                        workspace.numel() * workspace.element_size(),
                                        _ptr(y_slot), _ptr(y), _stream(stream)),
           "moe_verify_pass_fused")


def moe_verify_perslot(desc, weights: LayerWeightsC, x, n, topk_idx, topk_w, workspace, y_slot,
                       stream=None):
    _check(load().moe_verify_perslot(ctypes.byref(desc), ctypes.byref(weights), _ptr(x), n,
                                     _ptr(topk_idx), _ptr(topk_w), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(),
                                     _ptr(y_slot), _stream(stream)), "moe_verify_perslot")


def moe_verify_dedup(desc, weights: LayerWeightsC, x, n, u: UnionC, topk_w, workspace, y_slot,
                     stream=None):
    _check(load().moe_verify_dedup(ctypes.byref(desc), ctypes.byref(weights), _ptr(x), n,
                                   ctypes.byref(u), _ptr(topk_w), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _ptr(y_slot),
                                   _stream(stream)), "moe_verify_dedup")


def moe_verify_dedup_noalloc(desc, weights: LayerWeightsC, x, n, u: UnionC, topk_w, y_slot,
                             stream=None):
    """moe_verify_dedup without a workspace: scratch lives in the library's
    static device array (see include/moe_warp.h)."""
    _check(load().moe_verify_dedup_noalloc(ctypes.byref(desc), ctypes.byref(weights), _ptr(x), n,
                                           ctypes.byref(u), _ptr(topk_w), _ptr(y_slot),
                                           _stream(stream)), "moe_verify_dedup_noalloc")


def moe_noalloc_scratch_limit() -> int:
    return int(load().moe_noalloc_scratch_limit())


def moe_combine(desc, y_slot, n, y, stream=None):
    _check(load().moe_combine(ctypes.byref(desc), _ptr(y_slot), n, _ptr(y), _stream(stream)),
           "moe_combine")


def moe_diag_bounded_wait(limit_us: int, stream=None):
    _check(load().moe_diag_bounded_wait(limit_us, _stream(stream)), "moe_diag_bounded_wait")


def moe_last_device_error(stream=None) -> int:
    return int(load().moe_last_device_error(_stream(stream)))
