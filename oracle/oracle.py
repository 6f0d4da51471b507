"""Float64 CPU oracle of the MoE layer over one verification pass (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: imported by tests/, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``, never by the product package. It
shares no code with the CUDA library and imports nothing from it. The
arithmetic lives in ``moe_oracle.c`` (plain double-precision loops); this
module only marshals numpy arrays and composes per-token calls.

Weights are passed as numpy arrays: ``float32`` for fp32 layers, ``uint16``
(raw bfloat16 bit patterns) for bf16 layers.

Sources, as in moe_oracle.c: "Deep Dive into Mixture of Experts: From 1991 to
DeepSeek-V3" §1, §2 (top-k gating sketch) and §5 (shared experts); "Speculative
Decoding for Mixture-of-Experts Models: Expert Bytes, Kernel Bandwidth and the
Best Draft Length", abstract (per-slot and dedup bytes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into liboracle.so beside it (plain gcc, no FMA
    contraction, so x86 and Arm hosts give identical results)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
             "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def bind(path: str):
    """Load a compiled oracle library and declare its signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.oracle_gate_logits.argtypes = [I, I, I, P, P, P, P]
    lib.oracle_topk.argtypes = [I, I, I, P, P, P, P]
    lib.oracle_topk_biased.argtypes = [I, I, I, P, P, I, P, P, P]
    lib.oracle_expert_ffn.argtypes = [I, I, I, P, P, P, P, P]
    lib.oracle_moe_token.argtypes = [I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, P]
    lib.oracle_dense_token.argtypes = [I, I, I, I, I, P, P, P, P, P, P, P, P, P]
    lib.oracle_union.argtypes = [I, I, I, P, P, P, P, P, P]
    lib.oracle_bytes.argtypes = [I, I, I, I, I, I, I, P]
    for f in (lib.oracle_gate_logits, lib.oracle_topk, lib.oracle_topk_biased, lib.oracle_expert_ffn,
              lib.oracle_moe_token, lib.oracle_dense_token, lib.oracle_union,
              lib.oracle_bytes):
        f.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = bind(_LIB)
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _wdtype(w) -> int:
    if w.dtype == np.float32:
        return 0
    if w.dtype == np.uint16:
        return 1
    raise TypeError("weights must be float32 or uint16 (bf16 bits), got %s" % w.dtype)


def _check(rc, what):
    if rc != 0:
        raise RuntimeError("oracle %s failed with code %d" % (what, rc))


def gate_logits(x, w_router):
    """logits[t][e] = Σ_i x[t][i]·W_g[e][i] in float64, and Σ_i |x·W_g| per (t, e)."""
    x = _c(x, np.float32)
    wg = _c(w_router, np.float32)
    n, d = x.shape
    E = wg.shape[0]
    assert wg.shape[1] == d
    logits = np.empty((n, E), np.float64)
    absdot = np.empty((n, E), np.float64)
    _check(_load().oracle_gate_logits(d, E, n, _p(x), _p(wg), _p(logits), _p(absdot)), "gate")
    return logits, absdot


def topk(logits, k, bias=None, bias_in_weights=True):
    """Top-k (descending score, ties -> lower index), softmax over the k kept
    scores, and the smallest gap between consecutive sorted scores at
    positions 0..k per token. With a per-expert bias (DeepSeek-style routing
    sketch) the score is logit + bias; bias_in_weights=False takes the softmax
    over the kept experts' unbiased logits instead (bias for selection only)."""
    logits = _c(logits, np.float64)
    n, E = logits.shape
    idx = np.empty((n, k), np.int32)
    w = np.empty((n, k), np.float64)
    gap = np.empty((n,), np.float64)
    if bias is None:
        _check(_load().oracle_topk(E, k, n, _p(logits), _p(idx), _p(w), _p(gap)), "topk")
    else:
        b = _c(bias, np.float64)
        assert b.shape == (E,)
        _check(_load().oracle_topk_biased(E, k, n, _p(logits), _p(b), 1 if bias_in_weights else 0,
                                          _p(idx), _p(w), _p(gap)), "topk_biased")
    return idx, w, gap


def route(x, w_router, k, bias=None, bias_in_weights=True):
    """Gate GEMV + top-k + renormalised softmax (optionally with a per-expert
    routing bias, see topk). Returns a dict with idx, w, logits, absdot and
    gap (of the scores the selection compares)."""
    logits, absdot = gate_logits(x, w_router)
    idx, w, gap = topk(logits, k, bias, bias_in_weights)
    return {"idx": idx, "w": w, "logits": logits, "absdot": absdot, "gap": gap}


def expert_ffn(x, w_gate, w_up, w_down):
    """One expert on one hidden state: W_down(silu(W_gate x) ⊙ W_up x).
    w_gate, w_up: [I][d]; w_down: [d][I]."""
    wt = _wdtype(w_gate)
    I, d = w_gate.shape
    assert w_up.shape == (I, d) and w_down.shape == (d, I)
    xd = _c(x, np.float64)
    out = np.empty((d,), np.float64)
    wg, wu, wd = (_c(a, a.dtype) for a in (w_gate, w_up, w_down))
    _check(_load().oracle_expert_ffn(d, I, wt, _p(wg), _p(wu), _p(wd), _p(xd), _p(out)), "ffn")
    return out


def moe_tokens(x, idx, w, w_gate, w_up, w_down, ws_gate=None, ws_up=None, ws_down=None,
               tokens=None, slots=False):
    """Layer output for the listed tokens (all when tokens is None):
    y_t = Σ_shared FFN_s(x_t) + Σ_j w[t][j]·FFN_{idx[t][j]}(x_t).

    w_gate/w_up: [E][I][d]; w_down: [E][d][I]; ws_*: [s][...] or None.
    Returns y [len(tokens)][d] (float64) and, if slots, the per-slot outputs
    [len(tokens)][k+s][d] (slot j < k weighted by w[t][j], shared slots after)."""
    x = _c(x, np.float32)
    idx = _c(idx, np.int32)
    w = _c(w, np.float64)
    n, d = x.shape
    k = idx.shape[1]
    E, I, d2 = w_gate.shape
    assert d2 == d and w_down.shape == (E, d, I)
    wt = _wdtype(w_gate)
    s = 0 if ws_gate is None else ws_gate.shape[0]
    wg, wu, wd = (_c(a, a.dtype) for a in (w_gate, w_up, w_down))
    if s:
        sg, su, sd = (_c(a, a.dtype) for a in (ws_gate, ws_up, ws_down))
    else:
        sg = su = sd = None
    toks = list(range(n)) if tokens is None else list(tokens)
    y = np.empty((len(toks), d), np.float64)
    ys = np.empty((len(toks), k + s, d), np.float64) if slots else None
    lib = _load()
    for r, t in enumerate(toks):
        xt = x[t]
        it = idx[t]
        wt_ = w[t]
        yr = y[r]
        so = ys[r] if slots else None
        _check(lib.oracle_moe_token(d, I, k, s, wt, _p(wg), _p(wu), _p(wd), _p(sg), _p(su),
                                    _p(sd), _p(xt), _p(it), _p(wt_), _p(yr), _p(so)), "moe_token")
    return (y, ys) if slots else y


def dense_tokens(x, gate, w_gate, w_up, w_down, ws_gate=None, ws_up=None, ws_down=None):
    """Dense mixture (every expert runs, weighted by gate[t][e]) for all tokens."""
    x = _c(x, np.float32)
    gate = _c(gate, np.float64)
    n, d = x.shape
    E, I, _ = w_gate.shape
    wt = _wdtype(w_gate)
    s = 0 if ws_gate is None else ws_gate.shape[0]
    wg, wu, wd = (_c(a, a.dtype) for a in (w_gate, w_up, w_down))
    if s:
        sg, su, sd = (_c(a, a.dtype) for a in (ws_gate, ws_up, ws_down))
    else:
        sg = su = sd = None
    y = np.empty((n, d), np.float64)
    lib = _load()
    for t in range(n):
        _check(lib.oracle_dense_token(d, I, E, s, wt, _p(wg), _p(wu), _p(wd), _p(sg), _p(su),
                                      _p(sd), _p(x[t]), _p(gate[t]), _p(y[t])), "dense")
    return y


def union(idx, E):
    """Union of selected experts and the pairs grouped by (expert, token)."""
    idx = _c(idx, np.int32)
    n, k = idx.shape
    ids = np.empty((E,), np.int32)
    cnt = np.zeros((1,), np.int32)
    off = np.empty((E + 1,), np.int32)
    ptok = np.empty((n * k,), np.int32)
    pslot = np.empty((n * k,), np.int32)
    _check(_load().oracle_union(E, k, n, _p(idx), _p(ids), _p(cnt), _p(off), _p(ptok),
                                _p(pslot)), "union")
    u = int(cnt[0])
    return {"union_ids": ids[:u].copy(), "count": u, "offsets": off[:u + 1].copy(),
            "pair_tok": ptok, "pair_slot": pslot}


def bytes_per_pass(d, I, k, s, n, wdtype, union_count):
    """{per-slot, dedup, shared} requested expert-weight bytes of one pass."""
    b = np.zeros((3,), np.uint64)
    _check(_load().oracle_bytes(d, I, k, s, n, wdtype, union_count, _p(b)), "bytes")
    return [int(v) for v in b]
