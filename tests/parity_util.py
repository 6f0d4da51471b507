"""Helpers of the GPU parity tests: certified routing comparison, tolerance
checks, and host copies of the experts a sample of tokens selected.

Tolerances (fixed by the target the tests encode): max|err| ≤ 1e-5·rms(y)
for fp32-weight layers, ≤ 2e-2·rms(y) for bf16-weight / fp32-accumulate
layers; routing indices, union and byte counts bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

from moe_expert_layer_warp_gb300 import synth
from moe_expert_layer_warp_gb300.configs import W_F32
from oracle import oracle

U32 = 2.0 ** -24   # unit roundoff of fp32


def y_tol(shape) -> float:
    return 1e-5 if shape.wdtype == W_F32 else 2e-2


def logit_error_bound(orc_route: dict, d: int, bias=None) -> np.ndarray:
    """Upper bound on |fp32 compensated-dot logit − exact logit| per (t, e):
    rounding of the result (u·|l|) plus the compensated-dot remainder
    γ_d²·Σ|x_i·w_i| (Ogita, Rump and Oishi 2005, accurate dot product), with
    a factor 2 of slack for the lane-then-tree order of the partial sums.
    With a routing bias the score is fl(logit + bias): its rounding,
    u·(|l| + |b|), is added (again with a factor 2)."""
    gamma = d * U32 / (1.0 - d * U32)
    b = 2.0 * (U32 * np.abs(orc_route["logits"]) + gamma * gamma * orc_route["absdot"])
    if bias is not None:
        b = b + 2.0 * U32 * (np.abs(orc_route["logits"]) + np.abs(bias)[None, :])
    return b


def certified_tokens(orc_route: dict, d: int, bias=None) -> np.ndarray:
    """Tokens whose sorted scores at positions 0..k are separated by more than
    twice the GPU's error bound: for these the GPU's selection and order must
    equal the oracle's exactly."""
    b = logit_error_bound(orc_route, d, bias).max(axis=1)
    return orc_route["gap"] > 2.0 * b


def check_routing(gpu_idx: np.ndarray, gpu_w: np.ndarray, orc_route: dict, d: int, bias=None):
    """Bit-exact indices on certified tokens; on the others (near-ties within
    the error bound) the GPU's choice must be one an exact computation could
    make within that bound. Weights within 1e-5 absolute where indices agree.
    Returns the number of tie-ambiguous tokens."""
    cert = certified_tokens(orc_route, d, bias)
    bound = logit_error_bound(orc_route, d, bias)
    lg = orc_route["logits"] + (0.0 if bias is None else np.asarray(bias, np.float64)[None, :])
    amb = 0
    for t in range(gpu_idx.shape[0]):
        if cert[t]:
            np.testing.assert_array_equal(gpu_idx[t], orc_route["idx"][t], err_msg="token %d" % t)
        else:
            amb += 1
            k = gpu_idx.shape[1]
            assert len(set(gpu_idx[t].tolist())) == k
            kth = np.sort(lg[t])[::-1][k - 1]
            assert np.all(lg[t][gpu_idx[t]] >= kth - 4 * bound[t].max()), "token %d" % t
        if np.array_equal(gpu_idx[t], orc_route["idx"][t]):
            np.testing.assert_allclose(gpu_w[t], orc_route["w"][t], rtol=0, atol=1e-5)
    np.testing.assert_allclose(gpu_w.sum(axis=1), 1.0, rtol=0, atol=1e-5)
    return amb


def assert_close_rms(got: np.ndarray, ref: np.ndarray, tol: float, what: str, scale=None):
    """max|got − ref| ≤ tol · rms(scale), scale defaulting to ref. Slot outputs
    use rms(y) as their scale: the tolerance is stated on y."""
    rms = float(np.sqrt(np.mean(np.square(ref if scale is None else scale))))
    err = float(np.max(np.abs(got.astype(np.float64) - ref)))
    assert err <= tol * rms, "%s: max|err| %.3e > %.1e · rms %.3e" % (what, err, tol, rms)
    return err / rms


def host_layer_subset(L: synth.LayerWeights, experts):
    """Host copies (oracle form) of the listed routed experts and of every
    shared expert."""
    sel = torch.tensor(list(experts), dtype=torch.long, device=L.device)
    out = {
        "wg": synth.weights_numpy(L.w_gate.index_select(0, sel)),
        "wu": synth.weights_numpy(L.w_up.index_select(0, sel)),
        "wd": synth.weights_numpy(L.w_down.index_select(0, sel)),
        "sg": synth.weights_numpy(L.ws_gate), "su": synth.weights_numpy(L.ws_up),
        "sd": synth.weights_numpy(L.ws_down),
    }
    return out


def oracle_outputs(L: synth.LayerWeights, x: np.ndarray, orc_route: dict, tokens,
                   max_experts: int = 32):
    """Oracle y and per-slot outputs for the listed tokens (float64). The
    tokens are taken in chunks whose selected experts number at most
    max_experts (or one token's k), so that the host holds copies of only
    those experts at a time (a DeepSeek-V3-shaped expert is 88 MB)."""
    tokens = list(tokens)
    chunks, cur, cur_e = [], [], set()
    for t in tokens:
        e = set(orc_route["idx"][t].tolist())
        if cur and len(cur_e | e) > max_experts:
            chunks.append(cur)
            cur, cur_e = [], set()
        cur.append(t)
        cur_e |= e
    if cur:
        chunks.append(cur)
    ys_all, slots_all = [], []
    for ch in chunks:
        experts = sorted(set(orc_route["idx"][ch].ravel().tolist()))
        remap = {e: i for i, e in enumerate(experts)}
        H = host_layer_subset(L, experts)
        idx = np.vectorize(remap.get)(orc_route["idx"][ch]).astype(np.int32)
        y, ys = oracle.moe_tokens(x[ch], idx, orc_route["w"][ch], H["wg"], H["wu"], H["wd"],
                                  H["sg"], H["su"], H["sd"], slots=True)
        del H
        ys_all.append(y)
        slots_all.append(ys)
    return np.concatenate(ys_all), np.concatenate(slots_all)
