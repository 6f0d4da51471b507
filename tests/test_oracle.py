"""Pins of the float64 oracle against things other than itself.

Each test checks one oracle function against a brute force, a closed form, an
invariant fixed by the sources, or an independent library routine (torch
float64 linear/silu/softmax/topk), chosen so that a plausible slip in the
oracle (a transposed operand, a dropped term, a wrong index or sign, a wrong
tie order) fails at least one of them. tests/test_oracle_mutants.py plants
such slips in a copy of the oracle and checks that they are caught.

Sources: "Deep Dive into Mixture of Experts: From 1991 to DeepSeek-V3" §1
(dense mixture), §2 (top-k gating sketch: softmax over the kept logits), §5
(shared experts, unweighted); "Speculative Decoding for Mixture-of-Experts
Models: Expert Bytes, Kernel Bandwidth and the Best Draft Length", abstract
(per-slot bytes n·k·E_b, dedup bytes |U|·E_b).
"""
import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import oracle
from moe_expert_layer_warp_gb300 import synth
from moe_expert_layer_warp_gb300.configs import TINY, W_BF16, W_F32, LayerShape


def _t64(a):
    """numpy weights (float32 or bf16 bits) -> torch float64, exactly."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).double()
    return torch.from_numpy(np.ascontiguousarray(a)).double()


def _layer_np(shape, seed):
    L = synth.make_layer(shape, seed, "cpu")
    return {
        "wr": L.w_router.numpy(),
        "wg": synth.weights_numpy(L.w_gate), "wu": synth.weights_numpy(L.w_up),
        "wd": synth.weights_numpy(L.w_down),
        "sg": synth.weights_numpy(L.ws_gate), "su": synth.weights_numpy(L.ws_up),
        "sd": synth.weights_numpy(L.ws_down),
    }


def _torch_swiglu(x64, wg, wu, wd):
    return F.linear(F.silu(F.linear(x64, wg)) * F.linear(x64, wu), wd)


# ---------------------------------------------------------------- routing --

def test_gate_logits_match_torch_matmul():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((7, 96)).astype(np.float32)
    wr = rng.standard_normal((11, 96)).astype(np.float32)
    logits, absdot = oracle.gate_logits(x, wr)
    ref = torch.from_numpy(x).double() @ torch.from_numpy(wr).double().T
    np.testing.assert_allclose(logits, ref.numpy(), rtol=0, atol=1e-12)
    refabs = (torch.from_numpy(x).double().abs() @ torch.from_numpy(wr).double().abs().T)
    np.testing.assert_allclose(absdot, refabs.numpy(), rtol=1e-13, atol=0)


def _brute_topk_set(row, k):
    """Best k-subset by sum of logits; among equal sums the lexicographically
    smallest sorted index tuple."""
    best = None
    for c in itertools.combinations(range(len(row)), k):
        key = (-sum(row[list(c)]), c)
        if best is None or key < best:
            best = key
    return set(best[1])


@pytest.mark.parametrize("E,k", [(5, 1), (6, 2), (7, 3), (8, 4), (8, 8)])
def test_topk_equals_brute_force_with_ties(E, k):
    rng = np.random.default_rng(E * 10 + k)
    # few distinct values -> many exact ties at the selection boundary
    logits = rng.integers(-3, 3, size=(40, E)).astype(np.float64)
    idx, w, gap = oracle.topk(logits, k)
    for t in range(logits.shape[0]):
        assert set(idx[t].tolist()) == _brute_topk_set(logits[t], k)
        sel = logits[t][idx[t]]
        # descending logit, ascending index among equal logits
        for j in range(k - 1):
            assert sel[j] > sel[j + 1] or (sel[j] == sel[j + 1] and idx[t][j] < idx[t][j + 1])


def test_topk_matches_torch_topk_without_ties():
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((64, 256))
    idx, _, gap = oracle.topk(logits, 8)
    ref = torch.topk(torch.from_numpy(logits), 8, dim=1, sorted=True).indices.numpy()
    np.testing.assert_array_equal(idx, ref)
    srt = -np.sort(-logits, axis=1)
    np.testing.assert_allclose(gap, np.min(srt[:, :8] - srt[:, 1:9], axis=1), rtol=0, atol=0)


def test_duplicated_router_rows_tie_to_lower_index():
    rng = np.random.default_rng(3)
    d, E = 64, 8
    wr = rng.standard_normal((E, d)).astype(np.float32)
    wr[5] = wr[2]          # experts 2 and 5 always tie exactly
    wr[7] = wr[2]
    x = rng.standard_normal((50, d)).astype(np.float32)
    r = oracle.route(x, wr, 3)
    for t in range(50):
        row = r["idx"][t].tolist()
        for a, b in ((2, 5), (2, 7), (5, 7)):
            if b in row:
                assert a in row and row.index(a) < row.index(b)


def test_softmax_is_full_softmax_renormalised_over_selection():
    rng = np.random.default_rng(11)
    logits = rng.standard_normal((30, 64)) * 3.0
    for k in (1, 2, 6):
        idx, w, _ = oracle.topk(logits, k)
        p = torch.softmax(torch.from_numpy(logits), dim=1).numpy()
        sel = np.take_along_axis(p, idx.astype(np.int64), axis=1)
        np.testing.assert_allclose(w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-13, atol=0)
        np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-15)
        if k == 1:
            np.testing.assert_array_equal(w, 1.0)
        assert np.all(np.diff(w, axis=1) <= 0)   # descending logits -> descending weights


# ------------------------------------------------------------- expert FFN --

def test_expert_ffn_closed_form():
    """d=3, I=2, x = e_0: g = W_gate[:,0] = (0, ln 3), u = W_up[:,0] = (5, 2).
    silu(0) = 0 and silu(ln 3) = ln3/(1+1/3) = (3/4)·ln 3, so h = (0, 1.5·ln 3)
    and out_r = W_down[r][1]·1.5·ln 3 = (2, 4, 6)·1.5·ln 3 = (3, 6, 9)·ln 3.
    The other columns hold values that any misread index would pick up."""
    x = np.array([1.0, 0.0, 0.0])
    wg = np.array([[0.0, 7.0, -3.0], [math.log(3.0), 11.0, 13.0]], np.float32)
    wu = np.array([[5.0, -17.0, 19.0], [2.0, 23.0, -29.0]], np.float32)
    wd = np.array([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0]], np.float32)
    out = oracle.expert_ffn(x, wg, wu, wd)
    l3 = float(np.float32(math.log(3.0)))   # W_gate holds ln 3 rounded to float32
    expect = np.array([2.0, 4.0, 6.0]) * 2.0 * l3 / (1.0 + math.exp(-l3))
    np.testing.assert_allclose(out, expect, rtol=1e-15, atol=0)
    np.testing.assert_allclose(out, np.array([3.0, 6.0, 9.0]) * math.log(3.0), rtol=1e-6)


@pytest.mark.parametrize("wdtype", [W_F32, W_BF16])
def test_expert_ffn_matches_torch_swiglu(wdtype):
    shape = LayerShape(d=96, n_experts=3, top_k=1, inter=40, n_shared=0, wdtype=wdtype)
    L = _layer_np(shape, 21)
    x = np.random.default_rng(2).standard_normal(96)
    x64 = torch.from_numpy(x)
    for e in range(3):
        out = oracle.expert_ffn(x, L["wg"][e], L["wu"][e], L["wd"][e])
        ref = _torch_swiglu(x64, _t64(L["wg"][e]), _t64(L["wu"][e]), _t64(L["wd"][e]))
        np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------ layer output --

def _torch_layer(x, wr, k, L, s):
    """The whole layer from torch float64 library routines (topk, softmax,
    linear, silu) — independent of the oracle's C loops."""
    x64 = torch.from_numpy(x).double()
    logits = x64 @ torch.from_numpy(wr).double().T
    vals, idx = torch.topk(logits, k, dim=1, sorted=True)
    w = torch.softmax(vals, dim=1)
    y = torch.zeros_like(x64)
    for t in range(x.shape[0]):
        for j in range(k):
            e = int(idx[t, j])
            y[t] += w[t, j] * _torch_swiglu(x64[t], _t64(L["wg"][e]), _t64(L["wu"][e]),
                                            _t64(L["wd"][e]))
        for i in range(s):
            y[t] += _torch_swiglu(x64[t], _t64(L["sg"][i]), _t64(L["su"][i]), _t64(L["sd"][i]))
    return idx.numpy(), w.numpy(), y.numpy()


@pytest.mark.parametrize("wdtype,s", [(W_F32, 0), (W_BF16, 2)])
def test_layer_output_matches_torch_library_layer(wdtype, s):
    shape = LayerShape(d=64, n_experts=8, top_k=3, inter=48, n_shared=s, wdtype=wdtype)
    L = _layer_np(shape, 31)
    x = synth.make_pass(64, 5, 0.9, [9])
    r = oracle.route(x, L["wr"], 3)
    y, ys = oracle.moe_tokens(x, r["idx"], r["w"], L["wg"], L["wu"], L["wd"], L["sg"], L["su"],
                              L["sd"], slots=True)
    idx_ref, w_ref, y_ref = _torch_layer(x, L["wr"], 3, L, s)
    np.testing.assert_array_equal(r["idx"], idx_ref)
    np.testing.assert_allclose(r["w"], w_ref, rtol=1e-13, atol=0)
    np.testing.assert_allclose(y, y_ref, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(ys.sum(axis=1), y, rtol=1e-12, atol=1e-14)


def test_tiny_config_matches_torch_library_layer():
    shape = TINY.shape
    L = _layer_np(shape, TINY.weight_seed)
    x = synth.make_pass(shape.d, 4, 0.9, [TINY.x_seed_base])
    r = oracle.route(x, L["wr"], shape.top_k)
    y = oracle.moe_tokens(x, r["idx"], r["w"], L["wg"], L["wu"], L["wd"])
    idx_ref, w_ref, y_ref = _torch_layer(x, L["wr"], shape.top_k, L, 0)
    np.testing.assert_array_equal(r["idx"], idx_ref)
    np.testing.assert_allclose(y, y_ref, rtol=1e-11, atol=1e-13)


@pytest.mark.parametrize("s", [0, 1])
def test_dense_mixture_with_zero_weights_equals_sparse(s):
    """§1's dense mixture, with the sparse gate's weights on the selected
    experts and 0 elsewhere, equals the sparse output (both in the oracle and
    in an independent torch einsum over all experts)."""
    shape = LayerShape(d=64, n_experts=6, top_k=2, inter=32, n_shared=s, wdtype=W_BF16)
    L = _layer_np(shape, 41)
    x = synth.make_pass(64, 6, 0.5, [4])
    r = oracle.route(x, L["wr"], 2)
    gate = np.zeros((6, 6))
    for t in range(6):
        gate[t, r["idx"][t]] = r["w"][t]
    y_sparse = oracle.moe_tokens(x, r["idx"], r["w"], L["wg"], L["wu"], L["wd"], L["sg"],
                                 L["su"], L["sd"])
    y_dense = oracle.dense_tokens(x, gate, L["wg"], L["wu"], L["wd"], L["sg"], L["su"], L["sd"])
    np.testing.assert_allclose(y_dense, y_sparse, rtol=1e-12, atol=1e-14)
    x64 = torch.from_numpy(x).double()
    G = torch.einsum("td,eid->tei", x64, _t64(L["wg"]))
    U = torch.einsum("td,eid->tei", x64, _t64(L["wu"]))
    O = torch.einsum("tei,edi->ted", F.silu(G) * U, _t64(L["wd"]))
    y_ein = torch.einsum("te,ted->td", torch.from_numpy(gate), O)
    if s:
        GS = torch.einsum("td,sid->tsi", x64, _t64(L["sg"]))
        US = torch.einsum("td,sid->tsi", x64, _t64(L["su"]))
        y_ein = y_ein + torch.einsum("tsi,sdi->td", F.silu(GS) * US, _t64(L["sd"]))
    np.testing.assert_allclose(y_sparse, y_ein.numpy(), rtol=1e-11, atol=1e-13)


def test_shared_experts_are_unweighted_and_always_on():
    shape = LayerShape(d=64, n_experts=4, top_k=2, inter=32, n_shared=2, wdtype=W_F32)
    L = _layer_np(shape, 51)
    L["wd"][:] = 0.0      # routed experts contribute nothing
    x = synth.make_pass(64, 3, 0.0, [8])
    r = oracle.route(x, L["wr"], 2)
    y = oracle.moe_tokens(x, r["idx"], r["w"], L["wg"], L["wu"], L["wd"], L["sg"], L["su"],
                          L["sd"])
    x64 = torch.from_numpy(x).double()
    ref = sum(_torch_swiglu(x64, _t64(L["sg"][i]), _t64(L["su"][i]), _t64(L["sd"][i]))
              for i in range(2))
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------ union/bytes --

def test_union_matches_python_set_and_groups_pairs():
    rng = np.random.default_rng(13)
    for n, k, E in [(1, 6, 64), (9, 6, 64), (16, 2, 8), (64, 8, 256), (5, 3, 3)]:
        idx = np.stack([rng.permutation(E)[:k] for _ in range(n)]).astype(np.int32)
        u = oracle.union(idx, E)
        assert u["union_ids"].tolist() == sorted(set(idx.ravel().tolist()))
        assert k <= u["count"] <= min(E, n * k)
        off = u["offsets"]
        assert off[0] == 0 and off[-1] == n * k and np.all(np.diff(off) > 0)
        seen = set()
        for g, e in enumerate(u["union_ids"]):
            toks = u["pair_tok"][off[g]:off[g + 1]]
            assert np.all(np.diff(toks) > 0)            # tokens ascending within an expert
            for t, j in zip(toks, u["pair_slot"][off[g]:off[g + 1]]):
                assert idx[t, j] == e
                seen.add((int(t), int(j)))
        assert len(seen) == n * k                        # every pair exactly once


def test_bytes_closed_forms():
    for (d, I, k, s, wd) in [(2048, 1408, 6, 2, W_BF16), (4096, 14336, 2, 0, W_BF16),
                             (256, 512, 2, 0, W_F32), (7168, 2048, 8, 1, W_BF16)]:
        eb = 3 * d * I * (4 if wd == W_F32 else 2)
        for n in (1, 4, 9, 16):
            ucount = min(n * k, 7)
            ps, dd, sh = oracle.bytes_per_pass(d, I, k, s, n, wd, ucount)
            assert ps == n * k * eb and dd == ucount * eb and sh == s * eb
    # the sizes quoted for the workloads
    assert 3 * 2048 * 1408 * 2 == 17_301_504
    assert 3 * 4096 * 14336 * 2 == 352_321_536
    assert 3 * 7168 * 2048 * 2 == 88_080_384


def test_single_token_dedup_bytes_equal_perslot_bytes():
    shape = LayerShape(d=64, n_experts=16, top_k=4, inter=32, n_shared=1, wdtype=W_BF16)
    L = _layer_np(shape, 61)
    x = synth.make_pass(64, 1, 0.9, [1])
    r = oracle.route(x, L["wr"], 4)
    u = oracle.union(r["idx"], 16)
    ps, dd, _ = oracle.bytes_per_pass(64, 32, 4, 1, 1, W_BF16, u["count"])
    assert u["count"] == 4 and ps == dd


def test_identical_tokens_union_is_k():
    shape = LayerShape(d=64, n_experts=16, top_k=3, inter=32, n_shared=0, wdtype=W_BF16)
    L = _layer_np(shape, 71)
    x = np.repeat(synth.make_pass(64, 1, 0.0, [2]), 7, axis=0)   # rho -> 1
    r = oracle.route(x, L["wr"], 3)
    assert oracle.union(r["idx"], 16)["count"] == 3


def test_union_size_for_independent_tokens_is_plausible():
    """Loose statistical sanity (rho = 0): E|U| ≈ E·(1-(1-k/E)^n) for
    near-uniform routing."""
    shape = LayerShape(d=64, n_experts=64, top_k=6, inter=32, n_shared=0, wdtype=W_BF16)
    L = _layer_np(shape, 81)
    sizes = []
    for p in range(40):
        x = synth.make_pass(64, 8, 0.0, [1000 + p])
        sizes.append(oracle.union(oracle.route(x, L["wr"], 6)["idx"], 64)["count"])
    expect = 64 * (1 - (1 - 6 / 64) ** 8)
    assert abs(np.mean(sizes) - expect) < 0.2 * expect


# -- routing bias (DeepSeek-style routing sketch, §5) -------------------------
def _brute_topk(scores, k):
    """Indices of the k largest scores, ties to the lower index (plain sort)."""
    return [int(e) for e in sorted(range(len(scores)), key=lambda e: (-scores[e], e))[:k]]


def _softmax(v):
    v = np.asarray(v, np.float64)
    z = np.exp(v - v.max())
    return z / z.sum()


@pytest.mark.parametrize("bias_in_weights", [True, False])
def test_biased_topk_brute_force(bias_in_weights):
    """Selection on logit + bias; weights the softmax of the kept biased
    scores (the sketch as written) or of the kept unbiased logits."""
    rng = np.random.default_rng(11)
    E, k, n = 12, 3, 40
    # multiples of 1/8 so every sum is exact and ties occur
    logits = rng.integers(-16, 16, size=(n, E)) / 8.0
    bias = rng.integers(-8, 8, size=E) / 8.0
    idx, w, gap = oracle.topk(logits, k, bias, bias_in_weights)
    for t in range(n):
        sc = logits[t] + bias
        want = _brute_topk(sc, k)
        assert idx[t].tolist() == want
        vals = sc[want] if bias_in_weights else logits[t][want]
        np.testing.assert_allclose(w[t], _softmax(vals), rtol=0, atol=1e-15)
        srt = sorted(sc, reverse=True)
        assert gap[t] == min(srt[j] - srt[j + 1] for j in range(k))


def test_zero_bias_equals_unbiased_routing():
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((30, 16))
    a = oracle.topk(logits, 4)
    for mode in (True, False):
        b = oracle.topk(logits, 4, np.zeros(16), mode)
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])


def test_constant_bias_changes_nothing():
    """A bias equal on every expert shifts all scores alike: the selection is
    unchanged and so are the weights (softmax is shift invariant)."""
    rng = np.random.default_rng(5)
    logits = rng.integers(-40, 40, size=(25, 10)) / 4.0
    a = oracle.topk(logits, 3)
    for mode in (True, False):
        b = oracle.topk(logits, 3, np.full(10, 2.5), mode)
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_allclose(a[1], b[1], rtol=0, atol=1e-15)


def test_dominant_bias_forces_selection_and_modes_differ():
    """A bias far above every logit puts its expert first in every token's
    selection. With the bias in the weights that expert takes almost all
    the weight; with selection-only bias its weight follows its own logit."""
    rng = np.random.default_rng(9)
    logits = rng.standard_normal((20, 8))
    bias = np.zeros(8)
    bias[5] = 100.0
    idx_s, w_s, _ = oracle.topk(logits, 2, bias, True)
    idx_o, w_o, _ = oracle.topk(logits, 2, bias, False)
    assert (idx_s[:, 0] == 5).all() and (idx_o[:, 0] == 5).all()
    np.testing.assert_array_equal(idx_s, idx_o)
    assert (w_s[:, 1] < 1e-40).all()          # exp(-~100) relative to the first
    for t in range(20):
        np.testing.assert_allclose(w_o[t], _softmax(logits[t][idx_o[t]]), rtol=0, atol=1e-15)
    assert np.abs(w_o[:, 0] - w_s[:, 0]).max() > 0.1
