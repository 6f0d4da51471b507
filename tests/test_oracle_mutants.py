"""Plants plausible slips in a copy of the oracle (on the CPU) and checks that
the pins in test_oracle.py catch every one of them.

Each mutant is the oracle's C source with one textual edit, compiled into a
temporary library that replaces the oracle's for the duration of the check.
"""
import ctypes
import os
import subprocess

import pytest

import oracle.oracle as orc
import tests.test_oracle as pins
from moe_expert_layer_warp_gb300.configs import W_BF16, W_F32

MUTANTS = [
    ("silu applied to the up projection", "h[i] = silu(g) * u;", "h[i] = silu(u) * g;"),
    ("sigmoid instead of silu", "return z / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(-z));"),
    ("silu sign", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    ("W_down read transposed", "weight_at(wdown, wdtype, (size_t)r * I + i)",
     "weight_at(wdown, wdtype, (size_t)i * d + r)"),
    ("W_gate read transposed", "weight_at(wgate, wdtype, (size_t)i * d + c)",
     "weight_at(wgate, wdtype, (size_t)c * I + i)"),
    ("up uses the gate matrix", "u += weight_at(wup, wdtype", "u += weight_at(wgate, wdtype"),
    ("router read transposed", "(double)wg[(size_t)e * d + i]", "(double)wg[(size_t)i * E + e]"),
    ("ties to the higher index", "return (a->e < b->e) ? -1 : (a->e > b->e);",
     "return (a->e > b->e) ? -1 : (a->e < b->e);"),
    ("ascending instead of descending", "if (a->v > b->v) return -1;",
     "if (a->v > b->v) return 1;"),
    ("softmax numerator not shifted", "w[(size_t)t * k + j] = exp(u[j] - umax) / z;",
     "w[(size_t)t * k + j] = exp(u[j]) / z;"),
    ("softmax over one fewer logit", "for (int j = 0; j < k; ++j) z += exp(u[j] - umax);",
     "for (int j = 0; j + 1 < k; ++j) z += exp(u[j] - umax);"),
    ("routing bias ignored in the selection",
     "s[e].v = logits[(size_t)t * E + e] + (bias ? bias[e] : 0.0);",
     "s[e].v = logits[(size_t)t * E + e];"),
    ("selection-only bias also in the weights",
     "u[j] = (bias && !bias_in_weights) ? logits[(size_t)t * E + s[j].e] : s[j].v;",
     "u[j] = s[j].v;"),
    ("sketch weights without the bias",
     "u[j] = (bias && !bias_in_weights) ? logits[(size_t)t * E + s[j].e] : s[j].v;",
     "u[j] = bias ? logits[(size_t)t * E + s[j].e] : s[j].v;"),
    ("shared expert weighted by the first gate weight",
     "      y[r] += o[r];\n      if (slot_out) slot_out[(size_t)(k + i) * d + r] = o[r];",
     "      y[r] += w_t[0] * o[r];\n      if (slot_out) slot_out[(size_t)(k + i) * d + r] = o[r];"),
    ("routed expert unweighted", "y[r] += w_t[j] * o[r];", "y[r] += o[r];"),
    ("shared experts dropped", "for (int i = 0; i < s; ++i) {\n    oracle_expert_ffn(d, I, wdtype, (const char*)wsg + i * esz, (const char*)wsu + i * esz,\n                      (const char*)wsd + i * esz, xd, o);\n    for (int r = 0; r < d; ++r) {\n      y[r] += o[r];",
     "for (int i = 0; i < 0; ++i) {\n    oracle_expert_ffn(d, I, wdtype, (const char*)wsg + i * esz, (const char*)wsu + i * esz,\n                      (const char*)wsd + i * esz, xd, o);\n    for (int r = 0; r < d; ++r) {\n      y[r] += o[r];"),
    ("pairs ordered by slot, not token",
     "for (int t = 0; t < n; ++t)\n      for (int j = 0; j < k; ++j)\n        if (idx[(size_t)t * k + j] == e) {",
     "for (int j = 0; j < k; ++j)\n      for (int t = 0; t < n; ++t)\n        if (idx[(size_t)t * k + j] == e) {"),
    ("per-slot bytes miss the factor k", "bytes[0] = (uint64_t)n * (uint64_t)k * eb;",
     "bytes[0] = (uint64_t)n * eb;"),
    ("dedup bytes off by one", "bytes[1] = (uint64_t)union_count * eb;",
     "bytes[1] = (uint64_t)(union_count + 1) * eb;"),
    ("bf16 decoded from the wrong half", "((uint32_t)((const uint16_t*)w)[i]) << 16",
     "((uint32_t)((const uint16_t*)w)[i])"),
]

ALL_PINS = [
    pins.test_gate_logits_match_torch_matmul,
    lambda: pins.test_topk_equals_brute_force_with_ties(6, 2),
    lambda: pins.test_topk_equals_brute_force_with_ties(8, 4),
    pins.test_topk_matches_torch_topk_without_ties,
    pins.test_duplicated_router_rows_tie_to_lower_index,
    pins.test_softmax_is_full_softmax_renormalised_over_selection,
    lambda: pins.test_biased_topk_brute_force(True),
    lambda: pins.test_biased_topk_brute_force(False),
    pins.test_zero_bias_equals_unbiased_routing,
    pins.test_constant_bias_changes_nothing,
    pins.test_dominant_bias_forces_selection_and_modes_differ,
    pins.test_expert_ffn_closed_form,
    lambda: pins.test_expert_ffn_matches_torch_swiglu(W_F32),
    lambda: pins.test_expert_ffn_matches_torch_swiglu(W_BF16),
    lambda: pins.test_layer_output_matches_torch_library_layer(W_BF16, 2),
    pins.test_shared_experts_are_unweighted_and_always_on,
    lambda: pins.test_dense_mixture_with_zero_weights_equals_sparse(1),
    pins.test_union_matches_python_set_and_groups_pairs,
    pins.test_bytes_closed_forms,
]


def _compile(src_text, tmp_path, tag):
    src = tmp_path / ("mut_%s.c" % tag)
    so = tmp_path / ("libmut_%s.so" % tag)
    src.write_text(src_text)
    subprocess.check_call(["gcc", "-O1", "-ffp-contract=off", "-shared", "-fPIC", "-o", str(so),
                           str(src), "-lm"])
    return str(so)


def _caught(lib, monkeypatch):
    monkeypatch.setattr(orc, "_lib", lib)
    for pin in ALL_PINS:
        try:
            pin()
        except (AssertionError, RuntimeError, ValueError, IndexError):
            return True
    return False


def test_unmutated_copy_passes_every_pin(tmp_path, monkeypatch):
    with open(orc._SRC) as f:
        text = f.read()
    lib = orc.bind(_compile(text, tmp_path, "orig"))
    assert not _caught(lib, monkeypatch)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path, monkeypatch):
    with open(orc._SRC) as f:
        text = f.read()
    assert text.count(old) == 1, "mutation anchor must occur exactly once: %r" % old
    lib = orc.bind(_compile(text.replace(old, new), tmp_path, "m"))
    assert _caught(lib, monkeypatch), "pins did not catch: " + name
