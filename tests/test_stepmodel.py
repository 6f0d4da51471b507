"""Pins of the host step-time model against the pages' worked numbers and
closed forms, plus properties the method states.

Sources: "Is Speculative Decoding's Speedup a Hardware Problem or a Model
Problem?" (Hypothesis 1 and 2 tables); overdisp README, opening paragraph
(E[k]); "Speculative Decoding for Mixture-of-Experts Models: Expert Bytes,
Kernel Bandwidth and the Best Draft Length", abstract (ū < r criterion,
crossover, monotone staircase).
"""
import json
import os
import random

import numpy as np
import pytest

from moe_expert_layer_warp_gb300 import stepmodel as sm

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                   "speculative_worked_examples.json")))


def test_cost_ratio_from_flops():
    c = GOLD["cost_ratio_flops"]
    assert round(c["draft_flops_per_token"] / c["verifier_flops_per_token"], 4) == c["c_printed"]


@pytest.mark.parametrize("table", ["hypothesis1_theoretical", "hypothesis2_theoretical"])
def test_leviathan_table_values(table):
    tab = GOLD[table]
    for row in tab["rows"]:
        v = sm.leviathan_speedup(row["alpha"], row["gamma"], tab["c"])
        assert round(v, 2) == row["speedup"], (row, v)


def test_breakeven_span():
    b = GOLD["hypothesis2_breakeven"]
    lo = sm.breakeven_alpha(b["gamma_lo"], b["c"])
    hi = sm.breakeven_alpha(b["gamma_hi"], b["c"])
    assert round(100 * lo) == b["alpha_lo_percent"]
    assert round(100 * hi) == b["alpha_hi_percent"]
    seq = [sm.breakeven_alpha(g, b["c"]) for g in range(b["gamma_lo"], b["gamma_hi"] + 1)]
    assert all(a < b_ for a, b_ in zip(seq, seq[1:]))


def test_expected_tokens_limits_and_series():
    for g in range(0, 12):
        assert sm.expected_tokens(0.0, g) == 1.0
        assert sm.expected_tokens(1.0, g) == g + 1
        assert abs(sm.expected_tokens(1.0 - 1e-9, g) - (g + 1)) < 1e-6
        for a in (0.1, 0.5, 0.93):
            # capped geometric run: E[k] = Σ_{i=0}^{γ} α^i
            assert abs(sm.expected_tokens(a, g) - sum(a ** i for i in range(g + 1))) < 1e-12


def test_flat_verify_cost_reduces_to_leviathan():
    """With T(n) ≡ T(1) and t_draft = c·T(1), tokens/s relative to plain
    decoding is Leviathan's speedup."""
    T1 = 3.7e-3
    for a in (0.3, 0.6, 0.9):
        for g in (1, 4, 8):
            for c in (0.0, 0.1601, 0.5002):
                v = sm.tokens_per_second(a, g, lambda n: T1, c * T1) * T1
                assert abs(v - sm.leviathan_speedup(a, g, c)) < 1e-12


def test_dedup_faster_iff_u_below_r():
    """Step time per engine is B/BW + t_fix with the same t_fix: dedup has the
    smaller time exactly when ū < r."""
    rnd = random.Random(1)
    for _ in range(2000):
        ps = rnd.uniform(1e8, 1e10)
        dd = ps * rnd.uniform(0.05, 1.0)
        bw_ps = rnd.uniform(1e12, 8e12)
        bw_dd = bw_ps * rnd.uniform(0.2, 1.5)
        tf = rnd.uniform(0, 1e-5)
        t_ps = sm.EngineFit({1: bw_ps}, {1: tf}).layer_time(1, ps)
        t_dd = sm.EngineFit({1: bw_dd}, {1: tf}).layer_time(1, dd)
        u, r = dd / ps, bw_dd / bw_ps
        if abs(u - r) > 1e-9:
            assert (t_dd < t_ps) == sm.dedup_faster(u, r)


def test_crossover_is_first_n_where_u_below_r():
    ns = list(range(1, 10))
    u = {n: 1.0 / n ** 0.5 for n in ns}
    r = {n: 0.5 for n in ns}
    assert sm.crossover(ns, u, r) == 5          # 1/sqrt(5) = 0.447 < 0.5
    assert sm.crossover(ns, u, {n: 0.2 for n in ns}) is None


def test_staircase_is_monotone_in_alpha():
    rnd = random.Random(7)
    alphas = sm.acceptance_grid()
    assert len(alphas) == 22 and alphas[0] == 0.5 and abs(alphas[-1] - 0.95) < 1e-12
    for _ in range(200):
        # verify time increasing and concave-ish in n, as for byte-bound passes
        base = rnd.uniform(1e-4, 1e-2)
        slope = rnd.uniform(0.0, 0.3)
        T = {n: base * (1.0 + slope * (n - 1) ** rnd.uniform(0.5, 1.0)) for n in range(1, 17)}
        td = rnd.choice([0.0, 0.05, 0.1, 0.2]) * T[1]
        st = sm.staircase(alphas, sm.interpolated(T), td, 15)
        assert all(a <= b for a, b in zip(st, st[1:])), st


def test_best_draft_length_ties_go_to_smaller_gamma():
    # α = 0: every γ yields one token; with free drafting and flat T they tie
    assert sm.best_draft_length(0.0, lambda n: 1.0, 0.0, 8) == 0


def test_build_report_end_to_end():
    samples = {"perslot": {}, "dedup": {}}
    for n in range(1, 10):
        ps = n * 6 * 17_301_504 + 2 * 17_301_504
        dd = min(64, 6 + 2 * (n - 1)) * 17_301_504 + 2 * 17_301_504
        samples["perslot"][n] = [(ps, ps / 6.0e12)]
        samples["dedup"][n] = [(dd, dd / 5.0e12)]
    rep = sm.build_report(samples, {n: 5e-6 for n in range(1, 10)})
    d = rep.as_dict()
    assert d["r"][0] == pytest.approx(5.0 / 6.0)
    assert d["u_bar"][0] == pytest.approx(1.0)
    n_star = rep.crossover
    assert n_star is not None
    assert rep.u_bar[n_star] < rep.r[n_star]
    assert all(not (rep.u_bar[n] < rep.r[n]) for n in range(2, n_star))
    assert len(rep.gamma_star_best) == 22


def test_bandwidth_spread():
    assert sm.bandwidth_spread([(5.0, 1.0), (10.0, 2.0)]) == 0.0
    # rates 100 and 300 over equal time: BW = 200, spread 0.5
    assert sm.bandwidth_spread([(100.0, 1.0), (300.0, 1.0)]) == pytest.approx(0.5)


def test_saving_bound_holds_for_every_bandwidth_in_range():
    """Brute force over true bandwidths inside BW·[1−ε, 1+ε]: the saving's
    move never exceeds the bound, and the worst corner reaches most of it."""
    B_ps, bw_ps, e_ps = 3.0e9, 6.0e12, 0.08
    B_dd, bw_dd, e_dd = 1.2e9, 4.5e12, 0.15
    bound = sm.saving_bound(B_ps, bw_ps, e_ps, B_dd, bw_dd, e_dd)
    pred = B_ps / bw_ps - B_dd / bw_dd
    worst = 0.0
    for a in np.linspace(1 - e_ps, 1 + e_ps, 41):
        for b in np.linspace(1 - e_dd, 1 + e_dd, 41):
            worst = max(worst, abs(B_ps / (bw_ps * a) - B_dd / (bw_dd * b) - pred))
    assert worst <= bound * (1 + 1e-12)
    assert worst >= 0.75 * bound
    assert sm.saving_bound(B_ps, bw_ps, 0.0, B_dd, bw_dd, 0.0) == 0.0
    with pytest.raises(ValueError):
        sm.saving_bound(B_ps, bw_ps, 1.0, B_dd, bw_dd, 0.0)


def test_crossover_from_times():
    ns = list(range(1, 6))
    t_ps = {n: 10.0 * n for n in ns}
    t_dd = {n: 30.0 + 4.0 * n for n in ns}       # equal at n = 5: never strictly faster
    assert sm.crossover_from_times(ns, t_ps, t_dd) is None
    t_dd = {n: 12.0 + 5.0 * n for n in ns}       # n = 2: 22 > 20; n = 3: 27 < 30
    assert sm.crossover_from_times(ns, t_ps, t_dd) == 3
    # n = 1 never counts, even when dedup is faster there
    assert sm.crossover_from_times([1, 2], {1: 2.0, 2: 1.0}, {1: 1.0, 2: 3.0}) is None


def test_stack_check_agrees_with_itself_and_counts_misses():
    ns = list(range(1, 10))
    meas = {"perslot": {n: 100e-6 + 50e-6 * n for n in ns},
            "dedup": {n: 110e-6 + 30e-6 * n for n in ns}}
    bound = {n: 2e-6 for n in ns}
    chk = sm.StackCheck(ns, meas, meas, bound, sm.acceptance_grid(), 0.1601)
    d = chk.as_dict()
    assert d["saving_inside_bound"] == 9
    assert d["crossover_measured"] == d["crossover_predicted"] == 2
    assert d["gamma_star_within_one"] == 22
    assert d["gamma_star_measured"] == sorted(d["gamma_star_measured"])
    # predictions off by 5 µs on dedup at n = 4: that point leaves the bound
    pred = {"perslot": dict(meas["perslot"]), "dedup": dict(meas["dedup"])}
    pred["dedup"][4] += 5e-6
    chk = sm.StackCheck(ns, meas, pred, bound, sm.acceptance_grid(), 0.1601)
    assert chk.as_dict()["saving_inside_bound"] == 8


# -- non-geometric acceptance (overdisp README: block walk, p11 - p10) -------
def test_block_walk_hand_cases():
    a = [1, 1, 0, 1, 1, 1, 1, 0, 1]
    # g = 2: t=0 run 2 -> 3 tokens (t=3); t=3 run 2 -> 3 (t=6); t=6 run 1 -> 2 (t=8); t=8: 8+2 > 8
    assert sm.block_walk(a, 2) == (8, 3, 6)
    # g = 0: every position is a block of one verifier token
    assert sm.block_walk(a, 0) == (9, 9, 0)
    # g = 4: t=0 run 2 -> 3 (t=3); t=3 run 4 -> 5 (t=8); t=8: 8+4 > 8
    assert sm.block_walk(a, 4) == (8, 2, 8)
    assert sm.block_walk([0, 0, 0], 1) == (2, 2, 2)


def test_markov_yield_reduces_to_geometric_without_autocorrelation():
    for alpha in (0.1, 0.5, 0.77, 0.95):
        for g in range(0, 12):
            assert sm.markov_yield(alpha, 0.0, g) == pytest.approx(sm.expected_tokens(alpha, g),
                                                                   rel=1e-13)


def test_markov_rates_define_the_chain():
    p11, p10 = sm.markov_rates(0.9, 0.155)
    assert p11 - p10 == pytest.approx(0.155)
    assert p10 / (1 - p11 + p10) == pytest.approx(0.9)
    with pytest.raises(ValueError):
        sm.markov_rates(0.5, -1.5)           # p10 would exceed 1


@pytest.mark.parametrize("alpha,autocorr", [(0.6, 0.2), (0.9, 0.155), (0.94, 0.233), (0.8, -0.1)])
def test_block_walk_of_simulated_streams_matches_closed_form(alpha, autocorr):
    rng = np.random.default_rng(123)
    a = sm.markov_stream(300_000, alpha, autocorr, rng)
    assert a.mean() == pytest.approx(alpha, abs=0.01)
    prev = a[:-1].astype(bool)
    p11 = a[1:][prev].mean()
    p10 = a[1:][~prev].mean()
    assert p11 - p10 == pytest.approx(autocorr, abs=0.01)
    for g in (1, 3, 8):
        tok, blocks, drafted = sm.block_walk(a, g)
        assert drafted == g * blocks
        assert tok / blocks == pytest.approx(sm.markov_yield(alpha, autocorr, g), rel=0.01)


def test_positive_autocorrelation_lowers_the_yield_and_the_best_draft_length():
    """Over-dispersed acceptance yields fewer tokens per block than the i.i.d.
    formula at the same alpha (more so at longer drafts), and with a verify
    time that grows with the pass the best draft length does not move up."""
    for g in (2, 8, 16):
        assert sm.markov_yield(0.9, 0.2, g) < sm.expected_tokens(0.9, g)
    assert (sm.markov_yield(0.9, 0.2, 16) / sm.expected_tokens(0.9, 16) <
            sm.markov_yield(0.9, 0.2, 2) / sm.expected_tokens(0.9, 2))
    T = {n: 1.0 + 0.12 * (n - 1) for n in range(1, 17)}
    for alpha in (0.6, 0.75, 0.9, 0.95):
        g_iid = sm.best_draft_length_yield(lambda g: sm.expected_tokens(alpha, g),
                                           sm.interpolated(T), 0.05, 15)
        g_mk = sm.best_draft_length_yield(lambda g: sm.markov_yield(alpha, 0.2, g),
                                          sm.interpolated(T), 0.05, 15)
        assert g_mk <= g_iid
        assert g_iid == sm.best_draft_length(alpha, sm.interpolated(T), 0.05, 15)
