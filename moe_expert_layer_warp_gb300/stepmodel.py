"""Host step-time model of a speculative-decoding step on an MoE model.

Host analytics only: it consumes measured kernel times and byte counts and
runs no part of the layer itself.

Sources:
  [A] "Speculative Decoding for Mixture-of-Experts Models: Expert Bytes,
      Kernel Bandwidth and the Best Draft Length", abstract: a step's time is
      the bytes each kernel requests over its effective bandwidth, plus fixed
      time; dedup is faster exactly where its byte share ū(n) of the per-slot
      bytes is below its bandwidth ratio r(n); the crossover is the first pass
      size at which dedup is faster; the best draft length is a monotone
      staircase in the acceptance rate under geometric acceptance.
  [O] overdisp README (over-dispersed acceptance in greedy speculative
      decoding), opening paragraph: under i.i.d. acceptance with rate α a
      block of draft length γ yields E[k] = (1 − α^(γ+1))/(1 − α) tokens.
  [L] "Is Speculative Decoding's Speedup a Hardware Problem or a Model
      Problem?", Hypothesis 1: Leviathan et al.'s expected speedup
      (1 − α^(γ+1)) / ((1 − α)(γ·c + 1)) for a draft/verify cost ratio c.
  [W] overdisp README, method and results: a_t ∈ {0,1} says whether the
      draft's token at position t is accepted; a block walk over that stream
      gives, for a draft length g, the tokens each block advances (the
      accepted run, capped at g, plus the verifier's token) and the blocks;
      autocorrelation is p11 − p10 (accept after accept minus accept after
      reject); over-dispersed streams yield fewer tokens per block than the
      i.i.d. formula at the same α, and the best draft length moves down.
  [F] "Building a Terminal Based LLM Inference Internals Explorer - Part 3:
      Speculative Decoding", section "The Flow": one verification pass scores
      the γ drafts and the bonus position, n = γ + 1 tokens.

Readings (the abstract gives no formulas):
  - per engine e, the expert kernels' effective bandwidth at pass size n is
    BW_e(n) = Σ requested expert-weight bytes / Σ expert-kernel time over the
    measured passes; the step's time for one layer is
    T_e(n) = B_e(n)/BW_e(n) + t_fix(n), with t_fix (routing, union, combine)
    the same for both engines. B_e counts the bytes the engine's kernels
    request, shared experts included for both engines, so that
    ū(n) = mean B_dd / mean B_ps and dedup is faster ⇔ ū(n) < r(n) exactly.
  - a drafted token costs t_draft; a speculative step with draft length γ
    takes γ·t_draft + T(γ+1) and advances E[k](α, γ) tokens; plain decoding
    (γ = 0) advances 1 token in T(1). γ* maximises tokens per second, ties
    going to the smaller γ.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Callable, Dict, Iterable, List, Optional, Sequence


def expected_tokens(alpha: float, gamma: int) -> float:
    """[O] E[k] = (1 − α^(γ+1))/(1 − α), tokens a verification step yields
    (the accepted run plus the verifier's own token); γ+1 at α = 1."""
    if not 0.0 <= alpha <= 1.0 or gamma < 0:
        raise ValueError("need 0 <= alpha <= 1 and gamma >= 0")
    if alpha == 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def leviathan_speedup(alpha: float, gamma: int, c: float) -> float:
    """[L] expected speedup with a flat verify cost and draft cost ratio c."""
    return expected_tokens(alpha, gamma) / (gamma * c + 1.0)


def breakeven_alpha(gamma: int, c: float, tol: float = 1e-12) -> float:
    """Smallest α at which leviathan_speedup reaches 1 (bisection; the speedup
    is increasing in α)."""
    lo, hi = 0.0, 1.0
    if leviathan_speedup(hi, gamma, c) < 1.0:
        return float("nan")
    while hi - lo > tol:
        mid = 0.5 * (lo + hi)
        if leviathan_speedup(mid, gamma, c) >= 1.0:
            hi = mid
        else:
            lo = mid
    return hi


def effective_bandwidth(bytes_: Iterable[float], seconds: Iterable[float]) -> float:
    """[A] Σ requested bytes / Σ kernel time (bytes/s)."""
    b = float(sum(bytes_))
    s = float(sum(seconds))
    if s <= 0.0:
        raise ValueError("non-positive total time")
    return b / s


def byte_share(dedup_bytes: Iterable[float], perslot_bytes: Iterable[float]) -> float:
    """[A] ū(n): dedup bytes as a share of per-slot bytes (ratio of sums)."""
    ps = float(sum(perslot_bytes))
    if ps <= 0.0:
        raise ValueError("no per-slot bytes")
    return float(sum(dedup_bytes)) / ps


def dedup_faster(u_bar: float, r: float) -> bool:
    """[A] dedup is faster exactly where ū(n) < r(n)."""
    return u_bar < r


def crossover(ns: Sequence[int], u_bar: Dict[int, float], r: Dict[int, float]) -> Optional[int]:
    """[A] the first pass size n ≥ 2 at which dedup is faster, or None."""
    for n in sorted(ns):
        if n >= 2 and dedup_faster(u_bar[n], r[n]):
            return n
    return None


@dataclass
class EngineFit:
    """Per-engine fit: effective bandwidth per pass size and fixed time."""
    bw: Dict[int, float]                    # n -> bytes/s of the expert kernels
    t_fix: Dict[int, float]                 # n -> seconds (route + union + combine)
    bytes_per_layer: Dict[int, float] = field(default_factory=dict)  # n -> mean B_e(n)

    def layer_time(self, n: int, bytes_: Optional[float] = None) -> float:
        """[A] T_e(n) = B_e(n)/BW_e(n) + t_fix(n) for one layer."""
        b = self.bytes_per_layer[n] if bytes_ is None else bytes_
        return b / self.bw[n] + self.t_fix[n]


def step_time(fit: EngineFit, n: int, bytes_per_layer: Sequence[float]) -> float:
    """[A] a pass of n tokens through a stack: Σ_layers B_ℓ(n)/BW(n) + L·t_fix(n)."""
    return sum(b / fit.bw[n] for b in bytes_per_layer) + len(bytes_per_layer) * fit.t_fix[n]


def tokens_per_second(alpha: float, gamma: int, verify_time: Callable[[int], float],
                      t_draft: float) -> float:
    """Tokens advanced per second with draft length γ ([F]: n = γ+1)."""
    return expected_tokens(alpha, gamma) / (gamma * t_draft + verify_time(gamma + 1))


def speculation_faster(alpha: float, gamma: int, verify_time: Callable[[int], float],
                       t_draft: float) -> bool:
    """[A] speculation with draft length γ beats plain decoding:
    E[k](α,γ)/(γ·t_draft + T(γ+1)) > 1/T(1)."""
    return (tokens_per_second(alpha, gamma, verify_time, t_draft)
            > 1.0 / verify_time(1))


def best_draft_length(alpha: float, verify_time: Callable[[int], float], t_draft: float,
                      gamma_max: int) -> int:
    """[A] γ*(α) = argmax over γ ∈ {0..gamma_max} of tokens per second
    (γ = 0 is plain decoding); ties go to the smaller γ."""
    best_g, best_v = 0, tokens_per_second(alpha, 0, verify_time, t_draft)
    for g in range(1, gamma_max + 1):
        v = tokens_per_second(alpha, g, verify_time, t_draft)
        if v > best_v:
            best_g, best_v = g, v
    return best_g


def staircase(alphas: Sequence[float], verify_time: Callable[[int], float], t_draft: float,
              gamma_max: int) -> List[int]:
    """[A] γ*(α) over a grid of acceptance rates."""
    return [best_draft_length(a, verify_time, t_draft, gamma_max) for a in alphas]


def acceptance_grid(lo: float = 0.50, hi: float = 0.95, steps: int = 22) -> List[float]:
    """The 22 evenly spaced acceptance rates from 0.50 to 0.95."""
    return [lo + (hi - lo) * i / (steps - 1) for i in range(steps)]


def interpolated(times: Dict[int, float]) -> Callable[[int], float]:
    """A verify-time function over the measured pass sizes (n outside the
    measured range is rejected)."""
    def T(n: int) -> float:
        if n not in times:
            raise KeyError("pass size %d not measured" % n)
        return times[n]
    return T


@dataclass
class StepModelReport:
    ns: List[int]
    u_bar: Dict[int, float]
    r: Dict[int, float]
    bw_ps: Dict[int, float]
    bw_dd: Dict[int, float]
    t_fix: Dict[int, float]
    crossover: Optional[int]
    alphas: List[float]
    gamma_star_ps: List[int]
    gamma_star_dd: List[int]
    gamma_star_best: List[int]
    t_draft: float

    def as_dict(self) -> dict:
        return {
            "n": self.ns,
            "u_bar": [round(self.u_bar[n], 6) for n in self.ns],
            "r": [round(self.r[n], 6) for n in self.ns],
            "bw_perslot_GBs": [round(self.bw_ps[n] / 1e9, 2) for n in self.ns],
            "bw_dedup_GBs": [round(self.bw_dd[n] / 1e9, 2) for n in self.ns],
            "t_fix_us": [round(self.t_fix[n] * 1e6, 3) for n in self.ns],
            "crossover_n": self.crossover,
            "t_draft_us": round(self.t_draft * 1e6, 3),
            "alphas": [round(a, 5) for a in self.alphas],
            "gamma_star_perslot": self.gamma_star_ps,
            "gamma_star_dedup": self.gamma_star_dd,
            "gamma_star_best_engine": self.gamma_star_best,
        }


def build_report(samples: Dict[str, Dict[int, List[tuple]]], t_fix: Dict[int, float],
                 layers: int = 1, draft_cost_ratio: float = 0.0,
                 alphas: Optional[Sequence[float]] = None) -> StepModelReport:
    """Fit and evaluate the model from measured passes.

    samples[engine][n] = list of (requested_bytes, expert_kernel_seconds) per
    pass, engine in {"perslot", "dedup"}; t_fix[n] in seconds per layer.
    The draft cost per drafted token is draft_cost_ratio × T_best(1)."""
    ns = sorted(set(samples["perslot"]) & set(samples["dedup"]))
    bw_ps = {n: effective_bandwidth([b for b, _ in samples["perslot"][n]],
                                    [s for _, s in samples["perslot"][n]]) for n in ns}
    bw_dd = {n: effective_bandwidth([b for b, _ in samples["dedup"][n]],
                                    [s for _, s in samples["dedup"][n]]) for n in ns}
    u = {n: byte_share([b for b, _ in samples["dedup"][n]],
                       [b for b, _ in samples["perslot"][n]]) for n in ns}
    r = {n: bw_dd[n] / bw_ps[n] for n in ns}
    mean_b = {e: {n: sum(b for b, _ in samples[e][n]) / len(samples[e][n]) for n in ns}
              for e in ("perslot", "dedup")}
    fit_ps = EngineFit(bw_ps, t_fix, mean_b["perslot"])
    fit_dd = EngineFit(bw_dd, t_fix, mean_b["dedup"])
    T_ps = {n: layers * fit_ps.layer_time(n) for n in ns}
    T_dd = {n: layers * fit_dd.layer_time(n) for n in ns}
    T_best = {n: min(T_ps[n], T_dd[n]) for n in ns}
    if 1 not in T_best:
        raise ValueError("pass size 1 (plain decoding) must be measured")
    t_draft = draft_cost_ratio * T_best[1]
    gmax = max(ns) - 1
    al = list(alphas) if alphas is not None else acceptance_grid()
    return StepModelReport(
        ns=ns, u_bar=u, r=r, bw_ps=bw_ps, bw_dd=bw_dd, t_fix=dict(t_fix),
        crossover=crossover(ns, u, r), alphas=al,
        gamma_star_ps=staircase(al, interpolated(T_ps), t_draft, gmax),
        gamma_star_dd=staircase(al, interpolated(T_dd), t_draft, gmax),
        gamma_star_best=staircase(al, interpolated(T_best), t_draft, gmax),
        t_draft=t_draft)


# ------------------------------------------------------------ stack check --
def bandwidth_spread(samples: Sequence[tuple]) -> float:
    """Relative spread ε of a fit: max over the fitted passes of
    |b_i/s_i ÷ BW − 1|, BW = Σb/Σs. Used as the fit's bandwidth error."""
    bw = effective_bandwidth([b for b, _ in samples], [s for _, s in samples])
    return max(abs(b / s / bw - 1.0) for b, s in samples)


def saving_bound(bytes_ps: float, bw_ps: float, eps_ps: float, bytes_dd: float, bw_dd: float,
                 eps_dd: float) -> float:
    """[A] how far a bandwidth error moves the predicted saving T_ps − T_dd.

    Reading: if the true bandwidth of an engine lies in BW·[1−ε, 1+ε], its
    byte time B/BW_true lies within B/BW · ε/(1−ε) of the prediction; the
    fixed time is common to both engines and cancels in the saving, so the
    saving moves by at most the sum of the two engines' moves."""
    if not (0.0 <= eps_ps < 1.0 and 0.0 <= eps_dd < 1.0):
        raise ValueError("bandwidth error must lie in [0, 1)")
    return bytes_ps / bw_ps * eps_ps / (1.0 - eps_ps) + bytes_dd / bw_dd * eps_dd / (1.0 - eps_dd)


def crossover_from_times(ns: Sequence[int], t_ps: Dict[int, float],
                         t_dd: Dict[int, float]) -> Optional[int]:
    """[A] the first pass size n ≥ 2 at which the dedup pass takes less time."""
    for n in sorted(ns):
        if n >= 2 and t_dd[n] < t_ps[n]:
            return n
    return None


@dataclass
class StackCheck:
    """Predicted against measured stack passes at one hidden-state correlation."""
    ns: List[int]
    measured: Dict[str, Dict[int, float]]     # engine -> n -> seconds
    predicted: Dict[str, Dict[int, float]]
    bound: Dict[int, float]                   # n -> saving bound (seconds)
    alphas: List[float]
    draft_cost_ratio: float

    def saving(self, which: str) -> Dict[int, float]:
        t = self.measured if which == "measured" else self.predicted
        return {n: t["perslot"][n] - t["dedup"][n] for n in self.ns}

    def inside_bound(self) -> Dict[int, bool]:
        sm_, sp = self.saving("measured"), self.saving("predicted")
        return {n: abs(sm_[n] - sp[n]) <= self.bound[n] for n in self.ns}

    def gamma_star(self, which: str) -> List[int]:
        """γ*(α) over the grid with the faster engine at each n; a drafted
        token costs draft_cost_ratio × the n = 1 pass."""
        t = self.measured if which == "measured" else self.predicted
        best = {n: min(t["perslot"][n], t["dedup"][n]) for n in self.ns}
        return staircase(self.alphas, interpolated(best), self.draft_cost_ratio * best[1],
                         max(self.ns) - 1)

    def as_dict(self) -> dict:
        gm, gp = self.gamma_star("measured"), self.gamma_star("predicted")
        ins = self.inside_bound()
        us = lambda d: [round(d[n] * 1e6, 2) for n in self.ns]  # noqa: E731
        return {
            "n": self.ns,
            "measured_us": {e: us(self.measured[e]) for e in ("perslot", "dedup")},
            "predicted_us": {e: us(self.predicted[e]) for e in ("perslot", "dedup")},
            "saving_measured_us": us(self.saving("measured")),
            "saving_predicted_us": us(self.saving("predicted")),
            "saving_bound_us": us(self.bound),
            "saving_inside_bound": sum(ins.values()), "points": len(self.ns),
            "crossover_measured": crossover_from_times(self.ns, self.measured["perslot"],
                                                       self.measured["dedup"]),
            "crossover_predicted": crossover_from_times(self.ns, self.predicted["perslot"],
                                                        self.predicted["dedup"]),
            "draft_cost_ratio": self.draft_cost_ratio,
            "gamma_star_measured": gm, "gamma_star_predicted": gp,
            "gamma_star_within_one": sum(abs(a - b) <= 1 for a, b in zip(gm, gp)),
        }


# ------------------------------------------------ non-geometric acceptance --
def block_walk(a: Sequence[int], g: int):
    """[W] Walks an accept stream with draft length g: a block starting at
    position t advances r + 1 positions, r = the run of accepted drafts from
    t capped at g (the verifier supplies the token at t + r); the next block
    starts at t + r + 1. Returns (tokens, blocks, drafted) over the whole
    blocks that fit in the stream."""
    if g < 0:
        raise ValueError("draft length must be >= 0")
    n = len(a)
    t = tokens = blocks = 0
    while t + g < n:           # the block's drafts and the verifier's position fit
        r = 0
        while r < g and a[t + r]:
            r += 1
        tokens += r + 1
        blocks += 1
        t += r + 1
    return tokens, blocks, blocks * g


def markov_rates(alpha: float, autocorr: float):
    """(p11, p10) of a two-state accept chain with stationary acceptance α
    and autocorrelation p11 − p10 = autocorr: α = p10 / (1 − p11 + p10)."""
    p10 = alpha * (1.0 - autocorr)
    p11 = p10 + autocorr
    if not (0.0 <= p10 <= 1.0 and 0.0 <= p11 <= 1.0):
        raise ValueError("no chain with alpha=%g, autocorr=%g" % (alpha, autocorr))
    return p11, p10


def markov_stream(n: int, alpha: float, autocorr: float, rng) -> "np.ndarray":
    """A seeded accept stream of length n from the two-state chain, started
    in its stationary distribution."""
    import numpy as np
    p11, p10 = markov_rates(alpha, autocorr)
    u = rng.random(n)
    a = np.empty(n, np.int8)
    prev = u[0] < alpha
    a[0] = prev
    for t in range(1, n):
        prev = u[t] < (p11 if prev else p10)
        a[t] = prev
    return a


def markov_yield(alpha: float, autocorr: float, g: int) -> float:
    """Closed-form tokens per block of the block walk over the two-state
    chain (renewal-reward over the block's start state s = the acceptance of
    the position before it). From s the first draft is accepted with
    r_s = p11 or p10 and each next one with p11, so E[k|s] = 1 + r_s·(1 −
    p11^g)/(1 − p11); the next block starts in state 1 only when all g drafts
    were accepted and the verifier's position was accepted too, P = r_s·p11^g.
    With p11 = p10 = α this is (1 − α^(g+1))/(1 − α)."""
    p, q = markov_rates(alpha, autocorr)
    if g == 0:
        return 1.0
    run = g if p == 1.0 else (1.0 - p ** g) / (1.0 - p)
    e1, e0 = 1.0 + p * run, 1.0 + q * run
    pi1 = q * p ** g / (1.0 - p ** (g + 1) + q * p ** g)
    return pi1 * e1 + (1.0 - pi1) * e0


def best_draft_length_yield(yield_fn: Callable[[int], float], verify_time: Callable[[int], float],
                            t_draft: float, gamma_max: int) -> int:
    """γ* = argmax over γ ∈ {0..gamma_max} of yield(γ) / (γ·t_draft + T(γ+1)),
    ties to the smaller γ, for any tokens-per-block function."""
    best_g, best_v = 0, yield_fn(0) / verify_time(1)
    for g in range(1, gamma_max + 1):
        v = yield_fn(g) / (g * t_draft + verify_time(g + 1))
        if v > best_v:
            best_g, best_v = g, v
    return best_g
