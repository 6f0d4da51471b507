"""Benchmark: verify-pass tokens/s and expert-weight HBM GB/s, dedup vs
per-slot, on the DeepSeek-V2-Lite-shaped 26-layer MoE stack (expert layers
only: d=2048, 64 routed experts top-6 + 2 shared, SwiGLU I=1408, bf16 weights,
fp32 accumulate; 29.7 GB of expert weights).

One step = one verification pass at every pass size n = 1..9 (AR(1) hidden
states, rho = 0.9) through all 26 layers, once with each engine (per-slot and
dedup): 18 stack passes, 468 layer passes, 90 tokens. Every layer is fed the
same pass (attention and residuals are outside the path). Each layer's
weights (1.14 GB) are far larger than L2 and consecutive layers read different
weights, so every layer reads its expert weights cold from HBM. The step is
captured once in a CUDA graph and replayed.

Besides the headline the line carries the per-call breakdown of the layers'
passes (the step-time model's inputs), the stack check (the model fitted on
one layer run alone against the measured stack, at four hidden-state
correlations), and per-pass-size tables of the Mixtral- and DeepSeek-V3-shaped
layers.

Prints one JSON line (rank 0). ``--impl reference`` times the float64 CPU
oracle on the same workload instead (a bounded sample per step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verify-pass tokens/s and expert-weight HBM GB/s vs 8 TB/s, dedup vs per-slot"
UNIT = "tokens/s"
LAYERS = 26
WORKLOAD = ("deepseek-v2-lite-shaped 26-layer MoE stack (expert layers only, each fed the same "
            "pass): d=2048, 64 routed experts top-6 + 2 shared, SwiGLU I=1408, bf16 weights / "
            "fp32 accumulate, 29.7 GB of expert weights; verify passes n=1..9 at rho=0.9 through "
            "all 26 layers with the per-slot and the dedup engine")
HEADLINE_RHO = 0.9
N_PASSES_PER_N = 2        # distinct hidden-state passes per n, alternated across steps
EXPERT_BYTES = 3 * 2048 * 1408 * 2
BREAKDOWN_PASSES = 8      # passes per (pass size, engine) in the per-call breakdown
BREAKDOWN_ROUNDS = 9      # replays of each breakdown graph (median taken)
SPIN_CYCLES = 2_000_000   # ~1 ms of device spin before a timed pass: the host queues the whole
                          # pass meanwhile, so no launch waits on the host inside the timed span


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-extras", action="store_true",
                   help="skip the stack check and the other workloads' tables (profiling runs)")
    p.add_argument("--case", default=None,
                   help="profiling case WORKLOAD:ENGINE:N (e.g. v2lite:perslot:1): runs "
                        "--passes passes of one layer and prints their mean time")
    p.add_argument("--passes", type=int, default=4)
    p.add_argument("--sweep", default=None, choices=["tiny", "v2lite", "mixtral", "v3"],
                   help="one layer of WORKLOAD at every pass size and rho of that workload, "
                        "both engines: requested bytes, time and bandwidth per n, r(n), the "
                        "byte share and the crossover")
    p.add_argument("--rho", type=float, default=None, help="--sweep: this rho only")
    p.add_argument("--stack", action="store_true",
                   help="only the stack check: fit the step-time model on one layer run "
                        "alone, predict the stack's passes and compare with measured ones")
    p.add_argument("--calls", default=None, choices=["v2lite", "mixtral", "v3"],
                   help="for an ncu DRAM capture: one layer of WORKLOAD at rho = 0.9, one "
                        "per-slot and one dedup pass at each pass size; prints each expert "
                        "call's requested bytes in launch order")
    p.add_argument("--dram-record", nargs=2, metavar=("CALLS_JSON", "NCU_CSV"), default=None,
                   help="write profiles/dram_expert_calls_<workload>.txt from a --calls "
                        "output and the ncu csv of the same command")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed
    region (every 200 ms)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        import tempfile
        self.path = os.environ.get("MOE_CLOCKS_LOG") or os.path.join(
            tempfile.gettempdir(), "moe_clocks_rank%d.csv" % gpu_index)

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [s.strip() for s in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------- across ranks --
def max_over_ranks(x: float, dev) -> float:
    """The largest of every rank's x (all ranks call it; one process: x)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def job_value(world: int, tokens_per_step: int, ms_step: float) -> float:
    """Whole-job tokens/s: every rank processes tokens_per_step per step, and
    the job's step takes the slowest rank's time."""
    return world * tokens_per_step / (ms_step * 1e-3)


# ------------------------------------------------------------- our engine --
def build_stack(dev):
    """The 26 layers (seed 1000 + layer), one PassRunner each, and the
    headline's hidden-state passes: N_PASSES_PER_N per pass size at rho 0.9."""
    import torch
    from moe_expert_layer_warp_gb300 import configs, synth
    from moe_expert_layer_warp_gb300.layer import PassRunner
    w = configs.V2_LITE_STACK
    assert w.layers == LAYERS and HEADLINE_RHO in w.rhos
    layers = [synth.make_layer(w.shape, w.weight_seed + l, dev) for l in range(w.layers)]
    runners = [PassRunner(L, max(w.pass_sizes)) for L in layers]
    xs = {}
    for n in w.pass_sizes:
        xs[n] = [torch.from_numpy(synth.make_pass(w.shape.d, n, HEADLINE_RHO,
                                                  [w.x_seed_base + 1000 * q + n]))
                 .to(dev) for q in range(N_PASSES_PER_N)]
    return w, runners, xs


def step_plan(w, step_idx):
    """(n, engine, x variant) of the 18 stack passes of a step."""
    return [(n, eng, step_idx % N_PASSES_PER_N) for n in w.pass_sizes
            for eng in ("perslot", "dedup")]


def enqueue_step(w, runners, xs, step_idx, stream):
    for n, eng, q in step_plan(w, step_idx):
        for R in runners:
            R.forward(xs[n][q], eng, stream)


def kernels_per_pass():
    # moe_verify_pass: the gate GEMV (which also does the expert call's prep
    # work), the top-k/union kernel (which also gathers the dedup rows), one
    # expert kernel (tensor-core or CUDA-core, chosen per call), the combine
    return 2 + 1 + 1


def capture_graph(fn):
    """Captures fn(stream) into a CUDA graph on a side stream."""
    import torch
    cur = torch.cuda.current_stream()
    s = torch.cuda.Stream()
    s.wait_stream(cur)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn(s)
    cur.wait_stream(s)
    torch.cuda.synchronize()
    return g


def time_graphs(graphs, rounds):
    """Replays the graphs round-robin `rounds` times on the current stream,
    each replay between CUDA events after a device spin that covers the host's
    launch; returns each graph's median replay time in seconds."""
    import torch
    stream = torch.cuda.current_stream()
    evs = []
    for _ in range(rounds):
        for i, g in enumerate(graphs):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(SPIN_CYCLES // 4)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            evs.append((i, e0, e1))
    torch.cuda.synchronize()
    ts = [[] for _ in graphs]
    for i, e0, e1 in evs:
        ts[i].append(e0.elapsed_time(e1) * 1e-3)
    return [statistics.median(t) for t in ts]


def requested(R, eng):
    """Requested expert-weight bytes of the runner's last pass with `eng`:
    per-slot n·k·E_b or dedup |U|·E_b, plus the shared experts' s·E_b."""
    b = [int(v) for v in R.bytes.cpu().tolist()]
    return (b[0] if eng == "perslot" else b[1]) + b[2]


def unique_bytes(R):
    """The runner's last pass's distinct expert bytes, |U|·E_b + s·E_b."""
    b = [int(v) for v in R.bytes.cpu().tolist()]
    return b[1] + b[2]


def measure_breakdown(w, runners, xs):
    """The expert call's time inside pipelined passes, per pass size and
    engine, on the stack's layers. BREAKDOWN_PASSES passes (pass i on layer
    i, so consecutive passes read different weights) run back to back, as in
    the headline step, in one CUDA graph: the whole passes (moe_verify_pass:
    route, union, expert call, combine), and in a second graph their
    routing, union and combine alone. The two graphs are replayed
    round-robin between CUDA events on the stream; a pass's time is the
    first graph's median over the passes it holds, the fixed time the
    second's, the expert call's time their difference. Returns samples for
    the step-time model (each pass's requested bytes with the call time per
    pass), the fixed and pass times and the passes' unique bytes."""
    samples = {"perslot": {n: [] for n in w.pass_sizes}, "dedup": {n: [] for n in w.pass_sizes}}
    uniq = {"perslot": {n: [] for n in w.pass_sizes}, "dedup": {n: [] for n in w.pass_sizes}}
    tfix = {n: [] for n in w.pass_sizes}
    pass_ms = {"perslot": {n: [] for n in w.pass_sizes}, "dedup": {n: [] for n in w.pass_sizes}}
    import torch
    stream = torch.cuda.current_stream()
    for n in w.pass_sizes:
        for eng in ("perslot", "dedup"):
            plan = [(i % len(runners), i % N_PASSES_PER_N) for i in range(BREAKDOWN_PASSES)]
            reqs = []
            for li, q in plan:          # requested bytes of each pass (routing is deterministic)
                R = runners[li]
                R.forward(xs[n][q], eng, stream)
                reqs.append(requested(R, eng))
                uniq[eng][n].append(unique_bytes(R))

            def chain(s, with_expert):
                for li, q in plan:
                    R, x = runners[li], xs[n][q]
                    if with_expert:      # the whole pass, as the user calls it
                        R.forward(x, eng, s)
                    else:                # its fixed part: routing, union and combine
                        R.route_union(x, s)
                        R.combine(n, s)
            ga = capture_graph(lambda s: chain(s, True))
            gb = capture_graph(lambda s: chain(s, False))
            ta, tb = time_graphs([ga, gb], BREAKDOWN_ROUNDS)
            k = len(plan)
            call = max(ta - tb, 1e-9) / k
            for i in range(k):
                samples[eng][n].append((reqs[i], call))
            tfix[n].append(tb / k)
            pass_ms[eng][n].append(ta / k * 1e3)
            del ga, gb
    t_fix = {n: statistics.median(v) for n, v in tfix.items()}
    return samples, t_fix, pass_ms, uniq


FUSED_PASSES = 4   # passes per (pass size, engine) in the fused-combine comparison


def measure_fused(w, runners, xs):
    """Pass time with the combine as a launch of its own (moe_verify_pass)
    and fused into the expert kernel (moe_verify_pass_fused), per pass size
    and engine: FUSED_PASSES passes on as many layers back to back in one
    CUDA graph each way, replayed round-robin between CUDA events; medians
    per pass in microseconds."""
    out = {"separate_us": {}, "fused_us": {}}
    for eng in ("perslot", "dedup"):
        sep, fus = [], []
        for n in w.pass_sizes:
            plan = [(i % len(runners), i % N_PASSES_PER_N) for i in range(FUSED_PASSES)]

            def chain(s, fused):
                for li, q in plan:
                    runners[li].forward(xs[n][q], eng, s, fused=fused)
            ga = capture_graph(lambda s: chain(s, False))
            gb = capture_graph(lambda s: chain(s, True))
            ta, tb = time_graphs([ga, gb], BREAKDOWN_ROUNDS)
            sep.append(round(ta / len(plan) * 1e6, 2))
            fus.append(round(tb / len(plan) * 1e6, 2))
            del ga, gb
        out["separate_us"][eng] = sep
        out["fused_us"][eng] = fus
    return out


def e2e_measure(w, runners, xs, steps, warmup):
    """End to end through the public API with host buffers, as a serving loop
    runs it: each step uploads all its passes' hidden states from pinned host
    memory in one copy, runs every stack pass (PassRunner.forward — one
    moe_verify_pass call — per layer, each writing its y into the step's
    [layer][row] output block) and reads the whole block back to pinned host
    memory in one copy. One CUDA graph per step variant holds the upload, the
    passes and the read-back; every step replays one, so every copy runs
    every step inside the timed region."""
    import torch
    stream = torch.cuda.current_stream()
    dev = xs[w.pass_sizes[0]][0].device
    d = w.shape.d
    n_variants = N_PASSES_PER_N
    plans = [step_plan(w, v) for v in range(n_variants)]
    rows = sum(n for n, _, _ in plans[0])
    L = len(runners)
    hx = []
    for v in range(n_variants):
        blk = torch.empty((rows, d), dtype=torch.float32).pin_memory()
        r = 0
        for n, _, q in plans[v]:
            blk[r:r + n].copy_(xs[n][q].cpu())
            r += n
        hx.append(blk)
    hy = [torch.empty((L, rows, d), dtype=torch.float32).pin_memory() for _ in range(n_variants)]
    dx = torch.empty((rows, d), dtype=torch.float32, device=dev)
    dy = torch.empty((L, rows, d), dtype=torch.float32, device=dev)
    h2d = rows * d * 4
    d2h = L * rows * d * 4

    def capture_step(v, cap):
        dx.copy_(hx[v], non_blocking=True)
        r = 0
        for n, eng, q in plans[v]:
            for li, R in enumerate(runners):
                R.forward(dx[r:r + n], eng, cap, out=dy[li, r:r + n])
            r += n
        hy[v].copy_(dy, non_blocking=True)

    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    graphs = []
    with torch.cuda.stream(cap):
        for v in range(n_variants):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                capture_step(v, cap)
            graphs.append(g)
    stream.wait_stream(cap)
    for i in range(max(warmup, n_variants)):
        graphs[i % n_variants].replay()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        graphs[i % n_variants].replay()
    t1.record(stream)
    t1.synchronize()
    return t0.elapsed_time(t1) / steps, h2d, d2h


def e2e_measure_eager(w, runners, xs, steps, warmup):
    """End to end through the public API called pass by pass from Python, with
    host buffers: every stack pass copies its hidden states from pinned host
    memory, runs the 26 layers (one moe_verify_pass call each) and reads the
    26 layers' y back to pinned host memory, inside the timed region. The
    copies run on a copy stream ordered against the compute stream by events,
    so a pass's upload overlaps the previous pass and its read-back the next
    (double-buffered device and host buffers). Returns the device time per
    step and the host's issue time per step."""
    import torch
    stream = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    dev = xs[w.pass_sizes[0]][0].device
    d, L = w.shape.d, len(runners)
    hx = {n: [x.cpu().pin_memory() for x in xs[n]] for n in xs}
    hy = {n: [torch.empty((L, n, d), dtype=torch.float32).pin_memory() for _ in range(2)]
          for n in xs}
    dx = {n: [torch.empty((n, d), dtype=torch.float32, device=dev) for _ in range(2)] for n in xs}
    dy = {n: [torch.empty((L, n, d), dtype=torch.float32, device=dev) for _ in range(2)]
          for n in xs}
    h2d = sum(2 * n * d * 4 for n in w.pass_sizes)
    d2h = sum(2 * L * n * d * 4 for n in w.pass_sizes)
    state = {"i": 0, "done": [None, None]}

    def one(step_idx):
        for n, eng, q in step_plan(w, step_idx):
            b = state["i"] & 1
            state["i"] += 1
            with torch.cuda.stream(copy):
                if state["done"][b] is not None:
                    copy.wait_event(state["done"][b])   # buffer b's previous pass is read back
                dx[n][b].copy_(hx[n][q], non_blocking=True)
                up = torch.cuda.Event()
                up.record(copy)
            stream.wait_event(up)
            for li, R in enumerate(runners):
                R.forward(dx[n][b], eng, stream, out=dy[n][b][li])
            fin = torch.cuda.Event()
            fin.record(stream)
            with torch.cuda.stream(copy):
                copy.wait_event(fin)
                hy[n][b].copy_(dy[n][b], non_blocking=True)
                rd = torch.cuda.Event()
                rd.record(copy)
            state["done"][b] = rd

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    copy.wait_event(t0)
    h0 = time.perf_counter()
    for i in range(steps):
        one(i)
    host_ms = (time.perf_counter() - h0) * 1e3 / steps
    stream.wait_stream(copy)
    t1.record(stream)
    t1.synchronize()
    ms = t0.elapsed_time(t1) / steps
    return ms, h2d, d2h, host_ms


# -------------------------------------------------- committed DRAM records --
TRAFFIC_SOURCES = ("expert_stream.cu", "expert_mma.cu", "engine.cu", "plan.cuh", "common.cuh",
                   "launch.h", "tcgen05.cuh", "tmap.h", "api.cu", "route_union.cu")


def _code_only(text: str) -> str:
    """C/C++ source without its comments and with whitespace runs collapsed,
    so that the hash below changes with the code, not with its comments."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash() -> str:
    """sha256 (first 16 hex digits) over the code of the expert call's
    sources (comments excluded): every kernel of a pass and the choice
    between the expert kernels."""
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES:
        path = os.path.join(ROOT, "moe_expert_layer_warp_gb300", "csrc", f)
        h.update(_code_only(open(path, encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def dram_record_path(workload: str) -> str:
    return os.path.join(ROOT, "profiles", "dram_expert_calls_%s.txt" % workload)


def load_dram_record(workload: str, check_hash: bool = True):
    """The ``key: value`` lines of a committed ncu DRAM record (one expert
    call per pass size and engine), if its counters were taken on the
    current kernel sources; else None. Values are int lists."""
    path = dram_record_path(workload)
    if not os.path.exists(path):
        return None
    rec = {}
    for line in open(path):
        if ":" in line and not line.startswith((" ", "#")):
            k, v = line.split(":", 1)
            rec[k.strip()] = v.strip()
    if check_hash and rec.get("sources_sha256_16") != kernel_source_hash():
        return None
    out = {"rho": float(rec.get("rho", "nan")), "sources_sha256_16": rec.get("sources_sha256_16")}
    try:
        for key in ("n", "perslot_requested", "perslot_dram", "dedup_requested", "dedup_dram"):
            out[key] = [int(t) for t in rec[key].split(",")]
    except (KeyError, ValueError):
        return None
    if not all(len(out[k]) == len(out["n"]) for k in out if isinstance(out[k], list)):
        return None
    return out


def dram_factor(workload: str):
    """DRAM bytes of an expert call over its pass's unique expert bytes (the
    union's, |U|·E_b + s·E_b, which is what the dedup engine requests), per
    engine and pass size, from the record, when it was taken on the current
    sources; else None. Both engines read each distinct expert of a pass
    from DRAM about once — the per-slot engine runs the slots of one expert
    side by side, so L2 serves the repeats — so the factor is near 1 and
    does not depend on the routing; the record's rho is stated beside it."""
    rec = load_dram_record(workload)
    if rec is None:
        return None
    return {e: {n: rec[e + "_dram"][i] / rec["dedup_requested"][i]
                for i, n in enumerate(rec["n"])} for e in ("perslot", "dedup")}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        j = json.load(open(path))
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ------------------------------------------------------------- CPU oracle --
_ORC = {}   # state of a spawned oracle worker


def _oracle_worker_init(paths, k, E, passes):
    """Spawned worker: maps the layer's weights (read-only .npy memmaps, one
    copy in the page cache for all workers) and binds the oracle library."""
    from oracle import oracle
    _ORC["H"] = {name: np.load(p, mmap_mode="r") for name, p in paths.items()}
    _ORC.update(k=k, E=E, passes=passes, routes={}, orc=oracle)


def _oracle_token(task):
    """The oracle's routing of the pass (once per worker and pass) and its
    layer output for one token of it."""
    n, t = task
    orc, H, x = _ORC["orc"], _ORC["H"], _ORC["passes"][n]
    r = _ORC["routes"].get(n)
    if r is None:
        r = orc.route(x, H["wr"], _ORC["k"])
        orc.union(r["idx"], _ORC["E"])
        _ORC["routes"][n] = r
    orc.moe_tokens(x, r["idx"], r["w"], H["wg"], H["wu"], H["wd"], H["sg"], H["su"], H["sd"],
                   tokens=[t])
    return 1


class OracleHost:
    """The float64 oracle, as it stands, on one layer of the stack (layer 0;
    every layer has the same shape, so the oracle's cost per token and layer
    is the same for all 26): one thread in this process, or one spawned worker
    process per host core (spawn, never fork: this process may hold a CUDA
    context). Stack tokens/s = token-layers/s ÷ 26."""

    def __init__(self):
        import tempfile
        from moe_expert_layer_warp_gb300 import configs, synth
        w = configs.V2_LITE_STACK
        self.w = w
        L = synth.make_layer(w.shape, w.weight_seed, "cpu")
        self.H = {k: synth.weights_numpy(getattr(L, a)) for k, a in
                  (("wg", "w_gate"), ("wu", "w_up"), ("wd", "w_down"), ("sg", "ws_gate"),
                   ("su", "ws_up"), ("sd", "ws_down"))}
        self.H["wr"] = L.w_router.numpy()
        del L
        self.passes = {n: synth.make_pass(w.shape.d, n, HEADLINE_RHO, [w.x_seed_base + n])
                       for n in w.pass_sizes}
        self.order = [(n, t) for n in w.pass_sizes for t in range(n)]
        self.tmp = tempfile.mkdtemp(prefix="moe_oracle_")
        self.pool = None
        self.procs = 1

    def single(self, tasks):
        """Seconds for the tasks on one thread of this process."""
        _oracle_worker_init({}, self.w.shape.top_k, self.w.shape.n_experts, self.passes)
        _ORC["H"] = self.H
        t0 = time.perf_counter()
        for task in tasks:
            _oracle_token(task)
        return time.perf_counter() - t0

    def start_pool(self, procs=None):
        import multiprocessing as mp
        self.procs = procs or os.cpu_count() or 1
        paths = {}
        for name, arr in self.H.items():
            paths[name] = os.path.join(self.tmp, name + ".npy")
            np.save(paths[name], arr)
        ctx = mp.get_context("spawn")
        self.pool = ctx.Pool(self.procs, initializer=_oracle_worker_init,
                             initargs=(paths, self.w.shape.top_k, self.w.shape.n_experts,
                                       self.passes))
        self.pool.map(_oracle_token, [(1, 0)] * self.procs, chunksize=1)   # start and warm

    def parallel(self, tasks):
        """Seconds for the tasks spread over the worker processes."""
        t0 = time.perf_counter()
        self.pool.map(_oracle_token, tasks, chunksize=1)
        return time.perf_counter() - t0

    def close(self):
        import shutil
        if self.pool is not None:
            self.pool.close()
            self.pool.join()
        shutil.rmtree(self.tmp, ignore_errors=True)


def cpu_baseline_sample(budget_s=10.0):
    """The oracle as it stands on this host's cores, on a bounded sample of
    the workload: every token of one pass at each n = 1..9 (45 tokens)
    through layer 0 of the stack, first on one thread, then repeated over one
    worker per core until about budget_s; stack tokens/s = token-layers/s ÷
    26. Returns the cpu_baseline dict."""
    host = OracleHost()
    try:
        t1 = host.single(host.order)
        one = len(host.order) / t1 / LAYERS
        host.start_pool()
        t = host.parallel(host.order)
        reps = max(1, int(budget_s / max(t, 1e-3)))
        tasks = host.order * reps
        tp = host.parallel(tasks)
        many = len(tasks) / tp / LAYERS
    finally:
        host.close()
    return {"value": round(many, 4), "unit": UNIT, "cores": host.procs, "kind": "oracle",
            "sample": "float64 oracle (routing of each pass, layer output per token) on %d worker "
                      "processes, one per host core: every token of one pass at each n = 1..9 "
                      "through layer 0 of the stack, %d times (%d token-layers, %.1f s); stack "
                      "tokens/s = token-layers/s / 26 (every layer has the same shape)" % (
                          host.procs, reps, len(tasks), tp),
            "single_thread": {"value": round(one, 4), "cores": 1,
                              "sample": "the same 45 token-layers on one thread (%.1f s)" % t1}}


# ------------------------------------------------------------ stack check --
STACK_DRAFT_COST_RATIO = 0.1601   # draft/verify cost ratio c the pages derive from FLOPs
STACK_FIT_PASSES = 4   # held-out passes (own seeds) per (rho, n) for the bandwidth fit
STACK_DEPTHS = (1, 4, 13, 26)     # partial stacks whose crossover is predicted and measured
STACK_AUTOCORR = 0.155   # within-stream acceptance autocorrelation p11 - p10 (pooled, overdisp)
STACK_REPS = 3


def stack_check(w, runners, dev):
    """Per rho in {0, 0.5, 0.9, 0.99}: the bandwidths fitted on layer 0's
    expert call run alone over STACK_FIT_PASSES held-out passes (own seeds),
    each pass a CUDA graph behind an L2 flush (a 256 MB read) timed with and
    without its expert call; each stack pass (and its first 1, 4 and 13
    layers) predicted from every layer's requested bytes over those
    bandwidths plus the fixed time, and compared with the measured stack
    pass: the saving against its bound, the crossover per depth and the best
    draft length, under i.i.d. and autocorrelated acceptance. Returns the
    report dict."""
    import torch
    from moe_expert_layer_warp_gb300 import api, stepmodel, synth
    stream = torch.cuda.current_stream()
    # read (not written) to flush L2: the flush leaves clean lines behind, as
    # the previous layer's weights do inside a stack pass
    flush = torch.zeros(64 << 20, dtype=torch.float32, device=dev)
    engines = ("perslot", "dedup")

    def make_x(ri, rho, n, f):
        return torch.from_numpy(synth.make_pass(w.shape.d, n, rho, [
            w.x_seed_base + 100 * ri + 10000 * f + n])).to(dev)

    xs = {(ri, n): make_x(ri, rho, n, 0) for ri, rho in enumerate(w.rhos) for n in w.pass_sizes}
    fit_xs = {(ri, n): [make_x(ri, rho, n, 1 + f) for f in range(STACK_FIT_PASSES)]
              for ri, rho in enumerate(w.rhos) for n in w.pass_sizes}

    for (ri, n), x in xs.items():          # warm-up: every pass once through the stack,
        for eng in engines:                # every fitted pass once through layer 0
            for R in runners:
                R.forward(x, eng, stream)
            for xf in fit_xs[(ri, n)]:
                runners[0].forward(xf, eng, stream)
    torch.cuda.synchronize()
    if api.moe_last_device_error() != api.MOE_OK:
        raise RuntimeError("device error during the stack check's warm-up")

    R0 = runners[0]
    g_flush = capture_graph(lambda s: flush.sum())
    per_rho, fits_out = [], []
    for ri, rho in enumerate(w.rhos):
        samples = {e: {n: [] for n in w.pass_sizes} for e in engines}
        tfix = {n: [] for n in w.pass_sizes}
        t_flush = time_graphs([g_flush], 2 * BREAKDOWN_ROUNDS)[0]
        for n in w.pass_sizes:
            for eng in engines:
                reqs = []
                for x in fit_xs[(ri, n)]:
                    R0.forward(x, eng, stream)
                    reqs.append(requested(R0, eng))

                def one(s, x, with_expert):
                    flush.sum()
                    if with_expert:
                        R0.forward(x, eng, s)
                    else:
                        R0.route_union(x, s)
                        R0.combine(n, s)
                ga = [capture_graph(lambda s, x=x: one(s, x, True)) for x in fit_xs[(ri, n)]]
                gb = [capture_graph(lambda s, x=x: one(s, x, False)) for x in fit_xs[(ri, n)]]
                t = time_graphs(ga + gb, BREAKDOWN_ROUNDS)
                k = len(ga)
                for i in range(k):
                    samples[eng][n].append((reqs[i], max(t[i] - t[k + i], 1e-9)))
                    tfix[n].append(max(t[k + i] - t_flush, 0.0))
                del ga, gb
        t_fix = {n: statistics.median(v) for n, v in tfix.items()}
        fits = {e: stepmodel.EngineFit({n: stepmodel.effective_bandwidth(
            [b for b, _ in samples[e][n]], [t for _, t in samples[e][n]]) for n in w.pass_sizes},
            t_fix) for e in engines}
        eps = {e: {n: stepmodel.bandwidth_spread(samples[e][n]) for n in w.pass_sizes}
               for e in engines}
        fits_out.append({
            "rho": rho,
            "bw_perslot_GBs": [round(fits["perslot"].bw[n] / 1e9, 1) for n in w.pass_sizes],
            "bw_dedup_GBs": [round(fits["dedup"].bw[n] / 1e9, 1) for n in w.pass_sizes],
            "eps_perslot": [round(eps["perslot"][n], 4) for n in w.pass_sizes],
            "eps_dedup": [round(eps["dedup"][n], 4) for n in w.pass_sizes],
            "t_fix_us": [round(t_fix[n] * 1e6, 2) for n in w.pass_sizes]})
        meas_d = {L: {e: {} for e in engines} for L in STACK_DEPTHS}
        pred_d = {L: {e: {} for e in engines} for L in STACK_DEPTHS}
        bound = {}
        for n in w.pass_sizes:
            x = xs[(ri, n)]
            lb = {}
            for eng in engines:
                for L in STACK_DEPTHS:
                    ts = []
                    for rep in range(STACK_REPS):
                        e0 = torch.cuda.Event(enable_timing=True)
                        e1 = torch.cuda.Event(enable_timing=True)
                        torch.cuda._sleep(8 * SPIN_CYCLES)   # host queues the stack meanwhile
                        e0.record(stream)
                        for R in runners[:L]:
                            R.forward(x, eng, stream)
                        e1.record(stream)
                        torch.cuda.synchronize()
                        ts.append(e0.elapsed_time(e1) * 1e-3)
                    meas_d[L][eng][n] = statistics.median(ts)
                lb[eng] = [requested(R, eng) for R in runners]
                for L in STACK_DEPTHS:
                    pred_d[L][eng][n] = stepmodel.step_time(fits[eng], n, lb[eng][:L])
            bound[n] = stepmodel.saving_bound(sum(lb["perslot"]), fits["perslot"].bw[n],
                                              eps["perslot"][n], sum(lb["dedup"]),
                                              fits["dedup"].bw[n], eps["dedup"][n])
        meas, pred = meas_d[w.layers], pred_d[w.layers]
        chk = stepmodel.StackCheck(list(w.pass_sizes), meas, pred, bound,
                                   stepmodel.acceptance_grid(), STACK_DRAFT_COST_RATIO)
        d = chk.as_dict()
        d["rho"] = rho
        ns = list(w.pass_sizes)
        d["crossover_by_depth"] = [
            {"layers": L,
             "measured": stepmodel.crossover_from_times(ns, meas_d[L]["perslot"], meas_d[L]["dedup"]),
             "predicted": stepmodel.crossover_from_times(ns, pred_d[L]["perslot"],
                                                         pred_d[L]["dedup"])}
            for L in STACK_DEPTHS]
        # best draft length under i.i.d. and over-dispersed (two-state Markov)
        # acceptance, on the measured stack's best-engine pass times
        best = {n: min(meas["perslot"][n], meas["dedup"][n]) for n in ns}
        T = stepmodel.interpolated(best)
        td = STACK_DRAFT_COST_RATIO * best[1]
        alphas = stepmodel.acceptance_grid()
        g_iid = [stepmodel.best_draft_length_yield(
            lambda g, a=a: stepmodel.expected_tokens(a, g), T, td, max(ns) - 1) for a in alphas]
        g_mk = [stepmodel.best_draft_length_yield(
            lambda g, a=a: stepmodel.markov_yield(a, STACK_AUTOCORR, g), T, td, max(ns) - 1)
            for a in alphas]
        d["non_geometric"] = {
            "autocorr_p11_minus_p10": STACK_AUTOCORR,
            "gamma_star_iid": g_iid, "gamma_star_markov": g_mk,
            "shift": [b - a for a, b in zip(g_iid, g_mk)],
            "yield_ratio_markov_over_iid_at_0.90": [
                round(stepmodel.markov_yield(0.9, STACK_AUTOCORR, g) /
                      stepmodel.expected_tokens(0.9, g), 4) for g in range(1, max(ns))]}
        per_rho.append(d)
    if api.moe_last_device_error() != api.MOE_OK:
        raise RuntimeError("device error in the stack passes")
    summary = {
        "saving_inside_bound": "%d of %d" % (sum(d["saving_inside_bound"] for d in per_rho),
                                             sum(d["points"] for d in per_rho)),
        "crossover_predicted_equals_measured_by_depth": "%d of %d" % (
            sum(c["measured"] == c["predicted"] for d in per_rho for c in d["crossover_by_depth"]),
            sum(len(d["crossover_by_depth"]) for d in per_rho)),
        "crossover_within_one_pass_size_by_depth": "%d of %d" % (
            sum(_within_one(c["measured"], c["predicted"], max(w.pass_sizes))
                for d in per_rho for c in d["crossover_by_depth"]),
            sum(len(d["crossover_by_depth"]) for d in per_rho)),
        "gamma_star_within_one": "%d of %d" % (sum(d["gamma_star_within_one"] for d in per_rho),
                                               sum(len(d["gamma_star_measured"]) for d in per_rho)),
    }
    return {"stack": "deepseek-v2-lite-shaped 26-layer MoE stack (expert layers only, each fed "
                     "the same pass), bf16 weights, %.1f GB of expert weights" % (
                         w.layers * (w.shape.n_experts + w.shape.n_shared) * EXPERT_BYTES / 1e9),
            "fit": {"layer": 0, "passes_per_point": STACK_FIT_PASSES,
                    "l2": "flushed (256 MB read) before each fitted pass", "per_rho": fits_out},
            "summary": summary, "per_rho": per_rho}


def best_engine_rate(stack):
    """Stack tokens/s of a pass at each n = 1..9 with the faster engine at
    that n, from the stack check's measured 26-layer passes at the headline
    rho (each a single pass timed between CUDA events, not graph-replayed);
    None without the stack check."""
    if not stack:
        return None
    for d in stack["per_rho"]:
        if abs(d["rho"] - HEADLINE_RHO) < 1e-9:
            ps, dd = d["measured_us"]["perslot"], d["measured_us"]["dedup"]
            best = [min(a, b) for a, b in zip(ps, dd)]
            return {"tokens_per_s": round(sum(d["n"]) / (sum(best) * 1e-6), 2),
                    "engine_by_n": ["dedup" if b < a else "perslot" for a, b in zip(ps, dd)],
                    "per_slot_only_tokens_per_s": round(sum(d["n"]) / (sum(ps) * 1e-6), 2),
                    "dedup_only_tokens_per_s": round(sum(d["n"]) / (sum(dd) * 1e-6), 2),
                    "what": "one stack pass at each n = 1..9 (rho %.2f) with the faster engine at "
                            "each n, from the stack check's measured passes" % HEADLINE_RHO}
    return None


def _within_one(a, b, n_max):
    """Crossovers within one pass size; "never" (None) counts as n_max + 1."""
    a = n_max + 1 if a is None else a
    b = n_max + 1 if b is None else b
    return abs(a - b) <= 1


# ------------------------------------------------------ per-n layer tables --
CASES = {"tiny": "TINY", "v2lite": "V2_LITE", "mixtral": "MIXTRAL", "v3": "V3"}
SWEEP_PASSES = 2    # distinct hidden-state passes per (rho, n)


def sweep_workload(name, rhos=None, passes=SWEEP_PASSES):
    """One layer of a workload at each of its pass sizes and rhos through
    both engines; each pass a CUDA graph behind an L2 flush (a 256 MB read),
    timed with and without its expert call. Returns one dict per rho:
    requested bytes, expert-call time and bandwidth per n and engine, the
    DRAM bandwidth where a committed capture at that rho covers the current
    kernels, the byte share u(n), the bandwidth ratio r(n) and the
    crossover."""
    import torch
    from moe_expert_layer_warp_gb300 import api, configs, stepmodel, synth
    from moe_expert_layer_warp_gb300.layer import PassRunner
    w = getattr(configs, CASES[name])
    sh = w.shape
    L = synth.make_layer(sh, w.weight_seed, "cuda")
    R = PassRunner(L, max(w.pass_sizes) * w.streams)
    st = torch.cuda.current_stream()
    flush = torch.zeros(64 << 20, dtype=torch.float32, device="cuda")
    t_flush = time_graphs([capture_graph(lambda s: flush.sum())], 6)[0]
    engines = ("perslot", "dedup")
    peak = peaks()[0]
    out = []
    for rho in (rhos if rhos is not None else w.rhos):
        samples = {e: {n: [] for n in w.pass_sizes} for e in engines}
        uniq = {e: {n: [] for n in w.pass_sizes} for e in engines}
        tfix = {n: [] for n in w.pass_sizes}
        for n in w.pass_sizes:
            for f in range(passes):
                x = torch.from_numpy(synth.make_pass(sh.d, n, rho, [
                    w.x_seed_base + 5000 + 97 * f + 13 * s for s in range(w.streams)])).cuda()
                m = x.shape[0]
                for eng in engines:
                    R.forward(x, eng, st)
                    req = requested(R, eng)
                    uniq[eng][n].append(unique_bytes(R))

                    def one(s, with_expert):
                        flush.sum()
                        if with_expert:
                            R.forward(x, eng, s)
                        else:
                            R.route_union(x, s)
                            R.combine(m, s)
                    ga = capture_graph(lambda s: one(s, True))
                    gb = capture_graph(lambda s: one(s, False))
                    ta, tb = time_graphs([ga, gb], 3)
                    samples[eng][n].append((req, max(ta - tb, 1e-9)))
                    tfix[n].append(max(tb - t_flush, 0.0))
                    del ga, gb
        if api.moe_last_device_error() != api.MOE_OK:
            raise RuntimeError("device error in the sweep")
        ns = list(w.pass_sizes)
        bw = {e: {n: stepmodel.effective_bandwidth([b for b, _ in samples[e][n]],
                                                   [t for _, t in samples[e][n]]) for n in ns}
              for e in engines}
        u = {n: stepmodel.byte_share([b for b, _ in samples["dedup"][n]],
                                     [b for b, _ in samples["perslot"][n]]) for n in ns}
        r = {n: bw["dedup"][n] / bw["perslot"][n] for n in ns}
        line = {"workload": w.name, "rho": rho, "streams": w.streams, "n": ns,
                "passes_per_point": passes,
                "timing": "expert call inside a CUDA-graph-replayed pass behind a 256 MB L2 "
                          "flush (graph with minus graph without the call)",
                "peak_GBs": peak}
        fac = dram_factor(name)
        for eng in engines:
            gbs = [bw[eng][n] / 1e9 for n in ns]
            f = [fac[eng].get(n * w.streams) if fac else None for n in ns]
            dram = [None if fn is None else sum(uniq[eng][n]) * fn /
                    sum(t for _, t in samples[eng][n]) / 1e9 for n, fn in zip(ns, f)]
            line[eng] = {
                "requested_MB": [round(sum(b for b, _ in samples[eng][n]) / len(samples[eng][n])
                                       / 1e6, 1) for n in ns],
                "expert_us": [round(sum(t for _, t in samples[eng][n]) / len(samples[eng][n])
                                    * 1e6, 2) for n in ns],
                "GBs": [round(g, 1) for g in gbs],
                "frac_of_peak": [round(g / peak, 3) for g in gbs],
                "dram_GBs": [None if v is None else round(v, 1) for v in dram],
                "dram_frac_of_peak": [None if v is None else round(v / peak, 3) for v in dram]}
        line["dram_source"] = (os.path.relpath(dram_record_path(name), ROOT) + ": DRAM bytes = "
                               "each pass's unique expert bytes x the factor ncu measured per "
                               "engine and n on one call (rho %s)" % load_dram_record(name)["rho"]
                               if fac else "no capture on these sources")
        line.update({"u_bar": [round(u[n], 6) for n in ns], "r": [round(r[n], 6) for n in ns],
                     "crossover_n": stepmodel.crossover(ns, u, r),
                     "t_fix_us": [round(statistics.median(tfix[n]) * 1e6, 2) for n in ns]})
        out.append(line)
    del R, L
    torch.cuda.empty_cache()
    return out


# -------------------------------------------------------------- our arm --
def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from __graft_entry__ import build
    build()
    from moe_expert_layer_warp_gb300 import api, stepmodel

    w, runners, xs = build_stack(dev)
    stream = torch.cuda.current_stream()
    tokens_per_step = 2 * sum(w.pass_sizes)
    passes_per_step = 2 * len(w.pass_sizes) * len(runners)

    # warm-up (also configures the kernels before graph capture)
    for i in range(max(3, args.warmup)):
        enqueue_step(w, runners, xs, i, stream)
    torch.cuda.synchronize()
    st = api.moe_last_device_error()
    if st != api.MOE_OK:
        raise RuntimeError("device error during warm-up: %s" % api.status_str(st))

    # one graph per step variant (the x variant depends on the step index)
    graphs = []
    cap_stream = torch.cuda.Stream()
    cap_stream.wait_stream(stream)
    with torch.cuda.stream(cap_stream):
        for v in range(N_PASSES_PER_N):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap_stream):
                enqueue_step(w, runners, xs, v, cap_stream)
            graphs.append(g)
    stream.wait_stream(cap_stream)
    torch.cuda.synchronize()
    for v in range(N_PASSES_PER_N):
        graphs[v].replay()
    torch.cuda.synchronize()

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        graphs[i % N_PASSES_PER_N].replay()
    e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms_step = max_over_ranks(e0.elapsed_time(e1) / args.steps, dev)
    value = job_value(world, tokens_per_step, ms_step)
    del graphs

    st = api.moe_last_device_error()
    if st != api.MOE_OK:
        raise RuntimeError("device error in the timed region: %s" % api.status_str(st))

    # per-call breakdown on the stack's layers (outside the timed region)
    samples, t_fix, pass_ms, uniq = measure_breakdown(w, runners, xs)
    rep = stepmodel.build_report(samples, t_fix, layers=len(runners))
    fused = measure_fused(w, runners, xs)
    e2e_ms, h2d, d2h = e2e_measure(w, runners, xs, max(3, args.steps // 2), 3)
    e2e_ms = max_over_ranks(e2e_ms, dev)
    eager_ms, _, _, eager_host_ms = e2e_measure_eager(w, runners, xs, max(3, args.steps // 4), 2)
    eager_ms = max_over_ranks(eager_ms, dev)

    stack = None
    tables = None
    if not args.no_extras and rank == 0:
        stack = stack_check(w, runners, dev)
    del runners, xs
    torch.cuda.empty_cache()
    if not args.no_extras and rank == 0:
        tables = {"mixtral": sweep_workload("mixtral"), "v3": sweep_workload("v3")}

    if rank != 0:
        return
    peak, peak_kind = peaks()
    ns = list(w.pass_sizes)
    sh = w.shape
    fac = dram_factor("v2lite")
    per_engine = {}
    req_b, dram_b, call_s, ncalls = 0.0, 0.0, 0.0, 0
    for eng in ("perslot", "dedup"):
        gbs = [sum(b for b, _ in samples[eng][n]) / sum(s for _, s in samples[eng][n]) / 1e9
               for n in ns]
        dram = ([sum(uniq[eng][n]) * fac[eng][n] / sum(s for _, s in samples[eng][n]) / 1e9
                 for n in ns] if fac else None)
        per_engine[eng] = {
            "tokens_per_s_one_layer": [round(n / (statistics.median(pass_ms[eng][n]) * 1e-3), 1)
                                       for n in ns],
            "pass_us": [round(statistics.median(pass_ms[eng][n]) * 1e3, 2) for n in ns],
            "expert_us": [round(sum(s for _, s in samples[eng][n]) / len(samples[eng][n]) * 1e6, 2)
                          for n in ns],
            "requested_MB": [round(sum(b for b, _ in samples[eng][n]) / len(samples[eng][n]) / 1e6,
                                   1) for n in ns],
            "expert_GBs": [round(g, 1) for g in gbs],
            "expert_frac_of_peak": [round(g / peak, 3) for g in gbs],
            "dram_GBs": [round(g, 1) for g in dram] if dram else None,
        }
        if dram:
            per_engine[eng]["dram_frac_of_peak"] = [round(v / peak, 3) for v in dram]
        for n in ns:
            act = n * sh.d * 4 + n * (sh.top_k + sh.n_shared) * sh.d * 4
            for (b, s), u in zip(samples[eng][n], uniq[eng][n]):
                req_b += b + act
                dram_b += (u * fac[eng][n] if fac else float("nan")) + act
                call_s += s
                ncalls += 1
    achieved = req_b / call_s / 1e9
    achieved_dram = dram_b / call_s / 1e9 if fac else None
    cpu = None if args.no_cpu_baseline else cpu_baseline_sample()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1/sqrt(fan_in)) weights, AR(1) hidden states)",
        "config": {"workload": WORKLOAD, "layers": LAYERS,
                   "tokens_per_step": tokens_per_step, "stack_passes_per_step": 2 * len(ns),
                   "layer_passes_per_step": passes_per_step, "pass_sizes": ns,
                   "rho": HEADLINE_RHO,
                   "l2": "inputs larger than L2: 26 layers of 1.14 GB, each layer pass reads "
                         "another layer's weights than the one before it",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "timing": "CUDA-graph replay of each step, CUDA events on the stream"},
        "roofline": {"kernel": "expert call: expert_mma_kernel (tensor cores) or "
                               "expert_engine_kernel (CUDA cores), chosen per call; up/gate and "
                               "down of every group (a whole pass runs no prep kernel)",
                     "bound": "hbm",
                     "bytes": "requested: the call's expert-weight bytes as the method counts them "
                              "(per-slot n*k*E_b + s*E_b, dedup |U|*E_b + s*E_b) plus its "
                              "activations; per-slot requests of a repeated expert can be served "
                              "by L2, so frac can exceed 1; frac_dram counts DRAM bytes instead",
                     "achieved": round(achieved, 1), "peak": peak, "peak_source": peak_kind,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "achieved_dram": None if achieved_dram is None else round(achieved_dram, 1),
                     "frac_dram": None if achieved_dram is None else round(achieved_dram / peak, 4),
                     "traffic": None if not fac else int(round(dram_b / ncalls)),
                     "traffic_source": (os.path.relpath(dram_record_path("v2lite"), ROOT) +
                                        ": DRAM bytes per call = the pass's unique expert bytes "
                                        "x the factor ncu measured per engine and n (1.000-1.021)"
                                        if fac else "no capture on these sources"),
                     "calls": ncalls, "call_us_mean": round(call_s / ncalls * 1e6, 2)},
        "cpu_baseline": cpu,
        "e2e": {"value": round(job_value(world, tokens_per_step, e2e_ms), 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "path": "PassRunner.forward (moe_verify_pass) per layer, one pinned upload of "
                        "the step's hidden states and one read-back of all 26 layers' outputs, "
                        "captured per step variant in a CUDA graph"},
        "gpu_launches": args.steps * passes_per_step * kernels_per_pass(),
        "e2e_eager": {"value": round(job_value(world, tokens_per_step, eager_ms), 2),
                      "unit": UNIT, "host_issue_ms_per_step": round(eager_host_ms, 4),
                      "note": "the same passes and copies issued call by call from Python"},
        "clocks": clk,
        "layer_breakdown": {
            "what": "8 layer passes back to back (each on another layer of the stack) in one "
                    "CUDA graph per point, times per pass; expert call = graph with minus graph "
                    "without the calls; t_fix = routing, union and combine",
            "engines": per_engine, "stepmodel": rep.as_dict(),
            "fused_combine": dict(fused, what="layer passes back to back (graph replay, %d passes "
                                  "on as many layers, time per pass) with the combine as a launch of its own "
                                  "(moe_verify_pass, the headline's path) and fused into the "
                                  "expert kernel's last phase (moe_verify_pass_fused)"
                                  % FUSED_PASSES)},
        "stack_check": stack,
        "best_engine": best_engine_rate(stack),
        "tables": tables,
    }
    print(json.dumps(line), flush=True)


def run_reference(args):
    """The reference arm: the float64 oracle, as it stands, on this host's
    cores (one spawned worker per core), each step a bounded sample of the
    workload: tokens of the n = 1..9 passes through layer 0 of the stack,
    scaled to stack tokens (÷ 26). Rank 0 alone runs it."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    host = OracleHost()
    try:
        host.start_pool()
        t = host.parallel(host.order)                      # 45 token-layers
        budget = min(10.0, 150.0 / max(1, args.steps + args.warmup))
        per_step = max(1, min(2 * len(host.order), int(budget / max(t, 1e-3) * len(host.order))))
        order = (host.order * 2)[:per_step]
        for _ in range(args.warmup):
            host.parallel(order)
        el = sum(host.parallel(order) for _ in range(args.steps)) / args.steps
    finally:
        host.close()
    v = per_step / LAYERS / el
    desc = ("float64 oracle on the host (%d worker processes, one per core): per step, %d "
            "token-layers (tokens of the n=1..9 passes through layer 0 of the stack, with each "
            "pass's routing), counted as %d/26 stack tokens" % (host.procs, per_step, per_step))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 5), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens_per_step": round(per_step / LAYERS, 4)},
        "cpu_baseline": {"kind": "oracle", "cores": host.procs, "sample": desc,
                         "value": round(v, 5), "unit": UNIT},
        "e2e": {"value": round(v, 5), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def run_stack(args):
    """The stack check alone (26 layers), one JSON line."""
    import torch
    from __graft_entry__ import build
    build()
    from moe_expert_layer_warp_gb300 import configs, synth
    from moe_expert_layer_warp_gb300.layer import PassRunner
    w = configs.V2_LITE_STACK
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    layers = [synth.make_layer(w.shape, w.weight_seed + l, dev) for l in range(w.layers)]
    runners = [PassRunner(L, max(w.pass_sizes)) for L in layers]
    print(json.dumps(stack_check(w, runners, dev)), flush=True)


def run_case(args):
    """A small single-layer case for profilers: one layer, a few passes, no
    replicas. Prints the expert call's time inside a graph-replayed pass and
    alone between CUDA events."""
    import torch
    from __graft_entry__ import build
    build()
    from moe_expert_layer_warp_gb300 import api, configs, synth
    from moe_expert_layer_warp_gb300.layer import PassRunner
    wname, eng, n = args.case.split(":")
    w = getattr(configs, CASES[wname])
    n = int(n)
    L = synth.make_layer(w.shape, w.weight_seed, "cuda")
    x = torch.from_numpy(synth.make_pass(w.shape.d, n, w.rhos[-1],
                                         [w.x_seed_base + s for s in range(w.streams)])).cuda()
    R = PassRunner(L, x.shape[0])
    st = torch.cuda.current_stream()
    # the call inside a pass: a CUDA graph of flush (256 MB read), route,
    # union, expert call and combine, against the same graph without the call
    flush = torch.zeros(64 << 20, dtype=torch.float32, device="cuda")
    R.forward(x, eng, st)

    def one(s, with_expert):
        flush.sum()
        if with_expert:
            R.forward(x, eng, s)
        else:
            R.route_union(x, s)
            R.combine(x.shape[0], s)
    ga = capture_graph(lambda s: one(s, True))
    gb = capture_graph(lambda s: one(s, False))
    ta, tb = time_graphs([ga, gb], args.passes)
    # and alone between CUDA events (adds the events' and launch latency)
    ts = []
    for _ in range(args.passes):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        torch.cuda._sleep(SPIN_CYCLES)      # device busy while the host queues the pass
        R.route_union(x, st)
        e[0].record(st)
        R.experts(x, eng, st)
        e[1].record(st)
        R.combine(x.shape[0], st)
        torch.cuda.synchronize()
        ts.append(e[0].elapsed_time(e[1]))
    if api.moe_last_device_error() != api.MOE_OK:
        raise RuntimeError("device error")
    req = requested(R, eng)
    ms = (ta - tb) * 1e3
    ms_ev = statistics.median(ts)
    print(json.dumps({"case": args.case, "tokens": x.shape[0], "engine_ms": round(ms, 4),
                      "requested_bytes": req, "GBs": round(req / ms / 1e6, 1),
                      "engine_ms_events": round(ms_ev, 4),
                      "GBs_events": round(req / ms_ev / 1e6, 1),
                      "union": int(R.union_count.item())}))


def run_sweep(args):
    for line in sweep_workload(args.sweep, None if args.rho is None else [args.rho]):
        print(json.dumps(line), flush=True)


# ------------------------------------------------- DRAM capture and record --
DRAM_RHO = 0.9
DRAM_CALL_WORKLOADS = {"v2lite": ("V2_LITE_STACK", 0), "mixtral": ("MIXTRAL", 0), "v3": ("V3", 0)}


def run_calls(args):
    """For an ncu DRAM capture of the expert calls: one layer of the
    workload (the stack's layer 0 for v2lite) at rho = DRAM_RHO; at each pass
    size one per-slot pass, then one dedup pass. Prints the requested bytes
    of each expert call in launch order, as JSON."""
    import torch
    from __graft_entry__ import build
    build()
    from moe_expert_layer_warp_gb300 import api, configs, synth
    from moe_expert_layer_warp_gb300.layer import PassRunner
    cname, _ = DRAM_CALL_WORKLOADS[args.calls]
    w = getattr(configs, cname)
    L = synth.make_layer(w.shape, w.weight_seed, "cuda")
    R = PassRunner(L, max(w.pass_sizes) * w.streams)
    st = torch.cuda.current_stream()
    calls = []
    for n in w.pass_sizes:
        x = torch.from_numpy(synth.make_pass(w.shape.d, n, DRAM_RHO, [
            w.x_seed_base + 7000 + 13 * s for s in range(w.streams)])).cuda()
        for eng in ("perslot", "dedup"):
            R.forward(x, eng, st)
            torch.cuda.synchronize()
            calls.append({"n": n * w.streams, "engine": eng, "requested": requested(R, eng)})
    if api.moe_last_device_error() != api.MOE_OK:
        raise RuntimeError("device error")
    print(json.dumps({"workload": args.calls, "rho": DRAM_RHO, "calls": calls,
                      "sources_sha256_16": kernel_source_hash()}), flush=True)


def run_dram_record(args):
    """Writes profiles/dram_expert_calls_<workload>.txt from the JSON that
    --calls printed and the ncu csv (dram__bytes_read.sum and
    dram__bytes_write.sum of the expert kernels, one launch per call, in
    launch order) of the same command."""
    import csv
    calls_json, csv_path = args.dram_record
    c = json.load(open(calls_json))
    rows = list(csv.reader(l for l in open(csv_path) if l.startswith('"')))
    head = rows[0]
    ki, mi, vi, ii = (head.index(k) for k in ("Kernel Name", "Metric Name", "Metric Value", "ID"))
    per = {}
    names = {}
    for r in rows[1:]:
        if not re.search(r"expert_(mma|engine)_kernel", r[ki]):
            continue
        per.setdefault(int(r[ii]), 0)
        names[int(r[ii])] = r[ki].split("(")[0].split("::")[-1]
        if r[mi] in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            v = float(r[vi].replace(",", ""))
            unit = r[head.index("Metric Unit")]
            scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}[unit]
            per[int(r[ii])] += v * scale
    ids = sorted(per)
    if len(ids) != len(c["calls"]):
        raise SystemExit("%d expert-kernel launches in the csv, %d calls in the JSON"
                         % (len(ids), len(c["calls"])))
    tab = {"perslot": {}, "dedup": {}}
    for i, call in zip(ids, c["calls"]):
        tab[call["engine"]][call["n"]] = (call["requested"], int(round(per[i])), names[i])
    ns = sorted(tab["perslot"])
    path = dram_record_path(c["workload"])
    with open(path, "w") as f:
        f.write("# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one expert call per\n"
                "# pass size and engine, %s-shaped layer, rho = %s, each call a cold pass of its own\n"
                "# (routing differs from the bench's passes, so bench.py uses the ratio of DRAM bytes\n"
                "# to the pass's unique expert bytes, per engine and n, and scales each of its own\n"
                "# passes' unique bytes by it).\n"
                "# Used only while sources_sha256_16 matches the code of the kernel sources\n"
                "# (bench.kernel_source_hash()).\n#\n"
                "# Command (GB300, after the same command exited 0 without ncu):\n"
                "#   python bench.py --calls %s > calls.json &&\n"
                "#   ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum --clock-control none \\\n"
                "#       -k regex:\"expert_(mma|engine)_kernel\" --csv --log-file dram.csv \\\n"
                "#       python bench.py --calls %s\n"
                "#   python bench.py --dram-record calls.json dram.csv\n"
                "# The two metrics take one ncu pass per launch (nothing is saved or restored).\n#\n"
                "# n  engine   kernel                 requested MB   DRAM MB   DRAM/requested\n"
                % (c["workload"], c["rho"], c["workload"], c["workload"]))
        for eng in ("perslot", "dedup"):
            for n in ns:
                rq, dr, kn = tab[eng][n]
                f.write("# %2d %-8s %-22s %12.1f %9.1f %8.3f\n" % (n, eng, kn, rq / 1e6, dr / 1e6,
                                                                 dr / rq))
        f.write("sources_sha256_16: %s\n" % c["sources_sha256_16"])
        f.write("rho: %s\n" % c["rho"])
        f.write("n: %s\n" % ",".join(str(n) for n in ns))
        for eng in ("perslot", "dedup"):
            f.write("%s_requested: %s\n" % (eng, ",".join(str(tab[eng][n][0]) for n in ns)))
            f.write("%s_dram: %s\n" % (eng, ",".join(str(tab[eng][n][1]) for n in ns)))
    print("wrote", os.path.relpath(path, ROOT))


def main():
    args = parse_args()
    if args.dram_record:
        run_dram_record(args)
    elif args.calls:
        run_calls(args)
    elif args.sweep:
        run_sweep(args)
    elif args.case:
        run_case(args)
    elif args.stack:
        run_stack(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
