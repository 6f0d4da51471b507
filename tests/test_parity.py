"""GPU parity: the CUDA path through the C ABI against the float64 oracle on
the same seeded inputs.

Small layers are compared on every output element; they span several row
tiles and K stages with ragged K tails, groups split beyond 8 tokens, k = E,
k = 1, the largest pass (n·k = 512), the most shared experts (4, split into
sub-groups past 32 tokens), the most experts and largest top-k (256, 16),
the smallest dimensions (d = I = 64), n = 1 and identical tokens. The five
workload shapes run at full size in the launch configuration the benchmark
times and are compared with the oracle on every token — the V2-Lite layer at
every pass size, two layers of the 26-layer stack, the Mixtral layer at
n = 1, 2, 8 and 16 (rho = 0) and at n = 5 and 12 (rho = 0.99, large dedup
groups), and the V3 layer's 64 tokens — except one Mixtral pass (n = 16,
rho = 0.9), sampled on its last token (routing, union and bytes on every
token).
Both engines are checked, and against each other.
"""
import gc

import numpy as np
import pytest
import torch

from moe_expert_layer_warp_gb300 import configs, synth
from moe_expert_layer_warp_gb300.configs import LayerShape, W_BF16, W_F32
from moe_expert_layer_warp_gb300.layer import DEDUP, PERSLOT, PassRunner
from oracle import oracle
from tests import parity_util as pu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from moe_expert_layer_warp_gb300 import api, build
    build.build()
    api.load()
    yield
    gc.collect()
    torch.cuda.empty_cache()


def run_both(L, x_np, runner=None):
    """Runs the pass through both engines; returns host copies of everything."""
    dev = L.device
    n = x_np.shape[0]
    R = runner or PassRunner(L, n)
    x = torch.from_numpy(x_np).to(dev)
    out = {}
    y_ps = R.forward(x, PERSLOT).cpu().numpy()
    slots_ps = R.slots(n).cpu().numpy()
    idx, w = (t.cpu().numpy() for t in R.routing(n))
    u = {k: (v.cpu().numpy() if torch.is_tensor(v) else v) for k, v in R.union(n).items()}
    y_dd = R.forward(x, DEDUP).cpu().numpy()
    slots_dd = R.slots(n).cpu().numpy()
    # the pass with the combine fused into the expert kernel: the same y, bit for bit
    for eng, y_ref in ((PERSLOT, y_ps), (DEDUP, y_dd)):
        R.y.fill_(float("nan"))
        y_f = R.forward(x, eng, fused=True).cpu().numpy()
        np.testing.assert_array_equal(y_f.view(np.uint32), y_ref.view(np.uint32),
                                      err_msg="fused combine, %s" % eng)
    from moe_expert_layer_warp_gb300 import api
    assert api.moe_last_device_error() == api.MOE_OK
    out.update(y_ps=y_ps, y_dd=y_dd, slots_ps=slots_ps, slots_dd=slots_dd, idx=idx, w=w, u=u)
    return out


def check_pass(L, x_np, tokens=None, runner=None):
    sh = L.shape
    g = run_both(L, x_np, runner)
    orc = oracle.route(x_np, L.w_router.cpu().numpy(), sh.top_k)
    amb = pu.check_routing(g["idx"], g["w"], orc, sh.d)
    assert amb <= max(1, x_np.shape[0] // 20), "too many tie-ambiguous tokens: %d" % amb
    n = x_np.shape[0]
    if amb == 0:
        ou = oracle.union(orc["idx"], sh.n_experts)
        u = g["u"]
        assert u["count"] == ou["count"]
        np.testing.assert_array_equal(u["union_ids"], ou["union_ids"])
        np.testing.assert_array_equal(u["offsets"], ou["offsets"])
        np.testing.assert_array_equal(u["pair_tok"], ou["pair_tok"])
        np.testing.assert_array_equal(u["pair_slot"], ou["pair_slot"])
        b = oracle.bytes_per_pass(sh.d, sh.inter, sh.top_k, sh.n_shared, n, sh.wdtype,
                                  ou["count"])
        assert [int(v) for v in u["bytes"]] == b
    toks = list(range(n)) if tokens is None else list(tokens)
    y_o, slots_o = pu.oracle_outputs(L, x_np, orc, toks)
    tol = pu.y_tol(sh)
    pu.assert_close_rms(g["y_ps"][toks], y_o, tol, "per-slot y")
    pu.assert_close_rms(g["y_dd"][toks], y_o, tol, "dedup y")
    pu.assert_close_rms(g["slots_ps"][toks], slots_o, tol, "per-slot slots", scale=y_o)
    pu.assert_close_rms(g["slots_dd"][toks], slots_o, tol, "dedup slots", scale=y_o)
    ref = g["y_ps"].astype(np.float64)
    pu.assert_close_rms(g["y_dd"], ref, tol, "dedup vs per-slot")
    return g


SMALL = [
    ("f32-ragged", LayerShape(192, 6, 3, 256, 1, W_F32), [1, 2, 7]),
    ("bf16-ragged", LayerShape(576, 16, 4, 320, 1, W_BF16), [1, 5, 16, 33]),
    ("k-equals-E", LayerShape(128, 4, 4, 128, 0, W_BF16), [3]),
    ("top-1", LayerShape(128, 8, 1, 64, 2, W_F32), [5]),
    ("max-pairs", LayerShape(256, 32, 4, 128, 1, W_BF16), [128]),
    ("max-shared", LayerShape(256, 16, 2, 192, 4, W_BF16), [1, 40]),
    ("max-experts-top16", LayerShape(128, 256, 16, 64, 1, W_F32), [3, 32]),
    ("min-dims", LayerShape(64, 8, 2, 64, 1, W_BF16), [1, 9]),
]


@pytest.mark.parametrize("name,shape,ns", SMALL, ids=[s[0] for s in SMALL])
def test_small_layers_every_element(name, shape, ns):
    L = synth.make_layer(shape, 17, "cuda")
    R = PassRunner(L, max(ns))
    for n in ns:
        x = synth.make_pass(shape.d, n, 0.9, [123 + n])
        check_pass(L, x, runner=R)


def _rearranged(L, order):
    """Layer L with its W_gate / W_up storage rearranged: "up-below-gate"
    puts both in one buffer, W_up first (the CUDA-core kernel then reads the
    pair through one map based at W_up); "gate-is-up" passes one array as
    both (a distance of zero: the kernel loads the two as separate boxes)."""
    def arrange(g, u):
        if g is None:
            return None, None
        if order == "up-below-gate":
            buf = torch.empty((2,) + tuple(g.shape), dtype=g.dtype, device=g.device)
            buf[0].copy_(u)
            buf[1].copy_(g)
            return buf[1], buf[0]
        return g, g
    wg, wu = arrange(L.w_gate, L.w_up)
    sg, su = arrange(L.ws_gate, L.ws_up)
    return synth.LayerWeights(L.shape, L.w_router, wg, wu, L.w_down, sg, su, L.ws_down)


@pytest.mark.parametrize("order", ["up-below-gate", "gate-is-up"])
@pytest.mark.parametrize("shape", [LayerShape(192, 6, 3, 256, 1, W_F32),
                                   LayerShape(576, 16, 4, 320, 2, W_BF16)],
                         ids=["f32", "bf16"])
def test_gate_up_storage(order, shape):
    """Where W_gate and W_up lie relative to each other decides how the
    CUDA-core kernel loads them; every arrangement gives the oracle's result."""
    L = _rearranged(synth.make_layer(shape, 29, "cuda"), order)
    R = PassRunner(L, 5)
    for n in (1, 5):
        check_pass(L, synth.make_pass(shape.d, n, 0.9, [321 + n]), runner=R)


def test_tiny_workload_every_element():
    w = configs.TINY
    L = synth.make_layer(w.shape, w.weight_seed, "cuda")
    x = synth.make_pass(w.shape.d, w.pass_sizes[0], w.rhos[0], [w.x_seed_base])
    check_pass(L, x)


@pytest.mark.parametrize("bias_in_weights", [True, False], ids=["bias-in-weights", "selection-only"])
def test_biased_routing_and_layer(bias_in_weights):
    """moe_route_biased (DeepSeek-style routing bias) against the oracle:
    certified tokens bit-exact, weights to 1e-5, and the layer output of both
    engines with that routing within the bf16 tolerance."""
    shape = LayerShape(512, 32, 4, 256, 1, W_BF16)
    L = synth.make_layer(shape, 41, "cuda")
    n = 17
    x = synth.make_pass(shape.d, n, 0.5, [91])
    wr = L.w_router.cpu().numpy()
    spread = float(np.std(oracle.gate_logits(x, wr)[0]))
    bias = (np.random.default_rng(7).standard_normal(shape.n_experts) * spread).astype(np.float32)
    R = PassRunner(L, n, bias=torch.from_numpy(bias).cuda(), bias_in_weights=bias_in_weights)
    xt = torch.from_numpy(x).cuda()
    y_ps = R.forward(xt, PERSLOT).cpu().numpy()
    idx, w = (t.cpu().numpy() for t in R.routing(n))
    y_dd = R.forward(xt, DEDUP).cpu().numpy()
    from moe_expert_layer_warp_gb300 import api
    assert api.moe_last_device_error() == api.MOE_OK
    orc = oracle.route(x, wr, shape.top_k, bias.astype(np.float64), bias_in_weights)
    amb = pu.check_routing(idx, w, orc, shape.d, bias.astype(np.float64))
    assert amb <= 1
    toks = [t for t in range(n) if np.array_equal(idx[t], orc["idx"][t])]
    y_o, _ = pu.oracle_outputs(L, x, orc, toks)
    pu.assert_close_rms(y_ps[toks], y_o, pu.y_tol(shape), "biased per-slot y")
    pu.assert_close_rms(y_dd[toks], y_o, pu.y_tol(shape), "biased dedup y")


@pytest.mark.parametrize("shape,n,bias_mode", [
    (LayerShape(2048, 64, 6, 1408, 2, W_BF16), 9, None),
    (LayerShape(256, 32, 4, 128, 1, W_BF16), 128, None),        # n·k = 512, four token rounds
    (LayerShape(128, 256, 16, 64, 1, W_F32), 32, None),         # E = 256, k = 16
    (LayerShape(512, 32, 4, 256, 1, W_BF16), 17, 1),
    (LayerShape(512, 32, 4, 256, 1, W_BF16), 17, 0),
    (LayerShape(128, 8, 1, 64, 2, W_F32), 1, None),
], ids=["v2lite-n9", "max-pairs", "max-experts-top16", "bias-in-weights", "selection-only",
        "top1-n1"])
def test_route_union_equals_separate_calls(shape, n, bias_mode):
    """moe_route_union (top-k inside the union's CTA) against moe_route or
    moe_route_biased followed by moe_build_union: every routing and union
    output bit for bit, on the same inputs."""
    L = synth.make_layer(shape, 57, "cuda")
    x = torch.from_numpy(synth.make_pass(shape.d, n, 0.7, [123])).cuda()
    bias = None
    if bias_mode is not None:
        bias = torch.from_numpy(np.random.default_rng(3).standard_normal(shape.n_experts)
                                .astype(np.float32) * 0.05).cuda()
    R = PassRunner(L, n, bias=bias, bias_in_weights=bool(bias_mode))

    def outputs():
        idx, w = (t.cpu().numpy().copy() for t in R.routing(n))
        u = {k: (v.cpu().numpy().copy() if torch.is_tensor(v) else v)
             for k, v in R.union(n).items()}
        return idx, w, u

    for t in (R.topk_idx, R.topk_w, R.union_ids, R.offsets, R.pair_tok, R.pair_slot):
        t.fill_(-7)
    R.route(x)
    R.build_union(n)
    a = outputs()
    for t in (R.topk_idx, R.topk_w, R.union_ids, R.offsets, R.pair_tok, R.pair_slot):
        t.fill_(-7)
    R.route_union(x)
    b = outputs()
    from moe_expert_layer_warp_gb300 import api
    assert api.moe_last_device_error() == api.MOE_OK
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1].view(np.uint32), b[1].view(np.uint32))
    assert a[2]["count"] == b[2]["count"]
    for key in ("union_ids", "offsets", "pair_tok", "pair_slot", "bytes"):
        np.testing.assert_array_equal(a[2][key], b[2][key])


@pytest.mark.parametrize("shape", [LayerShape(256, 64, 6, 128, 1, W_BF16),
                                   LayerShape(128, 256, 16, 64, 1, W_F32)],
                         ids=["E64-top6", "E256-top16"])
def test_exact_ties_go_to_the_lower_index(shape):
    """Experts 2i and 2i+1 get identical gate rows, so their logits are
    bitwise equal: the selection takes the lower index first and every
    selected odd expert follows its even twin, as the oracle orders them."""
    L = synth.make_layer(shape, 61, "cuda")
    L.w_router[1::2] = L.w_router[0::2]
    n = 16
    x = synth.make_pass(shape.d, n, 0.0, [5])
    R = PassRunner(L, n)
    R.route_union(torch.from_numpy(x).cuda())
    idx, w = (t.cpu().numpy() for t in R.routing(n))
    from moe_expert_layer_warp_gb300 import api
    assert api.moe_last_device_error() == api.MOE_OK
    orc = oracle.route(x, L.w_router.cpu().numpy(), shape.top_k)
    np.testing.assert_array_equal(idx, orc["idx"])
    for t in range(n):
        for j, e in enumerate(idx[t]):
            if e % 2 == 1:
                assert j > 0 and idx[t][j - 1] == e - 1, (t, idx[t])
    np.testing.assert_allclose(w, orc["w"], rtol=0, atol=1e-5)
    pairs = w.reshape(n, shape.top_k // 2, 2)
    np.testing.assert_array_equal(pairs[:, :, 0], pairs[:, :, 1])


@pytest.mark.parametrize("shape", [LayerShape(576, 16, 4, 320, 1, W_BF16),
                                   LayerShape(192, 6, 3, 256, 2, W_F32)], ids=["bf16", "f32"])
@pytest.mark.parametrize("bias_mode", [None, 0], ids=["plain", "selection-only-bias"])
@pytest.mark.parametrize("fused", [False, True], ids=["verify-pass", "verify-pass-fused"])
def test_verify_pass_equals_single_calls(bias_mode, shape, fused):
    """forward() — one moe_verify_pass call, or one moe_verify_pass_fused
    call (the combine as the expert kernel's last phase) — against
    moe_route_union, moe_verify_* and moe_combine made one by one: y, slot
    outputs, the selection and its weights, and the union bit for bit, for
    both engines."""
    L = synth.make_layer(shape, 71, "cuda")
    n = 11
    x = torch.from_numpy(synth.make_pass(shape.d, n, 0.9, [19])).cuda()
    bias = None
    if bias_mode is not None:
        bias = torch.from_numpy(np.random.default_rng(4).standard_normal(shape.n_experts)
                                .astype(np.float32) * 0.05).cuda()
    R = PassRunner(L, n, bias=bias, bias_in_weights=bool(bias_mode))

    def poison_routing():
        for t in (R.topk_idx, R.pair_tok, R.pair_slot, R.union_ids, R.offsets, R.union_count):
            t.fill_(-7)
        R.topk_w.fill_(float("nan"))
        R.bytes.fill_(-7)

    for eng in (PERSLOT, DEDUP):
        R.y.fill_(float("nan"))     # an element the fused combine missed would stay NaN
        poison_routing()            # and so would routing outputs the pass did not write
        y1 = R.forward(x, eng, fused=fused).cpu().numpy().copy()
        s1 = R.slots(n).cpu().numpy().copy()
        i1 = R.routing(n)[0].cpu().numpy().copy()
        w1 = R.routing(n)[1].cpu().numpy().copy()
        u1 = {k: (v.cpu().numpy().copy() if torch.is_tensor(v) else v)
              for k, v in R.union(n).items()}
        R.y.fill_(-1.0)
        R.y_slot.fill_(-1.0)
        poison_routing()
        R.route_union(x)
        R.experts(x, eng)
        R.combine(n)
        y2 = R.y[: n * shape.d].view(n, shape.d).cpu().numpy()
        from moe_expert_layer_warp_gb300 import api
        assert api.moe_last_device_error() == api.MOE_OK
        np.testing.assert_array_equal(y1.view(np.uint32), y2.view(np.uint32))
        np.testing.assert_array_equal(s1.view(np.uint32), R.slots(n).cpu().numpy().view(np.uint32))
        np.testing.assert_array_equal(i1, R.routing(n)[0].cpu().numpy())
        np.testing.assert_array_equal(w1.view(np.uint32),
                                      R.routing(n)[1].cpu().numpy().view(np.uint32))
        u2 = R.union(n)
        assert u1["count"] == u2["count"]
        for key in ("union_ids", "offsets", "pair_tok", "pair_slot", "bytes"):
            np.testing.assert_array_equal(u1[key], u2[key].cpu().numpy(), err_msg=key)


@pytest.mark.parametrize("name,shape,ns", [SMALL[0], SMALL[1], SMALL[6]],
                         ids=[SMALL[0][0], SMALL[1][0], SMALL[6][0]])
def test_gate_logits_within_certified_bound(name, shape, ns):
    """moe_gate (the gate GEMV alone) against the oracle's float64 logits:
    every logit within the certified error bound of the compensated fp32
    dot, and bit for bit the logits moe_route_union leaves in the workspace
    (the same kernel)."""
    L = synth.make_layer(shape, 23, "cuda")
    R = PassRunner(L, max(ns))
    E = shape.n_experts
    for n in ns:
        x_np = synth.make_pass(shape.d, n, 0.5, [31 + n])
        x = torch.from_numpy(x_np).cuda()
        R.logits.fill_(float("nan"))
        R.gate(x)
        got = R.logits[: n * E].view(n, E).cpu().numpy().astype(np.float64)
        orc = oracle.route(x_np, L.w_router.cpu().numpy(), shape.top_k)
        bound = pu.logit_error_bound(orc, shape.d)
        assert np.all(np.abs(got - orc["logits"]) <= bound), "n=%d" % n
        R.route_union(x)
        ws = R.workspace[: n * E * 4].view(torch.float32).view(n, E).cpu().numpy()
        np.testing.assert_array_equal(got.astype(np.float32).view(np.uint32), ws.view(np.uint32))


def test_identical_tokens_select_k_experts():
    shape = LayerShape(512, 32, 4, 256, 1, W_BF16)
    L = synth.make_layer(shape, 5, "cuda")
    x = np.repeat(synth.make_pass(512, 1, 0.0, [3]), 9, axis=0)
    g = check_pass(L, x)
    assert g["u"]["count"] == 4


def test_repeated_runs_are_bitwise_identical():
    shape = LayerShape(576, 16, 4, 320, 1, W_BF16)
    L = synth.make_layer(shape, 29, "cuda")
    x = synth.make_pass(576, 11, 0.9, [77])
    a = run_both(L, x)
    b = run_both(L, x)
    for key in ("y_ps", "y_dd", "idx", "w"):
        np.testing.assert_array_equal(a[key], b[key])


def _workload_pass(w, n, rho, p):
    seeds = [w.x_seed_base + w.streams * p + s for s in range(w.streams)]
    return synth.make_pass(w.shape.d, n, rho, seeds)


def test_v2_lite_layer_full_size():
    """Every pass size, every token."""
    w = configs.V2_LITE
    L = synth.make_layer(w.shape, w.weight_seed, "cuda")
    R = PassRunner(L, max(w.pass_sizes))
    for n in w.pass_sizes:
        x = _workload_pass(w, n, w.rhos[0], 0)
        check_pass(L, x, runner=R)
    del L, R
    torch.cuda.empty_cache()


def test_mixtral_layer_full_size():
    w = configs.MIXTRAL
    L = synth.make_layer(w.shape, w.weight_seed, "cuda")
    R = PassRunner(L, max(w.pass_sizes))
    # n = 16 at rho = 0 (the most distinct experts) and n <= 8 on every
    # token; n = 16 at rho = 0.9 on its last token; n = 5 and 12 at rho = 0.99
    # (nearly identical tokens: dedup groups of five and twelve tokens on the
    # tensor cores) on every token
    for n, rho in [(1, 0.9), (2, 0.0), (8, 0.5), (16, 0.9), (16, 0.0), (5, 0.99), (12, 0.99)]:
        x = _workload_pass(w, n, rho, 0)
        check_pass(L, x, tokens=[n - 1] if (n, rho) == (16, 0.9) else None, runner=R)
    del L, R
    torch.cuda.empty_cache()


def test_v3_layer_full_size():
    w = configs.V3
    L = synth.make_layer(w.shape, w.weight_seed, "cuda")
    x = _workload_pass(w, w.pass_sizes[0], w.rhos[0], 0)
    check_pass(L, x)     # all 64 tokens
    del L
    torch.cuda.empty_cache()


def test_v2_lite_stack_layers_full_size():
    """Two layers of the 26-layer stack (first and last seeds), each on the
    same pass, as the stack runs them."""
    w = configs.V2_LITE_STACK
    for layer in (0, w.layers - 1):
        L = synth.make_layer(w.shape, w.weight_seed + layer, "cuda")
        x = _workload_pass(w, 9, 0.99, 0)
        check_pass(L, x)
        del L
        torch.cuda.empty_cache()


@pytest.mark.parametrize("shape,ns", [(LayerShape(576, 16, 4, 320, 1, W_BF16), [5, 16]),
                                      (LayerShape(192, 6, 3, 256, 1, W_F32), [7]),
                                      (LayerShape(2048, 64, 6, 1408, 2, W_BF16), [9])],
                         ids=["bf16-ragged", "f32-ragged", "v2-lite"])
def test_pass_reads_nothing_stale_from_the_workspace(shape, ns):
    """A pass writes every workspace byte it reads (counters, converted and
    gathered rows, activations, partial sums) before reading it: the same
    pass over a workspace of zeros and over one of 0xFF bytes (NaN as float,
    -1 as int), with y_slot and y set to NaN, gives the same y bit for bit,
    through both engines, with the combine separate and fused."""
    L = synth.make_layer(shape, 29, "cuda")
    R = PassRunner(L, max(ns))
    for n in ns:
        x = torch.from_numpy(synth.make_pass(shape.d, n, 0.9, [431 + n])).cuda()
        for eng in (PERSLOT, DEDUP):
            for fused in (False, True):
                ys = []
                for fill in (0, 255):
                    R.workspace.fill_(fill)
                    R.y_slot.fill_(float("nan"))
                    R.y.fill_(float("nan"))
                    ys.append(R.forward(x, eng, fused=fused).cpu().numpy().copy())
                np.testing.assert_array_equal(ys[1].view(np.uint32), ys[0].view(np.uint32),
                                              err_msg="n=%d %s fused=%s" % (n, eng, fused))
                assert np.all(np.isfinite(ys[0]))
    from moe_expert_layer_warp_gb300 import api
    assert api.moe_last_device_error() == api.MOE_OK
    del L, R
    torch.cuda.empty_cache()


@pytest.mark.parametrize("min_m", ["1000", "1", "3"],
                         ids=["cuda-core-only", "tensor-core-only", "both-kernels-in-one-call"])
def test_small_layers_on_each_expert_kernel(min_m):
    """bf16 calls pick one expert kernel by size; MOE_MMA_MIN_M (read once per
    process, hence a child process) forces every group of the same small
    layers onto the CUDA-core kernel (1000) or the tensor-core kernel (1),
    cutting tiles along K wherever they are few, or splits one call's groups
    between the two kernels by size (3: groups of three or more tokens on
    the tensor cores), so that both kernels add to the same fused-combine
    counts."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, MOE_MMA_MIN_M=min_m)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "tests/test_parity.py::test_small_layers_every_element",
                        "tests/test_parity.py::test_gate_up_storage",
                        "tests/test_parity.py::test_identical_tokens_select_k_experts",
                        "tests/test_parity.py::test_repeated_runs_are_bitwise_identical",
                        "tests/test_parity.py::test_verify_pass_equals_single_calls",
                        "tests/test_parity.py::test_pass_reads_nothing_stale_from_the_workspace"],
                       cwd=root, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
