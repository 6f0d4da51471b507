"""Host-only checks of the C ABI: the library builds and loads, it exports
every function include/moe_warp.h declares, and bad arguments are rejected on
the host before any launch (these calls touch no GPU)."""
import ctypes
import os
import re

import pytest

from moe_expert_layer_warp_gb300 import api, build
from moe_expert_layer_warp_gb300.configs import ALL, LayerShape, W_BF16

CC_SYNC_INTS = 1 + 512 + 4 * 32   # CUDA-core kernel: job counter + per-entry tile counts
MMA_SYNC_INTS = 1 + 528 + 2 * 4096   # tensor-core kernel: job counter, per-entry tile counts,
                                     # per-phase arrival counts of K pieces
MMA_PART_BYTES = 24 << 20            # tensor-core kernel partial sums (bf16 layers only)
HEADER_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


def _declared():
    names = []
    for h in sorted(os.listdir(HEADER_DIR)):
        if h.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", text,
                                re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return api.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "moe_route" in names and "moe_verify_dedup" in names
    for n in names:
        assert hasattr(lib, n), "libmoewarp.so does not export %s" % n
    assert set(api.EXPORTED) <= set(names)


def test_workspace_bytes_closed_form(lib):
    for w in ALL:
        sh = w.shape
        n = max(w.pass_sizes) * w.streams
        got = api.moe_workspace_bytes(api.make_desc(sh), n)
        a256 = lambda v: (v + 255) // 256 * 256
        hrows = n * sh.top_k + sh.n_shared * n
        want = (a256(n * sh.n_experts * 4) + a256(hrows * sh.inter * 4) + a256(2 * hrows * sh.inter * 2)
                + a256(n * sh.top_k * sh.d * 4) + a256(2 * n * sh.top_k * sh.d * 2)
                + a256(2 * n * sh.d * 2) + a256(n * sh.d * 4) + a256(CC_SYNC_INTS * 4)
                + a256(MMA_SYNC_INTS * 4) + 256
                + (MMA_PART_BYTES if sh.wdtype == W_BF16 else 0))
        assert got == want, w.name


def test_invalid_shapes_are_rejected(lib):
    bad = [LayerShape(2048, 64, 0, 1408, 2, W_BF16),     # k = 0
           LayerShape(2048, 4, 6, 1408, 2, W_BF16),      # k > E
           LayerShape(2048, 300, 6, 1408, 2, W_BF16),    # E > 256
           LayerShape(2048, 64, 6, 1408, 9, W_BF16),     # s > 4
           LayerShape(2000, 64, 6, 1408, 2, W_BF16),     # d not a multiple of 64
           LayerShape(2048, 64, 6, 1408, 2, 7)]          # unknown dtype
    for sh in bad:
        assert api.moe_workspace_bytes(api.make_desc(sh), 4) == 0
    good = api.make_desc(LayerShape(2048, 64, 6, 1408, 2, W_BF16))
    assert api.moe_workspace_bytes(good, 0) == 0        # n < 1
    assert api.moe_workspace_bytes(good, 86) == 0       # n·k > 512
    assert api.moe_workspace_bytes(good, 85) > 0


def test_null_and_misaligned_pointers_return_einval(lib):
    d = api.make_desc(LayerShape(256, 8, 2, 512, 0, 0))
    z = ctypes.c_void_p(0)
    one = ctypes.c_void_p(4096)
    odd = ctypes.c_void_p(4096 + 4)
    st = lib.moe_route(ctypes.byref(d), z, one, 4, one, one, one, 1 << 20, z)
    assert st == api.MOE_EINVAL
    st = lib.moe_route(ctypes.byref(d), one, odd, 4, one, one, one, 1 << 20, z)
    assert st == api.MOE_EINVAL
    st = lib.moe_route(ctypes.byref(d), one, one, 4, one, one, ctypes.c_void_p(4096 + 64),
                       1 << 20, z)   # workspace not 256-byte aligned
    assert st == api.MOE_EINVAL
    st = lib.moe_route(ctypes.byref(d), one, one, 4, one, one, one, 16, z)   # too small
    assert st == api.MOE_EINVAL
    u = api.UnionC()
    assert lib.moe_build_union(ctypes.byref(d), one, 4, ctypes.byref(u), z) == api.MOE_EINVAL
    w = api.LayerWeightsC()
    assert lib.moe_verify_perslot(ctypes.byref(d), ctypes.byref(w), one, 4, one, one, one,
                                  1 << 20, one, z) == api.MOE_EINVAL
    assert lib.moe_verify_dedup(ctypes.byref(d), ctypes.byref(w), one, 4, ctypes.byref(u), one,
                                one, 1 << 20, one, z) == api.MOE_EINVAL
    assert lib.moe_combine(ctypes.byref(d), z, 4, one, z) == api.MOE_EINVAL
    assert lib.moe_combine(ctypes.byref(d), one, 0, one, z) == api.MOE_EINVAL
    # moe_gate: null router, x or logits; misaligned x or logits; n out of range
    assert lib.moe_gate(ctypes.byref(d), z, one, 4, one, z) == api.MOE_EINVAL
    assert lib.moe_gate(ctypes.byref(d), one, z, 4, one, z) == api.MOE_EINVAL
    assert lib.moe_gate(ctypes.byref(d), one, one, 4, z, z) == api.MOE_EINVAL
    assert lib.moe_gate(ctypes.byref(d), one, odd, 4, one, z) == api.MOE_EINVAL
    assert lib.moe_gate(ctypes.byref(d), one, one, 4, ctypes.c_void_p(4096 + 2), z) == api.MOE_EINVAL
    assert lib.moe_gate(ctypes.byref(d), one, one, 0, one, z) == api.MOE_EINVAL


def test_status_strings(lib):
    for s in range(6):
        assert api.status_str(s).startswith("MOE_")


def test_biased_route_rejects_bad_mode_and_misaligned_bias(lib):
    desc = api.make_desc(LayerShape(256, 8, 2, 512, 0, W_BF16))
    one = ctypes.c_void_p(4096)
    ws = ctypes.c_void_p(1 << 20)
    big = 1 << 30
    f = lib.moe_route_biased
    assert f(ctypes.byref(desc), one, one, 2, one, 4, one, one, ws, big, None) == api.MOE_EINVAL
    assert f(ctypes.byref(desc), one, ctypes.c_void_p(4098), 1, one, 4, one, one, ws, big,
             None) == api.MOE_EINVAL


def test_route_union_checks_both_calls_arguments(lib):
    desc = api.make_desc(LayerShape(256, 8, 2, 512, 0, W_BF16))
    one = ctypes.c_void_p(4096)
    ws = ctypes.c_void_p(1 << 20)
    big = 1 << 30
    p = ctypes.c_void_p(8192)
    u = api.UnionC(p, p, p, p, p, p)
    f = lib.moe_route_union
    # the union's outputs must all be given
    empty = api.UnionC()
    assert f(ctypes.byref(desc), one, None, 1, one, 4, one, one, ctypes.byref(empty), ws, big,
             None) == api.MOE_EINVAL
    # the routing checks: mode, bias alignment, null x, n out of range, workspace size
    assert f(ctypes.byref(desc), one, one, 2, one, 4, one, one, ctypes.byref(u), ws, big,
             None) == api.MOE_EINVAL
    assert f(ctypes.byref(desc), one, ctypes.c_void_p(4098), 1, one, 4, one, one,
             ctypes.byref(u), ws, big, None) == api.MOE_EINVAL
    assert f(ctypes.byref(desc), one, None, 1, None, 4, one, one, ctypes.byref(u), ws, big,
             None) == api.MOE_EINVAL
    assert f(ctypes.byref(desc), one, None, 1, one, 0, one, one, ctypes.byref(u), ws, big,
             None) == api.MOE_EINVAL
    assert f(ctypes.byref(desc), one, None, 1, one, 4, one, one, ctypes.byref(u), ws, 16,
             None) == api.MOE_EINVAL
    # byte counters must be 8-byte aligned
    odd = api.UnionC(p, p, p, p, p, ctypes.c_void_p(8196))
    assert f(ctypes.byref(desc), one, None, 1, one, 4, one, one, ctypes.byref(odd), ws, big,
             None) == api.MOE_EINVAL


def test_verify_pass_rejects_bad_engine_and_missing_outputs(lib):
    desc = api.make_desc(LayerShape(256, 8, 2, 512, 0, W_BF16))
    one = ctypes.c_void_p(4096)
    p = ctypes.c_void_p(8192)
    u = api.UnionC(p, p, p, p, p, p)
    w = api.LayerWeightsC()
    f = lib.moe_verify_pass
    args = lambda wref, engine, y_slot, y: (ctypes.byref(desc), wref, None, 1, one, 4, engine, one,
                                           one, ctypes.byref(u), ctypes.c_void_p(1 << 20), 1 << 30,
                                           y_slot, y, None)
    assert f(*args(ctypes.byref(w), 2, one, one)) == api.MOE_EINVAL      # unknown engine
    assert f(*args(ctypes.byref(w), -1, one, one)) == api.MOE_EINVAL
    assert f(*args(None, 0, one, one)) == api.MOE_EINVAL                 # no weights
    assert f(*args(ctypes.byref(w), 1, None, one)) == api.MOE_EINVAL     # no y_slot
    assert f(*args(ctypes.byref(w), 1, one, None)) == api.MOE_EINVAL     # no y
    # the routing's own checks run first: W_g (weights.w_router) is NULL here
    assert f(*args(ctypes.byref(w), 0, one, one)) == api.MOE_EINVAL


def test_noalloc_refusals_each_say_why(lib):
    """Every host-side refusal of moe_verify_dedup_noalloc writes its own
    reason, so a caller never reads one left over from an earlier call."""
    f = lib.moe_verify_dedup_noalloc
    desc = api.make_desc(LayerShape(256, 8, 2, 512, 0, W_BF16))
    one = ctypes.c_void_p(4096)
    p = ctypes.c_void_p(8192)
    u = api.UnionC(p, p, p, p, p, p)
    w = api.LayerWeightsC(one, one, one, one)
    msg = lambda: lib.moe_last_cuda_error_string().decode()
    bad = api.make_desc(LayerShape(256, 8, 9, 512, 0, W_BF16))          # k > E
    assert f(ctypes.byref(bad), ctypes.byref(w), one, 4, ctypes.byref(u), one, one,
             None) == api.MOE_EINVAL
    assert "descriptor" in msg()
    assert f(ctypes.byref(desc), ctypes.byref(w), one, 0, ctypes.byref(u), one, one,
             None) == api.MOE_EINVAL
    assert "pass size" in msg()
    assert f(ctypes.byref(desc), ctypes.byref(api.LayerWeightsC()), one, 4, ctypes.byref(u), one,
             one, None) == api.MOE_EINVAL
    assert "weight" in msg()
    assert f(ctypes.byref(desc), ctypes.byref(w), None, 4, ctypes.byref(u), one, one,
             None) == api.MOE_EINVAL
    assert "x" in msg() and "weight" not in msg()
    assert f(ctypes.byref(desc), ctypes.byref(w), one, 4, ctypes.byref(api.UnionC()), one, one,
             None) == api.MOE_EINVAL
    assert "union" in msg()


def test_noalloc_size_refusal_comes_before_pointer_checks(lib):
    """A pass above the static maximum is refused for its size whatever else
    is wrong with the call (the caller learns first that it needs a
    workspace)."""
    big = api.make_desc(LayerShape(7168, 256, 8, 2048, 1, W_BF16))
    one = ctypes.c_void_p(4096)
    st = lib.moe_verify_dedup_noalloc(ctypes.byref(big), ctypes.byref(api.LayerWeightsC()), one, 64,
                                      ctypes.byref(api.UnionC()), one, one, None)
    assert st == api.MOE_EINVAL
    assert "static maximum" in lib.moe_last_cuda_error_string().decode()
