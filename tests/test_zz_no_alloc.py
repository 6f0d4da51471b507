"""The allocation-free dedup entry point (moe_verify_dedup_noalloc).

Some callers cannot allocate device memory — a plugin whose host framework
owns every GPU buffer, or a serving loop that must not allocate after
start-up — so the library offers the dedup engine with its scratch in a
static device array instead of a caller workspace. This checks, through the
C ABI, that two calls in a row (on different passes, so stale scratch from the
first call would show in the second) give the same slot outputs as
moe_verify_dedup with a workspace, within the tolerance the parity tests use,
and that a pass too large for the static array is refused with a clear error.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from moe_expert_layer_warp_gb300.configs import LayerShape, W_BF16, W_F32

pytestmark = pytest.mark.gpu

CASES = [
    ("v2lite-shape-n9", LayerShape(2048, 64, 6, 1408, 2, W_BF16), 9, 2e-2),
    ("fp32-n5", LayerShape(256, 8, 2, 512, 1, W_F32), 5, 1e-5),
]


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from moe_expert_layer_warp_gb300 import api, build
    build.build()
    return api


@pytest.mark.parametrize("name,shape,n,tol", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_workspace_engine_on_two_calls(lib, name, shape, n, tol):
    from moe_expert_layer_warp_gb300 import synth
    from moe_expert_layer_warp_gb300.layer import PassRunner
    api = lib
    L = synth.make_layer(shape, 41, "cuda")
    R = PassRunner(L, n)
    stream = torch.cuda.current_stream()
    S = shape.top_k + shape.n_shared
    y_na = torch.empty(n * S * shape.d, dtype=torch.float32, device="cuda")
    for call, seed in enumerate((501, 502)):
        x = torch.from_numpy(synth.make_pass(shape.d, n, 0.9, [seed])).cuda()
        R.route(x, stream)
        R.build_union(n, stream)
        R.experts(x, "dedup", stream)                      # existing entry point, workspace
        ref = R.slots(n).clone()
        y_na.fill_(float("nan"))
        api.moe_verify_dedup_noalloc(R.desc, R.wc, x, n, R.u, R.topk_w, y_na, stream)
        assert api.moe_last_device_error() == api.MOE_OK
        got = y_na.view(n, S, shape.d).double().cpu().numpy()
        want = ref.double().cpu().numpy()
        assert np.all(np.isfinite(got)), "call %d left outputs unwritten" % call
        rms = float(np.sqrt(np.mean(want ** 2)))
        err = float(np.max(np.abs(got - want)))
        assert err <= tol * rms, "call %d: max|err| %.3e > %.1e·rms %.3e" % (call, err, tol, rms)


def test_noalloc_rejects_pass_above_static_limit(lib):
    api = lib
    # DeepSeek-V3-shaped layer at 64 tokens: about 68 MB of scratch (routing,
    # activations, gathered rows and the 24 MiB partial-sum region), twice
    # the static array
    big = LayerShape(7168, 256, 8, 2048, 1, W_BF16)
    desc = api.make_desc(big)
    need = api.moe_workspace_bytes(desc, 64)
    assert need > api.moe_noalloc_scratch_limit(), (need, api.moe_noalloc_scratch_limit())
    u = api.UnionC()
    w = api.LayerWeightsC()
    one = ctypes.c_void_p(4096)
    st = api.load().moe_verify_dedup_noalloc(ctypes.byref(desc), ctypes.byref(w), one, 64,
                                             ctypes.byref(u), one, one, None)
    assert st == api.MOE_EINVAL
    msg = api.load().moe_last_cuda_error_string().decode()
    assert "static maximum" in msg and str(need) in msg
