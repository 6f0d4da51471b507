"""Failure detection without faulting the GPU.

Host side: bad arguments are rejected before any launch (tests/test_abi.py).
Device side: every wait in the kernels is bounded; here a diagnostic kernel
waits on an mbarrier that nothing arrives on, with a 2 ms limit. The test
checks that the timeout is reported through moe_last_device_error, that the
error word is cleared after it is read, and that the context still runs a
full verification pass correctly afterwards.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from moe_expert_layer_warp_gb300 import api, build, configs, synth
    from moe_expert_layer_warp_gb300.layer import PassRunner
    from oracle import oracle
    build.build()
    assert api.moe_last_device_error() == api.MOE_OK
    api.moe_diag_bounded_wait(2000)
    assert api.moe_last_device_error() == api.MOE_ETIMEOUT
    assert api.moe_last_device_error() == api.MOE_OK          # the word was cleared
    w = configs.TINY
    L = synth.make_layer(w.shape, w.weight_seed, "cuda")
    x_np = synth.make_pass(w.shape.d, 4, 0.9, [w.x_seed_base])
    y = PassRunner(L, 4).forward(torch.from_numpy(x_np).cuda(), "dedup").cpu().numpy()
    assert api.moe_last_device_error() == api.MOE_OK
    r = oracle.route(x_np, L.w_router.cpu().numpy(), w.shape.top_k)
    y_o = oracle.moe_tokens(x_np, r["idx"], r["w"], synth.weights_numpy(L.w_gate),
                            synth.weights_numpy(L.w_up), synth.weights_numpy(L.w_down))
    assert np.max(np.abs(y - y_o)) <= 1e-5 * np.sqrt(np.mean(y_o ** 2))


def test_bounded_wait_rejects_limits_out_of_range():
    from moe_expert_layer_warp_gb300 import api, build
    build.build()
    lib = api.load()
    assert lib.moe_diag_bounded_wait(0, None) == api.MOE_EINVAL
    assert lib.moe_diag_bounded_wait(2_000_000, None) == api.MOE_EINVAL


def test_expert_index_out_of_range_is_reported_not_read():
    """A per-slot call given an expert index outside [0, E) (a caller's bug):
    the kernel's own check records it and reads expert 0 instead, so nothing
    is read out of bounds; moe_last_device_error reports MOE_EDEVICE, and the
    next pass is correct."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from moe_expert_layer_warp_gb300 import api, build, synth
    from moe_expert_layer_warp_gb300.configs import LayerShape, W_BF16
    from moe_expert_layer_warp_gb300.layer import PassRunner
    from oracle import oracle
    build.build()
    assert api.moe_last_device_error() == api.MOE_OK
    shape = LayerShape(576, 16, 4, 320, 1, W_BF16)
    L = synth.make_layer(shape, 13, "cuda")
    n = 5
    R = PassRunner(L, n)
    x_np = synth.make_pass(shape.d, n, 0.9, [77])
    x = torch.from_numpy(x_np).cuda()
    R.route_union(x)
    R.topk_idx[3] = shape.n_experts + 83                     # not an expert of this layer
    R.experts(x, "perslot")
    assert api.moe_last_device_error() == api.MOE_EDEVICE
    assert api.moe_last_device_error() == api.MOE_OK          # the word was cleared
    y = R.forward(x, "perslot").cpu().numpy()
    assert api.moe_last_device_error() == api.MOE_OK
    r = oracle.route(x_np, L.w_router.cpu().numpy(), shape.top_k)
    y_o = oracle.moe_tokens(x_np, r["idx"], r["w"], synth.weights_numpy(L.w_gate),
                            synth.weights_numpy(L.w_up), synth.weights_numpy(L.w_down),
                            synth.weights_numpy(L.ws_gate), synth.weights_numpy(L.ws_up),
                            synth.weights_numpy(L.ws_down))
    assert np.max(np.abs(y - y_o)) <= 2e-2 * np.sqrt(np.mean(y_o ** 2))
