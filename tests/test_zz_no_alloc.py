"""moe_router_noalloc: the router for callers that cannot allocate device
memory (it uses the library's static device scratch instead of a workspace).

Its results must equal those of moe_router run with a caller-provided
workspace -- the same kernels on the same inputs -- on two calls in a row
(the second call finds the first call's contents in the shared scratch).
Collected last on purpose, so a run that stops at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from _gpu_common import TOL_WEIGHTS, lib, need_gpu, rel_max_err, workspace

pytestmark = pytest.mark.gpu


def _reference(fgs, cfg, T, g):
    ws, nws = workspace(cfg, T)
    idx = torch.empty((T, cfg.K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, cfg.K), dtype=torch.float32, device="cuda")
    fgs.moe_router(cfg, T, g["x"], g["W_r"], g["bias"], idx, w, ws, nws)
    assert fgs.moe_get_device_status(ws) == 0
    return idx.cpu().numpy(), w.cpu().numpy()


def _noalloc(fgs, cfg, T, g):
    idx = torch.full((T, cfg.K), -1, dtype=torch.int32, device="cuda")
    w = torch.full((T, cfg.K), -1.0, dtype=torch.float32, device="cuda")
    # straight through the C ABI
    st = fgs.lib.moe_router_noalloc(ctypes.byref(cfg), T, g["x"].data_ptr(), g["W_r"].data_ptr(),
                                    g["bias"].data_ptr(), idx.data_ptr(), w.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream)
    assert st == 0, fgs.moe_last_error_detail()
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy()


def test_noalloc_router_matches_workspace_router_twice():
    need_gpu()
    fgs = lib()
    cases = [
        synth.shape("k2_router"),                                        # T = 4096, E = 384
        synth.custom(name="grouped", T=300, d_model=7168, E_routed=384, K=8, n_group=8,
                     topk_group=4, router_only=True, x_dist="clusters32"),
    ]
    for shape in cases:  # two calls in a row on the shared scratch
        g = synth.generate(shape, device="cuda", weights=False)
        cfg = fgs.config(shape, d_ff=0)
        T = g["x"].shape[0]
        ref_idx, ref_w = _reference(fgs, cfg, T, g)
        got_idx, got_w = _noalloc(fgs, cfg, T, g)
        np.testing.assert_array_equal(got_idx, ref_idx)
        assert rel_max_err(got_w, ref_w) <= TOL_WEIGHTS


@pytest.mark.parametrize("name,T", [("k2_router", 9000), ("k3_latent", 2048), ("k3_latent", 4096)])
def test_noalloc_router_with_fewer_k_parts(name, T):
    """Sizes where moe_router's own count of K parts would overflow the
    static scratch: the call runs with fewer parts, so its logits are summed
    in another grouping.  On every token whose selection margin (oracle, fp64)
    exceeds the fp32 error of the logits both calls select the oracle's
    experts; the weights agree within the gate-weight tolerance; two calls
    in a row return the same result."""
    need_gpu()
    fgs = lib()
    import oracle
    from _gpu_common import GAP_MIN, by_expert, np64
    base = synth.shape(name)
    shape = synth.custom(name=f"{name}_T{T}", T=T, d_model=base.d_model, E_routed=base.E_routed,
                         K=base.K, n_group=base.n_group, topk_group=base.topk_group,
                         bias_range=base.bias_range, router_only=True)
    g = synth.generate(shape, device="cuda", weights=False)
    cfg = fgs.config(shape, d_ff=0)
    ref_idx, ref_w = _reference(fgs, cfg, T, g)
    got_idx, got_w = _noalloc(fgs, cfg, T, g)
    again_idx, again_w = _noalloc(fgs, cfg, T, g)
    np.testing.assert_array_equal(again_idx, got_idx)
    np.testing.assert_array_equal(again_w, got_w)
    r = oracle.router_from_x(np64(g["x"]), np64(g["W_r"]), g["bias"].cpu().numpy(), shape.K,
                             shape.n_group, shape.topk_group)
    clear = r["gap"] > GAP_MIN
    assert clear.mean() > 0.9
    want = by_expert(r["idx"])[clear]
    np.testing.assert_array_equal(by_expert(got_idx)[clear], want)
    np.testing.assert_array_equal(by_expert(ref_idx)[clear], want)
    same = (by_expert(got_idx) == by_expert(ref_idx)).all(axis=1)
    assert rel_max_err(by_expert(got_idx, got_w)[1][same], by_expert(ref_idx, ref_w)[1][same]) \
        <= TOL_WEIGHTS


def test_noalloc_router_rejects_oversized_problems():
    need_gpu()
    fgs = lib()
    shape = synth.shape("k3_latent")
    cfg = fgs.config(shape, d_ff=0)
    T = 8192  # E = 896: above the T <= 7972 bound
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    st = fgs.lib.moe_router_noalloc(ctypes.byref(cfg), T, dummy.data_ptr(), dummy.data_ptr(),
                                    dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), None)
    assert st == 4  # MOE_ERR_WORKSPACE, returned before anything is enqueued
    assert "static scratch" in fgs.moe_last_error_detail()
