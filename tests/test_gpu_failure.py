"""Failure detection on the GPU without a fault: one of the library's
bounded device waits is made to run out (a barrier nothing arrives at), the
status word reports MOE_ERR_TIMEOUT, and the same context then runs a layer
forward that matches the oracle."""
import time

import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu_common import TOL_BF16, by_expert, lib, need_gpu, np64, rel_max_err, workspace

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_context_stays_usable():
    need_gpu()
    fgs = lib()
    shape = synth.custom(name="after_timeout", T=64, d_model=256, E_routed=16, K=4, E_shared=1,
                         d_ff=128, d_ff_shared=128)
    cfg = fgs.config(shape)
    ws, nws = workspace(cfg, shape.T)
    assert fgs.moe_get_device_status(ws) == 0
    t0 = time.time()
    fgs.moe_selftest_bounded_wait(ws)
    assert fgs.moe_get_device_status(ws) == 6  # MOE_ERR_TIMEOUT (reading clears it)
    elapsed = time.time() - t0
    assert 1.5 < elapsed < 30.0, elapsed       # the 2 s limit, not a hang
    assert fgs.moe_get_device_status(ws) == 0

    g = synth.generate(shape, device="cuda")
    y = torch.empty((shape.T, shape.d_model), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((shape.T, shape.K), dtype=torch.int32, device="cuda")
    fgs.moe_layer_forward(cfg, shape.T, g["x"], g["W_r"], g["bias"], g["W_gate_up"], g["W_down"],
                          g["Ws_gate_up"], g["Ws_down"], None, None, y, idx, None, None, ws, nws)
    assert fgs.moe_get_device_status(ws) == 0
    f64 = lambda t: t.detach().cpu().to(torch.float64).numpy()  # noqa: E731
    ref = oracle.moe_layer_tokens(f64(g["x"]), f64(g["W_r"]), g["bias"].cpu().numpy(),
                                  g["W_gate_up"], g["W_down"], g["Ws_gate_up"], g["Ws_down"],
                                  shape.K, to_f64=f64)
    got_set = by_expert(idx.cpu().numpy())
    ref_set = by_expert(ref["idx"])
    clear = ref["gap"] > 1e-5
    np.testing.assert_array_equal(got_set[clear], ref_set[clear])
    same = (got_set == ref_set).all(axis=1)
    assert rel_max_err(np64(y)[same], ref["y"][same]) <= TOL_BF16


def test_selftest_needs_a_workspace():
    need_gpu()
    fgs = lib()
    with pytest.raises(fgs.MoeError) as ei:
        fgs.moe_selftest_bounded_wait(None)
    assert ei.value.status == 4
