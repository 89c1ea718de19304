"""Whole-layer parity (moe_layer_forward) against the oracle.

Small configurations are compared on every token; the K2 decode, K2 prefill
and K3 latent configurations run at full size, in the launch configuration
the benchmark times, and are compared on a sample of tokens the oracle
evaluates one by one (its cost is one fp64 upcast per selected expert)."""
import gc

import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu_common import (GAP_MIN, TOL_BF16, TOL_F32, by_expert, lib, need_gpu, np64,
                         rel_max_err, rows_covering_experts, to_f64_cpu, workspace)

pytestmark = pytest.mark.gpu


def _forward(shape, g, packed=False):
    fgs = lib()
    cfg = fgs.config(shape)
    if packed:  # weights rearranged once into the order the tensor cores stream
        cfg.weight_layout = fgs.MOE_WEIGHTS_PACKED
        g = fgs.pack_layer_weights(g)
    T = g["x"].shape[0]
    ws, nws = workspace(cfg, T)
    y = torch.empty((T, shape.d_model), dtype=g["x"].dtype, device="cuda")
    idx = torch.empty((T, shape.K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, shape.K), dtype=torch.float32, device="cuda")
    counts = torch.empty(shape.E_routed, dtype=torch.int32, device="cuda")
    fgs.moe_layer_forward(cfg, T, g["x"], g["W_r"], g["bias"], g["W_gate_up"], g["W_down"],
                          g.get("Ws_gate_up"), g.get("Ws_down"), g.get("W_lat_down"),
                          g.get("W_lat_up"), y, idx, w, counts, ws, nws)
    assert fgs.moe_get_device_status(ws) == 0
    return y, idx, w, counts


def _oracle(shape, g, rows):
    x = np64(g["x"][rows])
    return oracle.moe_layer_tokens(
        x, np64(g["W_r"]), g["bias"].cpu().numpy(), g["W_gate_up"], g["W_down"],
        g.get("Ws_gate_up"), g.get("Ws_down"), shape.K, shape.n_group, shape.topk_group,
        shape.routed_scaling_factor, shape.norm_topk_prob,
        W_lat_down64=np64(g["W_lat_down"]) if shape.d_latent else None,
        W_lat_up64=np64(g["W_lat_up"]) if shape.d_latent else None,
        to_f64=to_f64_cpu)


def _compare(shape, g, y, idx, w, counts, rows, tol):
    ref = _oracle(shape, g, rows)
    clear = ref["gap"] > GAP_MIN
    got_set, got_w = by_expert(idx.cpu().numpy()[rows], w.cpu().numpy()[rows])
    ref_set, ref_w = by_expert(ref["idx"], ref["w"])
    np.testing.assert_array_equal(got_set[clear], ref_set[clear])
    assert rel_max_err(got_w[clear], ref_w[clear]) <= 1e-4
    # rows whose selected set matches are compared on the layer output
    same = (got_set == ref_set).all(axis=1)
    assert same.mean() > 0.9
    assert rel_max_err(np64(y[rows])[same], ref["y"][same]) <= tol
    assert int(counts.sum()) == g["x"].shape[0] * shape.K


SMALL = [
    synth.shape("tiny"),
    synth.custom(name="small_grouped", T=256, d_model=512, E_routed=32, K=4, E_shared=1,
                 d_ff=256, d_ff_shared=128, n_group=4, topk_group=2, x_dist="clusters32"),
    synth.custom(name="small_k3", T=200, d_model=512, d_latent=256, E_routed=16, K=4,
                 E_shared=2, d_ff=128, d_ff_shared=128),
    synth.custom(name="small_noshared", T=33, d_model=256, E_routed=8, K=2, d_ff=64),
    # edge cases: one token; top-1 with no shared expert; one token past the
    # small-batch tile switch, with an odd number of 128-row weight tiles in
    # both passes (d_ff 192 -> 3 gate/up tiles, d_model 384 -> 3 down tiles)
    synth.custom(name="one_token", T=1, d_model=256, E_routed=8, K=2, E_shared=1, d_ff=64,
                 d_ff_shared=64),
    synth.custom(name="top1", T=300, d_model=256, E_routed=16, K=1, d_ff=128),
    synth.custom(name="tile_switch_odd_tiles", T=257, d_model=384, E_routed=12, K=3,
                 E_shared=1, d_ff=192, d_ff_shared=128),
]


@pytest.mark.parametrize("packed", [False, True], ids=["natural", "packed"])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: s.name)
def test_layer_small_every_token(shape, packed):
    need_gpu()
    if packed and shape.dtype == "f32":
        pytest.skip("packed weights are bf16 only")
    g = synth.generate(shape, device="cuda")
    y, idx, w, counts = _forward(shape, g, packed)
    rows = np.arange(shape.T)
    _compare(shape, g, y, idx, w, counts, rows, TOL_F32 if shape.dtype == "f32" else TOL_BF16)


@pytest.mark.parametrize("name", ["k2_decode", "k2_prefill", "k3_latent"])
def test_layer_full_size_sampled(name):
    """Full-size layers in the benchmark's launch configuration.  The output
    is compared element by element with the oracle on every token at decode
    size, and otherwise on the tokens that reach every expert's every row
    tile (first, last and every 128th slot of each expert), so that each
    expert's weights, each token tile and each ragged tail is checked."""
    need_gpu()
    shape = synth.shape(name)
    g = synth.generate(shape, device="cuda")
    try:
        y, idx, w, counts = _forward(shape, g, packed=True)
        torch.cuda.synchronize()
        T = shape.T
        rows = (np.arange(T) if T <= 256 else
                rows_covering_experts(idx.cpu().numpy(), shape.E_routed, shape.K))
        _compare(shape, g, y, idx, w, counts, rows, TOL_BF16)
        # the routing of every token on the gap criterion
        r = oracle.router_from_x(np64(g["x"]), np64(g["W_r"]), g["bias"].cpu().numpy(), shape.K,
                                 shape.n_group, shape.topk_group)
        clear = r["gap"] > GAP_MIN
        np.testing.assert_array_equal(by_expert(idx.cpu().numpy())[clear], by_expert(r["idx"])[clear])
        assert np.isfinite(np64(y)).all()
    finally:
        del g
        gc.collect()
        torch.cuda.empty_cache()


@pytest.mark.parametrize("y_pinned", [True, False], ids=["y_pinned", "y_pageable"])
@pytest.mark.parametrize("shape", [SMALL[1], SMALL[2]], ids=lambda s: s.name)
def test_layer_forward_host_pipelined_calls(shape, y_pinned):
    """Three host-buffer calls in a row on one workspace (their x copies go
    through alternating staging buffers, overlapping the previous forward)
    each return what the device-buffer forward returns for the same x.  A
    pinned y is written by the layer's last kernel directly (the combine for
    the K2 form, the latent up-projection for K3); a pageable one is staged
    and copied."""
    need_gpu()
    fgs = lib()
    g = synth.generate(shape, device="cuda")
    cfg = fgs.config(shape)
    T = shape.T
    ws, nws = workspace(cfg, T)
    xs = [synth.generate(shape, device="cuda", seed=s, weights=False)["x"] for s in (1, 2, 3)]
    ys_host = [torch.full((T, shape.d_model), float("nan"), dtype=xs[0].dtype) for _ in xs]
    if y_pinned:
        ys_host = [y.pin_memory() for y in ys_host]
    xs_host = [x.cpu().pin_memory() for x in xs]
    for xh, yh in zip(xs_host, ys_host):  # enqueued back to back, no synchronisation
        fgs.moe_layer_forward_host(cfg, T, xh, g["W_r"], g["bias"], g["W_gate_up"], g["W_down"],
                                   g.get("Ws_gate_up"), g.get("Ws_down"), g.get("W_lat_down"),
                                   g.get("W_lat_up"), yh, ws, nws)
    torch.cuda.synchronize()
    assert fgs.moe_get_device_status(ws) == 0
    for x, yh in zip(xs, ys_host):
        ws2, nws2 = workspace(cfg, T)
        y = torch.empty((T, shape.d_model), dtype=x.dtype, device="cuda")
        fgs.moe_layer_forward(cfg, T, x, g["W_r"], g["bias"], g["W_gate_up"], g["W_down"],
                              g.get("Ws_gate_up"), g.get("Ws_down"), g.get("W_lat_down"),
                              g.get("W_lat_up"), y, None, None, None, ws2, nws2)
        torch.cuda.synchronize()
        assert torch.equal(yh, y.cpu())


@pytest.mark.parametrize("same_y", [False, True], ids=["own_y", "shared_y"])
@pytest.mark.parametrize("shape", SMALL[1:3], ids=lambda s: s.name)
def test_layer_host_pipelined(shape, same_y):
    """moe_layer_forward_host_pipelined: each call's y reaches its y_host by
    the next call (or the flush) and equals the device-buffer forward's, bit
    for bit; a y_host shared by all calls ends with the last call's y."""
    need_gpu()
    fgs = lib()
    g = synth.generate(shape, device="cuda")
    cfg = fgs.config(shape)
    T = shape.T
    ws, nws = workspace(cfg, T)
    xs = [synth.generate(shape, device="cuda", seed=s, weights=False)["x"] for s in (1, 2, 3, 4)]
    xs_host = [x.cpu().pin_memory() for x in xs]
    n_y = 1 if same_y else len(xs)
    ys_host = [torch.full((T, shape.d_model), float("nan"), dtype=xs[0].dtype).pin_memory()
               for _ in range(n_y)]
    stream = torch.cuda.Stream()
    for i, xh in enumerate(xs_host):  # enqueued back to back
        fgs.moe_layer_forward_host_pipelined(cfg, T, xh, g["W_r"], g["bias"], g["W_gate_up"],
                                             g["W_down"], g.get("Ws_gate_up"), g.get("Ws_down"),
                                             g.get("W_lat_down"), g.get("W_lat_up"),
                                             ys_host[i % n_y], ws, nws, stream=stream)
    fgs.moe_layer_forward_host_flush(ws, stream=stream)
    stream.synchronize()
    assert fgs.moe_get_device_status(ws) == 0
    want = []
    for x in xs:
        ws2, nws2 = workspace(cfg, T)
        y = torch.empty((T, shape.d_model), dtype=x.dtype, device="cuda")
        fgs.moe_layer_forward(cfg, T, x, g["W_r"], g["bias"], g["W_gate_up"], g["W_down"],
                              g.get("Ws_gate_up"), g.get("Ws_down"), g.get("W_lat_down"),
                              g.get("W_lat_up"), y, None, None, None, ws2, nws2)
        torch.cuda.synchronize()
        want.append(y.cpu())
    if same_y:
        assert torch.equal(ys_host[0], want[-1])
    else:
        for yh, y in zip(ys_host, want):
            assert torch.equal(yh, y)
    fgs.moe_layer_forward_host_release(ws)


@pytest.mark.parametrize("shape", SMALL[1:3], ids=lambda s: s.name)
def test_layer_with_presplit_router_weight(shape):
    """The layer forward with the router weight split once
    (MOE_ROUTER_WEIGHT_SPLIT) returns exactly what it returns with fp32 W_r."""
    need_gpu()
    fgs = lib()
    g = synth.generate(shape, device="cuda")
    y0, idx0, w0, c0 = _forward(shape, g)
    cfg = fgs.config(shape, router_weight=fgs.MOE_ROUTER_WEIGHT_SPLIT)
    g_s = dict(g)
    g_s["W_r"] = fgs.split_router_weight(cfg, g["W_r"])
    T = g["x"].shape[0]
    ws, nws = workspace(cfg, T)
    y = torch.empty_like(y0)
    idx, w, counts = torch.empty_like(idx0), torch.empty_like(w0), torch.empty_like(c0)
    fgs.moe_layer_forward(cfg, T, g_s["x"], g_s["W_r"], g_s["bias"], g_s["W_gate_up"],
                          g_s["W_down"], g_s.get("Ws_gate_up"), g_s.get("Ws_down"),
                          g_s.get("W_lat_down"), g_s.get("W_lat_up"), y, idx, w, counts, ws, nws)
    torch.cuda.synchronize()
    assert fgs.moe_get_device_status(ws) == 0
    for a, b in ((y, y0), (idx, idx0), (w, w0), (counts, c0)):
        assert torch.equal(a, b)


@pytest.mark.parametrize("weights_in", ["combine", "experts"])
@pytest.mark.parametrize("shape", [SMALL[1], SMALL[5]], ids=lambda s: s.name)
def test_layer_composed_from_the_public_calls(shape, weights_in):
    """moe_router -> moe_permute -> moe_grouped_swiglu -> moe_combine, each
    through the C ABI, equals the oracle layer.  With the gate weights applied
    in the combine (NULL to the experts) the result is the layer forward's,
    bit for bit; applied in the experts' epilogue (NULL to the combine) they
    scale each expert row before it is rounded to bf16."""
    need_gpu()
    fgs = lib()
    g = synth.generate(shape, device="cuda")
    cfg = fgs.config(shape)
    T, K, E, d, S = shape.T, shape.K, shape.E_routed, shape.d_model, shape.E_shared
    ws, nws = workspace(cfg, T)
    dev = dict(device="cuda")
    idx = torch.empty((T, K), dtype=torch.int32, **dev)
    w = torch.empty((T, K), dtype=torch.float32, **dev)
    fgs.moe_router(cfg, T, g["x"], g["W_r"], g["bias"], idx, w, ws, nws)
    counts = torch.empty(E, dtype=torch.int32, **dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, **dev)
    perm = torch.empty(T * K, dtype=torch.int32, **dev)
    inv = torch.empty(T * K, dtype=torch.int32, **dev)
    fgs.moe_permute(cfg, T, idx, counts, offsets, perm, inv, ws, nws)
    Y = torch.empty((T * K, d), dtype=g["x"].dtype, **dev)
    Ysh = torch.empty((S, T, d), dtype=g["x"].dtype, **dev) if S else None
    in_experts = weights_in == "experts"
    fgs.moe_grouped_swiglu(cfg, T, g["x"], offsets, perm, w if in_experts else None,
                           g["W_gate_up"], g["W_down"], g["x"] if S else None,
                           g.get("Ws_gate_up"), g.get("Ws_down"), Y, Ysh, ws, nws)
    y = torch.empty((T, d), dtype=g["x"].dtype, **dev)
    fgs.moe_combine(cfg, T, Y, inv, None if in_experts else w, Ysh, y)
    torch.cuda.synchronize()
    assert fgs.moe_get_device_status(ws) == 0
    _compare(shape, g, y, idx, w, counts, np.arange(T), TOL_BF16)
    if not in_experts:
        y_layer, idx_l, w_l, counts_l = _forward(shape, g)
        torch.cuda.synchronize()
        assert torch.equal(idx, idx_l) and torch.equal(w, w_l)
        assert torch.equal(y, y_layer)


def test_layer_forward_host_release_starts_afresh():
    """After moe_layer_forward_host_release, host-buffer calls on the same
    workspace run again (on new state) and still return the device-buffer
    forward's result."""
    need_gpu()
    fgs = lib()
    shape = SMALL[1]
    g = synth.generate(shape, device="cuda")
    cfg = fgs.config(shape)
    T = shape.T
    ws, nws = workspace(cfg, T)
    x_host = g["x"].cpu().pin_memory()
    y_ref, _, _, _ = _forward(shape, g)
    for _ in range(2):
        y_host = torch.full((T, shape.d_model), float("nan"), dtype=g["x"].dtype).pin_memory()
        for _ in range(3):
            fgs.moe_layer_forward_host(cfg, T, x_host, g["W_r"], g["bias"], g["W_gate_up"],
                                       g["W_down"], g.get("Ws_gate_up"), g.get("Ws_down"), None,
                                       None, y_host, ws, nws)
        torch.cuda.synchronize()
        assert torch.equal(y_host, y_ref.cpu())
        fgs.moe_layer_forward_host_release(ws)
    fgs.moe_layer_forward_host_release(ws)  # releasing twice is harmless
