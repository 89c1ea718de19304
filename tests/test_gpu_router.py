"""Router parity on the GPU: moe_router_from_logits bit-exact against the
oracle on shared fp32 logits; moe_router (fused GEMM) on the gap criterion."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu_common import (GAP_MIN, TOL_WEIGHTS, by_expert, lib, need_gpu, np64, rel_max_err,
                         workspace)

pytestmark = pytest.mark.gpu

# (E, K, n_group, topk_group)
ROUTER_SHAPES = [(16, 4, 1, 1), (384, 8, 1, 1), (384, 8, 8, 4), (896, 16, 1, 1), (64, 6, 4, 2),
                 (32, 32, 1, 1), (8, 1, 1, 1), (96, 9, 3, 1)]


def _logits(kind, T, E, gen):
    if kind == "normal":
        return torch.randn((T, E), generator=gen) * 1.5
    if kind == "grid":  # distinct values on a 2^-10 grid: no near-ties
        base = (torch.arange(E, dtype=torch.float32) - E / 2) * 2.0 ** -10 * 7
        return torch.stack([base[torch.randperm(E, generator=gen)] for _ in range(T)])
    if kind == "ties":  # few distinct values: many exact ties, broken by index
        vals = torch.tensor([-1.0, -0.5, 0.0, 0.25, 0.5, 1.0])
        return vals[torch.randint(0, len(vals), (T, E), generator=gen)]
    if kind == "crowded":  # scores packed within 1e-5: every fast value is near a threshold
        return 0.3 + torch.rand((T, E), generator=gen) * 1e-5
    if kind == "wide":  # logits beyond the fast range mixed with ordinary ones
        return torch.randn((T, E), generator=gen) * 40.0
    raise ValueError(kind)


@pytest.mark.parametrize("shape", ROUTER_SHAPES, ids=lambda s: "E%d_K%d_G%d_%d" % s)
@pytest.mark.parametrize("kind", ["normal", "grid", "ties", "crowded", "wide"])
@pytest.mark.parametrize("T", [1, 37, 1000])
def test_router_from_logits_bit_exact(shape, kind, T):
    need_gpu()
    fgs = lib()
    E, K, G, Gk = shape
    seed = E * 1000 + K * 10 + G + 7 * T + 100000 * ["normal", "grid", "ties", "crowded",
                                                      "wide"].index(kind)
    gen = torch.Generator().manual_seed(seed)
    z = _logits(kind, T, E, gen).float()
    b = torch.zeros(E) if kind != "normal" else (torch.rand(E, generator=gen) - 0.5) * 0.3
    cfg = fgs.config(d_model=128, E_routed=E, K=K, n_group=G, topk_group=Gk)
    idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K), dtype=torch.float32, device="cuda")
    fgs.moe_router_from_logits(cfg, T, z.cuda(), b.cuda(), idx, w)
    torch.cuda.synchronize()
    ref = oracle.router_from_logits(z.numpy(), b.numpy(), K, G, Gk)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref["idx"])
    assert rel_max_err(w.cpu().numpy(), ref["w"]) <= TOL_WEIGHTS


def _check_router_from_x(cfg_shape, x, W_r, bias, tensor_cores=True):
    fgs = lib()
    T = x.shape[0]
    cfg = fgs.config(cfg_shape, d_ff=0)
    idx = torch.empty((T, cfg.K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, cfg.K), dtype=torch.float32, device="cuda")
    if tensor_cores:  # a workspace selects the split-bf16 tensor-core GEMM for bf16 x
        ws, nws = workspace(cfg, T)
        fgs.moe_router(cfg, T, x, W_r, bias, idx, w, ws, nws)
        assert fgs.moe_get_device_status(ws) == 0
    else:             # no workspace: the fused fp32 CUDA-core kernel
        fgs.moe_router(cfg, T, x, W_r, bias, idx, w)
    torch.cuda.synchronize()
    ref = oracle.router_from_x(np64(x), np64(W_r), bias.cpu().numpy(), cfg.K, cfg.n_group,
                               cfg.topk_group)
    got_idx = idx.cpu().numpy()
    clear = ref["gap"] > GAP_MIN
    assert clear.mean() > 0.98, "the inputs should leave almost every token with a clear margin"
    got_set, got_w = by_expert(got_idx, w.cpu().numpy())
    ref_set, ref_w = by_expert(ref["idx"], ref["w"])
    np.testing.assert_array_equal(got_set[clear], ref_set[clear])
    assert rel_max_err(got_w[clear], ref_w[clear]) <= TOL_WEIGHTS
    # every token, clear or not, selects K distinct valid experts
    assert ((got_idx >= 0) & (got_idx < cfg.E_routed)).all()
    srt = np.sort(got_idx, axis=1)
    assert (np.diff(srt, axis=1) > 0).all()


@pytest.mark.parametrize("tensor_cores", [True, False], ids=["split_bf16_tc", "fp32_ffma"])
@pytest.mark.parametrize("name,T", [("tiny", None), ("k2_router", None), ("k2_prefill", 700),
                                    ("k3_latent", 300)])
def test_router_matches_oracle(name, T, tensor_cores):
    need_gpu()
    shape = synth.shape(name)
    g = synth.generate(shape, device="cuda", T=T, weights=False)
    _check_router_from_x(shape, g["x"], g["W_r"], g["bias"], tensor_cores)


@pytest.mark.parametrize("parts,tile,name,T", [(5, 256, "k2_prefill", 700), (7, 128, "k3_latent", 300),
                                           (1, 256, "k2_router", 600), (48, 32, "k2_decode", 100)])
def test_router_uneven_k_parts(parts, tile, name, T):
    """The tensor-core router with K part counts that split the d / 64 k
    steps unevenly (112 = 22 + 22 + 23 + 22 + 23 at 5 parts), a single part,
    and 48 parts of 2-3 k steps, each with its token tile, against the oracle
    (gap criterion), in a child process: the overrides are read once per
    process."""
    need_gpu()
    import os
    import subprocess
    import sys
    env = dict(os.environ, FGS_ROUTER_KSPLIT=str(parts), FGS_ROUTER_TILE=str(tile))
    here = os.path.dirname(os.path.abspath(__file__))
    r = subprocess.run([sys.executable, os.path.join(here, "_router_env_case.py"), name, str(T)],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]


@pytest.mark.parametrize("tensor_cores", [True, False], ids=["split_bf16_tc", "fp32_ffma"])
def test_router_ragged_tokens_and_small_E(tensor_cores):
    need_gpu()
    for T, E, K, G, Gk in [(1, 16, 4, 1, 1), (65, 40, 5, 4, 2), (130, 130, 7, 1, 1),
                           (300, 200, 6, 1, 1), (77, 1024, 32, 8, 4), (513, 1024, 32, 1, 1)]:
        shape = synth.custom(T=T, d_model=256, E_routed=E, K=K, n_group=G, topk_group=Gk,
                             router_only=True)
        g = synth.generate(shape, device="cuda", seed=T + E)
        _check_router_from_x(shape, g["x"], g["W_r"], g["bias"], tensor_cores)


def test_dense_gates_from_router_outputs():
    """G [T, E] from the router's own outputs equals the oracle's spreading
    of those outputs exactly (its entries are copies)."""
    need_gpu()
    fgs = lib()
    shape = synth.custom(name="dense_g", T=300, d_model=512, E_routed=64, K=6, n_group=8,
                         topk_group=3, router_only=True, x_dist="clusters32")
    g = synth.generate(shape, device="cuda", weights=False)
    cfg = fgs.config(shape, d_ff=0)
    T = shape.T
    ws, nws = workspace(cfg, T)
    idx = torch.empty((T, shape.K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, shape.K), dtype=torch.float32, device="cuda")
    fgs.moe_router(cfg, T, g["x"], g["W_r"], g["bias"], idx, w, ws, nws)
    G = torch.full((T, shape.E_routed), -1.0, dtype=torch.float32, device="cuda")
    fgs.moe_dense_gates(cfg, T, idx, w, G)
    torch.cuda.synchronize()
    want = oracle.dense_gates(idx.cpu().numpy(), w.cpu().numpy().astype(np.float64),
                              shape.E_routed)
    np.testing.assert_array_equal(G.cpu().numpy().astype(np.float64), want)


@pytest.mark.parametrize("T,K,E", [(4096, 8, 384), (7, 3, 16), (128, 16, 896)])
def test_bias_update_bit_exact(T, K, E):
    need_gpu()
    fgs = lib()
    gen = torch.Generator().manual_seed(T + K + E)
    counts = torch.multinomial(torch.ones(E), T * K, replacement=True, generator=gen)
    counts = torch.bincount(counts, minlength=E).to(torch.int32)
    counts[: min(E, 4)] = T * K // E  # some experts exactly at the mean load
    bias = (torch.rand(E, generator=gen) - 0.5).to(torch.float32)
    cfg = fgs.config(d_model=128, E_routed=E, K=K)
    b_dev = bias.cuda()
    for _ in range(3):  # three batches with the same loads
        fgs.moe_update_bias(cfg, T, counts.cuda(), 1e-3, b_dev)
    torch.cuda.synchronize()
    want = bias.numpy()
    for _ in range(3):
        want = oracle.aux_free_bias_update(want, counts.numpy(), T, K, 1e-3)
    np.testing.assert_array_equal(b_dev.cpu().numpy(), want)


@pytest.mark.parametrize("T,E,K,grid", [(4096, 896, 16, False), (8192, 384, 8, False),
                                        (37, 12, 3, True), (1, 16, 4, False), (300, 32, 32, True)])
def test_quantile_bias_update_bit_exact(T, E, K, grid):
    """Quantile Balancing on the GPU equals the oracle bit for bit: the
    thresholds (order statistics of each expert's fp32 scores) and the
    updated bias, over two batches in a row with rates 1 and 0.3; a coarse
    logit grid makes many scores tie."""
    need_gpu()
    fgs = lib()
    gen = torch.Generator().manual_seed(T * 7 + E)
    z = torch.randn((T, E), generator=gen) * 1.5 + torch.linspace(-1, 1, E)
    if grid:
        z = torch.round(z * 4) / 4
    z = z.to(torch.float32)
    bias = ((torch.rand(E, generator=gen) - 0.5) * 0.2).to(torch.float32)
    cfg = fgs.config(d_model=128, E_routed=E, K=K)
    b_dev = bias.cuda()
    theta = torch.empty(E, dtype=torch.float32, device="cuda")
    want_b = bias.numpy()
    for rate in (1.0, 0.3):
        fgs.moe_quantile_bias_update(cfg, T, z.cuda(), rate, theta, b_dev)
        torch.cuda.synchronize()
        want_theta, want_b = oracle.quantile_bias_update(z.numpy(), want_b, K, rate)
        np.testing.assert_array_equal(theta.cpu().numpy(), want_theta)
        np.testing.assert_array_equal(b_dev.cpu().numpy(), want_b)


@pytest.mark.parametrize("name,T", [("k2_router", 700), ("k3_latent", 300), ("k2_decode", None)])
def test_presplit_router_weight_is_bit_identical(name, T):
    """A router weight split once (MOE_ROUTER_WEIGHT_SPLIT) gives the same
    indices and weights, bit for bit, as the fp32 weight split per call;
    through moe_router, moe_router_noalloc and the layer forward."""
    need_gpu()
    fgs = lib()
    shape = synth.shape(name)
    T = T or shape.T
    g = synth.generate(shape, device="cuda", T=T, weights=False)
    cfg = fgs.config(shape, d_ff=0)
    cfg_s = fgs.config(shape, d_ff=0, router_weight=fgs.MOE_ROUTER_WEIGHT_SPLIT)
    W_s = fgs.split_router_weight(cfg_s, g["W_r"])
    ws, nws = workspace(cfg, T)
    outs = []
    for c, W in ((cfg, g["W_r"]), (cfg_s, W_s)):
        idx = torch.empty((T, c.K), dtype=torch.int32, device="cuda")
        w = torch.empty((T, c.K), dtype=torch.float32, device="cuda")
        fgs.moe_router(c, T, g["x"], W, g["bias"], idx, w, ws, nws)
        idx2, w2 = idx.clone(), w.clone()
        fgs.moe_router_noalloc(c, T, g["x"], W, g["bias"], idx2, w2)
        torch.cuda.synchronize()
        assert fgs.moe_get_device_status(ws) == 0
        outs.append((idx.cpu(), w.cpu(), idx2.cpu(), w2.cpu()))
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
    assert torch.equal(outs[0][0], outs[0][2]) and torch.equal(outs[0][1], outs[0][3])
