"""FP8 block-scaled expert weights (MOE_WEIGHTS_PACKED_FP8) against the oracle.

The packed bank is checked byte for byte against the layout moe.h documents,
rebuilt here on the CPU.  Layer outputs are compared with the oracle's FP8
layer (each selected expert dequantised exactly in fp64): every token of the
small configurations, and sampled tokens of the full-size FP8 configurations
in the launch configuration the benchmark times.  The GPU rounds each
weight once to bf16 (code value x scale) before the tensor cores, so the
bf16 output bound applies."""
import gc

import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu_common import (GAP_MIN, TOL_BF16, by_expert, lib, need_gpu, np64, rel_max_err,
                         rows_covering_experts, workspace)

pytestmark = pytest.mark.gpu

BANKS = ("W_gate_up", "W_down", "Ws_gate_up", "Ws_down")


def _expected_packed(kind, q, s):
    """The packed bytes moe.h specifies, built on the CPU from codes q
    [G, R, C] and scales s [G, R/128, C/128]."""
    G, R, C = q.shape
    ks_n, a128 = C // 64, R // 128
    tiles = []
    recs = []
    for g in range(G):
        for u in range((a128 + 1) // 2):
            pair = [t for t in (2 * u, 2 * u + 1) if t < a128]
            for ks in range(ks_n):
                for t in pair:
                    tile = np.empty((128, 64), dtype=np.uint8)
                    for r in range(128):
                        if kind == 0:  # gate/up interleave
                            src = ((r >> 4) & 1) * (R // 2) + 64 * t + 16 * (r >> 5) + (r & 15)
                        else:
                            src = 128 * t + r
                        row = q[g, src, 64 * ks:64 * ks + 64].reshape(8, 8)
                        for c in range(8):
                            tile[r, 8 * (c ^ (r & 7)):8 * (c ^ (r & 7)) + 8] = row[c]
                    tiles.append(tile.reshape(-1))
                rec = np.zeros(4, dtype=np.float32)
                for a, t in enumerate(pair):
                    if kind == 0:
                        rb = ((64 * t) // 128, (R // 2 + 64 * t) // 128)
                    else:
                        rb = (t, t)
                    rec[2 * a] = s[g, rb[0], ks // 2]
                    rec[2 * a + 1] = s[g, rb[1], ks // 2]
                recs.append(rec)
    return np.concatenate(tiles), np.stack(recs).reshape(-1)


@pytest.mark.parametrize("kind,R,C", [(0, 384, 256), (1, 384, 256), (1, 256, 128)],
                         ids=["gate_up_odd_tiles", "plain_odd_tiles", "plain"])
def test_pack_fp8_matches_documented_layout(kind, R, C):
    need_gpu()
    fgs = lib()
    gen = torch.Generator(device="cpu").manual_seed(R + C + kind)
    G = 2
    q = torch.randint(0, 256, (G, R, C), generator=gen, dtype=torch.uint8)
    s = torch.rand((G, R // 128, C // 128), generator=gen, dtype=torch.float32)
    nbytes = fgs.moe_packed_fp8_bytes(G, R, C)
    dst = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    fgs.moe_pack_weights_fp8(kind, G, R, C, q.cuda(), s.cuda(), dst)
    torch.cuda.synchronize()
    want_tiles, want_recs = _expected_packed(kind, q.numpy(), s.numpy())
    got = dst.cpu().numpy()
    n = G * R * C
    assert nbytes == n + want_recs.size * 4
    np.testing.assert_array_equal(got[:n], want_tiles)
    np.testing.assert_array_equal(got[n:].view(np.float32), want_recs)


def _forward(shape, g):
    fgs = lib()
    cfg = fgs.config(shape)
    assert cfg.weight_layout == fgs.MOE_WEIGHTS_PACKED_FP8
    gp = fgs.pack_layer_weights_fp8(g)
    T = g["x"].shape[0]
    ws, nws = workspace(cfg, T)
    y = torch.empty((T, shape.d_model), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((T, shape.K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, shape.K), dtype=torch.float32, device="cuda")
    counts = torch.empty(shape.E_routed, dtype=torch.int32, device="cuda")
    fgs.moe_layer_forward(cfg, T, gp["x"], gp["W_r"], gp["bias"], gp["W_gate_up"], gp["W_down"],
                          gp.get("Ws_gate_up"), gp.get("Ws_down"), gp.get("W_lat_down"),
                          gp.get("W_lat_up"), y, idx, w, counts, ws, nws)
    assert fgs.moe_get_device_status(ws) == 0
    return y, idx, w, counts


class _Bank:
    """Index an FP8 bank per expert, copying only that expert to the host."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, e):
        return self.t[e].cpu().numpy()

    def __len__(self):
        return self.t.shape[0]


def _oracle(shape, g, rows):
    b = {k: _Bank(g[k]) if k in g else None
         for k in [n + sfx for n in BANKS for sfx in ("_q", "_s")]}
    return oracle.moe_layer_tokens_fp8(
        np64(g["x"][rows]), np64(g["W_r"]), g["bias"].cpu().numpy(),
        b["W_gate_up_q"], b["W_gate_up_s"], b["W_down_q"], b["W_down_s"],
        b.get("Ws_gate_up_q"), b.get("Ws_gate_up_s"), b.get("Ws_down_q"), b.get("Ws_down_s"),
        K=shape.K, n_group=shape.n_group, topk_group=shape.topk_group,
        scale=shape.routed_scaling_factor, norm_topk_prob=shape.norm_topk_prob,
        W_lat_down64=np64(g["W_lat_down"]) if shape.d_latent else None,
        W_lat_up64=np64(g["W_lat_up"]) if shape.d_latent else None)


def _compare(shape, g, y, idx, w, counts, rows):
    ref = _oracle(shape, g, rows)
    clear = ref["gap"] > GAP_MIN
    got_set, got_w = by_expert(idx.cpu().numpy()[rows], w.cpu().numpy()[rows])
    ref_set, ref_w = by_expert(ref["idx"], ref["w"])
    np.testing.assert_array_equal(got_set[clear], ref_set[clear])
    assert rel_max_err(got_w[clear], ref_w[clear]) <= 1e-4
    same = (got_set == ref_set).all(axis=1)
    assert same.mean() > 0.9
    assert rel_max_err(np64(y[rows])[same], ref["y"][same]) <= TOL_BF16
    assert int(counts.sum()) == g["x"].shape[0] * shape.K


SMALL = [
    synth.custom(name="fp8_grouped", T=256, d_model=512, E_routed=32, K=4, E_shared=1,
                 d_ff=256, d_ff_shared=128, n_group=4, topk_group=2, x_dist="clusters32",
                 weights="fp8"),
    # d_model 384: three 128-row down tiles, so the last pair has one tile
    # (gate/up tiles are 64 features, always an even count with d_ff % 128)
    synth.custom(name="fp8_odd_tiles", T=300, d_model=384, E_routed=12, K=3, E_shared=1,
                 d_ff=256, d_ff_shared=128, weights="fp8"),
    synth.custom(name="fp8_k3", T=200, d_model=512, d_latent=256, E_routed=16, K=4, E_shared=2,
                 d_ff=128, d_ff_shared=128, weights="fp8"),
    synth.custom(name="fp8_one_token", T=1, d_model=256, E_routed=8, K=2, E_shared=1, d_ff=128,
                 d_ff_shared=128, weights="fp8"),
    # few experts, many tokens: experts of several 256-row tiles
    synth.custom(name="fp8_multi_tile", T=700, d_model=256, E_routed=4, K=2, d_ff=128,
                 weights="fp8"),
]


# token tiles of 32 rows (T <= 256): the weights go through TMEM unless
# FGS_FP8_TMEM=0 keeps them in shared memory
FP8_ENV_SHAPES = [
    synth.custom(name="fp8_env_grouped", T=256, d_model=512, E_routed=32, K=4, E_shared=1,
                 d_ff=256, d_ff_shared=128, n_group=4, topk_group=2, x_dist="clusters32",
                 weights="fp8"),
    synth.custom(name="fp8_env_odd_tiles", T=200, d_model=384, E_routed=12, K=3, E_shared=1,
                 d_ff=256, d_ff_shared=128, weights="fp8"),
    synth.custom(name="fp8_env_k3", T=128, d_model=512, d_latent=256, E_routed=16, K=4,
                 E_shared=2, d_ff=128, d_ff_shared=128, weights="fp8"),
]


@pytest.mark.parametrize("case", range(len(FP8_ENV_SHAPES)),
                         ids=[s.name for s in FP8_ENV_SHAPES])
def test_fp8_weights_in_tmem_equal_shared_memory_form(case):
    """The two FP8 forms apply the same arithmetic to each code, so the
    layer's output bytes are identical whether the converters write the bf16
    weights into TMEM or into shared memory (each form in its own process:
    the library reads the override once)."""
    need_gpu()
    import os
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    out = {}
    for tmem in ("1", "0"):
        env = dict(os.environ, FGS_FP8_TMEM=tmem)
        r = subprocess.run([sys.executable, os.path.join(here, "_fp8_env_case.py"), str(case)],
                           env=env, capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
        line = [ln for ln in r.stdout.splitlines() if ln.startswith("digest ")][-1].split()
        assert line[2] == "1", "non-finite output"
        out[tmem] = line[1]
    assert out["1"] == out["0"]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: s.name)
def test_layer_fp8_small_every_token(shape):
    need_gpu()
    g = synth.generate(shape, device="cuda")
    y, idx, w, counts = _forward(shape, g)
    _compare(shape, g, y, idx, w, counts, np.arange(shape.T))


@pytest.mark.parametrize("name", ["k2_decode_fp8", "k2_prefill_fp8", "k3_latent_fp8"])
def test_layer_fp8_full_size_sampled(name):
    need_gpu()
    shape = synth.shape(name)
    g = synth.generate(shape, device="cuda")
    try:
        y, idx, w, counts = _forward(shape, g)
        torch.cuda.synchronize()
        # the oracle dequantises every expert the compared tokens select, in
        # fp64 (seconds each): four evenly spaced tokens, and the tokens at
        # the first, last and every 128th slot of the two largest experts
        # (both of their row tiles and their ragged tails)
        rows = np.unique(np.concatenate([
            np.linspace(0, shape.T - 1, 4).astype(np.int64),
            rows_covering_experts(idx.cpu().numpy(), shape.E_routed, shape.K, largest=2)]))
        _compare(shape, g, y, idx, w, counts, rows)
        assert np.isfinite(np64(y)).all()
    finally:
        del g
        gc.collect()
        torch.cuda.empty_cache()


def test_fp8_layout_rejects_unaligned_widths():
    need_gpu()
    fgs = lib()
    shape = synth.custom(name="fp8_bad", T=8, d_model=256, E_routed=8, K=2, d_ff=192,
                         weights="fp8")
    cfg = fgs.config(shape)
    assert fgs.moe_validate_config(cfg, 8) == 2  # MOE_ERR_UNSUPPORTED_SHAPE


def test_layer_fp8_host_buffers():
    """moe_layer_forward_host with FP8 banks returns what the device-buffer
    forward returns (pinned x and y; y written by the combine directly)."""
    need_gpu()
    fgs = lib()
    shape = SMALL[0]
    g = synth.generate(shape, device="cuda")
    cfg = fgs.config(shape)
    gp = fgs.pack_layer_weights_fp8(g)
    T = shape.T
    ws, nws = workspace(cfg, T)
    x_host = g["x"].cpu().pin_memory()
    y_host = torch.full((T, shape.d_model), float("nan"), dtype=torch.bfloat16).pin_memory()
    fgs.moe_layer_forward_host(cfg, T, x_host, gp["W_r"], gp["bias"], gp["W_gate_up"],
                               gp["W_down"], gp.get("Ws_gate_up"), gp.get("Ws_down"), None, None,
                               y_host, ws, nws)
    torch.cuda.synchronize()
    assert fgs.moe_get_device_status(ws) == 0
    y, idx, w, counts = _forward(shape, g)
    torch.cuda.synchronize()
    assert torch.equal(y_host, y.cpu())
