"""Run moe_layer_forward on seeded synthetic inputs of any shape, for
profiling (e.g. under ncu on a case small enough to capture).

    python -m fine_grained_sparse_gb300.run_layer --T 2048 --E 32 --K 8 --d 7168 \
        --F 2048 --S 1 --G 8 --Gk 4 --iters 2
"""
from __future__ import annotations

import argparse
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

import fine_grained_sparse_gb300 as fgs  # noqa: E402


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--T", type=int, default=2048)
    ap.add_argument("--d", type=int, default=7168)
    ap.add_argument("--E", type=int, default=32)
    ap.add_argument("--K", type=int, default=8)
    ap.add_argument("--F", type=int, default=2048)
    ap.add_argument("--S", type=int, default=1)
    ap.add_argument("--Fs", type=int, default=0)
    ap.add_argument("--G", type=int, default=1)
    ap.add_argument("--Gk", type=int, default=1)
    ap.add_argument("--L", type=int, default=0)
    ap.add_argument("--x-dist", default="clusters32")
    ap.add_argument("--iters", type=int, default=2)
    ap.add_argument("--natural", action="store_true", help="natural (unpacked) weight layout")
    ap.add_argument("--router-only", action="store_true",
                    help="run moe_router alone (no expert weights are made)")
    a = ap.parse_args(argv)
    shape = synth.custom(name="profile_case", T=a.T, d_model=a.d, E_routed=a.E, K=a.K,
                         E_shared=a.S, d_ff=a.F, d_ff_shared=a.Fs or a.F, n_group=a.G,
                         topk_group=a.Gk, d_latent=a.L, x_dist=a.x_dist)
    if a.router_only:
        return run_router(shape, a)
    g = synth.generate(shape, device="cuda")
    cfg = fgs.config(shape)
    if not a.natural:
        cfg.weight_layout = fgs.MOE_WEIGHTS_PACKED
        g = fgs.pack_layer_weights(g)
    nws = fgs.moe_workspace_size(cfg, a.T)
    ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
    y = torch.empty((a.T, a.d), dtype=torch.bfloat16, device="cuda")
    for _ in range(a.iters):
        fgs.moe_layer_forward(cfg, a.T, g["x"], g["W_r"], g["bias"], g["W_gate_up"], g["W_down"],
                              g.get("Ws_gate_up"), g.get("Ws_down"), g.get("W_lat_down"),
                              g.get("W_lat_up"), y, None, None, None, ws, nws)
    status = fgs.moe_get_device_status(ws)
    if status:
        raise SystemExit("device status: " + fgs.moe_status_string(status))
    print("ok", float(y.float().abs().mean()))


def run_router(shape, a):
    x = synth.activations(shape, "cuda")
    W_r, bias = synth.router_params(shape, "cuda")
    cfg = fgs.config(shape)
    nws = fgs.moe_workspace_size(cfg, a.T)
    ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
    idx = torch.empty((a.T, a.K), dtype=torch.int32, device="cuda")
    w = torch.empty((a.T, a.K), dtype=torch.float32, device="cuda")
    for _ in range(a.iters):
        fgs.moe_router(cfg, a.T, x, W_r, bias, idx, w, ws, nws)
    status = fgs.moe_get_device_status(ws)
    if status:
        raise SystemExit("device status: " + fgs.moe_status_string(status))
    print("ok", float(w.sum()) / a.T)


if __name__ == "__main__":
    main()
