"""Grouped SwiGLU experts (tensor-core bf16 path and fp32 CUDA-core path)
against the oracle's expert math, slot by slot."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu_common import TOL_BF16, TOL_F32, lib, need_gpu, np64, rel_max_err, workspace

pytestmark = pytest.mark.gpu


def _case(T, d, E, K, F, S, Fs, dtype, seed, skew=False):
    shape = synth.custom(T=T, d_model=d, E_routed=E, K=K, E_shared=S, d_ff=F, d_ff_shared=Fs,
                         dtype=dtype)
    g = synth.generate(shape, device="cuda", seed=seed)
    gen = torch.Generator().manual_seed(seed)
    wts = torch.ones(E)
    if skew:
        wts[:K] = 50.0
    idx = torch.stack([torch.multinomial(wts, K, replacement=False, generator=gen)
                       for _ in range(T)])
    topk_w = torch.rand((T, K), generator=gen) + 0.1
    return shape, g, idx.numpy(), topk_w


def _run(shape, g, idx, topk_w):
    fgs = lib()
    T, K, E = shape.T, shape.K, shape.E_routed
    cfg = fgs.config(shape)
    p = oracle.permute(idx, E)
    ws, nws = workspace(cfg, T)
    dt = g["x"].dtype
    Y = torch.empty((T * K, shape.d_model), dtype=dt, device="cuda")
    S = shape.E_shared
    Ys = torch.empty((S, T, shape.d_model), dtype=dt, device="cuda") if S else None
    fgs.moe_grouped_swiglu(
        cfg, T, g["x"], torch.from_numpy(p["offsets"].astype(np.int32)).cuda(),
        torch.from_numpy(p["perm"].astype(np.int32)).cuda(), topk_w.cuda(), g["W_gate_up"],
        g["W_down"], g["x"] if S else None, g.get("Ws_gate_up"), g.get("Ws_down"), Y, Ys, ws, nws)
    assert fgs.moe_get_device_status(ws) == 0
    return p, Y, Ys


def _reference(shape, g, idx, topk_w, p):
    T, K, F = shape.T, shape.K, shape.d_ff
    x = np64(g["x"])
    Wgu, Wd = np64(g["W_gate_up"]), np64(g["W_down"])
    Yref = np.zeros((T * K, shape.d_model))
    for e in range(shape.E_routed):
        slots = np.arange(p["offsets"][e], p["offsets"][e + 1])
        if slots.size == 0:
            continue
        j = p["perm"][slots]
        t, k = j // K, j % K
        Yref[slots] = topk_w.numpy()[t, k][:, None] * oracle.swiglu_expert(
            x[t], Wgu[e, :F], Wgu[e, F:], Wd[e])
    Ysref = None
    if shape.E_shared:
        Fs = shape.d_ff_shared
        Sgu, Sd = np64(g["Ws_gate_up"]), np64(g["Ws_down"])
        Ysref = np.stack([oracle.swiglu_expert(x, Sgu[s, :Fs], Sgu[s, Fs:], Sd[s])
                          for s in range(shape.E_shared)])
    return Yref, Ysref


CASES = [
    # T, d, E, K, F, S, Fs, skew   -- several k-steps, output blocks and ragged tails
    (100, 256, 8, 2, 128, 1, 64, False),
    (600, 384, 4, 2, 192, 1, 128, False),     # experts with > 256 rows: 2 token tiles
    (37, 512, 16, 4, 64, 2, 128, True),       # T <= 64: 64-row token tile
    (130, 256, 64, 8, 128, 0, 0, False),      # no shared expert, many 1-3 row experts
    (1, 128, 4, 2, 64, 1, 64, False),         # a single token
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "T%d_d%d_E%d_K%d_F%d_S%d" % c[:6])
def test_grouped_swiglu_bf16(case):
    need_gpu()
    T, d, E, K, F, S, Fs, skew = case
    shape, g, idx, topk_w = _case(T, d, E, K, F, S, Fs, "bf16", seed=T + d + E, skew=skew)
    p, Y, Ys = _run(shape, g, idx, topk_w)
    Yref, Ysref = _reference(shape, g, idx, topk_w, p)
    assert rel_max_err(np64(Y), Yref) <= TOL_BF16
    if S:
        assert rel_max_err(np64(Ys), Ysref) <= TOL_BF16


@pytest.mark.parametrize("case", [(64, 256, 16, 4, 64, 1, 64, False), (45, 96, 6, 3, 40, 2, 24, True)])
def test_grouped_swiglu_f32(case):
    need_gpu()
    T, d, E, K, F, S, Fs, skew = case
    shape, g, idx, topk_w = _case(T, d, E, K, F, S, Fs, "f32", seed=T + d, skew=skew)
    p, Y, Ys = _run(shape, g, idx, topk_w)
    Yref, Ysref = _reference(shape, g, idx, topk_w, p)
    assert rel_max_err(np64(Y), Yref) <= TOL_F32
    assert rel_max_err(np64(Ys), Ysref) <= TOL_F32


def test_linear_bf16():
    need_gpu()
    fgs = lib()
    gen = torch.Generator(device="cuda").manual_seed(3)
    for T, i, o in [(5, 256, 384), (300, 512, 256)]:
        x = torch.randn((T, i), generator=gen, device="cuda").bfloat16()
        W = (torch.randn((o, i), generator=gen, device="cuda") * 0.05).bfloat16()
        add = torch.randn((T, o), generator=gen, device="cuda").bfloat16()
        y = torch.empty((T, o), dtype=torch.bfloat16, device="cuda")
        ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
        fgs.moe_linear(T, i, o, x, W, add, y, ws, 4096)
        torch.cuda.synchronize()
        want = np64(x) @ np64(W).T + np64(add)
        assert rel_max_err(np64(y), want) <= TOL_BF16


def _pack_reference(W: torch.Tensor, gate_up: bool) -> torch.Tensor:
    """The documented MOE_WEIGHTS_PACKED order, written with torch indexing."""
    G, R, C = W.shape
    a128, ks = R // 128, C // 64
    r = torch.arange(128)
    rows = []
    for t in range(a128):
        if gate_up:
            F = R // 2
            rows.append(((r >> 4) & 1) * F + 64 * t + 16 * (r >> 5) + (r & 15))
        else:
            rows.append(128 * t + r)
    tiles = W[:, torch.cat(rows), :].reshape(G, a128, 128, ks, 8, 8)   # g, t, row, k-step, chunk, elem
    pos = torch.arange(8)
    chunk_at = pos[None, :] ^ (r[:, None] & 7)                           # [row, position] -> chunk
    idx = chunk_at[None, None, :, None, :, None].expand(G, a128, 128, ks, 8, 8)
    sw = torch.gather(tiles, 4, idx)                                     # swizzled tiles
    sw = sw.permute(0, 1, 3, 2, 4, 5)                                    # g, t, k-step, row, pos, elem
    out = []
    for g in range(G):
        for u in range((a128 + 1) // 2):
            for k in range(ks):
                for t in range(2 * u, min(2 * u + 2, a128)):
                    out.append(sw[g, t, k].reshape(-1))
    return torch.cat(out).reshape(G, R, C)


@pytest.mark.parametrize("gate_up", [True, False])
@pytest.mark.parametrize("G,R,C", [(2, 256, 128), (3, 384, 192), (1, 128, 64)])
def test_pack_weights_layout(gate_up, G, R, C):
    need_gpu()
    fgs = lib()
    W = torch.randn((G, R, C), generator=torch.Generator().manual_seed(R + C)).bfloat16()
    dst = torch.empty_like(W, device="cuda")
    fgs.moe_pack_weights(fgs.MOE_PACK_GATE_UP if gate_up else fgs.MOE_PACK_PLAIN, G, R, C,
                         W.cuda(), dst)
    torch.cuda.synchronize()
    assert torch.equal(dst.cpu(), _pack_reference(W, gate_up))


@pytest.mark.parametrize("case", CASES[:4], ids=lambda c: "T%d_d%d_E%d_K%d_F%d_S%d" % c[:6])
def test_grouped_swiglu_packed_equals_natural(case):
    """The packed layout feeds the tensor cores the same operands: bit-exact."""
    need_gpu()
    fgs = lib()
    T, d, E, K, F, S, Fs, skew = case
    shape, g, idx, topk_w = _case(T, d, E, K, F, S, Fs, "bf16", seed=T + d + E, skew=skew)
    p, Y, Ys = _run(shape, g, idx, topk_w)
    gp = fgs.pack_layer_weights(g)
    cfg = fgs.config(shape, weight_layout=fgs.MOE_WEIGHTS_PACKED)
    ws, nws = workspace(cfg, T)
    Y2 = torch.empty_like(Y)
    Ys2 = torch.empty_like(Ys) if S else None
    fgs.moe_grouped_swiglu(
        cfg, T, g["x"], torch.from_numpy(p["offsets"].astype(np.int32)).cuda(),
        torch.from_numpy(p["perm"].astype(np.int32)).cuda(), topk_w.cuda(), gp["W_gate_up"],
        gp["W_down"], g["x"] if S else None, gp.get("Ws_gate_up"), gp.get("Ws_down"), Y2, Ys2,
        ws, nws)
    assert fgs.moe_get_device_status(ws) == 0
    assert torch.equal(Y, Y2)
    if S:
        assert torch.equal(Ys, Ys2)


@pytest.mark.parametrize("case", [(100, 256, 8, 2, 128, 1, 128, False),
                                  (600, 384, 4, 2, 256, 1, 128, False),
                                  (33, 512, 16, 4, 128, 2, 128, True)],
                         ids=lambda c: "T%d_d%d_E%d_K%d_F%d_S%d" % c[:6])
def test_grouped_swiglu_fp8(case):
    """moe_grouped_swiglu with FP8 block-scaled banks: the routed rows of Y
    carry their routing weight (applied in the FP8 down pass's epilogue)."""
    need_gpu()
    fgs = lib()
    T, d, E, K, F, S, Fs, skew = case
    shape = synth.custom(T=T, d_model=d, E_routed=E, K=K, E_shared=S, d_ff=F, d_ff_shared=Fs,
                         weights="fp8")
    g = synth.generate(shape, device="cuda", seed=T + E)
    gen = torch.Generator().manual_seed(T + E)
    wts = torch.ones(E)
    if skew:
        wts[:K] = 50.0
    idx = torch.stack([torch.multinomial(wts, K, replacement=False, generator=gen)
                       for _ in range(T)]).numpy()
    topk_w = torch.rand((T, K), generator=gen) + 0.1
    cfg = fgs.config(shape)
    assert cfg.weight_layout == fgs.MOE_WEIGHTS_PACKED_FP8
    gp = fgs.pack_layer_weights_fp8(g)
    p = oracle.permute(idx, E)
    ws, nws = workspace(cfg, T)
    Y = torch.empty((T * K, d), dtype=torch.bfloat16, device="cuda")
    Ys = torch.empty((S, T, d), dtype=torch.bfloat16, device="cuda") if S else None
    fgs.moe_grouped_swiglu(
        cfg, T, g["x"], torch.from_numpy(p["offsets"].astype(np.int32)).cuda(),
        torch.from_numpy(p["perm"].astype(np.int32)).cuda(), topk_w.cuda(), gp["W_gate_up"],
        gp["W_down"], g["x"] if S else None, gp.get("Ws_gate_up"), gp.get("Ws_down"), Y, Ys, ws,
        nws)
    assert fgs.moe_get_device_status(ws) == 0
    x = np64(g["x"])
    host = {k: v.cpu().numpy() for k, v in g.items() if k.endswith(("_q", "_s"))}
    Yref = np.zeros((T * K, d))
    for e in range(E):
        slots = np.arange(p["offsets"][e], p["offsets"][e + 1])
        if slots.size == 0:
            continue
        j = p["perm"][slots]
        t, k = j // K, j % K
        gu = oracle.dequant_fp8_blocks(host["W_gate_up_q"][e], host["W_gate_up_s"][e])
        dn = oracle.dequant_fp8_blocks(host["W_down_q"][e], host["W_down_s"][e])
        Yref[slots] = topk_w.numpy()[t, k][:, None] * oracle.swiglu_expert(x[t], gu[:F], gu[F:], dn)
    assert rel_max_err(np64(Y), Yref) <= TOL_BF16
    for s in range(S):
        gu = oracle.dequant_fp8_blocks(host["Ws_gate_up_q"][s], host["Ws_gate_up_s"][s])
        dn = oracle.dequant_fp8_blocks(host["Ws_down_q"][s], host["Ws_down_s"][s])
        assert rel_max_err(np64(Ys[s]), oracle.swiglu_expert(x, gu[:Fs], gu[Fs:], dn)) <= TOL_BF16
