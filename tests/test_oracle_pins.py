"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each ``check_*`` function raises AssertionError on a mismatch.  The tests run
them on the oracle as written; ``test_planted_mistakes_are_caught`` plants
plausible mistakes in the oracle (on the CPU) and requires that some pin
fails for each one.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as Fnn

import oracle
from oracle import moe_oracle as mo
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# helpers written independently of the oracle
# --------------------------------------------------------------------------
def _dominates(ca, a, cb, b):
    """(value descending, index ascending) total order: does a come before b?"""
    return ca > cb or (ca == cb and a < b)


def _brute_topk(values, K):
    """The unique K-subset whose every member precedes every non-member."""
    n = len(values)
    found = []
    for sub in itertools.combinations(range(n), K):
        rest = [j for j in range(n) if j not in sub]
        if all(_dominates(values[a], a, values[b], b) for a in sub for b in rest):
            found.append(set(sub))
    assert len(found) == 1, found
    return found[0]


def _brute_group_select(c32, K, G, Gk):
    """Group-limited selection by enumeration (pairs for the top-2 sum)."""
    E = len(c32)
    gs = E // G
    gscore = []
    for j in range(G):
        members = range(j * gs, (j + 1) * gs)
        best = None
        for a, b in itertools.permutations(members, 2):
            v = np.float32(c32[a]) + np.float32(c32[b])
            best = v if best is None or v > best else best
        gscore.append(best)
    kept = _brute_topk(gscore, Gk)
    masked = [c32[e] if (e // gs) in kept else np.float32(0.0) for e in range(E)]
    return _brute_topk(masked, K), masked


def _dense_swiglu_torch(x, Wg, Wu, Wd):
    """Independent SwiGLU FFN via torch fp64 library routines."""
    xt = torch.as_tensor(x, dtype=torch.float64)
    h = Fnn.silu(Fnn.linear(xt, torch.as_tensor(Wg, dtype=torch.float64))) * \
        Fnn.linear(xt, torch.as_tensor(Wu, dtype=torch.float64))
    return Fnn.linear(h, torch.as_tensor(Wd, dtype=torch.float64)).numpy()


def _rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# checks
# --------------------------------------------------------------------------
def check_sigmoid_closed_forms():
    from scipy.special import expit
    assert oracle.sigmoid(0.0) == 0.5
    assert abs(oracle.sigmoid(math.log(3.0)) - 0.75) < 1e-15
    assert abs(oracle.sigmoid(-math.log(3.0)) - 0.25) < 1e-15
    z = _rng(0).normal(0, 4, 4096)
    s = oracle.sigmoid(z)
    np.testing.assert_allclose(s + oracle.sigmoid(-z), 1.0, rtol=0, atol=4.5e-16)
    np.testing.assert_allclose(s, expit(z), rtol=1e-14, atol=0)
    assert oracle.sigmoid(-1000.0) == 0.0 and oracle.sigmoid(1000.0) == 1.0


def check_silu():
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(math.log(3.0)) - 0.75 * math.log(3.0)) < 1e-15
    v = _rng(1).normal(0, 3, 4096)
    ref = Fnn.silu(torch.as_tensor(v, dtype=torch.float64)).numpy()
    np.testing.assert_allclose(oracle.silu(v), ref, rtol=1e-14, atol=1e-300)


def check_bf16_upcast():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0000, 0x8000, 0x7F7F], dtype=np.uint16)
    got = oracle.bf16_bits_to_f64(bits)
    assert got[0] == 1.0 and got[1] == -2.0 and got[2] == 1.0 + 2.0 ** -7
    assert got[3] == 0.0 and np.signbit(got[4])
    rnd = _rng(2).integers(0, 0x7F80, 2048).astype(np.uint16)
    tb = torch.from_numpy(rnd.astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.bf16_bits_to_f64(rnd), tb)


def check_biased_scores_fp32():
    z = _rng(3).normal(0, 1, (8, 40)).astype(np.float32)
    b = _rng(4).uniform(-0.1, 0.1, 40).astype(np.float32)
    c = oracle.biased_scores_f32(z, b)
    assert c.dtype == np.float32
    for t in range(8):
        for e in range(40):
            s = np.float32(1.0 / (1.0 + math.exp(-float(z[t, e]))))
            assert c[t, e] == np.float32(s + b[e])


def check_select_plain_bruteforce(n_cases=300):
    rng = _rng(5)
    for case in range(n_cases):
        E = int(rng.integers(2, 11))
        K = int(rng.integers(1, E + 1))
        # a coarse grid forces ties
        c = (rng.integers(-4, 5, E) * 0.125).astype(np.float32)
        idx, _ = oracle.select_experts(c[None, :], K)
        assert set(idx[0].tolist()) == _brute_topk(list(c), K)
        for a, b in zip(idx[0][:-1], idx[0][1:]):
            assert _dominates(c[a], a, c[b], b)


def check_select_grouped_bruteforce(n_cases=200):
    rng = _rng(6)
    for case in range(n_cases):
        E = 12
        G = int(rng.choice([2, 3, 4, 6]))
        Gk = int(rng.integers(1, G + 1))
        K = int(rng.integers(1, Gk * (E // G) + 1))
        c = (rng.integers(-3, 6, E) * 0.0625).astype(np.float32)
        idx, masked = oracle.select_experts(c[None, :], K, G, Gk)
        want, want_masked = _brute_group_select(c, K, G, Gk)
        assert set(idx[0].tolist()) == want, (c, G, Gk, K)
        np.testing.assert_array_equal(masked[0], np.array(want_masked, np.float32))


def check_group_special_cases():
    rng = _rng(7)
    c = rng.normal(0.5, 0.2, (64, 48)).astype(np.float32)
    plain, _ = oracle.select_experts(c, 8)
    one, _ = oracle.select_experts(c, 8, 1, 1)
    all_groups, _ = oracle.select_experts(c, 8, 8, 8)
    np.testing.assert_array_equal(plain, one)
    np.testing.assert_array_equal(plain, all_groups)


def check_masked_fill_is_literal_zero():
    # group 0 = experts 0..3, group 1 = experts 4..7; group 0 wins (0.9 > 0.5)
    c = np.array([[0.5, 0.4, -0.2, -0.3, 0.3, 0.2, 0.1, 0.05]], dtype=np.float32)
    idx, masked = oracle.select_experts(c, 4, 2, 1)
    assert idx[0].tolist() == [0, 1, 4, 5]
    assert masked[0, 4:].tolist() == [0.0] * 4


def check_weights():
    rng = _rng(8)
    T, E, K = 32, 24, 6
    z = rng.normal(0, 1, (T, E)).astype(np.float32)
    # bias large enough to reorder biased vs unbiased scores
    b = rng.uniform(-0.4, 0.4, E).astype(np.float32)
    r = oracle.router_from_logits(z, b, K)
    s = 1.0 / (1.0 + np.exp(-z.astype(np.float64)))
    np.testing.assert_allclose(r["w"].sum(1), 2.827, rtol=1e-12)
    # dense G of the Router page's fourth equation, gathered at the selection
    sel = np.zeros((T, E))
    np.put_along_axis(sel, r["idx"], 1.0, axis=1)
    G = 2.827 * s * sel / (s * sel).sum(1, keepdims=True)
    np.testing.assert_allclose(np.take_along_axis(G, r["idx"], 1), r["w"], rtol=1e-13)
    assert ((G > 0).sum(1) == K).all()
    # K = 1 and norm_topk_prob off: no renormalisation, scale still applied
    r1 = oracle.router_from_logits(z, b, 1)
    np.testing.assert_allclose(r1["w"][:, 0], 2.827 * np.take_along_axis(s, r1["idx"], 1)[:, 0], rtol=1e-14)
    rn = oracle.router_from_logits(z, b, K, norm_topk_prob=False)
    np.testing.assert_allclose(rn["w"], 2.827 * np.take_along_axis(s, rn["idx"], 1), rtol=1e-14)


def check_router_from_x():
    rng = _rng(9)
    x = rng.normal(0, 1, (5, 12))
    W = rng.uniform(-0.3, 0.3, (7, 12))
    b = rng.uniform(-0.1, 0.1, 7).astype(np.float32)
    r = oracle.router_from_x(x, W, b, 3)
    for t in range(5):
        for e in range(7):
            want = math.fsum(float(x[t, i]) * float(W[e, i]) for i in range(12))
            assert abs(r["z64"][t, e] - want) <= 1e-15 * max(1.0, abs(want))
    rl = oracle.router_from_logits(np.float32(r["z64"]), b, 3)
    np.testing.assert_array_equal(r["idx"], rl["idx"])


def check_permute():
    rng = _rng(10)
    for T, E, K in [(1, 4, 2), (9, 6, 3), (40, 16, 4), (33, 32, 8)]:
        idx = np.stack([rng.permutation(E)[:K] for _ in range(T)])
        p = oracle.permute(idx, E)
        perm, offsets = [], [0]
        for e in range(E):               # literal: expert-major, tokens ascending
            for t in range(T):
                for k in range(K):
                    if idx[t, k] == e:
                        perm.append(t * K + k)
            offsets.append(len(perm))
        np.testing.assert_array_equal(p["perm"], perm)
        np.testing.assert_array_equal(p["offsets"], offsets)
        np.testing.assert_array_equal(p["counts"], np.diff(offsets))
        assert p["counts"].sum() == T * K
        np.testing.assert_array_equal(p["perm"][p["inv"]], np.arange(T * K))
        np.testing.assert_array_equal(np.sort(p["perm"]), np.arange(T * K))


def check_swiglu_expert():
    rng = _rng(11)
    d, F, m = 24, 10, 7
    u = rng.normal(0, 1, (m, d))
    Wg, Wu, Wd = rng.normal(0, .2, (F, d)), rng.normal(0, .2, (F, d)), rng.normal(0, .2, (d, F))
    np.testing.assert_allclose(oracle.swiglu_expert(u, Wg, Wu, Wd),
                               _dense_swiglu_torch(u, Wg, Wu, Wd), rtol=1e-12, atol=1e-14)


def _small_bank(rng, E, F, d, std=0.2):
    return (rng.normal(0, std, (E, 2 * F, d)), rng.normal(0, std, (E, d, F)))


def check_dense_reduction():
    """E = K, zero router weight and bias: s = 1/2 everywhere, w = 2.827 / K."""
    rng = _rng(12)
    T, d, F, E = 6, 20, 8, 5
    x = rng.normal(0, 1, (T, d))
    Wgu, Wd = _small_bank(rng, E, F, d)
    Sgu, Sd = _small_bank(rng, 1, F, d)
    out = oracle.moe_layer_tokens(x, np.zeros((E, d)), np.zeros(E, np.float32),
                                  Wgu, Wd, Sgu, Sd, K=E)
    np.testing.assert_allclose(out["w"], 2.827 / E, rtol=1e-14)
    want = _dense_swiglu_torch(x, Sgu[0][:F], Sgu[0][F:], Sd[0])
    for e in range(E):
        want = want + (2.827 / E) * _dense_swiglu_torch(x, Wgu[e][:F], Wgu[e][F:], Wd[e])
    np.testing.assert_allclose(out["y"], want, rtol=1e-12, atol=1e-12)
    # E = K = 1: no renormalisation, w = 2.827 * sigmoid(0)
    out1 = oracle.moe_layer_tokens(x, np.zeros((1, d)), np.zeros(1, np.float32),
                                   Wgu[:1], Wd[:1], Sgu, Sd, K=1)
    want1 = _dense_swiglu_torch(x, Sgu[0][:F], Sgu[0][F:], Sd[0]) + \
        1.4135 * _dense_swiglu_torch(x, Wgu[0][:F], Wgu[0][F:], Wd[0])
    np.testing.assert_allclose(out1["y"], want1, rtol=1e-12, atol=1e-12)


def check_layer_routing_weights():
    """Routed part = sum_k w_k f_{idx_k}(x), token by token, with nonzero bias."""
    rng = _rng(13)
    T, d, F, E, K = 9, 16, 6, 8, 3
    x = rng.normal(0, 1, (T, d))
    Wr = rng.uniform(-0.25, 0.25, (E, d))
    b = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    Wgu, Wd = _small_bank(rng, E, F, d)
    out = oracle.moe_layer_tokens(x, Wr, b, Wgu, Wd, None, None, K=K)
    for t in range(T):
        y = np.zeros(d)
        for k in range(K):
            e = out["idx"][t, k]
            y += out["w"][t, k] * _dense_swiglu_torch(x[t:t + 1], Wgu[e][:F], Wgu[e][F:], Wd[e])[0]
        np.testing.assert_allclose(out["y"][t], y, rtol=1e-12, atol=1e-13)


def check_k3_composition():
    """Identity latent projections reduce the K3 form to the K2 form with
    zero-padded routed experts (same router input and shared experts)."""
    rng = _rng(14)
    T, d, L, F, E, K, S = 7, 12, 8, 5, 6, 2, 2
    x = rng.normal(0, 1, (T, d))
    Wr = rng.uniform(-0.3, 0.3, (E, d))
    b = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    Wgu, Wd = _small_bank(rng, E, F, L)
    Sgu, Sd = _small_bank(rng, S, F, d)
    Wdl = np.zeros((L, d))
    Wdl[:, :L] = np.eye(L)
    k3 = oracle.moe_layer_tokens(x, Wr, b, Wgu, Wd, Sgu, Sd, K=K,
                                 W_lat_down64=Wdl, W_lat_up64=Wdl.T)
    Pgu = np.zeros((E, 2 * F, d))
    Pgu[:, :, :L] = Wgu
    Pd = np.zeros((E, d, F))
    Pd[:, :L, :] = Wd
    k2 = oracle.moe_layer_tokens(x, Wr, b, Pgu, Pd, Sgu, Sd, K=K)
    np.testing.assert_array_equal(k3["idx"], k2["idx"])
    np.testing.assert_allclose(k3["y"], k2["y"], rtol=1e-12, atol=1e-13)
    # the latent map is really applied: a non-identity projection changes y
    k3b = oracle.moe_layer_tokens(x, Wr, b, Wgu, Wd, Sgu, Sd, K=K,
                                  W_lat_down64=2.0 * Wdl, W_lat_up64=Wdl.T)
    assert np.abs(k3b["y"] - k3["y"]).max() > 1e-3


def check_page_figures():
    vals = {}
    with open(os.path.join(GOLDEN, "pages_printed_figures.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                k, v = (s.strip() for s in line.split("="))
                vals[k] = float(v)
    k2 = synth.shape("k2_prefill")
    assert k2.d_model * k2.E_routed == vals["router_expert_scores_params"]
    assert k2.d_model * k2.E_routed + k2.E_routed == vals["router_params_per_instance"]
    assert vals["router_params_per_instance"] * vals["moe_blocks"] == vals["router_params_60_blocks"]
    for name in ("k2_router", "k2_decode", "k2_prefill"):
        c = synth.shape(name)
        assert (c.d_model, c.E_routed, c.K) == (vals["router_in_d"], vals["k2_routed_experts"],
                                                vals["k2_experts_per_token"])
        assert c.routed_scaling_factor == vals["routed_scaling_factor"] == oracle.ROUTED_SCALING_FACTOR
    for name in ("k2_decode", "k2_prefill"):
        assert synth.shape(name).E_shared == vals["k2_shared_experts"]
    k3 = synth.shape("k3_latent")
    assert (k3.d_model, k3.E_routed, k3.K, k3.E_shared, k3.d_latent, k3.d_ff) == (
        vals["k3_hidden"], vals["k3_routed_experts"], vals["k3_experts_per_token"],
        vals["k3_shared_experts"], vals["k3_latent"], vals["k3_intermediate"])
    # generated router tensors carry exactly the page's parameter count
    g = synth.generate(synth.custom(T=1, d_model=7168, E_routed=384, K=8, router_only=True))
    assert g["W_r"].numel() + g["bias"].numel() == vals["router_params_per_instance"]


def _brute_gap(c32, K, G, Gk):
    """Smallest margin of a token's decisions, by enumerating pairs: every
    selected vs every unselected masked score, and (G > 1, Gk < G) every kept
    vs every dropped group score (group scores by enumerating member pairs)."""
    E = len(c32)
    gs = E // G
    gscore = []
    for j in range(G):
        members = range(j * gs, (j + 1) * gs)
        gscore.append(max(np.float32(c32[a]) + np.float32(c32[b])
                          for a, b in itertools.permutations(members, 2)))
    kept = _brute_topk(gscore, Gk) if G > 1 else {0}
    masked = [c32[e] if (G == 1 or (e // gs) in kept) else np.float32(0.0) for e in range(E)]
    sel = _brute_topk(masked, K)
    gap = math.inf
    for a in sel:
        for b in set(range(E)) - sel:
            gap = min(gap, float(masked[a]) - float(masked[b]))
    if G > 1:
        for a in kept:
            for b in set(range(G)) - kept:
                gap = min(gap, float(gscore[a]) - float(gscore[b]))
    return gap


def check_gaps():
    c = np.array([[0.9, 0.5, 0.5 + 2 ** -20, 0.1]], dtype=np.float32)
    gap = oracle.selection_gaps(c, 2)
    assert gap[0] == pytest.approx(2 ** -20, rel=1e-6)
    assert oracle.selection_gaps(c, 4)[0] == np.inf
    # group limiting where the group decision binds: E = 8 in 4 groups of 2,
    # keep 2 groups, K = 2.  Group scores (both members summed) are 1.0,
    # 0.9375, 0.921875, 0.4375: groups 0 and 1 are kept with a margin of
    # 0.9375 - 0.921875 = 1/64; the masked scores 0.875, 0.125, 0.5, 0.4375,
    # 0, 0, 0, 0 select experts 0 and 2 with a margin of 0.5 - 0.4375 = 1/16.
    # The token's gap is the smaller one, exactly 1/64 (all values are exact
    # in fp32).
    cg = np.array([[0.875, 0.125, 0.5, 0.4375, 0.625, 0.296875, 0.25, 0.1875]],
                  dtype=np.float32)
    assert set(oracle.select_experts(cg, 2, 4, 2)[0][0].tolist()) == {0, 2}
    assert oracle.selection_gaps(cg, 2, 4, 2)[0] == 1.0 / 64
    # without group limiting the same scores decide only the expert top-2:
    # experts 0 and 4 (0.875, 0.625) against 0.5, margin 1/8
    assert oracle.selection_gaps(cg, 2)[0] == 0.125
    # the pairwise brute force on random tiny tokens, plain and grouped,
    # with many exact ties (values on a coarse grid)
    rng = _rng(21)
    for case in range(300):
        G = int(rng.choice([1, 2, 3, 4]))
        gs = int(rng.integers(2, 4))
        E = G * gs
        Gk = int(rng.integers(1, G + 1))
        K = int(rng.integers(1, min(E, Gk * gs) + 1)) if G > 1 else int(rng.integers(1, E + 1))
        c32 = (rng.integers(0, 24, E) / 16.0 - 0.25).astype(np.float32)
        got = oracle.selection_gaps(c32[None, :], K, G, Gk)[0]
        want = _brute_gap(list(c32), K, G, Gk)
        assert got == want, (case, c32, K, G, Gk, got, want)


def check_combine():
    """The combine of per-slot expert outputs equals the layer's routed sum:
    evaluating every expert on its dispatched rows (slot order of permute),
    combining them with the gate weights and adding the shared experts gives
    the y of moe_layer; and a hand case with K = 2."""
    Y = np.array([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0], [7.0, 8.0]])
    inv = np.array([2, 0, 3, 1])  # token 0: slots 2, 0; token 1: slots 3, 1
    w = np.array([[0.5, 0.25], [1.0, 2.0]])
    Ys = np.array([[[10.0, 20.0], [30.0, 40.0]]])
    y = oracle.combine(Y, inv, w, Ys)
    np.testing.assert_array_equal(y, [[0.5 * 5 + 0.25 * 1 + 10, 0.5 * 6 + 0.25 * 2 + 20],
                                      [7 + 2 * 3 + 30, 8 + 2 * 4 + 40]])
    rng = _rng(22)
    T, d, E, K, F = 12, 16, 6, 3, 8
    gu, dn = _small_bank(rng, E, F, d)
    sgu, sdn = _small_bank(rng, 1, F, d)
    x = rng.normal(size=(T, d))
    Wr = rng.normal(size=(E, d)) * 0.3
    b = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    ref = oracle.moe_layer_tokens(x, Wr, b, gu, dn, sgu, sdn, K)
    p = oracle.permute(ref["idx"], E)
    Yslot = np.zeros((T * K, d))
    for e in range(E):
        for r in range(p["offsets"][e], p["offsets"][e + 1]):
            t = p["perm"][r] // K
            Yslot[r] = oracle.swiglu_expert(x[t:t + 1], gu[e, :F], gu[e, F:], dn[e])[0]
    Ysh = oracle.swiglu_expert(x, sgu[0, :F], sgu[0, F:], sdn[0])[None]
    np.testing.assert_allclose(oracle.combine(Yslot, p["inv"], ref["w"], Ysh), ref["y"],
                               rtol=1e-12, atol=1e-12)


def check_dense_gates():
    """G [T, E] from a real routing: exactly K non-zero entries per row, at
    the selected experts, holding their weights; each row sums to the
    scaling factor when the weights are renormalised (the G equation's
    numerator over its denominator sums to 1)."""
    rng = np.random.default_rng(11)
    T, E, K = 40, 32, 4
    z = rng.normal(size=(T, E)).astype(np.float32)
    b = rng.uniform(-0.1, 0.1, size=E).astype(np.float32)
    r = oracle.router_from_logits(z, b, K)
    G = oracle.dense_gates(r["idx"], r["w"], E)
    assert G.shape == (T, E)
    assert ((G != 0).sum(axis=1) == K).all()
    for t in range(T):
        for k in range(K):
            assert G[t, r["idx"][t, k]] == r["w"][t, k]
    np.testing.assert_allclose(G.sum(axis=1), oracle.ROUTED_SCALING_FACTOR, rtol=1e-12)
    # without renormalisation a row holds scale * s of its selected experts
    r1 = oracle.router_from_logits(z, b, K, norm_topk_prob=False)
    G1 = oracle.dense_gates(r1["idx"], r1["w"], E)
    s = oracle.sigmoid(z.astype(np.float64))
    sel = G1 != 0
    np.testing.assert_allclose(G1[sel], oracle.ROUTED_SCALING_FACTOR * s[sel], rtol=1e-12)


def check_bias_update():
    """Special cases of the sign-only update with gamma: a batch whose loads
    all equal the mean leaves b unchanged bit for bit; when one expert takes
    every pair, its bias drops by gamma and every other rises by gamma; an
    expert's direction depends only on whether its load is above or below
    T K / E (here the mean, 2, is met by experts 1 and 2)."""
    g = np.float32(1e-3)
    b = np.array([0.25, -0.5, 0.125, 0.0], dtype=np.float32)
    T, K, E = 4, 2, 4                       # T K = 8 pairs, mean load 2
    same = oracle.aux_free_bias_update(b, [2, 2, 2, 2], T, K)
    assert same.dtype == np.float32 and (same == b).all()
    one = oracle.aux_free_bias_update(b, [8, 0, 0, 0], T, K)
    assert one[0] == np.float32(0.25) - g
    assert (one[1:] == b[1:] + g).all()
    mixed = oracle.aux_free_bias_update(b, [5, 2, 2, 0], T, K)
    assert mixed[0] < b[0] and mixed[1] == b[1] and mixed[2] == b[2] and mixed[3] > b[3]
    # many steps with a fixed imbalance move the biases linearly, in fp32
    bb = b.copy()
    for _ in range(10):
        bb = oracle.aux_free_bias_update(bb, [8, 0, 0, 0], T, K)
    assert abs(float(bb[0]) - (0.25 - 10e-3)) < 1e-6 and abs(float(bb[3]) - 10e-3) < 1e-6


def _scores_f32(z32):
    """fp32 router scores written out element by element: the fp64 logistic
    function of each logit, rounded once to fp32."""
    z32 = np.asarray(z32, dtype=np.float32)
    out = np.empty(z32.shape, dtype=np.float32)
    for idx in np.ndindex(z32.shape):
        out[idx] = np.float32(1.0 / (1.0 + math.exp(-float(z32[idx]))))
    return out


def check_quantile_bias():
    """Quantile Balancing (the K3 page's training-side bias update, read as
    documented in the oracle): the threshold is an order statistic of each
    expert's scores; equal score distributions need no correction; rate 0
    keeps the bias, rate 1 sets it to the common cut-off minus the
    threshold; one update makes a skewed batch's loads more even."""
    # thresholds against a counting definition: theta is a score of the
    # column with at least r scores >= theta and fewer than r scores > theta
    rng = _rng(31)
    for case in range(60):
        T = int(rng.integers(1, 40))
        E = int(rng.integers(1, 9))
        K = int(rng.integers(1, E + 1))
        z = (rng.integers(-8, 8, (T, E)) / 4.0).astype(np.float32)  # many ties
        b = rng.uniform(-0.1, 0.1, E).astype(np.float32)
        theta, nb = oracle.quantile_bias_update(z, b, K, rate=0.0)
        assert (nb == b).all()
        sc = _scores_f32(z)
        r = -(-(T * K) // E)
        for e in range(E):
            col = sc[:, e]
            assert theta[e] in col
            assert (col >= theta[e]).sum() >= r and (col > theta[e]).sum() < r
    # hand case: T = 4, E = 2, K = 1, so each expert's target is 2 tokens and
    # its threshold the 2nd largest score; the cut-off is their mean
    z = np.array([[2.0, -1.0], [1.5, -0.5], [-2.0, 0.5], [-1.0, 0.25]], dtype=np.float32)
    sc = _scores_f32(z)
    theta, nb = oracle.quantile_bias_update(z, np.zeros(2, np.float32), 1, rate=1.0)
    assert theta[0] == sc[1, 0] and theta[1] == sc[3, 1]
    tau = (float(theta[0]) + float(theta[1])) / 2
    assert nb[0] == np.float32(tau - float(theta[0])) and nb[1] == np.float32(tau - float(theta[1]))
    assert nb[0] < 0 < nb[1]  # the expert with the higher threshold is pushed down
    # columns that hold the same scores in other orders: one threshold, no
    # correction -- whatever the previous bias, rate 1 takes it to zero
    base = rng.normal(size=24).astype(np.float32)
    zc = np.stack([rng.permutation(base) for _ in range(6)], axis=1)
    b = rng.uniform(-0.1, 0.1, 6).astype(np.float32)
    theta, nb = oracle.quantile_bias_update(zc, b, 2, rate=1.0)
    assert (theta == theta[0]).all() and (nb == 0).all()
    _, half = oracle.quantile_bias_update(zc, b, 2, rate=0.5)
    np.testing.assert_array_equal(half, (b.astype(np.float64) * 0.5).astype(np.float32))
    # a batch routed unevenly (per-expert offsets in the logits): after one
    # rate-1 update the selection with the new bias spreads the same tokens
    # more evenly
    T, E, K = 512, 16, 2
    z = (rng.normal(size=(T, E)) + np.linspace(-1.5, 1.5, E)).astype(np.float32)
    c0 = oracle.biased_scores_f32(z, np.zeros(E, np.float32))
    load0 = np.bincount(oracle.select_experts(c0, K)[0].reshape(-1), minlength=E)
    _, nb = oracle.quantile_bias_update(z, np.zeros(E, np.float32), K, rate=1.0)
    load1 = np.bincount(oracle.select_experts(oracle.biased_scores_f32(z, nb), K)[0].reshape(-1),
                        minlength=E)
    assert load1.max() < 0.6 * load0.max() and load1.min() > 2 * max(load0.min(), 1)


ALL_CHECKS = [
    check_sigmoid_closed_forms, check_silu, check_bf16_upcast, check_biased_scores_fp32,
    check_select_plain_bruteforce, check_select_grouped_bruteforce, check_group_special_cases,
    check_masked_fill_is_literal_zero, check_weights, check_router_from_x, check_permute,
    check_swiglu_expert, check_dense_reduction, check_layer_routing_weights,
    check_k3_composition, check_page_figures, check_gaps, check_combine, check_dense_gates,
    check_bias_update, check_quantile_bias,
]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check()


# --------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail
# --------------------------------------------------------------------------
def _softmax_like(z):
    z = np.asarray(z, dtype=np.float64)
    return np.exp(z) / (1.0 + np.exp(z)) * (1 + 1e-3)


def _swapped_swiglu(u, Wg, Wu, Wd):
    u = np.asarray(u, np.float64)
    return (mo.silu(u @ np.asarray(Wu).T) * (u @ np.asarray(Wg).T)) @ np.asarray(Wd).T


def _weights_without_scale(s, K, scale=2.827, norm=True):
    s = np.asarray(s, np.float64)
    return s / s.sum(-1, keepdims=True)


def _group_top1(c32, n_group):
    T, E = c32.shape
    return np.sort(c32.reshape(T, n_group, E // n_group), axis=-1)[..., -1] * np.float32(2)


def _order_index_desc(values):
    n = values.shape[-1]
    position = np.broadcast_to(-np.arange(n), values.shape)
    return np.lexsort((position, -values), axis=-1)


def _permute_token_major(idx, E):
    p = mo._orig_permute(idx, E)
    flat = np.asarray(idx).reshape(-1)
    order = np.lexsort((-np.arange(flat.size), flat))
    p["perm"] = order
    p["inv"] = np.empty_like(order)
    p["inv"][order] = np.arange(order.size)
    return p


def _masked_neg_inf_select(c32, K, n_group=1, topk_group=1):
    c32 = np.asarray(c32, dtype=np.float32)
    T, E = c32.shape
    masked = c32.copy()
    if n_group > 1:
        gscore = mo.group_scores_f32(c32, n_group)
        kept = mo._canonical_order(gscore)[:, :topk_group]
        keep = np.zeros((T, n_group), dtype=bool)
        np.put_along_axis(keep, kept, True, axis=1)
        masked[~np.repeat(keep, E // n_group, axis=1)] = -np.inf
    return mo._canonical_order(masked)[:, :K].astype(np.int64), masked


def _biased_weights_router(z32, bias32, K, n_group=1, topk_group=1, scale=2.827, norm_topk_prob=True):
    out = mo._orig_router_from_logits(z32, bias32, K, n_group, topk_group, scale, norm_topk_prob)
    c = np.take_along_axis(out["c32"].astype(np.float64), out["idx"], 1)
    out["w"] = mo.router_weights(c, K, scale, norm_topk_prob)
    return out


def _dense_gates_transposed(idx, w, E):
    G = np.zeros((np.asarray(idx).shape[0], E))
    G[np.arange(G.shape[0])[:, None], np.asarray(idx)[:, ::-1]] = np.asarray(w)
    return G


def _bias_update_wrong_sign(bias32, counts, T, K, gamma=1e-3):
    return mo._orig_bias_update(bias32, counts, T, K, -gamma)


def _gaps_without_groups(c32, K, n_group=1, topk_group=1):
    return mo._orig_selection_gaps(c32, K, 1, 1) if n_group == 1 else \
        _expert_gap_only(c32, K, n_group, topk_group)


def _expert_gap_only(c32, K, n_group, topk_group):
    _, masked = mo.select_experts(np.asarray(c32, np.float32), K, n_group, topk_group)
    srt = -np.sort(-masked.astype(np.float64), axis=-1)
    return srt[:, K - 1] - srt[:, K] if K < masked.shape[1] else np.full(masked.shape[0], np.inf)


def _gaps_group_rank_shifted(c32, K, n_group=1, topk_group=1):
    gap = _expert_gap_only(c32, K, n_group, topk_group)
    if n_group > 1 and topk_group + 1 < n_group:  # one rank too far down
        g = -np.sort(-mo.group_scores_f32(np.asarray(c32, np.float32), n_group).astype(np.float64), -1)
        gap = np.minimum(gap, g[:, topk_group] - g[:, topk_group + 1])
    return gap


def _combine_by_perm(Y, inv, w, Y_shared=None):
    # reads Y through the inverse map's inverse (perm) instead of inv
    inv = np.asarray(inv)
    perm = np.empty_like(inv)
    perm[inv] = np.arange(inv.size)
    return mo._orig_combine(Y, perm, w, Y_shared)


def _qb_variant(z32, bias32, K, rate=1.0, rank_shift=0, sign=1, biased=False, smallest=False):
    z32 = np.asarray(z32, dtype=np.float32)
    T, E = z32.shape
    s32 = mo.round_f32(mo.sigmoid(z32.astype(np.float64)))
    if biased:
        s32 = s32 + np.asarray(bias32, np.float32)[None, :]
    r = min(T, -(-(T * K) // E) + rank_shift)
    srt = np.sort(s32, axis=0) if smallest else -np.sort(-s32, axis=0)
    theta = srt[r - 1].astype(np.float32)
    tau = sum(float(v) for v in theta) / E
    b = np.asarray(bias32, np.float32).astype(np.float64)
    new = b + float(np.float32(rate)) * (sign * (tau - theta.astype(np.float64)) - b)
    return theta, mo.round_f32(new)


MUTANTS = {
    "sigmoid_not_logistic": ("sigmoid", _softmax_like),
    "gate_up_swapped": ("swiglu_expert", _swapped_swiglu),
    "scaling_dropped": ("router_weights", _weights_without_scale),
    "group_score_top1": ("group_scores_f32", _group_top1),
    "ties_to_higher_index": ("_canonical_order", _order_index_desc),
    "permute_not_stable": ("permute", _permute_token_major),
    "masked_fill_neg_inf": ("select_experts", _masked_neg_inf_select),
    "weights_from_biased_scores": ("router_from_logits", _biased_weights_router),
    "dense_gates_misplaced": ("dense_gates", _dense_gates_transposed),
    "bias_update_wrong_sign": ("aux_free_bias_update", _bias_update_wrong_sign),
    "gaps_ignore_group_decision": ("selection_gaps", _gaps_without_groups),
    "gaps_group_rank_shifted": ("selection_gaps", _gaps_group_rank_shifted),
    "combine_reads_perm": ("combine", _combine_by_perm),
    "qb_rank_off_by_one": ("quantile_bias_update",
                           lambda z, b, K, rate=1.0: _qb_variant(z, b, K, rate, rank_shift=1)),
    "qb_sign_flipped": ("quantile_bias_update",
                        lambda z, b, K, rate=1.0: _qb_variant(z, b, K, rate, sign=-1)),
    "qb_quantile_of_biased_scores": ("quantile_bias_update",
                                     lambda z, b, K, rate=1.0: _qb_variant(z, b, K, rate,
                                                                           biased=True)),
    "qb_smallest_scores": ("quantile_bias_update",
                           lambda z, b, K, rate=1.0: _qb_variant(z, b, K, rate, smallest=True)),
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistakes_are_caught(mutant, monkeypatch):
    name, fn = MUTANTS[mutant]
    monkeypatch.setattr(mo, "_orig_permute", mo.permute, raising=False)
    monkeypatch.setattr(mo, "_orig_router_from_logits", mo.router_from_logits, raising=False)
    monkeypatch.setattr(mo, "_orig_bias_update", mo.aux_free_bias_update, raising=False)
    monkeypatch.setattr(mo, "_orig_selection_gaps", mo.selection_gaps, raising=False)
    monkeypatch.setattr(mo, "_orig_combine", mo.combine, raising=False)
    monkeypatch.setattr(mo, name, fn)
    # the package namespace re-exports the functions: patch it too
    if hasattr(oracle, name):
        monkeypatch.setattr(oracle, name, fn)
    failed = []
    for check in ALL_CHECKS:
        try:
            check()
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"no pin caught the planted mistake {mutant}"
