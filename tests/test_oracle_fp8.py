"""Pins of the oracle's FP8 block-scaled weight reading (CPU only).

The pages say only that the K2 checkpoint's tensors carry FP8 block scales
("Kimi K2 · Router · OpenModelAtlas", Parameters).  The oracle reads that as
OCP E4M3 codes with one fp32 multiplier per 128 x 128 block.  These tests pin
the decoder to torch's own float8_e4m3fn conversion and to the encoding's
closed forms, the block dequantisation to a brute-force loop, and the FP8
layer to the bf16 layer on weights that both forms hold exactly; each
planted mistake below must be caught by one of them.
"""
import numpy as np
import pytest
import torch

import oracle
import synth


def _codes():
    return np.arange(256, dtype=np.uint8)


def test_e4m3_matches_torch_float8_cast():
    c = _codes()
    want = torch.from_numpy(c.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_to_f64(c)
    np.testing.assert_array_equal(got, want)  # NaN positions compare equal too


def test_e4m3_closed_forms():
    v = oracle.e4m3_to_f64(_codes())
    assert v[0x00] == 0.0 and np.signbit(v[0x80])
    assert v[0x01] == 2.0 ** -9            # smallest subnormal
    assert v[0x07] == 7 * 2.0 ** -9        # largest subnormal
    assert v[0x08] == 2.0 ** -6            # smallest normal
    assert v[0x38] == 1.0                  # exponent field 7 = bias
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert np.isfinite(np.delete(v, [0x7F, 0xFF])).all()  # no infinities


def test_e4m3_order_sign_and_spacing():
    v = oracle.e4m3_to_f64(_codes())
    pos = v[:0x7F]
    assert (np.diff(pos) > 0).all()
    np.testing.assert_array_equal(v[0x81:0xFF], -v[0x01:0x7F])
    # within a binade the step is 2^(e - 7 - 3); subnormals step 2^-9
    for c in range(0x00, 0x7E):
        e = c >> 3
        step = 2.0 ** (max(e, 1) - 10)
        assert v[c + 1] - v[c] == step, hex(c)


def _brute_dequant(q, s, block=128):
    out = np.empty(q.shape, dtype=np.float64)
    vals = oracle.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    G, R, C = q.shape
    for g in range(G):
        for r in range(R):
            for c in range(C):
                out[g, r, c] = vals[q[g, r, c]] * float(s[g, r // block, c // block])
    return out


def _small_bank(seed=0, G=2, R=256, C=384):
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 256, size=(G, R, C), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    s = rng.uniform(0.5, 2.0, size=(G, -(-R // 128), -(-C // 128)))
    return q, s


@pytest.mark.parametrize("R,C", [(256, 384), (200, 136)], ids=["whole_blocks", "ragged_blocks"])
def test_dequant_blocks_brute_force(R, C):
    q, s = _small_bank(R=R, C=C)
    np.testing.assert_array_equal(oracle.dequant_fp8_blocks(q, s), _brute_dequant(q, s))


def _planted_transposed(q, s):
    # block index taken as (column block, row block)
    st = np.swapaxes(s, -1, -2)
    full = np.repeat(np.repeat(st, 128, -2), 128, -1)
    full = np.resize(full, q.shape) if full.shape != q.shape else full
    return oracle.e4m3_to_f64(q) * full


def _planted_row_block_only(q, s):
    # the column block index dropped: every column takes block column 0
    full = np.repeat(np.repeat(s[..., :1], 128, -2), q.shape[-1], -1)
    return oracle.e4m3_to_f64(q) * full[..., :q.shape[-2], :]


@pytest.mark.parametrize("mutant", [_planted_transposed, _planted_row_block_only])
def test_dequant_planted_mistakes_are_caught(mutant):
    q, s = _small_bank(seed=1, R=384, C=256)  # 3 x 2 blocks
    good = _brute_dequant(q, s)
    assert not np.array_equal(mutant(q, s), good)


def _exact_fp8_layer_case():
    """Banks whose block multipliers are powers of two, so every weight is
    exactly a bf16 number as well as code x scale."""
    shape = synth.custom(name="fp8pin", T=24, d_model=256, E_routed=6, K=2, E_shared=1,
                         d_ff=128, d_ff_shared=128, weights="fp8", x_dist="clusters32")
    g = synth.generate(shape)
    rng = np.random.default_rng(7)
    for k in [k for k in g if k.endswith("_s")]:
        g[k] = torch.from_numpy(2.0 ** rng.integers(-12, -6, size=tuple(g[k].shape))).float()
    return shape, g


def _np(t):
    return t.to(torch.float64).numpy() if t.dtype != torch.uint8 else t.numpy()


def test_fp8_layer_equals_bf16_layer_on_exact_weights():
    shape, g = _exact_fp8_layer_case()
    x = _np(g["x"])
    deq = {k: oracle.dequant_fp8_blocks(_np(g[k + "_q"]), _np(g[k + "_s"]))
           for k in ("W_gate_up", "W_down", "Ws_gate_up", "Ws_down")}
    for v in deq.values():  # every weight is a bf16 number
        np.testing.assert_array_equal(torch.from_numpy(v).to(torch.bfloat16).double().numpy(), v)
    common = dict(K=shape.K, n_group=shape.n_group, topk_group=shape.topk_group)
    ref = oracle.moe_layer_tokens(x, _np(g["W_r"]), _np(g["bias"]), deq["W_gate_up"],
                                  deq["W_down"], deq["Ws_gate_up"], deq["Ws_down"], **common)
    got = oracle.moe_layer_tokens_fp8(
        x, _np(g["W_r"]), _np(g["bias"]), _np(g["W_gate_up_q"]), _np(g["W_gate_up_s"]),
        _np(g["W_down_q"]), _np(g["W_down_s"]), _np(g["Ws_gate_up_q"]), _np(g["Ws_gate_up_s"]),
        _np(g["Ws_down_q"]), _np(g["Ws_down_s"]), **common)
    np.testing.assert_array_equal(got["idx"], ref["idx"])
    np.testing.assert_array_equal(got["y"], ref["y"])
    # a planted mistake: the gate and up halves' scale rows exchanged
    gs = _np(g["W_gate_up_s"]).copy()
    half = gs.shape[1] // 2
    gs = np.concatenate([gs[:, half:], gs[:, :half]], axis=1)
    bad = oracle.moe_layer_tokens_fp8(
        x, _np(g["W_r"]), _np(g["bias"]), _np(g["W_gate_up_q"]), gs,
        _np(g["W_down_q"]), _np(g["W_down_s"]), _np(g["Ws_gate_up_q"]), _np(g["Ws_gate_up_s"]),
        _np(g["Ws_down_q"]), _np(g["Ws_down_s"]), **common)
    assert not np.allclose(bad["y"], ref["y"])


def test_synth_fp8_checkpoint_has_no_nan_codes_and_normal_weights():
    shape = synth.custom(name="fp8stat", T=4, d_model=512, E_routed=2, K=1, d_ff=256,
                         weights="fp8")
    g = synth.generate(shape)
    q = g["W_gate_up_q"].numpy()
    assert not ((q & 0x7F) == 0x7F).any()
    w = oracle.dequant_fp8_blocks(q, g["W_gate_up_s"].numpy())
    assert 0.015 < w.std() < 0.03
