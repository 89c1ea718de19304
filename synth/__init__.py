"""Seeded synthetic inputs for the fine-grained MoE layer.

This module is the only code shared by the CUDA path's tests/benchmark and the
CPU oracle.  It draws random tensors and nothing else: no step of the layer's
arithmetic lives here.

Shapes follow the pages' statement of the layer:
  * Kimi K2 (d_model 7168, 384 routed experts, top-8, 1 shared expert) --
    "Kimi K2 MoE", section 2 (Derivation); "Kimi K2" (visual-learn), "Many
    experts, few used at a time"; "Kimi K2 · Router", parameter table
    (gate weight 7168 x 384 plus a 384-entry bias).
  * Kimi K3 (896 routed, top-16, 2 shared at 7168, latent 3584, intermediate
    3072) -- "Kimi K3's router picks 16 of 896 experts", K3 table.

Distributions: router weight kaiming-uniform with a = sqrt(5) (the pages'
``reset_parameters``), i.e. U(-1/sqrt(d), 1/sqrt(d)); selection bias uniform;
expert weights N(0, 0.02); activations N(0, 1) or a 32-cluster Gaussian
mixture (centres N(0, I), unit noise) so that routing is skewed.

Weight layouts (row-major, ``nn.Linear`` convention out x in):
  W_r         [E, d]            fp32
  bias        [E]               fp32
  W_gate_up   [E, 2F, d]        rows 0..F-1 gate, rows F..2F-1 up
  W_down      [E, d_out, F]
  Ws_gate_up  [S, 2Fs, d]       shared experts, same convention
  Ws_down     [S, d, Fs]
  W_lat_down  [L, d]            K3 latent down-projection (d -> L)
  W_lat_up    [d, L]            K3 latent up-projection (L -> d)
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch

__all__ = ["LayerShape", "CONFIGS", "SEEDS", "shape", "generate", "custom", "activations",
           "router_params", "routed_expert", "shared_expert", "latent_projections",
           "routed_expert_fp8", "shared_expert_fp8", "FP8_BLOCK"]


@dataclasses.dataclass(frozen=True)
class LayerShape:
    name: str
    T: int
    d_model: int
    E_routed: int
    K: int
    E_shared: int = 0
    d_ff: int = 0
    d_ff_shared: int = 0
    n_group: int = 1
    topk_group: int = 1
    routed_scaling_factor: float = 2.827
    norm_topk_prob: bool = True
    d_latent: int = 0
    dtype: str = "bf16"          # "f32" or "bf16": activations and expert weights
    x_dist: str = "normal"       # "normal" or "clusters32"
    bias_range: float = 0.1
    router_only: bool = False
    # "bf16", or "fp8": routed and shared expert weights as FP8 E4M3 codes
    # with one fp32 multiplier per 128 x 128 block (the K3 latent
    # projections stay bf16)
    weights: str = "bf16"

    @property
    def d_expert(self) -> int:
        """Width the routed experts work on (the latent width for K3)."""
        return self.d_latent if self.d_latent else self.d_model


CONFIGS: Dict[str, LayerShape] = {
    "tiny": LayerShape("tiny", T=64, d_model=256, E_routed=16, K=4, E_shared=1,
                       d_ff=64, d_ff_shared=64, dtype="f32", bias_range=0.1),
    "k2_router": LayerShape("k2_router", T=4096, d_model=7168, E_routed=384, K=8,
                            dtype="bf16", bias_range=0.05, router_only=True),
    "k2_decode": LayerShape("k2_decode", T=128, d_model=7168, E_routed=384, K=8,
                            E_shared=1, d_ff=2048, d_ff_shared=2048,
                            x_dist="clusters32", bias_range=0.1),
    "k2_prefill": LayerShape("k2_prefill", T=8192, d_model=7168, E_routed=384, K=8,
                             E_shared=1, d_ff=2048, d_ff_shared=2048, n_group=8,
                             topk_group=4, x_dist="clusters32", bias_range=0.1),
    "k3_latent": LayerShape("k3_latent", T=4096, d_model=7168, E_routed=896, K=16,
                            E_shared=2, d_ff=3072, d_ff_shared=3072, d_latent=3584,
                            bias_range=0.1),
}

for _n in ("k2_decode", "k2_prefill", "k3_latent"):
    CONFIGS[_n + "_fp8"] = dataclasses.replace(CONFIGS[_n], name=_n + "_fp8", weights="fp8")

# the FP8 forms draw x, W_r and the bias from their bf16 forms' seeds
SEEDS = {"tiny": 0, "k2_router": 1, "k2_decode": 2, "k2_prefill": 3, "k3_latent": 4,
         "k2_decode_fp8": 2, "k2_prefill_fp8": 3, "k3_latent_fp8": 4}


def shape(name: str) -> LayerShape:
    return CONFIGS[name]


def custom(**kw) -> LayerShape:
    kw.setdefault("name", "custom")
    return LayerShape(**kw)


def _wdtype(cfg: LayerShape) -> torch.dtype:
    return torch.float32 if cfg.dtype == "f32" else torch.bfloat16


# Every tensor has its own generator, seeded from (seed, stream id), so one
# expert's weights can be drawn without drawing the others.
_STREAM_X, _STREAM_WR, _STREAM_BIAS, _STREAM_LAT_DOWN, _STREAM_LAT_UP = 1, 2, 3, 4, 5
_STREAM_SHARED, _STREAM_ROUTED = 100, 1000
_STREAM_SHARED_FP8, _STREAM_ROUTED_FP8 = 500, 100000
FP8_BLOCK = 128
FP8_CODE_STD = 112.0  # codes ~ N(0, 112^2): the largest of a block's ~16k near 448


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed << 24) + stream)
    return g


def _normal(gen, shp, std, device, dtype):
    t = torch.randn(shp, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def _uniform(gen, shp, lo, hi, device):
    t = torch.rand(shp, generator=gen, device=device, dtype=torch.float32)
    return t.mul_(hi - lo).add_(lo)


def _seed(cfg: LayerShape, seed: Optional[int]) -> int:
    return SEEDS.get(cfg.name, 12345) if seed is None else seed


def activations(cfg: LayerShape, device="cpu", seed: Optional[int] = None,
                T: Optional[int] = None) -> torch.Tensor:
    """x [T, d_model]: N(0, 1), or a 32-cluster Gaussian mixture (centres
    N(0, I), cluster chosen uniformly, unit noise)."""
    T = cfg.T if T is None else T
    gen = _gen(_seed(cfg, seed), _STREAM_X, device)
    dt = _wdtype(cfg)
    if cfg.x_dist == "normal":
        return _normal(gen, (T, cfg.d_model), 1.0, device, dt)
    if cfg.x_dist == "clusters32":
        centres = torch.randn((32, cfg.d_model), generator=gen, device=device)
        which = torch.randint(0, 32, (T,), generator=gen, device=device)
        noise = torch.randn((T, cfg.d_model), generator=gen, device=device)
        return (centres[which] + noise).to(dt)
    raise ValueError(cfg.x_dist)


def router_params(cfg: LayerShape, device="cpu", seed: Optional[int] = None):
    """(W_r [E, d] fp32 kaiming-uniform with a = sqrt(5), bias [E] fp32)."""
    s = _seed(cfg, seed)
    d, E = cfg.d_model, cfg.E_routed
    bound = 1.0 / math.sqrt(d)  # kaiming_uniform(a=sqrt(5)): gain*sqrt(3/fan_in)
    W_r = _uniform(_gen(s, _STREAM_WR, device), (E, d), -bound, bound, device)
    bias = _uniform(_gen(s, _STREAM_BIAS, device), (E,), -cfg.bias_range, cfg.bias_range, device)
    return W_r, bias


def routed_expert(cfg: LayerShape, e: int, device="cpu", seed: Optional[int] = None):
    """(W_gate_up [2F, d_e], W_down [d_e, F]) of routed expert e, N(0, 0.02)."""
    g = _gen(_seed(cfg, seed), _STREAM_ROUTED + e, device)
    dt, de, F = _wdtype(cfg), cfg.d_expert, cfg.d_ff
    return _normal(g, (2 * F, de), 0.02, device, dt), _normal(g, (de, F), 0.02, device, dt)


def shared_expert(cfg: LayerShape, s_idx: int, device="cpu", seed: Optional[int] = None):
    """(Ws_gate_up [2Fs, d], Ws_down [d, Fs]) of shared expert s_idx."""
    g = _gen(_seed(cfg, seed), _STREAM_SHARED + s_idx, device)
    dt, d, Fs = _wdtype(cfg), cfg.d_model, cfg.d_ff_shared
    return _normal(g, (2 * Fs, d), 0.02, device, dt), _normal(g, (d, Fs), 0.02, device, dt)


def _fp8_matrix(gen, rows: int, cols: int, device):
    """A block-scaled FP8 E4M3 matrix: (codes [rows, cols] uint8, scales
    [ceil(rows/128), ceil(cols/128)] fp32).  Code values are drawn N(0, 112^2)
    clamped to +-448 and rounded to E4M3 by torch's float8 cast; the block
    multipliers U(0.5, 1.5) * 0.02 / 112, so the weights are about N(0, 0.02)."""
    v = torch.randn((rows, cols), generator=gen, device=device, dtype=torch.float32)
    codes = v.mul_(FP8_CODE_STD).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    nb = ((rows + FP8_BLOCK - 1) // FP8_BLOCK, (cols + FP8_BLOCK - 1) // FP8_BLOCK)
    scales = _uniform(gen, nb, 0.5, 1.5, device).mul_(0.02 / FP8_CODE_STD)
    return codes, scales


def routed_expert_fp8(cfg: LayerShape, e: int, device="cpu", seed: Optional[int] = None):
    """(gu codes [2F, d_e], gu scales, down codes [d_e, F], down scales) of
    routed expert e in the FP8 block-scaled form."""
    g = _gen(_seed(cfg, seed), _STREAM_ROUTED_FP8 + e, device)
    de, F = cfg.d_expert, cfg.d_ff
    return (*_fp8_matrix(g, 2 * F, de, device), *_fp8_matrix(g, de, F, device))


def shared_expert_fp8(cfg: LayerShape, s_idx: int, device="cpu", seed: Optional[int] = None):
    """(gu codes [2Fs, d], gu scales, down codes [d, Fs], down scales)."""
    g = _gen(_seed(cfg, seed), _STREAM_SHARED_FP8 + s_idx, device)
    d, Fs = cfg.d_model, cfg.d_ff_shared
    return (*_fp8_matrix(g, 2 * Fs, d, device), *_fp8_matrix(g, d, Fs, device))


def latent_projections(cfg: LayerShape, device="cpu", seed: Optional[int] = None):
    """(W_lat_down [L, d], W_lat_up [d, L]), N(0, 0.02)."""
    s, dt, d, L = _seed(cfg, seed), _wdtype(cfg), cfg.d_model, cfg.d_latent
    return (_normal(_gen(s, _STREAM_LAT_DOWN, device), (L, d), 0.02, device, dt),
            _normal(_gen(s, _STREAM_LAT_UP, device), (d, L), 0.02, device, dt))


def generate(cfg: LayerShape, device="cpu", seed: Optional[int] = None,
             T: Optional[int] = None, weights: bool = True) -> Dict[str, torch.Tensor]:
    """Draw every input of one layer call.  Deterministic for (seed, device)."""
    out: Dict[str, torch.Tensor] = {"x": activations(cfg, device, seed, T)}
    out["W_r"], out["bias"] = router_params(cfg, device, seed)
    if cfg.router_only or not weights:
        return out
    dt, de, F, E = _wdtype(cfg), cfg.d_expert, cfg.d_ff, cfg.E_routed
    if cfg.weights == "fp8":
        _generate_fp8(cfg, device, seed, out)
        if cfg.d_latent:
            out["W_lat_down"], out["W_lat_up"] = latent_projections(cfg, device, seed)
        return out
    W_gate_up = torch.empty((E, 2 * F, de), device=device, dtype=dt)
    W_down = torch.empty((E, de, F), device=device, dtype=dt)
    for e in range(E):
        W_gate_up[e], W_down[e] = routed_expert(cfg, e, device, seed)
    out["W_gate_up"], out["W_down"] = W_gate_up, W_down
    S, Fs = cfg.E_shared, cfg.d_ff_shared
    if S:
        Ws_gate_up = torch.empty((S, 2 * Fs, cfg.d_model), device=device, dtype=dt)
        Ws_down = torch.empty((S, cfg.d_model, Fs), device=device, dtype=dt)
        for s in range(S):
            Ws_gate_up[s], Ws_down[s] = shared_expert(cfg, s, device, seed)
        out["Ws_gate_up"], out["Ws_down"] = Ws_gate_up, Ws_down
    if cfg.d_latent:
        out["W_lat_down"], out["W_lat_up"] = latent_projections(cfg, device, seed)
    return out


def _bank(n: int, rows: int, cols: int, device):
    nb = ((rows + FP8_BLOCK - 1) // FP8_BLOCK, (cols + FP8_BLOCK - 1) // FP8_BLOCK)
    return (torch.empty((n, rows, cols), device=device, dtype=torch.uint8),
            torch.empty((n, *nb), device=device, dtype=torch.float32))


def _generate_fp8(cfg: LayerShape, device, seed, out: Dict[str, torch.Tensor]) -> None:
    """FP8 expert banks: W_gate_up_q/_s, W_down_q/_s and the shared experts'
    Ws_gate_up_q/_s, Ws_down_q/_s (codes uint8, block scales fp32)."""
    de, F, E = cfg.d_expert, cfg.d_ff, cfg.E_routed
    gq, gs = _bank(E, 2 * F, de, device)
    dq, ds = _bank(E, de, F, device)
    for e in range(E):
        gq[e], gs[e], dq[e], ds[e] = routed_expert_fp8(cfg, e, device, seed)
    out.update(W_gate_up_q=gq, W_gate_up_s=gs, W_down_q=dq, W_down_s=ds)
    S, Fs, d = cfg.E_shared, cfg.d_ff_shared, cfg.d_model
    if S:
        sgq, sgs = _bank(S, 2 * Fs, d, device)
        sdq, sds = _bank(S, d, Fs, device)
        for i in range(S):
            sgq[i], sgs[i], sdq[i], sds[i] = shared_expert_fp8(cfg, i, device, seed)
        out.update(Ws_gate_up_q=sgq, Ws_gate_up_s=sgs, Ws_down_q=sdq, Ws_down_s=sds)
