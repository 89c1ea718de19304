"""fp64 CPU oracle of the Kimi-K2-style fine-grained MoE layer forward.

TEST INFRASTRUCTURE: imported only by tests, the smoke check and the CPU
baseline leg of the benchmark.  Plain NumPy, fp64 for every floating-point
value the pages leave in real arithmetic; the expert-selection decision is
taken in fp32, the precision the pages' gate code computes it in (see
``biased_scores_f32``).

Sources (page title, then section / equation / listing):
  [Router]  "Kimi K2 · Router · OpenModelAtlas": the four equations under
            "All 4 steps" (z = x W_r, s = sigmoid(z), E_sel = top_8(s + b),
            G = 2.827 s E_sel / sum s E_sel), the in/out shapes, the parameter
            table, and the MoEGate listing (fp32 cast of x and W_r, sigmoid
            scoring, noaux_tc biased selection with n_group/topk_group group
            limiting, renormalisation with +1e-20, routed_scaling_factor).
  [K2MoE]   "Kimi K2 MoE" (llm-arch-kb): section 2 (DeepSeekMoE form, shared
            expert always on, SwiGLU experts with 3 d d_ff parameters),
            section 3 (output = shared(x) + routed, weights from the unbiased
            scores over the selected set).
  [K3]      "Kimi K3's router picks 16 of 896 experts": the K3 table and the
            Stable LatentMoE paragraph (routed experts see a 7168 -> 3584
            projection, their combined output is projected back to 7168, two
            shared experts stay at 7168).
  [Params]  "Kimi K2 · Router · OpenModelAtlas", section "Parameters": the
            note under the per-instance accounting says the checkpoint's
            tensors carry FP8 block scales.  The pages name neither the FP8
            encoding nor the block shape nor the scale's type; the reading
            taken (``e4m3_to_f64``, ``dequant_fp8_blocks``) is the OCP E4M3
            encoding with one fp32 multiplier per 128 x 128 block.

Where the pages leave a step open, the reading taken is stated next to the
code it shapes.
"""
from __future__ import annotations

from typing import Callable, Dict, Optional, Sequence, Tuple

import numpy as np

ROUTED_SCALING_FACTOR = 2.827  # [Router] "scaled by 2.827"; G equation
RENORM_EPS = 1e-20             # [Router] MoEGate.forward: denominator + 1e-20


# --------------------------------------------------------------------------
# elementary functions
# --------------------------------------------------------------------------
def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 numbers given as their 16-bit patterns."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def e4m3_to_f64(codes) -> np.ndarray:
    """Value of FP8 E4M3 numbers given as their 8-bit codes.

    [Params] reading: the OCP 8-bit floating-point E4M3 encoding -- bit 7
    the sign, bits 6..3 the exponent with bias 7, bits 2..0 the mantissa;
    exponent 0 is subnormal (m/8 * 2^-6); there are no infinities and
    S.1111.111 is NaN, so the largest magnitude is 1.75 * 2^8 = 448.
    """
    return _E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def _e4m3_values() -> np.ndarray:
    """The value of every code 0..255, from the field definitions above (a
    table, so that decoding a large bank is one lookup per code)."""
    c = np.arange(256, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64)))
    mag = np.where((e == 15) & ((c & 0x7) == 7), np.nan, mag)
    return sign * mag


_E4M3_TABLE = _e4m3_values()


FP8_BLOCK = 128  # [Params] reading: one scale per 128 x 128 block


def dequant_fp8_blocks(codes, scales, block: int = FP8_BLOCK) -> np.ndarray:
    """W[..., r, c] = e4m3(codes[..., r, c]) * scales[..., r // block, c // block], fp64.

    [Params] reading: a block-scaled FP8 matrix stores codes and one fp32
    multiplier per block x block tile of it (rows and columns counted from
    0); the weight is the code's value times its tile's multiplier.
    """
    q = e4m3_to_f64(codes)
    sc = np.asarray(scales, dtype=np.float64)
    R, C = q.shape[-2], q.shape[-1]
    if R % block == 0 and C % block == 0:  # each block times its scale, by broadcasting
        lead = q.shape[:-2]
        qb = q.reshape(*lead, R // block, block, C // block, block)
        return (qb * sc[..., :, None, :, None]).reshape(q.shape)
    full = np.repeat(np.repeat(sc, block, axis=-2), block, axis=-1)
    return q * full[..., :R, :C]


def sigmoid(z) -> np.ndarray:
    """s = 1 / (1 + exp(-z)) in fp64.  [Router] "All 4 steps", s = sigma(z)."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def silu(v) -> np.ndarray:
    """SiLU(v) = v * sigmoid(v), the gate non-linearity of a SwiGLU expert."""
    v = np.asarray(v, dtype=np.float64)
    return v * sigmoid(v)


def round_f32(a) -> np.ndarray:
    """Round fp64 values to the nearest fp32 (IEEE round-to-nearest-even)."""
    return np.asarray(a, dtype=np.float64).astype(np.float32)


# --------------------------------------------------------------------------
# router: selection
# --------------------------------------------------------------------------
def biased_scores_f32(z32, bias32) -> np.ndarray:
    """Selection scores c = s + b in fp32.

    [Router] MoEGate.forward casts x and W_r to fp32 before the linear map, so
    the logits, the sigmoid and the bias add are fp32 operations there.  The
    selection is a discrete decision, so it is taken in that precision here:
    s is sigmoid(z) computed in fp64 and rounded once to fp32 (the correctly
    rounded fp32 sigmoid), and c = fp32(s + b) is one IEEE fp32 addition.
    """
    z32 = np.asarray(z32, dtype=np.float32)
    s32 = round_f32(sigmoid(z32.astype(np.float64)))
    return s32 + np.asarray(bias32, dtype=np.float32)[None, :]


def _canonical_order(values: np.ndarray) -> np.ndarray:
    """Indices sorting the last axis by (value descending, index ascending).

    torch.topk(..., sorted=False) in the [Router] listing fixes the selected
    set but neither the order of the output nor how equal values are broken;
    this total order is the reading used on both sides.
    """
    n = values.shape[-1]
    position = np.broadcast_to(np.arange(n), values.shape)
    return np.lexsort((position, -values), axis=-1)


def group_scores_f32(c32: np.ndarray, n_group: int) -> np.ndarray:
    """Per group, the fp32 sum of its two largest selection scores.

    [Router] MoEGate.forward, group_scores: the scores are viewed as
    [n, n_group, E / n_group] (contiguous experts per group) and the top-2
    values of each group are summed.
    """
    T, E = c32.shape
    grouped = np.sort(c32.reshape(T, n_group, E // n_group), axis=-1)
    return grouped[..., -1] + grouped[..., -2]  # fp32 + fp32


def select_experts(c32: np.ndarray, K: int, n_group: int = 1,
                   topk_group: int = 1) -> Tuple[np.ndarray, np.ndarray]:
    """Biased (noaux_tc) top-K with optional group limiting.

    Returns (idx [T, K] int64 in canonical order, masked scores [T, E] fp32).
    [Router] "All 4 steps": E_sel = [i in top_K(s + b)]; MoEGate.forward: keep
    the topk_group groups with the largest group scores and fill the scores of
    every other expert with 0.0 (a literal 0.0, not -inf) before the top-K.
    With n_group == 1 the mask keeps everything.
    """
    c32 = np.asarray(c32, dtype=np.float32)
    T, E = c32.shape
    masked = c32.copy()
    if n_group > 1:
        gscore = group_scores_f32(c32, n_group)
        kept = _canonical_order(gscore)[:, :topk_group]
        keep_group = np.zeros((T, n_group), dtype=bool)
        np.put_along_axis(keep_group, kept, True, axis=1)
        keep_expert = np.repeat(keep_group, E // n_group, axis=1)
        masked[~keep_expert] = np.float32(0.0)
    idx = _canonical_order(masked)[:, :K]
    return idx.astype(np.int64), masked


def selection_gaps(c32: np.ndarray, K: int, n_group: int = 1,
                   topk_group: int = 1) -> np.ndarray:
    """Smallest margin (fp64) of any discrete decision taken for a token.

    The margin of the expert top-K is (K-th) - (K+1-th) masked score; with
    group limiting the group decision's margin, (topk_group-th) - (next) group
    score, also counts.  A token with a margin above the fp32 error of the
    logits has a unique selection under any faithful fp32 evaluation.
    """
    c32 = np.asarray(c32, dtype=np.float32)
    T, E = c32.shape
    _, masked = select_experts(c32, K, n_group, topk_group)
    srt = -np.sort(-masked.astype(np.float64), axis=-1)
    gap = np.full(T, np.inf)
    if K < E:
        gap = srt[:, K - 1] - srt[:, K]
    if n_group > 1 and topk_group < n_group:
        g = -np.sort(-group_scores_f32(c32, n_group).astype(np.float64), axis=-1)
        gap = np.minimum(gap, g[:, topk_group - 1] - g[:, topk_group])
    return gap


# --------------------------------------------------------------------------
# router: gate weights
# --------------------------------------------------------------------------
def router_weights(s_selected, K: int, scale: float = ROUTED_SCALING_FACTOR,
                   norm_topk_prob: bool = True) -> np.ndarray:
    """G restricted to the selected set, in fp64.

    [Router] G_i = 2.827 * s_i E_sel_i / sum_j s_j E_sel_j with the unbiased
    scores s (the bias only chooses, [K2MoE] section 3).  MoEGate.forward
    renormalises only when K > 1 and norm_topk_prob, adds 1e-20 to the
    denominator, and always multiplies by routed_scaling_factor.
    """
    s = np.asarray(s_selected, dtype=np.float64)
    if K > 1 and norm_topk_prob:
        s = s / (s.sum(axis=-1, keepdims=True) + RENORM_EPS)
    return s * scale


def router_from_logits(z32, bias32, K: int, n_group: int = 1, topk_group: int = 1,
                       scale: float = ROUTED_SCALING_FACTOR,
                       norm_topk_prob: bool = True) -> Dict[str, np.ndarray]:
    """Router steps 2-4 from given fp32 logits z [T, E]."""
    z32 = np.asarray(z32, dtype=np.float32)
    c32 = biased_scores_f32(z32, bias32)
    idx, _ = select_experts(c32, K, n_group, topk_group)
    s64 = sigmoid(z32.astype(np.float64))
    w = router_weights(np.take_along_axis(s64, idx, axis=1), K, scale, norm_topk_prob)
    return {"idx": idx, "w": w, "c32": c32,
            "gap": selection_gaps(c32, K, n_group, topk_group)}


def router_from_x(x64, W_r64, bias32, K: int, n_group: int = 1, topk_group: int = 1,
                  scale: float = ROUTED_SCALING_FACTOR,
                  norm_topk_prob: bool = True) -> Dict[str, np.ndarray]:
    """All four router steps from the hidden states.

    [Router] z = x_ffn W_r with W_r stored [E, d] (gate.weight); the product
    is exact up to fp64 rounding.  The selection sees z rounded to fp32 (the
    pages' logits are fp32); the weights use sigmoid of the fp64 logits.
    """
    x64 = np.asarray(x64, dtype=np.float64)
    W_r64 = np.asarray(W_r64, dtype=np.float64)
    z64 = x64 @ W_r64.T
    z32 = round_f32(z64)
    c32 = biased_scores_f32(z32, bias32)
    idx, _ = select_experts(c32, K, n_group, topk_group)
    s64 = sigmoid(z64)
    w = router_weights(np.take_along_axis(s64, idx, axis=1), K, scale, norm_topk_prob)
    return {"idx": idx, "w": w, "z64": z64, "c32": c32,
            "gap": selection_gaps(c32, K, n_group, topk_group)}


# --------------------------------------------------------------------------
# router: the dense gate matrix and the aux-loss-free bias update
# --------------------------------------------------------------------------
def dense_gates(idx, w, E: int) -> np.ndarray:
    """G [T, E]: each token's selected weights at their experts, 0 elsewhere.

    [Router] the "out: G [B batch, T positions, 384 experts]" shape and the
    Explanation: the implementation returns the K weights with their expert
    indices, and G spreads them over all E experts, zero for the others.
    """
    idx = np.asarray(idx)
    T = idx.shape[0]
    G = np.zeros((T, E))
    G[np.arange(T)[:, None], idx] = np.asarray(w, dtype=np.float64)
    return G


def aux_free_bias_update(bias32, counts, T: int, K: int, gamma: float = 1e-3) -> np.ndarray:
    """One sign-only update of the selection bias from one batch's loads.

    [K2MoE] "Routing-distribution diagnostics": the aux-loss-free bias keeps
    DeepSeek V3's schedule, gamma = 1e-3 and a sign-only update.  Reading:
    an expert that received more pairs than the mean load T K / E has its
    bias lowered by gamma, one that received fewer has it raised by gamma,
    one at the mean keeps it.  The comparison with the mean is made in
    integers (E * load against T * K); the bias is fp32 and the step is one
    fp32 addition of the fp32 gamma.
    """
    counts = np.asarray(counts, dtype=np.int64)
    E = counts.shape[0]
    step = np.sign(np.int64(T) * K - E * counts).astype(np.float64)
    g32 = np.float64(np.float32(gamma))
    return round_f32(np.asarray(bias32, dtype=np.float64) + g32 * step).astype(np.float32)


def quantile_bias_update(z32, bias32, K: int, rate: float = 1.0) -> Tuple[np.ndarray, np.ndarray]:
    """One Quantile Balancing update of the selection bias from one batch.

    [K3] "The router trains inside the main run": Quantile Balancing takes,
    per expert, the threshold at which that expert receives its target
    number of tokens from a quantile of the router scores, and updates the
    selection bias from it (training only; at inference the bias is fixed).
    The update rule is not printed; the reading taken:
      * target load n* = T K / E tokens per expert (every expert equal);
      * threshold theta_e = the ceil(n*)-th largest router score s_e(t) of
        the batch (the (1 - K/E) quantile of expert e's scores, taken as an
        order statistic), s = sigmoid(z) rounded once to fp32 (the scores the
        selection compares);
      * common cut-off tau = the mean of theta over the experts, summed in
        fp64 in expert order;
      * target bias b*_e = tau - theta_e, so that an expert's biased score
        at its threshold, theta_e + b*_e, is the common cut-off and its top
        n* tokens are the ones that reach tau;
      * b_e <- b_e + rate (b*_e - b_e), in fp64, rounded once to fp32
        (rate 1 sets the target bias).
    Returns (theta [E] fp32, new bias [E] fp32).
    """
    z32 = np.asarray(z32, dtype=np.float32)
    T, E = z32.shape
    s32 = round_f32(sigmoid(z32.astype(np.float64)))
    r = -(-(T * K) // E)  # ceil(T K / E), 1 <= r <= T
    theta = np.empty(E, dtype=np.float32)
    for e in range(E):
        theta[e] = np.sort(s32[:, e])[::-1][r - 1]
    total = 0.0
    for e in range(E):  # fixed order, fp64
        total += float(theta[e])
    tau = total / E
    b = np.asarray(bias32, dtype=np.float32).astype(np.float64)
    target = tau - theta.astype(np.float64)
    new = b + float(np.float32(rate)) * (target - b)
    return theta, round_f32(new)


# --------------------------------------------------------------------------
# dispatch (permute)
# --------------------------------------------------------------------------
def permute(idx, E: int) -> Dict[str, np.ndarray]:
    """Group the (token, slot) pairs by expert.

    [K2MoE] section 3 names the dispatch step without giving its body.
    Reading: expert-major order, and within an expert ascending token index
    (a stable sort of the flattened (t, k) list by expert id).  Entry j = t*K+k.
      counts[e]            number of pairs routed to e
      offsets[e]           exclusive prefix sum of counts (length E + 1)
      perm[offsets[e]+r]   the j of the r-th pair of expert e
      inv[j]               the slot holding pair j
    """
    idx = np.asarray(idx, dtype=np.int64)
    flat = idx.reshape(-1)
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    perm = np.argsort(flat, kind="stable").astype(np.int64)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size, dtype=np.int64)
    return {"counts": counts, "offsets": offsets, "perm": perm, "inv": inv}


def combine(Y, inv, w, Y_shared=None) -> np.ndarray:
    """y[t] = sum_k w[t, k] Y[inv[t K + k]] + sum_s Y_shared[s, t], in fp64.

    [K2MoE] section 3: the routed output is the gate-weighted sum of the
    selected experts' outputs, and the layer adds the shared expert's output
    (shared(x) + routed).  Y holds one expert output per slot (the dispatch
    order of ``permute``), inv maps pair t K + k to its slot, w [T, K] are the
    gate weights (ones when the rows of Y already carry them).
    """
    Y = np.asarray(Y, dtype=np.float64)
    inv = np.asarray(inv, dtype=np.int64)
    w = np.asarray(w, dtype=np.float64)
    T, K = w.shape
    y = np.zeros((T, Y.shape[1]))
    for t in range(T):
        for k in range(K):
            y[t] += w[t, k] * Y[inv[t * K + k]]
    if Y_shared is not None:
        y = y + np.asarray(Y_shared, dtype=np.float64).sum(axis=0)
    return y


# --------------------------------------------------------------------------
# experts and the layer
# --------------------------------------------------------------------------
def swiglu_expert(u64, W_gate64, W_up64, W_down64) -> np.ndarray:
    """f(u) = W_down (SiLU(W_gate u) * (W_up u)) for the rows of u, in fp64.

    [K2MoE] section 2 calls the experts SwiGLU FFNs with 3 d d_ff parameters
    (gate, up and down matrices, no biases); the formula itself is not
    printed, so this is the standard form.  Weights follow nn.Linear
    (out x in): W_gate, W_up [F, d], W_down [d, F].
    """
    u = np.asarray(u64, dtype=np.float64)
    gate = u @ np.asarray(W_gate64, dtype=np.float64).T
    up = u @ np.asarray(W_up64, dtype=np.float64).T
    return (silu(gate) * up) @ np.asarray(W_down64, dtype=np.float64).T


ExpertFn = Callable[[int], Tuple[np.ndarray, np.ndarray, np.ndarray]]


def moe_layer(x64, W_r64, bias32, routed: ExpertFn, shared: Optional[ExpertFn],
              n_shared: int, K: int, n_group: int = 1, topk_group: int = 1,
              scale: float = ROUTED_SCALING_FACTOR, norm_topk_prob: bool = True,
              W_lat_down64=None, W_lat_up64=None, E: Optional[int] = None,
              logits32=None) -> Dict[str, np.ndarray]:
    """Forward of the MoE layer for the token rows of x (tokens are independent).

    K2 form ([K2MoE] section 3): y = sum_s f_s(x) + sum_k w_k f_{idx_k}(x).
    K3 form ([K3], Stable LatentMoE): u = W_lat_down x; y = sum_s f_s(x) +
    W_lat_up (sum_k w_k f_{idx_k}(u)); the router reads the 7168-wide x.

    ``routed(e)`` / ``shared(s)`` return (W_gate, W_up, W_down) as fp64 arrays,
    so huge weight banks can be upcast one expert at a time.  ``logits32``
    replaces the router GEMM by given fp32 logits.
    """
    x64 = np.asarray(x64, dtype=np.float64)
    T = x64.shape[0]
    if logits32 is not None:
        r = router_from_logits(logits32, bias32, K, n_group, topk_group, scale, norm_topk_prob)
    else:
        r = router_from_x(x64, W_r64, bias32, K, n_group, topk_group, scale, norm_topk_prob)
    idx, w = r["idx"], r["w"]
    u = x64 if W_lat_down64 is None else x64 @ np.asarray(W_lat_down64, np.float64).T
    routed_out = np.zeros_like(u)
    for e in np.unique(idx):
        rows, slots = np.nonzero(idx == e)
        Wg, Wu, Wd = routed(int(e))
        routed_out[rows] += w[rows, slots][:, None] * swiglu_expert(u[rows], Wg, Wu, Wd)
    if W_lat_up64 is not None:
        routed_out = routed_out @ np.asarray(W_lat_up64, np.float64).T
    y = routed_out
    for s in range(n_shared):
        Wg, Wu, Wd = shared(s)
        y = y + swiglu_expert(x64, Wg, Wu, Wd)
    out = dict(r)
    out["y"] = y
    if E is not None:
        out.update(permute(idx, E))
    return out


def moe_layer_tokens(x64, W_r64, bias32, W_gate_up, W_down, Ws_gate_up, Ws_down,
                     K: int, n_group: int = 1, topk_group: int = 1,
                     scale: float = ROUTED_SCALING_FACTOR, norm_topk_prob: bool = True,
                     W_lat_down64=None, W_lat_up64=None,
                     to_f64: Callable = np.asarray) -> Dict[str, np.ndarray]:
    """``moe_layer`` over stacked weight banks.

    W_gate_up [E, 2F, d] holds the gate rows then the up rows of each expert;
    ``to_f64`` turns one expert's slice into an fp64 array (for bf16 banks it
    performs the exact upcast), so only the experts the given tokens select
    are ever converted.
    """
    def split(bank_gu, bank_d, e):
        gu = np.asarray(to_f64(bank_gu[e]), dtype=np.float64)
        F = gu.shape[0] // 2
        return gu[:F], gu[F:], np.asarray(to_f64(bank_d[e]), dtype=np.float64)

    n_shared = 0 if Ws_gate_up is None else len(Ws_gate_up)
    return moe_layer(
        x64, W_r64, bias32,
        routed=lambda e: split(W_gate_up, W_down, e),
        shared=(lambda s: split(Ws_gate_up, Ws_down, s)) if n_shared else None,
        n_shared=n_shared, K=K, n_group=n_group, topk_group=topk_group, scale=scale,
        norm_topk_prob=norm_topk_prob, W_lat_down64=W_lat_down64, W_lat_up64=W_lat_up64)


def moe_layer_tokens_fp8(x64, W_r64, bias32, gu_q, gu_s, dn_q, dn_s, sgu_q=None, sgu_s=None,
                         sdn_q=None, sdn_s=None, K: int = 8, n_group: int = 1,
                         topk_group: int = 1, scale: float = ROUTED_SCALING_FACTOR,
                         norm_topk_prob: bool = True, W_lat_down64=None,
                         W_lat_up64=None) -> Dict[str, np.ndarray]:
    """``moe_layer`` with FP8 block-scaled expert weights ([Params] reading).

    gu_q [E, 2F, d] uint8 codes with gu_s [E, 2F/128, d/128] fp32 scales
    (gate rows then up rows), dn_q [E, d, F] with dn_s [E, d/128, F/128]; the
    shared experts' banks likewise (or None).  Each selected expert is
    dequantised exactly in fp64 (``dequant_fp8_blocks``) and then runs the
    same fp64 SwiGLU as the bf16 form.
    """
    def split(q_gu, s_gu, q_dn, s_dn, e):
        gu = dequant_fp8_blocks(q_gu[e], s_gu[e])
        F = gu.shape[0] // 2
        return gu[:F], gu[F:], dequant_fp8_blocks(q_dn[e], s_dn[e])

    n_shared = 0 if sgu_q is None else len(sgu_q)
    return moe_layer(
        x64, W_r64, bias32,
        routed=lambda e: split(gu_q, gu_s, dn_q, dn_s, e),
        shared=(lambda s_: split(sgu_q, sgu_s, sdn_q, sdn_s, s_)) if n_shared else None,
        n_shared=n_shared, K=K, n_group=n_group, topk_group=topk_group, scale=scale,
        norm_topk_prob=norm_topk_prob, W_lat_down64=W_lat_down64, W_lat_up64=W_lat_up64)
