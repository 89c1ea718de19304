"""Fine-grained MoE layer forward (Kimi-K2 / Kimi-K3 shapes) on GB300.

A thin ctypes binding over the C ABI declared in ``include/moe.h``: every
function here has the C name, marshals tensors to pointers and raises
``MoeError`` on a non-zero status.  All arithmetic runs in the library's
CUDA kernels; there is no other implementation behind these names, and
importing the package fails when the library has not been built
(``python fine_grained_sparse_gb300/build.py``, or ``__graft_entry__.build()``).

Tensors are torch tensors on the current CUDA device (PyTorch provides the
device memory and the stream); plain integers are accepted as raw pointers.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

from .build import lib_path

__all__ = [
    "MoeError", "MoeConfig", "MOE_F32", "MOE_BF16", "MOE_STAGE_COUNT", "STATUS", "lib",
    "config", "moe_version", "moe_status_string", "moe_validate_config", "moe_workspace_size",
    "moe_get_device_status", "moe_router", "moe_router_from_logits", "moe_permute",
    "moe_grouped_swiglu", "moe_combine", "moe_linear", "moe_layer_forward",
    "moe_layer_forward_host", "moe_layer_forward_host_pipelined", "moe_layer_forward_host_flush",
    "moe_layer_forward_host_release", "moe_last_error_detail",
    "moe_pack_weights", "pack_layer_weights",
    "moe_router_noalloc", "moe_launch_count", "moe_dense_gates", "moe_update_bias",
    "moe_quantile_bias_update",
    "MOE_WEIGHTS_NATURAL", "MOE_WEIGHTS_PACKED", "MOE_PACK_GATE_UP", "MOE_PACK_PLAIN",
    "MOE_WEIGHTS_PACKED_FP8", "moe_packed_fp8_bytes", "moe_pack_weights_fp8",
    "pack_layer_weights_fp8", "moe_selftest_bounded_wait", "MOE_ROUTER_WEIGHT_F32",
    "MOE_ROUTER_WEIGHT_SPLIT", "moe_router_weight_split_bytes", "moe_split_router_weight",
    "split_router_weight",
]

MOE_F32, MOE_BF16 = 0, 1
MOE_WEIGHTS_NATURAL, MOE_WEIGHTS_PACKED, MOE_WEIGHTS_PACKED_FP8 = 0, 1, 2
MOE_PACK_GATE_UP, MOE_PACK_PLAIN = 0, 1
MOE_ROUTER_WEIGHT_F32, MOE_ROUTER_WEIGHT_SPLIT = 0, 1
MOE_STAGE_COUNT = 5
STAGE_NAMES = ("router", "dispatch", "expert_gate_up", "expert_down", "combine")
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE",
          3: "MOE_ERR_ALIGNMENT", 4: "MOE_ERR_WORKSPACE", 5: "MOE_ERR_CUDA",
          6: "MOE_ERR_TIMEOUT", 7: "MOE_ERR_DEVICE_INDEX"}


class MoeError(RuntimeError):
    def __init__(self, status: int, func: str, detail: str):
        self.status = status
        super().__init__(f"{func}: {STATUS.get(status, status)} ({detail})")


class MoeConfig(ctypes.Structure):
    _fields_ = [
        ("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("E_routed", ctypes.c_int32),
        ("E_shared", ctypes.c_int32), ("d_ff_shared", ctypes.c_int32), ("K", ctypes.c_int32),
        ("n_group", ctypes.c_int32), ("topk_group", ctypes.c_int32),
        ("routed_scaling_factor", ctypes.c_float), ("norm_topk_prob", ctypes.c_int32),
        ("d_latent", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("weight_layout", ctypes.c_int32), ("router_weight", ctypes.c_int32),
    ]


def _load():
    path = lib_path()
    if not os.path.exists(path):
        raise ImportError(
            f"fine_grained_sparse_gb300: CUDA library {path} is missing; build it with "
            "`python fine_grained_sparse_gb300/build.py`")
    return ctypes.CDLL(path)


lib = _load()

_P, _I32, _I64, _SZ, _F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
_CFG = ctypes.POINTER(MoeConfig)
_SIGS = {
    "moe_version": ([], _I32),
    "moe_launch_count": ([], ctypes.c_uint64),
    "moe_status_string": ([_I32], ctypes.c_char_p),
    "moe_last_error_detail": ([], ctypes.c_char_p),
    "moe_validate_config": ([_CFG, _I64], _I32),
    "moe_workspace_size": ([_CFG, _I64], _SZ),
    "moe_get_device_status": ([_P, _P], _I32),
    "moe_router": ([_CFG, _I64, _P, _P, _P, _P, _P, _P, _SZ, _P], _I32),
    "moe_router_from_logits": ([_CFG, _I64, _P, _P, _P, _P, _P], _I32),
    "moe_dense_gates": ([_CFG, _I64, _P, _P, _P, _P], _I32),
    "moe_update_bias": ([_CFG, _I64, _P, _F, _P, _P], _I32),
    "moe_quantile_bias_update": ([_CFG, _I64, _P, _F, _P, _P, _P], _I32),
    "moe_permute": ([_CFG, _I64, _P, _P, _P, _P, _P, _P, _SZ, _P], _I32),
    "moe_grouped_swiglu": ([_CFG, _I64] + [_P] * 12 + [_SZ, _P], _I32),
    "moe_combine": ([_CFG, _I64, _P, _P, _P, _P, _P, _P], _I32),
    "moe_linear": ([_I64, _I32, _I32, _P, _P, _P, _P, _P, _SZ, _P], _I32),
    "moe_pack_weights": ([_I32, _I64, _I64, _I64, _P, _P, _P], _I32),
    "moe_packed_fp8_bytes": ([_I64, _I64, _I64], _I64),
    "moe_selftest_bounded_wait": ([_P, _P], _I32),
    "moe_pack_weights_fp8": ([_I32, _I64, _I64, _I64, _P, _P, _P, _P], _I32),
    "moe_router_noalloc": ([_CFG, _I64, _P, _P, _P, _P, _P, _P], _I32),
    "moe_router_weight_split_bytes": ([_CFG], _SZ),
    "moe_split_router_weight": ([_CFG, _P, _P, _P], _I32),
    "moe_layer_forward": ([_CFG, _I64] + [_P] * 14 + [_SZ, _P, _P], _I32),
    "moe_layer_forward_host": ([_CFG, _I64] + [_P] * 11 + [_SZ, _P], _I32),
    "moe_layer_forward_host_pipelined": ([_CFG, _I64] + [_P] * 11 + [_SZ, _P], _I32),
    "moe_layer_forward_host_flush": ([_P, _P], _I32),
    "moe_layer_forward_host_release": ([_P], _I32),
}
for _name, (_args, _res) in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, func: str):
    if status != 0:
        raise MoeError(status, func, lib.moe_last_error_detail().decode())


def config(shape=None, **kw) -> MoeConfig:
    """MoeConfig from a ``synth.LayerShape``-like object and/or keywords."""
    vals = dict(d_model=0, d_ff=0, E_routed=0, E_shared=0, d_ff_shared=0, K=1, n_group=1,
                topk_group=1, routed_scaling_factor=2.827, norm_topk_prob=1, d_latent=0,
                dtype=MOE_BF16, weight_layout=MOE_WEIGHTS_NATURAL,
                router_weight=MOE_ROUTER_WEIGHT_F32)
    if shape is not None:
        for k in vals:
            if hasattr(shape, k):
                vals[k] = getattr(shape, k)
        if hasattr(shape, "dtype") and isinstance(shape.dtype, str):
            vals["dtype"] = MOE_F32 if shape.dtype == "f32" else MOE_BF16
        if getattr(shape, "router_only", False):
            vals["d_ff"] = 0
        if getattr(shape, "weights", "bf16") == "fp8":
            vals["weight_layout"] = MOE_WEIGHTS_PACKED_FP8
    vals.update(kw)
    vals["norm_topk_prob"] = int(bool(vals["norm_topk_prob"]))
    return MoeConfig(**vals)


def moe_version() -> int:
    return lib.moe_version()


def moe_launch_count() -> int:
    """Kernels the library has enqueued in this process so far."""
    return int(lib.moe_launch_count())


def moe_status_string(status: int) -> str:
    return lib.moe_status_string(status).decode()


def moe_last_error_detail() -> str:
    return lib.moe_last_error_detail().decode()


def moe_validate_config(cfg: MoeConfig, T: int) -> int:
    return lib.moe_validate_config(ctypes.byref(cfg), T)


def moe_workspace_size(cfg: MoeConfig, T: int) -> int:
    return lib.moe_workspace_size(ctypes.byref(cfg), T)


def moe_get_device_status(workspace, stream=None) -> int:
    return lib.moe_get_device_status(_ptr(workspace), _stream(stream))


def moe_router(cfg, T, x, W_r, bias, topk_idx, topk_w, workspace=None, ws_bytes=0, stream=None):
    _check(lib.moe_router(ctypes.byref(cfg), T, _ptr(x), _ptr(W_r), _ptr(bias), _ptr(topk_idx),
                          _ptr(topk_w), _ptr(workspace), ws_bytes, _stream(stream)), "moe_router")


def moe_dense_gates(cfg, T, topk_idx, topk_w, G, stream=None):
    """G [T, E] fp32: the routing weights at their experts, 0 elsewhere."""
    _check(lib.moe_dense_gates(ctypes.byref(cfg), T, _ptr(topk_idx), _ptr(topk_w), _ptr(G),
                               _stream(stream)), "moe_dense_gates")


def moe_update_bias(cfg, T, counts, gamma, bias, stream=None):
    """bias [E] fp32 in place: += gamma * sign(T K / E - counts)."""
    _check(lib.moe_update_bias(ctypes.byref(cfg), T, _ptr(counts), float(gamma), _ptr(bias),
                               _stream(stream)), "moe_update_bias")


def moe_quantile_bias_update(cfg, T, logits, rate, theta, bias, stream=None):
    """Quantile Balancing: theta [E] out, bias [E] fp32 updated in place."""
    _check(lib.moe_quantile_bias_update(ctypes.byref(cfg), T, _ptr(logits), float(rate),
                                        _ptr(theta), _ptr(bias), _stream(stream)),
           "moe_quantile_bias_update")


def moe_router_noalloc(cfg, T, x, W_r, bias, topk_idx, topk_w, stream=None):
    """moe_router on the library's static device scratch (no workspace)."""
    _check(lib.moe_router_noalloc(ctypes.byref(cfg), T, _ptr(x), _ptr(W_r), _ptr(bias),
                                  _ptr(topk_idx), _ptr(topk_w), _stream(stream)),
           "moe_router_noalloc")


def moe_router_from_logits(cfg, T, logits, bias, topk_idx, topk_w, stream=None):
    _check(lib.moe_router_from_logits(ctypes.byref(cfg), T, _ptr(logits), _ptr(bias),
                                      _ptr(topk_idx), _ptr(topk_w), _stream(stream)),
           "moe_router_from_logits")


def moe_permute(cfg, T, topk_idx, counts, offsets, perm, inv, workspace, ws_bytes, stream=None):
    _check(lib.moe_permute(ctypes.byref(cfg), T, _ptr(topk_idx), _ptr(counts), _ptr(offsets),
                           _ptr(perm), _ptr(inv), _ptr(workspace), ws_bytes, _stream(stream)),
           "moe_permute")


def moe_grouped_swiglu(cfg, T, x_e, offsets, perm, topk_w, W_gate_up, W_down, x_shared,
                       Ws_gate_up, Ws_down, Y, Y_shared, workspace, ws_bytes, stream=None):
    _check(lib.moe_grouped_swiglu(ctypes.byref(cfg), T, _ptr(x_e), _ptr(offsets), _ptr(perm),
                                  _ptr(topk_w), _ptr(W_gate_up), _ptr(W_down), _ptr(x_shared),
                                  _ptr(Ws_gate_up), _ptr(Ws_down), _ptr(Y), _ptr(Y_shared),
                                  _ptr(workspace), ws_bytes, _stream(stream)),
           "moe_grouped_swiglu")


def moe_combine(cfg, T, Y, inv, topk_w, Y_shared, y, stream=None):
    """y = sum_k w_k Y[inv] + sum_s Y_shared; topk_w None means weight 1 (the
    weights already in Y)."""
    _check(lib.moe_combine(ctypes.byref(cfg), T, _ptr(Y), _ptr(inv), _ptr(topk_w), _ptr(Y_shared),
                           _ptr(y), _stream(stream)), "moe_combine")


def moe_linear(T, in_features, out_features, x, W, add, y, workspace, ws_bytes, stream=None):
    _check(lib.moe_linear(T, in_features, out_features, _ptr(x), _ptr(W), _ptr(add), _ptr(y),
                          _ptr(workspace), ws_bytes, _stream(stream)), "moe_linear")


def moe_layer_forward(cfg, T, x, W_r, bias, W_gate_up, W_down, Ws_gate_up, Ws_down, W_lat_down,
                      W_lat_up, y, topk_idx_out=None, topk_w_out=None, counts_out=None,
                      workspace=None, ws_bytes=0, stage_events: Optional[Sequence] = None,
                      stream=None):
    ev_array = None
    if stage_events is not None:
        handles = []
        for e in stage_events:
            if e is None:  # this stage boundary is not recorded
                handles.append(None)
            elif hasattr(e, "cuda_event"):
                if not e.cuda_event:  # torch creates its events lazily, on first record
                    import torch
                    e.record(torch.cuda.current_stream() if stream is None else stream)
                handles.append(e.cuda_event)
            else:
                handles.append(int(e))
        if len(handles) != MOE_STAGE_COUNT + 1:
            raise ValueError("stage_events needs MOE_STAGE_COUNT + 1 events")
        ev_array = (ctypes.c_void_p * len(handles))(*handles)
    _check(lib.moe_layer_forward(ctypes.byref(cfg), T, _ptr(x), _ptr(W_r), _ptr(bias),
                                 _ptr(W_gate_up), _ptr(W_down), _ptr(Ws_gate_up), _ptr(Ws_down),
                                 _ptr(W_lat_down), _ptr(W_lat_up), _ptr(y), _ptr(topk_idx_out),
                                 _ptr(topk_w_out), _ptr(counts_out), _ptr(workspace), ws_bytes,
                                 ctypes.cast(ev_array, ctypes.c_void_p) if ev_array is not None else None,
                                 _stream(stream)), "moe_layer_forward")


def moe_layer_forward_host(cfg, T, x_host, W_r, bias, W_gate_up, W_down, Ws_gate_up, Ws_down,
                           W_lat_down, W_lat_up, y_host, workspace, ws_bytes, stream=None):
    _check(lib.moe_layer_forward_host(ctypes.byref(cfg), T, _ptr(x_host), _ptr(W_r), _ptr(bias),
                                      _ptr(W_gate_up), _ptr(W_down), _ptr(Ws_gate_up),
                                      _ptr(Ws_down), _ptr(W_lat_down), _ptr(W_lat_up),
                                      _ptr(y_host), _ptr(workspace), ws_bytes, _stream(stream)),
           "moe_layer_forward_host")


def moe_layer_forward_host_pipelined(cfg, T, x_host, W_r, bias, W_gate_up, W_down, Ws_gate_up,
                                     Ws_down, W_lat_down, W_lat_up, y_host, workspace, ws_bytes,
                                     stream=None):
    """moe_layer_forward_host whose y_host is valid once `stream` has passed
    the next such call on the workspace, or moe_layer_forward_host_flush."""
    _check(lib.moe_layer_forward_host_pipelined(
        ctypes.byref(cfg), T, _ptr(x_host), _ptr(W_r), _ptr(bias), _ptr(W_gate_up), _ptr(W_down),
        _ptr(Ws_gate_up), _ptr(Ws_down), _ptr(W_lat_down), _ptr(W_lat_up), _ptr(y_host),
        _ptr(workspace), ws_bytes, _stream(stream)), "moe_layer_forward_host_pipelined")


def moe_layer_forward_host_flush(workspace, stream=None):
    """Make `stream` wait for the latest pipelined call's copy of y."""
    _check(lib.moe_layer_forward_host_flush(_ptr(workspace), _stream(stream)),
           "moe_layer_forward_host_flush")


def moe_layer_forward_host_release(workspace):
    """Drop the library's per-workspace state of moe_layer_forward_host."""
    _check(lib.moe_layer_forward_host_release(_ptr(workspace)), "moe_layer_forward_host_release")


def moe_pack_weights(kind, groups, rows, cols, src, dst, stream=None):
    _check(lib.moe_pack_weights(kind, groups, rows, cols, _ptr(src), _ptr(dst), _stream(stream)),
           "moe_pack_weights")


def moe_router_weight_split_bytes(cfg) -> int:
    return int(lib.moe_router_weight_split_bytes(ctypes.byref(cfg)))


def moe_split_router_weight(cfg, W_r, W_split, stream=None):
    _check(lib.moe_split_router_weight(ctypes.byref(cfg), _ptr(W_r), _ptr(W_split),
                                       _stream(stream)), "moe_split_router_weight")


def split_router_weight(cfg, W_r, stream=None):
    """The MOE_ROUTER_WEIGHT_SPLIT form of an fp32 router weight on W_r's
    device: a new bf16 [E, 3 d] tensor, for a config whose router_weight is
    MOE_ROUTER_WEIGHT_SPLIT (a one-time load step)."""
    import torch
    out = torch.empty((cfg.E_routed, 3 * cfg.d_model), dtype=torch.bfloat16, device=W_r.device)
    moe_split_router_weight(cfg, W_r, out, stream)
    return out


def moe_selftest_bounded_wait(workspace, stream=None):
    """Enqueue one bounded device wait that runs out (about 2 s); the
    workspace status word then reads MOE_ERR_TIMEOUT."""
    _check(lib.moe_selftest_bounded_wait(_ptr(workspace), _stream(stream)),
           "moe_selftest_bounded_wait")


def moe_packed_fp8_bytes(groups, rows, cols) -> int:
    return int(lib.moe_packed_fp8_bytes(groups, rows, cols))


def moe_pack_weights_fp8(kind, groups, rows, cols, codes, scales, dst, stream=None):
    _check(lib.moe_pack_weights_fp8(kind, groups, rows, cols, _ptr(codes), _ptr(scales), _ptr(dst),
                                    _stream(stream)), "moe_pack_weights_fp8")


def pack_layer_weights_fp8(weights: dict, stream=None) -> dict:
    """The weights of one layer for a config whose weight_layout is
    MOE_WEIGHTS_PACKED_FP8: the FP8 banks (keys ``<bank>_q`` with codes and
    ``<bank>_s`` with block scales, as produced by ``synth.generate`` for an
    FP8 shape) packed into one uint8 buffer each under ``<bank>``, and the
    bf16 latent projections packed as by ``pack_layer_weights``."""
    import torch
    out = {k: v for k, v in weights.items() if not (k.endswith("_q") or k.endswith("_s"))}
    kinds = {"W_gate_up": MOE_PACK_GATE_UP, "Ws_gate_up": MOE_PACK_GATE_UP,
             "W_down": MOE_PACK_PLAIN, "Ws_down": MOE_PACK_PLAIN}
    for key, kind in kinds.items():
        q, sc = weights.get(key + "_q"), weights.get(key + "_s")
        if q is None:
            continue
        G, R, C = q.shape
        dst = torch.empty(moe_packed_fp8_bytes(G, R, C), dtype=torch.uint8, device=q.device)
        moe_pack_weights_fp8(kind, G, R, C, q.contiguous(), sc.contiguous(), dst, stream)
        out[key] = dst
    lat = {k: weights[k] for k in ("W_lat_down", "W_lat_up") if weights.get(k) is not None}
    if lat:
        out.update(pack_layer_weights(lat, stream))
    return out


def pack_layer_weights(weights: dict, stream=None) -> dict:
    """Copies of the bf16 weight banks of one layer (keys as produced by
    ``synth.generate``: W_gate_up, W_down, Ws_gate_up, Ws_down, W_lat_down,
    W_lat_up) in MOE_WEIGHTS_PACKED order; other entries are passed through.
    Use with a config whose weight_layout is MOE_WEIGHTS_PACKED."""
    import torch
    out = dict(weights)
    kinds = {"W_gate_up": MOE_PACK_GATE_UP, "Ws_gate_up": MOE_PACK_GATE_UP,
             "W_down": MOE_PACK_PLAIN, "Ws_down": MOE_PACK_PLAIN,
             "W_lat_down": MOE_PACK_PLAIN, "W_lat_up": MOE_PACK_PLAIN}
    for key, kind in kinds.items():
        w = weights.get(key)
        if w is None:
            continue
        w3 = w if w.dim() == 3 else w.unsqueeze(0)
        dst = torch.empty_like(w3)
        moe_pack_weights(kind, w3.shape[0], w3.shape[1], w3.shape[2], w3, dst, stream)
        out[key] = dst if w.dim() == 3 else dst.squeeze(0)
    return out
