"""The C-ABI library builds, loads without a GPU and exports every symbol the
public header declares; argument checks answer before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def fgs():
    import __graft_entry__
    __graft_entry__.build()
    import fine_grained_sparse_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("moe_router", "moe_router_from_logits", "moe_permute", "moe_grouped_swiglu",
                     "moe_combine", "moe_layer_forward", "moe_workspace_size"):
        assert required in names


def test_library_exports_every_declared_symbol(fgs):
    lib = ctypes.CDLL(fgs.lib_path())
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(fgs):
    assert fgs.moe_version() >= 100
    assert fgs.moe_launch_count() == fgs.moe_launch_count()  # no launch without a GPU
    for code in range(8):
        assert fgs.moe_status_string(code) != "unknown status"


def _k2(fgs, **kw):
    base = dict(d_model=7168, d_ff=2048, E_routed=384, E_shared=1, d_ff_shared=2048, K=8,
                n_group=8, topk_group=4, dtype=fgs.MOE_BF16)
    base.update(kw)
    return fgs.config(**base)


@pytest.mark.parametrize("kw,status", [
    ({}, 0),
    ({"K": 0}, 1),
    ({"K": 385}, 1),
    ({"E_routed": 1025, "n_group": 1, "topk_group": 1}, 1),
    ({"n_group": 5}, 1),                      # 384 % 5 != 0
    ({"topk_group": 9}, 1),
    ({"E_routed": 64, "n_group": 8, "topk_group": 1, "K": 9}, 1),  # K > topk_group * E / n_group
    ({"d_model": 7200}, 2),                   # bf16 path: d % 128
    ({"d_ff": 2000}, 2),
    ({"d_latent": 3000}, 2),
    ({"K": 33, "n_group": 1, "topk_group": 1}, 2),
    ({"dtype": 7}, 1),
])
def test_validate_config(fgs, kw, status):
    assert fgs.moe_validate_config(_k2(fgs, **kw), 8192) == status


def test_validate_rows(fgs):
    assert fgs.moe_validate_config(_k2(fgs), 0) == 1
    assert fgs.moe_validate_config(_k2(fgs), 1) == 0


def test_workspace_size_grows_with_T(fgs):
    cfg = _k2(fgs)
    a, b = fgs.moe_workspace_size(cfg, 128), fgs.moe_workspace_size(cfg, 8192)
    assert 0 < a < b
    assert fgs.moe_workspace_size(_k2(fgs, K=0), 128) == 0
    # the gathered rows alone: T*K rows of d bf16
    assert b > 8192 * 8 * 7168 * 2


def test_argument_errors_return_before_any_cuda_call(fgs):
    cfg = _k2(fgs)
    lib = fgs.lib
    # null pointers
    assert lib.moe_router(ctypes.byref(cfg), 16, None, None, None, None, None, None, 0, None) == 1
    # misaligned pointers (never dereferenced: the check comes first)
    bad = 0x1001
    assert lib.moe_router(ctypes.byref(cfg), 16, bad, 0x1000, 0x1000, 0x1000, 0x1000, None, 0,
                          None) == 3
    assert lib.moe_router_from_logits(ctypes.byref(cfg), 16, 0x1000, bad, 0x1000, 0x1000, None) == 3
    # workspace too small
    ws = fgs.moe_workspace_size(cfg, 16)
    assert lib.moe_layer_forward(ctypes.byref(cfg), 16, *([0x1000] * 10), None, None, None,
                                 0x1000, ws - 256, None, None) == 4
    assert "workspace" in fgs.moe_last_error_detail()
    # shape the bf16 path does not cover
    assert lib.moe_linear(16, 100, 128, 0x1000, 0x1000, None, 0x1000, 0x1000, 4096, None) == 2
    # invalid config reaches every entry point
    assert lib.moe_permute(ctypes.byref(_k2(fgs, K=0)), 16, *([0x1000] * 5), 0x1000, 4096, None) == 1


def test_python_binding_raises(fgs):
    cfg = _k2(fgs)
    with pytest.raises(fgs.MoeError) as ei:
        fgs.moe_router(cfg, 16, None, None, None, None, None, stream=0)
    assert ei.value.status == 1


@pytest.mark.parametrize("kw,status", [
    ({}, 0),
    ({"d_ff": 2048 - 64}, 2),       # FP8 blocks: d_ff % 128
    ({"d_ff_shared": 192}, 2),
    ({"d_model": 7168 + 64}, 2),    # d_model % 128 fails the bf16 rule first, also FP8's
    ({"d_latent": 3584}, 0),
    ({"d_latent": 3584 - 64}, 2),
    ({"dtype": 0}, 2),              # FP8 weights need bf16 activations
])
def test_validate_config_fp8_layout(fgs, kw, status):
    cfg = _k2(fgs, weight_layout=fgs.MOE_WEIGHTS_PACKED_FP8, **kw)
    assert fgs.moe_validate_config(cfg, 8192) == status


def test_packed_fp8_bytes(fgs):
    # codes, then one 16-byte record per (group, pair of 128-row tiles, 64-column k step)
    assert fgs.moe_packed_fp8_bytes(384, 4096, 7168) == 384 * 4096 * 7168 + 384 * 16 * 112 * 16
    assert fgs.moe_packed_fp8_bytes(2, 384, 256) == 2 * 384 * 256 + 2 * 2 * 4 * 16  # odd pair
    for bad in [(0, 128, 128), (1, 192, 128), (1, 128, 192), (1, 64, 128)]:
        assert fgs.moe_packed_fp8_bytes(*bad) == -1


def test_pack_fp8_argument_errors(fgs):
    lib = fgs.lib
    assert lib.moe_pack_weights_fp8(5, 1, 128, 128, 0x1000, 0x1000, 0x100000, None) == 1  # kind
    assert lib.moe_pack_weights_fp8(1, 1, 192, 128, 0x1000, 0x1000, 0x100000, None) == 2  # rows
    assert lib.moe_pack_weights_fp8(1, 1, 128, 128, 0x1001, 0x1000, 0x100000, None) == 3  # align
    assert lib.moe_pack_weights_fp8(1, 1, 128, 128, 0x1000, 0x1000, 0x1000, None) == 1  # overlap


def test_router_weight_split_form_argument_errors(fgs):
    lib = fgs.lib
    cfg = fgs.config(d_model=7168, E_routed=384, K=8)
    assert fgs.moe_router_weight_split_bytes(cfg) == 6 * 384 * 7168
    assert fgs.moe_router_weight_split_bytes(fgs.config(d_model=96, E_routed=16, K=4)) == 0
    split = fgs.config(d_model=256, E_routed=16, K=4, router_weight=fgs.MOE_ROUTER_WEIGHT_SPLIT)
    assert fgs.moe_validate_config(split, 64) == 0
    assert fgs.moe_validate_config(fgs.config(d_model=256, E_routed=16, K=4, router_weight=2), 64) == 1
    # moe_split_router_weight: shape, alignment and overlap checks
    bad_d = fgs.config(d_model=96, E_routed=16, K=4)
    assert lib.moe_split_router_weight(ctypes.byref(bad_d), 0x1000, 0x100000, None) == 2
    assert lib.moe_split_router_weight(ctypes.byref(split), 0x1004, 0x100000, None) == 3
    assert lib.moe_split_router_weight(ctypes.byref(split), 0x1000, 0x2000, None) == 1
    assert lib.moe_split_router_weight(ctypes.byref(split), None, 0x100000, None) == 1
    # the split form needs the tensor-core path: a workspace and bf16 x
    assert lib.moe_router(ctypes.byref(split), 64, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000,
                          None, 0, None) == 2
    split_f32 = fgs.config(d_model=256, E_routed=16, K=4, dtype=fgs.MOE_F32,
                           router_weight=fgs.MOE_ROUTER_WEIGHT_SPLIT)
    assert lib.moe_router(ctypes.byref(split_f32), 64, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000,
                          0x100000, 1 << 30, None) == 2


def test_combine_argument_errors(fgs):
    lib = fgs.lib
    cfg = _k2(fgs)
    # Y, inv, topk_w, Y_shared, y: null Y, then a misaligned topk_w
    assert lib.moe_combine(ctypes.byref(cfg), 16, None, 0x1000, None, None, 0x1000, None) == 1
    assert lib.moe_combine(ctypes.byref(cfg), 16, 0x1000, 0x1000, 0x1004, None, 0x1000, None) == 3
    # Y_shared with the latent form
    k3 = _k2(fgs, d_latent=3584, n_group=1, topk_group=1)
    assert lib.moe_combine(ctypes.byref(k3), 16, 0x1000, 0x1000, None, 0x2000, 0x3000, None) == 1


def test_host_pipeline_release_without_state(fgs):
    lib = fgs.lib
    assert lib.moe_layer_forward_host_release(None) == 1
    # a workspace that never went through moe_layer_forward_host: nothing to release
    assert lib.moe_layer_forward_host_release(0x1000) == 0
    # nothing pending: the flush enqueues nothing (no stream is touched)
    assert lib.moe_layer_forward_host_flush(None, None) == 1
    assert lib.moe_layer_forward_host_flush(0x1000, None) == 0


@pytest.mark.parametrize("E,T,split,ok", [
    (384, 32938, False, True), (384, 32939, False, False),
    (384, 43690, True, True), (384, 43691, True, False),
    (896, 7972, False, True), (896, 7973, False, False),
    (896, 18724, True, True), (896, 18725, True, False),
])
def test_noalloc_router_size_bound(fgs, E, T, split, ok):
    """moe_router_noalloc rejects a problem, before any CUDA call, exactly when
    even one K part overflows its 64 MiB scratch (the bound its header
    states); larger problems are rejected, smaller ones get past the check."""
    cfg = fgs.config(d_model=7168, E_routed=E, K=8,
                     router_weight=fgs.MOE_ROUTER_WEIGHT_SPLIT if split else 0)
    need = 256 + (0 if split else (6 * E * 7168 + 255) // 256 * 256) + \
        (4 * T * E + 255) // 256 * 256
    if ok:
        # accepted sizes would go on to the GPU: check the bound arithmetic only
        assert need <= 64 << 20
        return
    assert need > 64 << 20
    st = fgs.lib.moe_router_noalloc(ctypes.byref(cfg), T, 0x1000, 0x1000, 0x1000, 0x1000,
                                    0x1000, None)
    assert st == 4
    assert "static scratch" in fgs.moe_last_error_detail()


def test_quantile_bias_argument_errors(fgs):
    lib = fgs.lib
    cfg = fgs.config(d_model=128, E_routed=16, K=4)
    assert lib.moe_quantile_bias_update(ctypes.byref(cfg), 8, None, 1.0, 0x1000, 0x1000, None) == 1
    assert lib.moe_quantile_bias_update(ctypes.byref(cfg), 8, 0x1000, 1.5, 0x1000, 0x1000, None) == 1
    assert lib.moe_quantile_bias_update(ctypes.byref(cfg), 8, 0x1000, 1.0, 0x1004, 0x1000, None) == 3
