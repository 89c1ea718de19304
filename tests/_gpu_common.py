"""Shared helpers of the GPU parity tests (not collected as a test module)."""
import numpy as np
import pytest
import torch

cuda_ok = torch.cuda.is_available()


def need_gpu():
    if not cuda_ok:
        pytest.skip("no CUDA device")


def lib():
    import fine_grained_sparse_gb300 as fgs
    return fgs


def np64(t: torch.Tensor) -> np.ndarray:
    """Exact fp64 copy of a tensor's values (bf16 and fp32 upcast exactly)."""
    return t.detach().cpu().to(torch.float64).numpy()


def workspace(cfg, T):
    fgs = lib()
    n = fgs.moe_workspace_size(cfg, T)
    assert n > 0, fgs.moe_last_error_detail()
    return torch.zeros(n, dtype=torch.uint8, device="cuda"), n


def rel_max_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-300))


def to_f64_cpu(t: torch.Tensor) -> np.ndarray:
    """Oracle-side upcast of one weight slice: copied to the host first."""
    return t.detach().cpu().to(torch.float64).numpy()


# Tolerances (max |got - ref| / max |ref|)
#  * gate weights, fp32 router: the kernel computes sigmoid and the
#    renormalisation in fp64 and rounds once to fp32 (2^-24 relative); the
#    logits of the GEMM path differ from the oracle's fp64 logits by the fp32
#    accumulation error (~d * 2^-24 * |x||w| ~ 1e-6 relative to the logit).
#    1e-4 is the bound the layer is specified to.
TOL_WEIGHTS = 1e-4
#  * layer / expert outputs with bf16 experts: the expert inputs and weights
#    are exact bf16 values on both sides; the kernel rounds H (the SwiGLU
#    activation) and Y (each weighted expert output) to bf16 (2^-9 relative
#    each), so a K-term sum stays well inside 1e-2 of max |ref|.
TOL_BF16 = 1e-2
#  * layer outputs with fp32 experts: fp32 FMA accumulation over d_model and
#    d_ff terms (~1e-6 relative) plus fp32 expf in SiLU.
TOL_F32 = 1e-4
# Tokens whose K-th vs (K+1)-th biased score gap (or group gap) is below this
# may legitimately select differently when the logits come from the fp32 GEMM.
GAP_MIN = 1e-5


def by_expert(idx, w=None):
    """Selected sets in ascending expert order (and the weights aligned to
    them).  The order inside the selected set is a convention that near-equal
    scores may flip when the two sides' logits differ by rounding; the set is
    what the margin criterion fixes."""
    idx = np.asarray(idx)
    order = np.argsort(idx, axis=1, kind="stable")
    sidx = np.take_along_axis(idx, order, axis=1)
    if w is None:
        return sidx
    return sidx, np.take_along_axis(np.asarray(w), order, axis=1)


def rows_covering_experts(idx, E, K, largest=None, step=128):
    """Token rows that reach the row tiles of the expert GEMMs at full size:
    for each expert that received pairs (or only the ``largest`` ones by
    pair count), the tokens in its first and last slot and in every
    ``step``-th slot between them, so that each of its row tiles (at most 256
    rows) and its ragged tail are compared.  Slots follow the dispatch order
    (the oracle's permute of the device's expert indices, which the permute
    tests pin bit for bit)."""
    import oracle
    p = oracle.permute(np.asarray(idx), E)
    live = [e for e in range(E) if p["counts"][e] > 0]
    if largest is not None:
        live = sorted(live, key=lambda e: -int(p["counts"][e]))[:largest]
    rows = set()
    for e in live:
        m = int(p["counts"][e])
        o = int(p["offsets"][e])
        for r in sorted(set(list(range(0, m, step)) + [m - 1])):
            rows.add(int(p["perm"][o + r]) // K)
    return np.array(sorted(rows), dtype=np.int64)
