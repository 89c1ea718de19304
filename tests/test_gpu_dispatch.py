"""Dispatch (moe_permute) and combine parity on the GPU: bit-exact integers."""
import numpy as np
import pytest
import torch

import oracle
from _gpu_common import lib, need_gpu, np64, rel_max_err, workspace

pytestmark = pytest.mark.gpu


def _distinct_idx(T, E, K, gen, skew=False):
    if skew:  # most tokens share a handful of experts
        w = torch.ones(E)
        w[: max(K, 4)] = 200.0
    else:
        w = torch.ones(E)
    return torch.stack([torch.multinomial(w, K, replacement=False, generator=gen)
                        for _ in range(T)]).to(torch.int32)


def _run_permute(idx, E, K):
    fgs = lib()
    T = idx.shape[0]
    cfg = fgs.config(d_model=128, E_routed=E, K=K)
    ws, nws = workspace(cfg, T)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * K, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * K, dtype=torch.int32, device="cuda")
    fgs.moe_permute(cfg, T, idx.cuda(), counts, offsets, perm, inv, ws, nws)
    status = fgs.moe_get_device_status(ws)
    return status, counts.cpu().numpy(), offsets.cpu().numpy(), perm.cpu().numpy(), inv.cpu().numpy()


@pytest.mark.parametrize("T,E,K,skew", [(1, 4, 2, False), (7, 16, 4, False), (300, 384, 8, False),
                                        (8192, 384, 8, True), (4096, 896, 16, False),
                                        (33, 8, 8, False), (1000, 64, 1, True)])
def test_permute_bit_exact(T, E, K, skew):
    need_gpu()
    gen = torch.Generator().manual_seed(T * 31 + E)
    idx = _distinct_idx(T, E, K, gen, skew)
    status, counts, offsets, perm, inv = _run_permute(idx, E, K)
    assert status == 0
    ref = oracle.permute(idx.numpy(), E)
    np.testing.assert_array_equal(counts, ref["counts"])
    np.testing.assert_array_equal(offsets, ref["offsets"])
    np.testing.assert_array_equal(perm, ref["perm"])
    np.testing.assert_array_equal(inv, ref["inv"])


def test_permute_reports_bad_index():
    """An expert index outside [0, E) is reported, its pair left out of the
    counts and its inv entry set to -1; a combine over that inv stays inside
    Y and sums the token's remaining pairs."""
    need_gpu()
    fgs = lib()
    idx = torch.tensor([[0, 1], [2, 9], [3, 1]], dtype=torch.int32)  # 9 >= E = 4
    status, counts, offsets, perm, inv = _run_permute(idx, 4, 2)
    assert status == 7  # MOE_ERR_DEVICE_INDEX
    assert counts.sum() == 5 and offsets[-1] == 5
    assert inv[3] == -1
    good = np.array([0, 1, 2, 4, 5])
    ref = oracle.permute(idx.numpy().reshape(-1)[good].reshape(-1, 1), 4)
    np.testing.assert_array_equal(counts, ref["counts"])
    # the valid pairs keep the slots the oracle gives them
    np.testing.assert_array_equal(inv[good], ref["inv"])
    T, K, d = 3, 2, 128
    gen = torch.Generator().manual_seed(9)
    Y = torch.randn((T * K, d), generator=gen).to(torch.bfloat16)
    w = torch.rand((T, K), generator=gen)
    cfg = fgs.config(d_model=d, d_ff=64, E_routed=4, K=K)
    y = torch.full((T, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    fgs.moe_combine(cfg, T, Y.cuda(), torch.from_numpy(inv).cuda(), w.cuda(), None, y)
    torch.cuda.synchronize()
    inv_ok = np.where(inv >= 0, inv, 0)
    w_ok = np.where(inv.reshape(T, K) >= 0, w.numpy(), 0.0)
    want = oracle.combine(np64(Y), inv_ok, w_ok)
    got = np64(y)
    assert np.isfinite(got).all()
    assert rel_max_err(got, want) <= 2 ** -8


@pytest.mark.parametrize("weighted", [False, True], ids=["weights_in_Y", "weights_in_combine"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_combine(dtype, weighted):
    """moe_combine against the oracle's combine over the oracle's permute:
    y[t] = sum_k w[t, k] Y[inv[t K + k]] + sum_s Y_shared[s, t]."""
    need_gpu()
    fgs = lib()
    T, K, d, S = 77, 4, 256, 2
    gen = torch.Generator().manual_seed(5)
    idx = _distinct_idx(T, 12, K, gen)
    ref_p = oracle.permute(idx.numpy(), 12)
    Y = torch.randn((T * K, d), generator=gen).to(dtype)
    Ys = torch.randn((S, T, d), generator=gen).to(dtype)
    w = torch.rand((T, K), generator=gen) * 2.827 if weighted else None
    cfg = fgs.config(d_model=d, d_ff=64, E_routed=12, E_shared=S, d_ff_shared=64, K=K,
                     dtype=fgs.MOE_BF16 if dtype == torch.bfloat16 else fgs.MOE_F32)
    y = torch.empty((T, d), dtype=dtype, device="cuda")
    inv = torch.from_numpy(ref_p["inv"].astype(np.int32)).cuda()
    fgs.moe_combine(cfg, T, Y.cuda(), inv, w.cuda() if weighted else None, Ys.cuda(), y)
    torch.cuda.synchronize()
    want = oracle.combine(np64(Y), ref_p["inv"], w.numpy() if weighted else np.ones((T, K)),
                          np64(Ys))
    # bf16: one rounding of the fp32 sum (2^-9) plus fp32 summation error
    tol = 2 ** -8 if dtype == torch.bfloat16 else 1e-6
    assert rel_max_err(np64(y), want) <= tol
