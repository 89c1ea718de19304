"""Expert-parallel dispatch and combine (fine_grained_sparse_gb300.expert_parallel)
on gloo ranks on the CPU.

Each rank routes its own tokens (the oracle's router), orders the (token,
slot) pairs with the oracle's permute, and sends the dispatched rows to the
ranks that own their experts.  Every rank evaluates only its own experts (the
oracle's SwiGLU) on the rows it received, sends the outputs back, and
combines them with its own inv and gate weights.  The result must equal the
single-process oracle layer on that rank's tokens, and the exchange plans of
the ranks must agree with one another.
"""
import json
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _layer(seed, E, d, F):
    rng = np.random.default_rng(seed)
    gu = rng.normal(0, 0.2, (E, 2 * F, d))
    dn = rng.normal(0, 0.2, (E, d, F))
    sgu = rng.normal(0, 0.2, (1, 2 * F, d))
    sdn = rng.normal(0, 0.2, (1, d, F))
    Wr = rng.normal(0, 0.3, (E, d))
    b = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    return gu, dn, sgu, sdn, Wr, b


def _rank_main(rank, world, port, E, K, out_dir):
    import torch.distributed as dist
    import oracle
    from fine_grained_sparse_gb300 import expert_parallel as ep

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    d, F = 16, 8
    gu, dn, sgu, sdn, Wr, b = _layer(7, E, d, F)
    T = 23 + 9 * rank  # ranks hold different numbers of tokens
    x = np.random.default_rng(100 + rank).normal(size=(T, d))
    r = oracle.router_from_x(x, Wr, b, K)
    p = oracle.permute(r["idx"], E)
    rows = torch.as_tensor(x[p["perm"] // K])  # dispatched rows, slot order
    plan = ep.plan_dispatch(p["counts"], E)
    local = ep.dispatch_rows(rows, plan).numpy()
    e0, e1 = ep.expert_range(E, world, rank)
    out = np.zeros_like(local)
    for j, e in enumerate(range(e0, e1)):
        a, z = plan.local_offsets[j], plan.local_offsets[j + 1]
        if z > a:
            out[a:z] = oracle.swiglu_expert(local[a:z], gu[e, :F], gu[e, F:], dn[e])
    back = ep.return_rows(torch.as_tensor(out), plan).numpy()
    Ysh = oracle.swiglu_expert(x, sgu[0, :F], sgu[0, F:], sdn[0])[None]
    y = oracle.combine(back, p["inv"], r["w"], Ysh)
    ref = oracle.moe_layer_tokens(x, Wr, b, gu, dn, sgu, sdn, K)
    res = {"err": float(np.abs(y - ref["y"]).max() / np.abs(ref["y"]).max()),
           "send": plan.send_splits, "recv": plan.recv_splits,
           "counts_from": plan.counts_from.tolist(), "counts": p["counts"].tolist(),
           "local_rows": int(plan.local_offsets[-1]), "T": T}
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(res, f)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()  # the ranks import the package, which loads the library


@pytest.mark.parametrize("world,E,K", [(2, 8, 2), (2, 12, 3), (3, 12, 4)])
def test_expert_parallel_matches_single_process_layer(tmp_path, world, E, K):
    mp.start_processes(_rank_main, args=(world, _free_port(), E, K, str(tmp_path)),
                       nprocs=world, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    per = E // world
    for q, rq in enumerate(res):
        assert rq["err"] <= 1e-12
        # rank q receives from p exactly what p sends to q, per expert
        for p, rp in enumerate(res):
            assert rq["recv"][p] == rp["send"][q]
            assert rq["counts_from"][p] == rp["counts"][q * per:(q + 1) * per]
        assert sum(rq["send"]) == rq["T"] * K
        assert rq["local_rows"] == sum(rq["recv"])


def test_expert_range_partition():
    from fine_grained_sparse_gb300 import expert_parallel as ep
    assert [ep.expert_range(384, 8, q) for q in (0, 7)] == [(0, 48), (336, 384)]
    with pytest.raises(ValueError):
        ep.expert_range(10, 4, 0)
