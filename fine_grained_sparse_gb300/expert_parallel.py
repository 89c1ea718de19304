"""Expert-parallel dispatch and combine across ranks: the exchange plan and
the two all-to-all transfers around the expert GEMMs.

"Kimi K2" (visual-learn), "Many experts, few used at a time": the experts a
token selects live on other chips, and the exchange between chips costs
time; "Kimi K3's router picks 16 of 896 experts", closing sections: K3 needs
dedicated communication infrastructure for FFN routing and is deployed on 64
or more accelerators.  This module holds the host side of that exchange; the
per-rank work (router, dispatch order, expert GEMMs, combine) is the
single-GPU library's.

Layout.  Experts are split contiguously over the W ranks of the group: rank q
owns experts [q E / W, (q + 1) E / W) (E divisible by W).  moe_permute orders
a rank's dispatched rows expert-major, so the rows bound for rank q are one
contiguous run of slots, [offsets[q E / W], offsets[(q + 1) E / W]).

Exchange.  (1) Every rank sends each peer the per-expert counts of the
peer's experts (one small all-to-all), so the receiver knows, per source
rank, how many rows each of its experts gets.  (2) The dispatched rows go
out with one all-to-all whose send splits are the row counts per destination
and whose receive splits are the row counts per source.  They arrive
source-major (all rows from rank 0, expert-major among them, then rank 1,
...); ``Plan.local_order`` regroups them expert-major (each local expert's
rows from rank 0, then rank 1, ...), the order the grouped GEMM reads with
``Plan.local_offsets``.  (3) The experts' outputs go back through the inverse
of that regrouping and the reverse all-to-all, and land in the sender's slot
order, where moe_combine sums them with the sender's own inv and gate
weights.

Tensors may live on the CPU (gloo) or a GPU (NCCL); counts travel as int64.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Tuple

import numpy as np

__all__ = ["Plan", "expert_range", "plan_dispatch", "dispatch_rows", "return_rows"]


def expert_range(E: int, world: int, rank: int) -> Tuple[int, int]:
    """[first, last) experts of ``rank`` under the contiguous split."""
    if world < 1 or E % world:
        raise ValueError(f"{E} experts do not split evenly over {world} ranks")
    per = E // world
    return rank * per, (rank + 1) * per


@dataclasses.dataclass
class Plan:
    world: int
    rank: int
    E: int
    send_splits: List[int]        # rows this rank sends to each rank (its slot order)
    recv_splits: List[int]        # rows this rank receives from each rank
    counts_from: np.ndarray       # [world, E / world]: rows per (source, local expert)
    local_counts: np.ndarray      # [E / world]: rows per local expert
    local_offsets: np.ndarray     # [E / world + 1]: expert-major offsets of the local rows
    local_order: np.ndarray       # expert-major position -> position in the received rows


def plan_dispatch(counts, E: int, group=None, device="cpu") -> Plan:
    """The exchange plan from this rank's per-expert counts (moe_permute's
    ``counts``).  Collective over ``group``: every rank calls it."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    counts = np.asarray(counts, dtype=np.int64).reshape(-1)
    if counts.size != E:
        raise ValueError("counts must hold one entry per routed expert")
    per = expert_range(E, world, 0)[1]
    send_splits = [int(counts[q * per:(q + 1) * per].sum()) for q in range(world)]
    # each peer gets the counts of its own experts
    out = torch.empty(E, dtype=torch.int64, device=device)
    dist.all_to_all_single(out, torch.as_tensor(counts, device=device), [per] * world,
                           [per] * world, group=group)
    counts_from = out.cpu().numpy().reshape(world, per)
    recv_splits = [int(v) for v in counts_from.sum(axis=1)]
    local_counts = counts_from.sum(axis=0)
    local_offsets = np.concatenate([[0], np.cumsum(local_counts)]).astype(np.int64)
    # received rows: source p's block starts at src_start[p]; inside it the
    # rows of local expert j start at src_start[p] + sum_{i<j} counts_from[p, i]
    src_start = np.concatenate([[0], np.cumsum(recv_splits)[:-1]]).astype(np.int64)
    within = np.concatenate([np.zeros((world, 1), np.int64), np.cumsum(counts_from, axis=1)[:, :-1]],
                            axis=1)
    order = np.empty(int(local_offsets[-1]), dtype=np.int64)
    pos = 0
    for j in range(per):
        for p in range(world):
            n = int(counts_from[p, j])
            start = int(src_start[p] + within[p, j])
            order[pos:pos + n] = np.arange(start, start + n)
            pos += n
    return Plan(world, rank, E, send_splits, recv_splits, counts_from, local_counts,
                local_offsets, order)


def dispatch_rows(rows, plan: Plan, group=None):
    """Send this rank's dispatched rows (slot order, [sum(send_splits), D])
    to the experts' owners; returns the rows of this rank's experts,
    expert-major ([sum(local_counts), D])."""
    import torch
    import torch.distributed as dist

    recv = rows.new_empty((sum(plan.recv_splits),) + tuple(rows.shape[1:]))
    dist.all_to_all_single(recv, rows.contiguous(), plan.recv_splits, plan.send_splits,
                           group=group)
    return recv[torch.as_tensor(plan.local_order, device=recv.device)]


def return_rows(local_out, plan: Plan, group=None):
    """The inverse of ``dispatch_rows``: this rank's experts' outputs
    (expert-major) back to the ranks that sent the rows; returns this rank's
    rows in its own slot order ([sum(send_splits), D])."""
    import torch
    import torch.distributed as dist

    by_source = torch.empty_like(local_out)
    by_source[torch.as_tensor(plan.local_order, device=local_out.device)] = local_out
    back = local_out.new_empty((sum(plan.send_splits),) + tuple(local_out.shape[1:]))
    dist.all_to_all_single(back, by_source, plan.send_splits, plan.recv_splits, group=group)
    return back
