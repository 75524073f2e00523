"""Expert-parallel sharding of the MoE layer: the partition, the dispatch plan
and the two all-to-all exchanges (host-side bookkeeping over torch.distributed).

The layer's tokens are independent, so the plain multi-GPU form is replicas
(every rank holds all experts and its own tokens; no collective).  Expert
parallelism instead splits the experts: with G ranks, rank r owns the
contiguous experts [r E / G, (r + 1) E / G) (E divisible by G); the router and
the shared expert are replicated, and every rank routes its own tokens.  A
layer then runs as:

1. route (on each rank, its own tokens): idx [T, k] ascending, w [T, k];
2. dispatch: every pick (t, j) is a row x_t sent to the owner of idx[t, j].
   Rows leave in the stable order (owner, expert, token), so each destination
   receives, from each source, its rows already grouped by expert with tokens
   ascending.  One all-to-all of the per-destination counts, then one
   all-to-all of the rows (and of their expert ids).  Remote rows land in a
   local buffer before any expert GEMM reads them;
3. local experts: the received rows, regrouped by (local expert, source rank,
   arrival order) -- a stable permutation -- run through the grouped expert
   FFNs as one expert group each;
4. combine: the expert outputs go back with the reverse all-to-all (the same
   counts, transposed), are put back into pick order (t, j), and each token sums
   w[t, j] * o_j over j in ascending expert order, plus its shared expert's
   output computed locally.

Exchanges use no multicast and no peer memory; each is a plain
``all_to_all_single`` with split sizes (NCCL on GPUs, gloo on CPU).  This module
moves rows and indices only: it does none of the layer's arithmetic (no router,
no FFN, no weighted sum).  "Optimizing on-device inference for Apple Silicon",
section "Keeping expert routing on the GPU": the same histogram / prefix /
stable-scatter grouping, here applied once per destination rank and once per
local expert.
"""
from __future__ import annotations

import dataclasses

import torch
import torch.distributed as dist


def experts_per_rank(n_experts: int, world: int) -> int:
    if world < 1 or n_experts % world != 0:
        raise ValueError(f"{n_experts} experts do not split evenly over {world} ranks")
    return n_experts // world


def expert_owner(expert: torch.Tensor, n_experts: int, world: int) -> torch.Tensor:
    """Rank that owns each expert id (contiguous blocks of E / G experts)."""
    return torch.div(expert, experts_per_rank(n_experts, world), rounding_mode="floor")


@dataclasses.dataclass
class DispatchPlan:
    """Where every pick of this rank's tokens goes, and how many rows move.

    order        [T k] int64: flat pick ids t k + j in sending order
                 (owner rank, expert, token ascending)
    send_counts  [G] rows sent to each rank
    recv_counts  [G] rows received from each rank (after ``exchange_counts``)
    """

    order: torch.Tensor
    send_counts: list
    recv_counts: list | None = None


def plan_dispatch(idx: torch.Tensor, n_experts: int, world: int) -> DispatchPlan:
    """Sending order of the picks of idx [T, k] and the per-destination counts."""
    T, k = idx.shape
    e = idx.reshape(-1).to(torch.int64)
    t = torch.arange(T, dtype=torch.int64).repeat_interleave(k)
    owner = expert_owner(e, n_experts, world)
    key = (owner * n_experts + e) * max(T, 1) + t
    order = torch.sort(key, stable=True).indices
    counts = torch.bincount(owner, minlength=world)
    return DispatchPlan(order=order, send_counts=[int(c) for c in counts])


def exchange_counts(plan: DispatchPlan, group=None) -> DispatchPlan:
    """All-to-all of the per-destination row counts: fills ``plan.recv_counts``."""
    world = dist.get_world_size(group)
    send = torch.tensor(plan.send_counts, dtype=torch.int64)
    recv = torch.empty(world, dtype=torch.int64)
    dist.all_to_all_single(recv, send, group=group)
    plan.recv_counts = [int(c) for c in recv]
    return plan


def dispatch(x: torch.Tensor, idx: torch.Tensor, n_experts: int, group=None):
    """Send each pick's token row to the rank owning its expert.

    x [T, d] (any dtype), idx [T, k].  Returns (plan, rows [R, d], experts [R])
    where R = sum(plan.recv_counts) and the received rows come grouped by
    source rank, each source's rows in (expert, token) order."""
    world = dist.get_world_size(group)
    T, k = idx.shape
    plan = exchange_counts(plan_dispatch(idx, n_experts, world), group)
    tok = torch.div(plan.order, k, rounding_mode="floor")
    send_rows = x[tok].contiguous()
    send_e = idx.reshape(-1).to(torch.int64)[plan.order].contiguous()
    n_recv = sum(plan.recv_counts)
    rows = torch.empty((n_recv, x.shape[1]), dtype=x.dtype)
    experts = torch.empty(n_recv, dtype=torch.int64)
    dist.all_to_all_single(rows, send_rows, plan.recv_counts, plan.send_counts, group=group)
    dist.all_to_all_single(experts, send_e, plan.recv_counts, plan.send_counts, group=group)
    return plan, rows, experts


def local_groups(experts: torch.Tensor, first_expert: int, n_local: int):
    """Regroup received rows by local expert, stably (expert, arrival order).

    Returns (counts [n_local], offsets [n_local + 1], perm [R]): perm lists the
    received row indices of local expert 0, then 1, ... in arrival order (which
    is source rank, then token)."""
    local = experts - first_expert
    if local.numel() and (int(local.min()) < 0 or int(local.max()) >= n_local):
        raise ValueError("a received row names an expert this rank does not own")
    perm = torch.sort(local, stable=True).indices
    counts = torch.bincount(local, minlength=n_local)
    offsets = torch.zeros(n_local + 1, dtype=torch.int64)
    offsets[1:] = torch.cumsum(counts, 0)
    return counts, offsets, perm


def combine_rows(out_rows: torch.Tensor, plan: DispatchPlan, T: int, k: int, group=None) -> torch.Tensor:
    """Return each expert output row to the rank that sent the pick.

    out_rows [R, d]: the output for each received row, in the order the rows
    were received.  Returns per_pick [T, k, d] on the sending rank: the output
    of pick (t, j), ready for the weighted sum over j."""
    d = out_rows.shape[1]
    back = torch.empty((T * k, d), dtype=out_rows.dtype)
    dist.all_to_all_single(back, out_rows.contiguous(), plan.send_counts, plan.recv_counts, group=group)
    per_pick = torch.empty_like(back)
    per_pick[plan.order] = back
    return per_pick.reshape(T, k, d)
