"""Expert-parallel (EP) and expert-tensor-parallel (ETP) exchange bookkeeping
for a token-level MoE dispatcher whose experts are spread over ranks.

MoE Parallel Folding (arXiv 2504.14960) study notes, "method overview": after
the router and the permutation, an All-to-All-V sends every expert's rows to
the rank that holds the expert; with expert tensor parallelism an
AllGather-V collects the rows of an F-sharded expert over its group and a
ReduceScatter-V sums the partial outputs and hands each rank its own rows
back; the reverse All-to-All-V returns the outputs before the un-permutation.

On one GPU every one of these exchanges is the identity, and libmoe runs all E
experts locally. This module is the host-side logic for E experts over the
ranks of a torch.distributed group (gloo on CPU, NCCL on GPU):

- split sizes from the per-expert `counts` that moe_permute returns (the
  permuted rows are expert-major, so the rows for each rank are contiguous);
- the All-to-All-V of rows and its reverse;
- the chunk reordering between "by source rank, then expert" (the order in
  which rows arrive) and "by local expert, then source rank" (the order the
  grouped GEMM wants, so that each local expert's rows are contiguous);
- AllGather-V and ReduceScatter-V over an ETP group, the latter summing the
  partials in rank order (deterministic, the same on every backend).

Rows are torch tensors [n, d] on any device the group's backend supports.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch
import torch.distributed as dist


def chunk_order(sizes: torch.Tensor) -> torch.Tensor:
    """Row indices that reorder chunks laid out as sizes[a, b] (a-major: all
    chunks of a = 0 first) into b-major order (chunk (0,0), (1,0), ..., then
    (0,1), (1,1), ...). sizes is a 2-D int64 CPU tensor of chunk row counts."""
    A, B = sizes.shape
    flat = sizes.reshape(-1)
    starts = torch.zeros_like(flat)
    if flat.numel() > 1:
        starts[1:] = torch.cumsum(flat, 0)[:-1]
    starts = starts.reshape(A, B)
    parts = [torch.arange(int(starts[a, b]), int(starts[a, b] + sizes[a, b]), dtype=torch.int64)
             for b in range(B) for a in range(A)]
    if not parts:
        return torch.zeros(0, dtype=torch.int64)
    return torch.cat(parts)


@dataclass
class EPPlan:
    """Who sends how many rows to whom, for one layer call on one rank."""
    world: int
    rank: int
    experts_per_rank: int
    send_counts: torch.Tensor     # [world, E_local]: my rows for expert (j, e) on rank j
    recv_counts: torch.Tensor     # [world, E_local]: rows from rank src for my expert e
    send_splits: list             # rows to each rank
    recv_splits: list             # rows from each rank
    local_counts: torch.Tensor    # [E_local]: rows of each local expert over all sources
    local_offsets: torch.Tensor   # [E_local + 1] int32 prefix (moe_expert_ffn's offsets)
    to_expert_major: torch.Tensor     # received order -> (local expert, source) order
    from_expert_major: torch.Tensor   # its inverse


def ep_plan(counts: torch.Tensor, group=None) -> EPPlan:
    """Exchange the per-expert counts (a small All-to-All) and derive every
    split size. counts: [E] per-expert row counts of this rank's permuted rows
    (moe_permute's output); E must divide evenly over the group's ranks, rank j
    holding experts [j*E/world, (j+1)*E/world)."""
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    E = int(counts.numel())
    if E % world != 0:
        raise ValueError(f"{E} experts do not divide over {world} ranks")
    El = E // world
    send = counts.to(torch.int64).reshape(world, El).contiguous()
    recv = torch.empty_like(send)
    dist.all_to_all_single(recv, send, group=group)
    send_c, recv_c = send.cpu(), recv.cpu()
    local = recv_c.sum(0)
    offs = torch.zeros(El + 1, dtype=torch.int32)
    offs[1:] = torch.cumsum(local, 0).to(torch.int32)
    fwd = chunk_order(recv_c)
    inv = torch.empty_like(fwd)
    inv[fwd] = torch.arange(fwd.numel(), dtype=torch.int64)
    return EPPlan(world, rank, El, send_c, recv_c, send_c.sum(1).tolist(), recv_c.sum(1).tolist(),
                  local, offs, fwd, inv)


def ep_dispatch(Xp: torch.Tensor, plan: EPPlan, group=None) -> torch.Tensor:
    """All-to-All-V of this rank's expert-major rows Xp[:n_kept] to the ranks
    that hold their experts; returns the received rows in local-expert-major
    order (plan.local_offsets delimit the experts)."""
    n = sum(plan.send_splits)
    out = Xp.new_empty((sum(plan.recv_splits),) + tuple(Xp.shape[1:]))
    dist.all_to_all_single(out, Xp[:n].contiguous(), output_split_sizes=plan.recv_splits,
                           input_split_sizes=plan.send_splits, group=group)
    return out.index_select(0, plan.to_expert_major.to(out.device))


def ep_combine(Y_local: torch.Tensor, plan: EPPlan, group=None) -> torch.Tensor:
    """Reverse of ep_dispatch: local-expert-major output rows go back to the
    ranks they came from; returns this rank's rows in its own expert-major
    order (the layout moe_unpermute reads)."""
    by_source = Y_local.index_select(0, plan.from_expert_major.to(Y_local.device)).contiguous()
    out = Y_local.new_empty((sum(plan.send_splits),) + tuple(Y_local.shape[1:]))
    dist.all_to_all_single(out, by_source, output_split_sizes=plan.send_splits,
                           input_split_sizes=plan.recv_splits, group=group)
    return out


def etp_allgather_v(rows: torch.Tensor, counts: torch.Tensor, group=None):
    """AllGather-V over an ETP group whose ranks all hold the same experts
    (each an F-shard of them). rows: this rank's expert-major rows, counts
    [E] their per-expert counts. Returns (gathered rows in expert-major order
    over the group's ranks, gathered counts [world, E], the reorder indices)."""
    world = dist.get_world_size(group)
    E = int(counts.numel())
    c = counts.to(torch.int64).reshape(1, E)
    allc = [torch.empty_like(c) for _ in range(world)]
    dist.all_gather(allc, c, group=group)
    allc = torch.cat(allc).cpu()                      # [world, E]
    sizes = allc.sum(1)
    mx = int(sizes.max()) if world else 0
    n = int(sizes[dist.get_rank(group)])
    pad = rows.new_zeros((mx,) + tuple(rows.shape[1:]))
    pad[:n] = rows[:n]
    bufs = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(bufs, pad, group=group)
    flat = torch.cat([bufs[r][: int(sizes[r])] for r in range(world)])
    order = chunk_order(allc)                         # (rank, expert) -> (expert, rank)
    return flat.index_select(0, order.to(flat.device)), allc, order


def etp_reduce_scatter_v(partial: torch.Tensor, allc: torch.Tensor, order: torch.Tensor,
                         group=None) -> torch.Tensor:
    """ReduceScatter-V matching etp_allgather_v: partial [sum(allc), ...] in
    expert-major order holds this rank's F-shard contribution for every
    gathered row; returns the sum over the group's ranks (added in rank order)
    of the rows this rank contributed, in its own expert-major order."""
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    parts = [torch.empty_like(partial) for _ in range(world)]
    dist.all_gather(parts, partial.contiguous(), group=group)
    total = parts[0].clone()
    for r in range(1, world):
        total += parts[r]
    inv = torch.empty_like(order)
    inv[order] = torch.arange(order.numel(), dtype=torch.int64)
    by_rank = total.index_select(0, inv.to(total.device))
    sizes = allc.sum(1)
    start = int(sizes[:rank].sum())
    return by_rank[start:start + int(sizes[rank])]
