"""Host-side plan of an expert-parallel group (the C ABI's mok_ep_* calls do all row movement).

"Mixture-of-Kittens(MoK)란? ..." (alltoptrend), section 4 (1): one schedule table, built from every
rank's routing, drives the pull dispatch and the push combine of both passes.  Before the first
call each rank needs (a) the partition -- which tokens and experts it holds, (b) every rank's routing
ids, which on GPUs without shared memory arrive by an all-gather over the process group (on one GPU,
or over peer-mapped memory, the library reads the peers' buffers directly), and (c) the sizes of
the buffers it allocates.  This module computes those; it holds no layer arithmetic.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Partition:
    world: int
    rank: int
    tokens_per_rank: int
    experts_per_rank: int

    @property
    def tokens(self) -> range:
        return range(self.rank * self.tokens_per_rank, (self.rank + 1) * self.tokens_per_rank)

    @property
    def experts(self) -> range:
        return range(self.rank * self.experts_per_rank, (self.rank + 1) * self.experts_per_rank)


def partition(T: int, E: int, world: int, rank: int, max_ranks: int = 8) -> Partition:
    """Even split of T tokens and E experts over `world` ranks (rank r: tokens [r T/world, ...) and
    experts [r E/world, ...))."""
    if not 1 <= world <= max_ranks:
        raise ValueError(f"world must be in [1, {max_ranks}]")
    if not 0 <= rank < world:
        raise ValueError("rank outside the group")
    if T % world or E % world:
        raise ValueError("T and E must be multiples of the group size")
    return Partition(world, rank, T // world, E // world)


def exchange_routing(topk_ids_local: torch.Tensor, group=None) -> torch.Tensor:
    """Every rank's [tokens_per_rank, K] routing ids, concatenated in rank order ([T, K]), by an
    all-gather over the process group (CPU tensors with gloo, device tensors with NCCL)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    parts = [torch.empty_like(topk_ids_local) for _ in range(world)]
    dist.all_gather(parts, topk_ids_local.contiguous(), group=group)
    return torch.cat(parts)


def dispatch_counts(topk_ids_group: np.ndarray, part: Partition) -> np.ndarray:
    """[world (holding the token), world (owning the expert)]: slots each rank's tokens send to each
    rank's experts -- the rows every pull dispatch moves (ids outside the group's experts count
    nowhere: they are skipped)."""
    ids = np.asarray(topk_ids_group).reshape(part.world, -1)
    E = part.world * part.experts_per_rank
    out = np.zeros((part.world, part.world), np.int64)
    for src in range(part.world):
        valid = ids[src][(ids[src] >= 0) & (ids[src] < E)]
        out[src] = np.bincount(valid // part.experts_per_rank, minlength=part.world)
    return out


def buffer_bytes(mok, cfg, shape_group, part: Partition) -> dict:
    """Device bytes one rank allocates: its workspace and forward context (shape: the group's T,
    this rank's experts), and its receive buffers of expert outputs and of dX rows."""
    shape = mok.make_shape(shape_group.T, shape_group.H, shape_group.I, part.experts_per_rank, shape_group.K)
    recv = part.tokens_per_rank * shape_group.K * shape_group.H * 2
    return dict(workspace=mok.mok_workspace_bytes(cfg, shape), fwd_ctx=mok.mok_fwd_ctx_bytes(cfg, shape),
                y_recv=recv, dx_recv=recv)
