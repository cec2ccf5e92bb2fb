"""Query-row sharding of the selection across a process group.

"NVIDIA/Megatron-LM pull request #8299", section "Change", and "NovaSky-AI/SkyRL
pull request #2422", Summary: query rows are independent (a row's selection
depends on its own query and the shared pooled keys only), so each of G ranks
selects a contiguous range of rows and one all-gather of the int32 pool ids
rebuilds the [T, budget] tensor on every rank; pool expansion, tail append and
mask filtering then run on the gathered ids. This module holds the host side of
that path: the split, the gather and the reassembly. Every selection step still
runs in the CUDA library (kpool_select_ex with a row range, then kpool_expand).

Two things differ from the pages. The split balances causal work rather than
row counts (kpool_balanced_row_split): under the causal mask an even split of
rows gives the last rank about 2G - 1 times the first rank's pairs. And since
the ranges then differ in length, the gather pads every shard to the longest
one and the reassembly drops the padding.

The collective is torch.distributed's all_gather (NCCL between GPUs, gloo on
CPUs); nothing here uses multicast memory.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import kpool as K


def row_bounds(cu_seqlens, kpool: int, world: int, row_weight: int = 0) -> list:
    """Bounds [0, b1, ..., T] of `world` contiguous row ranges of near-equal work (host list)."""
    return K.kpool_balanced_row_split(cu_seqlens, kpool, world, row_weight)


def gather_pool_ids(local_ids: torch.Tensor, bounds: list, group=None) -> torch.Tensor:
    """All-gather each rank's pool ids [b[r+1] - b[r], budget] (int32) into [T, budget] on every
    rank. Shards are padded with -1 to the longest range for the collective, then trimmed."""
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    if len(bounds) != world + 1:
        raise ValueError(f"{world} ranks need {world + 1} bounds, got {len(bounds)}")
    sizes = [bounds[r + 1] - bounds[r] for r in range(world)]
    if local_ids.dim() != 2 or local_ids.shape[0] != sizes[rank] or local_ids.dtype != torch.int32:
        raise ValueError(f"rank {rank} must hold [{sizes[rank]}, budget] int32 pool ids, "
                         f"got {tuple(local_ids.shape)} {local_ids.dtype}")
    budget = local_ids.shape[1]
    r_max = max(sizes)
    padded = torch.full((r_max, budget), -1, dtype=torch.int32, device=local_ids.device)
    padded[: sizes[rank]] = local_ids
    parts = [torch.empty_like(padded) for _ in range(world)]
    dist.all_gather(parts, padded, group=group)
    return torch.cat([parts[r][: sizes[r]] for r in range(world)], dim=0)


def sharded_select(q, k, w, cu_seqlens, kpool: int, index_topk: int, scale: float, group=None,
                   row_weight: int = 0, workspace=None, stream=None):
    """The whole selection with the query rows split over the ranks of `group`.

    Every rank holds the whole batch's q, k, w and cu_seqlens (the indexer is replicated, as in
    the pages' shard plan); each selects its range of rows with kpool_select_ex, the pool ids are
    all-gathered, and every rank expands the gathered ids. Returns (pool_ids [T, budget],
    token_ids [T, index_topk + kpool]), equal to the unsharded kpool_select's bit for bit."""
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    bounds = row_bounds(cu_seqlens.cpu(), kpool, world, row_weight)
    lo, hi = bounds[rank], bounds[rank + 1]
    local_ids, _, _ = K.kpool_select_ex(q, k, w, cu_seqlens, kpool, index_topk, scale, workspace=workspace,
                                        stream=stream, row_range=(lo, hi))
    pool_ids = gather_pool_ids(local_ids, bounds, group)
    token_ids = K.kpool_expand(pool_ids, cu_seqlens, kpool, index_topk, stream=stream)
    return pool_ids, token_ids
