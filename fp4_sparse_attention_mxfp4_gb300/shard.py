"""Host side of key-sharded decode ("Score a DSA sparse indexer in FP4", section "Decode context
parallelism": each rank scores its own shard of a sequence's keys, keeps its local top-k, and the
ranks' candidates are gathered and merged into the row's top-k).

A shard is a contiguous key range of every sequence, starting on a 128-key tile (the decode
scorer's unit of keys). Shard w of W takes the tiles [tiles * w / W, tiles * (w + 1) / W) of a
sequence, so the shards partition its keys in order. On one GPU the shards are scored by
separate decode calls over range schedules; across ranks each rank scores its own shard and
``gather_candidates`` all-gathers the lists before ``idx_fp4_merge_candidates``. Everything here
is bookkeeping: the scoring and the merge run in the library's kernels.
"""
from __future__ import annotations

import numpy as np

TILE = 128  # keys per scorer tile: a shard's first key is a multiple of it


def shard_ranges(ctx_lens, world: int, tile: int = TILE):
    """Key ranges of each shard: a list of `world` pairs (key_begin, key_end) of int32 arrays [B]."""
    if world < 1:
        raise ValueError("world must be >= 1")
    ctx = np.asarray(ctx_lens, dtype=np.int64)
    if np.any(ctx < 0):
        raise ValueError("context lengths must be >= 0")
    tiles = -(-ctx // tile)
    out = []
    for w in range(world):
        begin = np.minimum(tiles * w // world * tile, ctx)
        end = np.minimum(tiles * (w + 1) // world * tile, ctx)
        out.append((begin.astype(np.int32), end.astype(np.int32)))
    return out


def gather_candidates(topk_idx, topk_val, group=None):
    """All-gather every rank's [rows, k] candidate lists over torch.distributed: returns
    (idx [world, rows, k], val [world, rows, k]) stacked in rank order."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    idx = [torch.empty_like(topk_idx) for _ in range(world)]
    val = [torch.empty_like(topk_val) for _ in range(world)]
    dist.all_gather(idx, topk_idx.contiguous(), group=group)
    dist.all_gather(val, topk_val.contiguous(), group=group)
    return torch.stack(idx), torch.stack(val)
