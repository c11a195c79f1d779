"""Record-range split of one CSA2 decode layer across devices (one process per device).

A long context's records can be cut into contiguous ranges, one per rank: a record's indexer
score needs only that record's key, and the row's top-K is a subset of the union of every
range's own top-K.  Rank k holds records [first_k, first_k + count_k) of every sequence (their
indexer keys and latents); the queries, head weights, window rows and sinks are on every rank
and one rank (the window owner) attends to the window.  A rank's steps:

  1. the scores of its range (csa2_index_scores over the range's keys, visibility clipped to
     the range),
  2. the range's exact top-K candidates (csa2_shard_candidates),
  3. all-gather of every range's candidates, and their merge into the row's top-K
     (csa2_merge_candidates: the same indices on every rank, bit for bit),
  4. attention partials over the selected records of its range, and the window on the owner
     (csa2_sparse_attn_partial),
  5. all-gather of the partials and their merge: sink, normalisation, inverse RoPE
     (csa2_attn_merge).

The collective is `torch.distributed.all_gather` (any backend); the compute steps are the
library's calls (`LibrarySteps`).  `split_full_layer` runs one rank's steps;
`emulate_split` runs every range on one device in turn, with concatenation in place of the
gathers.  Nothing here computes: the steps are calls, the rest is arranging their arguments.
"""
from __future__ import annotations

import torch

from . import (attn_merge, index_scores, merge_candidates, shard_candidates, sparse_attn_partial)


def record_ranges(n_records: int, n_parts: int) -> list[tuple[int, int]]:
    """Contiguous, balanced ranges [(first, count)] covering records 0 .. n_records - 1."""
    if n_parts < 1 or n_records < n_parts:
        raise ValueError("need at least one record per range")
    base, extra = divmod(n_records, n_parts)
    out, first = [], 0
    for k in range(n_parts):
        count = base + (1 if k < extra else 0)
        out.append((first, count))
        first += count
    return out


class LibrarySteps:
    """The compute steps as library calls (the CUDA path)."""

    def scores(self, local, n_visible):
        return index_scores(local["q_idx"], local["w"], local["k_idx"], local["k_scale"], local["seq_of_row"],
                            n_visible)

    def candidates(self, scores, n_visible, K, first):
        return shard_candidates(scores, n_visible, K, first)

    def merge(self, scores, pos, cnt, K):
        return merge_candidates(scores, pos, cnt, K)

    def partial(self, local, idx, first, count, skip_window):
        return sparse_attn_partial(local["q"], local["q_pos"], local["seq_of_row"], local["lat"], local["lat_scale"],
                                   idx, local["swa"], local["swa_scale"], local["swa_pos0"], local["window"],
                                   local["theta"], local["softmax_scale"], range_first=first, range_count=count,
                                   skip_window=skip_window)

    def attn_merge(self, part_o, part_ml, local):
        return attn_merge(part_o, part_ml, local["q_pos"], local["sink"], local["theta"])


def all_gather_stack(t: torch.Tensor, group=None) -> torch.Tensor:
    """Every rank's `t`, stacked along a new leading dimension in rank order."""
    import torch.distributed as dist
    parts = [torch.empty_like(t) for _ in range(dist.get_world_size(group))]
    dist.all_gather(parts, t.contiguous(), group=group)
    return torch.stack(parts)


def clipped_visibility(n_visible: torch.Tensor, first: int, count: int) -> torch.Tensor:
    """Visible records of each row inside [first, first + count), as the range's own count."""
    return (n_visible.to(torch.int64) - first).clamp(0, count).to(torch.int32)


def split_full_layer(local: dict, first: int, count: int, K: int, rank: int, world: int, steps=None,
                     gather=all_gather_stack, window_owner: int | None = None):
    """One rank's share of a FULL layer over a record-range split: returns the row's top-K
    indices (global positions, identical on every rank), the attention output and the sink
    mass (identical on every rank).

    `local` holds this rank's range of records ("k_idx", "k_scale", "lat", "lat_scale" with
    `count` records per sequence) and the full query-side inputs ("q_idx", "w", "q", "q_pos",
    "seq_of_row", "n_visible", "swa", "swa_scale", "swa_pos0", "window", "sink", "theta",
    "softmax_scale")."""
    steps = LibrarySteps() if steps is None else steps
    owner = world - 1 if window_owner is None else window_owner
    n_vis = clipped_visibility(local["n_visible"], first, count)
    sc = steps.scores(local, n_vis)
    cs, cp, cc = steps.candidates(sc, n_vis, K, first)
    idx = steps.merge(gather(cs), gather(cp), gather(cc), K)
    part_o, part_ml = steps.partial(local, idx, first, count, rank != owner)
    out, sink_mass = steps.attn_merge(gather(part_o), gather(part_ml), local)
    return idx, out, sink_mass


def emulate_split(shards: list[dict], ranges: list[tuple[int, int]], K: int, steps=None,
                  window_owner: int | None = None):
    """Every range of the split on one device in turn (the gathers become concatenations):
    `shards[k]` is range k's `local` dict.  Same results as `split_full_layer` on each rank."""
    steps = LibrarySteps() if steps is None else steps
    world = len(ranges)
    owner = world - 1 if window_owner is None else window_owner
    cands = []
    for local, (first, count) in zip(shards, ranges):
        n_vis = clipped_visibility(local["n_visible"], first, count)
        cands.append(steps.candidates(steps.scores(local, n_vis), n_vis, K, first))
    idx = steps.merge(torch.stack([c[0] for c in cands]), torch.stack([c[1] for c in cands]),
                      torch.stack([c[2] for c in cands]), K)
    parts = [steps.partial(local, idx, first, count, k != owner)
             for k, (local, (first, count)) in enumerate(zip(shards, ranges))]
    out, sink_mass = steps.attn_merge(torch.stack([p[0] for p in parts]), torch.stack([p[1] for p in parts]), shards[0])
    return idx, out, sink_mass
