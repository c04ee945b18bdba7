"""Splitting one block-sparse attention workload across GPUs.

Every (batch entry, head) pair of block-sparse attention is independent: a
block-row's softmax and output touch that pair's rows only ("question on
blocksparse", openai/triton issue 117: the softmax reduces each row across
the row's own blocks).  One workload [Z, H, S, D] on a layout [H, nb, nb]
is therefore cut into contiguous ranges of the flattened pair index
u = z * H + h, each range balanced by the number of present blocks (the work
of a pair), with no exchange between the ranges.

A rank runs its range [u0, u1) as one call with batch 1 and u1 - u0 "heads":
the dense tensors viewed as [1, Z*H, S, D] and sliced to [1, u1-u0, S, D],
and the layout of those pairs' heads stacked into [u1-u0, nb, nb]
(`shard_layout`).
"""

from __future__ import annotations

import numpy as np


def pair_weights(layout: np.ndarray, Z: int) -> np.ndarray:
    """Present blocks of every pair u = z * H + h (length Z * H)."""
    per_head = np.asarray(layout).reshape(layout.shape[0], -1).sum(axis=1).astype(np.int64)
    return np.tile(per_head, Z)


def balanced_ranges(weights: np.ndarray, world: int) -> list[tuple[int, int]]:
    """Cut 0..n-1 into `world` contiguous ranges [u0, u1) whose weight sums are
    balanced: boundary r is the first index whose prefix sum reaches
    r / world of the total.  Every index lies in exactly one range, and no
    range exceeds total / world by more than the heaviest single weight."""
    w = np.asarray(weights, dtype=np.int64)
    n = w.size
    if world < 1:
        raise ValueError("world must be >= 1")
    prefix = np.concatenate([[0], np.cumsum(w)])
    total = int(prefix[-1])
    bounds = [0]
    for r in range(1, world):
        target = total * r / world
        # first k with prefix[k] >= target, never before the previous boundary
        k = int(np.searchsorted(prefix, target, side="left"))
        bounds.append(min(max(k, bounds[-1]), n))
    bounds.append(n)
    return [(bounds[r], bounds[r + 1]) for r in range(world)]


def shard_layout(layout: np.ndarray, Z: int, rank: int, world: int):
    """(u0, u1, sub_layout) of this rank: its pairs [u0, u1) and the layout of
    their heads stacked in pair order ([u1 - u0, nb, nb], possibly empty)."""
    lay = np.asarray(layout)
    H = lay.shape[0]
    u0, u1 = balanced_ranges(pair_weights(lay, Z), world)[rank]
    heads = np.arange(u0, u1) % H
    return u0, u1, np.ascontiguousarray(lay[heads])


# ------------------------------------------------------ DSD / DDS shards ----
#
# DSD (C = A_sp B, output rows follow A_sp's block-rows) shards over
# block-rows, DDS (C = A B_sp, output columns follow B_sp's block-columns)
# over block-columns; each rank produces disjoint output rows / columns, so
# the pieces are the result with no reduction.  A rank's problem is a layout
# of the same shape with every block outside its lines removed, and the
# sparse operand restricted to the blocks that remain (block order is
# row-major (h, i, j), so the remaining blocks keep their relative order).

def line_weights(layout: np.ndarray, orient: int) -> np.ndarray:
    """Present blocks of every line, flattened over heads: block-rows
    (orient 0, index h * nb + i) or block-columns (orient 1, h * nb + j)."""
    lay = np.asarray(layout)
    counts = lay.sum(axis=2 if orient == 0 else 1)  # [H, nb]
    return counts.reshape(-1).astype(np.int64)


def shard_lines(layout: np.ndarray, orient: int, rank: int, world: int):
    """(l0, l1, sub_layout, block_ids) of this rank: its lines [l0, l1) in the
    flattened (h, line) order, the layout with every other line's blocks
    removed, and the ids (row-major (h, i, j) ranks in the full layout) of
    the blocks it keeps, ascending -- the rows of the sparse operand it
    takes, in the sub-layout's own block order."""
    lay = np.asarray(layout)
    H, nb = lay.shape[0], lay.shape[1]
    l0, l1 = balanced_ranges(line_weights(lay, orient), world)[rank]
    keep = np.zeros((H, nb), dtype=bool)
    keep.reshape(-1)[l0:l1] = True
    sub = lay.copy()
    if orient == 0:
        sub[~keep] = 0                                   # rows outside [l0, l1)
    else:
        sub = np.where(keep[:, None, :], sub, 0).astype(lay.dtype)  # columns outside
    ids = np.flatnonzero(sub[lay.astype(bool)])          # the kept blocks' full-layout ids, ascending
    return l0, l1, np.ascontiguousarray(sub), ids
