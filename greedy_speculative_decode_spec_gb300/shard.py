"""Merging per-shard LM-head argmaxes when the vocabulary is split across ranks.

Each rank runs `spec_lmhead_argmax` on its slice W[v0:v1] of the weight and obtains, per
row, the slice's maximum logit and the lowest slice index attaining it. Offsetting the
index by v0 and keeping, per row, the largest maximum with the lowest global index among
equal maxima gives the unsharded result (lowest index wins ties: span-02
`engine/crates/model/src/spec.rs`, `greedy_logprob`). One all-gather of these pairs
(8 bytes per row per rank) is the whole exchange.
"""
from __future__ import annotations

import numpy as np


def shard_bounds(V: int, world: int, rank: int) -> tuple[int, int]:
    """The contiguous vocabulary slice [v0, v1) of `rank` (sizes differ by at most one)."""
    base, extra = divmod(V, world)
    v0 = rank * base + min(rank, extra)
    return v0, v0 + base + (1 if rank < extra else 0)


def merge_shard_argmax(max_logit: np.ndarray, global_ids: np.ndarray) -> np.ndarray:
    """max_logit, global_ids: [world][M] (fp32 maxima, global ids, -1 for a failed row).
    Returns the merged ids [M]."""
    max_logit = np.asarray(max_logit, dtype=np.float32)
    global_ids = np.asarray(global_ids, dtype=np.int64)
    world, M = max_logit.shape
    out = np.full(M, -1, dtype=np.int64)
    for m in range(M):
        best = None
        for r in range(world):
            i = int(global_ids[r, m])
            if i < 0:
                best = None
                break
            key = (float(max_logit[r, m]), -i)
            if best is None or key > best:
                best = key
        if best is not None:
            out[m] = -best[1]
    return out
