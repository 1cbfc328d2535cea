"""Sequence sharding of one packed verify batch over ranks (host logic only).

The verify step is independent per sequence: sequence b reads only its own
target rows, draft rows and uniforms (positions k_offsets[b] + b .. of the
target-row arrays, k_offsets[b] .. of the draft-row arrays).  A batch
therefore splits over ranks into contiguous sequence ranges with no data
exchange; each rank calls spec_verify on its slice with rebased offsets and
the outputs concatenate back in rank order.

Ranges are balanced by logit rows (target + draft), which is what the
streaming pass costs, not by sequence count.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Shard:
    """Sequences [b0, b1) of the batch, and the row ranges they own."""
    b0: int
    b1: int
    draft_rows: tuple[int, int]   # rows of draft_logits / draft_tokens / u_accept
    target_rows: tuple[int, int]  # rows of target_logits / u_resample / out_tokens
    k_offsets: np.ndarray         # rebased prefix sums, int32 [b1 - b0 + 1]

    @property
    def B(self) -> int:
        return self.b1 - self.b0


def shard_ranges(k_offsets, world: int) -> list[tuple[int, int]]:
    """Split sequences into `world` contiguous ranges with about equal logit
    rows each (sequence b costs 2 k_b + 1 rows).  Ranges may be empty when
    world > B."""
    ko = np.asarray(k_offsets, dtype=np.int64)
    B = ko.size - 1
    if B < 0 or world < 1:
        raise ValueError("k_offsets must have B + 1 entries and world >= 1")
    # rows before sequence b: draft rows ko[b] plus target rows ko[b] + b
    cum = 2 * ko + np.arange(B + 1)
    total = cum[-1]
    cuts = [0]
    for r in range(1, world):
        goal = total * r / world
        b = int(np.searchsorted(cum, goal, side="left"))
        b = min(max(b, cuts[-1]), B)
        cuts.append(b)
    cuts.append(B)
    return [(cuts[r], cuts[r + 1]) for r in range(world)]


def make_shard(k_offsets, b0: int, b1: int) -> Shard:
    ko = np.asarray(k_offsets, dtype=np.int64)
    if not (0 <= b0 <= b1 <= ko.size - 1):
        raise ValueError(f"bad sequence range [{b0}, {b1})")
    d = (int(ko[b0]), int(ko[b1]))
    t = (int(ko[b0]) + b0, int(ko[b1]) + b1)
    return Shard(b0, b1, d, t, (ko[b0:b1 + 1] - ko[b0]).astype(np.int32))


def shard_for_rank(k_offsets, world: int, rank: int) -> Shard:
    b0, b1 = shard_ranges(k_offsets, world)[rank]
    return make_shard(k_offsets, b0, b1)
