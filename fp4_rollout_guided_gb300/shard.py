"""Host-side work division across ranks (one process per GPU).

The hot path has no exchange step: every NVFP4 block depends only on its own
values and its segment's global scale.  Two plans are offered:

* ``weak``: each rank runs its own full copy of the workload (its own
  rollout stream, seeded by rank); units = all ranks' elements.
* ``strong``: the training segments of one workload are split into
  contiguous whole-segment ranges, balanced by element count, so that no
  segment (and no global scale) is split and no collective is needed.
"""
from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass(frozen=True)
class Shard:
    rank: int
    world: int
    seed: int
    seg_lo: int   # first training segment of this rank (strong plan)
    seg_hi: int   # one past the last


def weak_plan(world: int, rank: int, base_seed: int = 0) -> Shard:
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    return Shard(rank, world, base_seed + rank, 0, -1)


def strong_plan(seg_rows: np.ndarray, world: int, rank: int) -> Shard:
    """Contiguous whole-segment ranges with near-equal row counts."""
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    seg_rows = np.asarray(seg_rows, dtype=np.int64)
    n = len(seg_rows) - 1
    total = int(seg_rows[-1])
    # cut at the segment boundary nearest each rank's ideal start row
    cuts = [0]
    for k in range(1, world):
        ideal = total * k / world
        j = int(np.argmin(np.abs(seg_rows - ideal)))
        cuts.append(max(cuts[-1], min(j, n)))
    cuts.append(n)
    return Shard(rank, world, 0, cuts[rank], cuts[rank + 1])
