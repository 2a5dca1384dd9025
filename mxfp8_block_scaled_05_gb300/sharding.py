"""Host-side work splitting for running the quantizer on several ranks.

The weight-synchronization pass ("End-to-End MXFP8 RL on Blackwell", section "The
grid, byte for byte": the synced weights must equal the learner's forward weights byte
for byte, including under tensor-parallel sharding) is embarrassingly parallel: every
32-block is independent. Two splits keep the bytes identical to the unsharded
quantization:
  * whole weights assigned to ranks (no exchange at all);
  * row shards of one weight whose boundaries are multiples of 128, so that each shard's
    swizzled scale tiles are exactly a contiguous slice of the whole weight's tiles.
No data-path collective is involved; ranks only agree on the plan.
"""
from __future__ import annotations


def row_shards(rows: int, world: int, align: int = 128):
    """[start, end) row ranges, one per rank, boundaries at multiples of `align`, as even
    as that allows; trailing ranks may get empty ranges."""
    if rows < 0 or world <= 0 or align <= 0:
        raise ValueError("rows >= 0, world > 0, align > 0 required")
    tiles = (rows + align - 1) // align
    per, extra = divmod(tiles, world)
    out, t = [], 0
    for r in range(world):
        n = per + (1 if r < extra else 0)
        lo, hi = min(t * align, rows), min((t + n) * align, rows)
        out.append((lo, hi))
        t += n
    return out


def assign_weights(sizes, world: int):
    """Longest-processing-time-first assignment of whole weights (by element count) to
    ranks. Returns one list of weight indices per rank, each in ascending order."""
    if world <= 0:
        raise ValueError("world > 0 required")
    loads = [0] * world
    parts = [[] for _ in range(world)]
    for i in sorted(range(len(sizes)), key=lambda j: (-sizes[j], j)):
        r = min(range(world), key=lambda q: (loads[q], q))
        parts[r].append(i)
        loads[r] += sizes[i]
    return [sorted(p) for p in parts]
