"""Seeded random workload structures for the randomized parity tests.

Each case draws a handful of outputs with random fusion groups, shapes
(ragged in both dimensions, 16-byte rows or not), FSDP shard splits (empty
shards included), formats, destination ranks and tensor-parallel slices.
Shapes and bookkeeping only; no arithmetic of the stage.
"""
from __future__ import annotations

import random

from .configs import TILE, Output, Param, ValueRecipe, Workload


def _split(rng: random.Random, rows: int, shards: int) -> tuple:
    """A random dim-0 split of rows into `shards` parts (zeros allowed)."""
    cuts = sorted(rng.randint(0, rows) for _ in range(shards - 1))
    edges = [0] + cuts + [rows]
    return tuple(edges[i + 1] - edges[i] for i in range(shards))


def _slice(rng: random.Random, extent: int, dim: int):
    """Random 128-aligned ranges of [0, extent): a random non-empty set of
    blocks, as runs of consecutive blocks in random order, the run holding
    a ragged last block placed last."""
    nb = -(-extent // TILE)
    blocks = sorted(rng.sample(range(nb), rng.randint(1, nb)))
    runs, cur = [], [blocks[0]]
    for b in blocks[1:]:
        if b == cur[-1] + 1 and rng.random() < 0.7:
            cur.append(b)
        else:
            runs.append(cur)
            cur = [b]
    runs.append(cur)
    rng.shuffle(runs)
    if extent % TILE:
        tail = [r for r in runs if r[-1] == nb - 1]
        runs = [r for r in runs if r[-1] != nb - 1] + tail
    ranges = tuple((r[0] * TILE, min(extent, (r[-1] + 1) * TILE) - r[0] * TILE) for r in runs)
    return (dim, ranges)


def random_workload(seed: int, max_outputs: int = 5) -> Workload:
    rng = random.Random(seed)
    ranks = rng.randint(1, 4)
    shards = rng.randint(1, 5)
    params, outputs = [], []
    for o in range(rng.randint(1, max_outputs)):
        cols = rng.choice([1, 2, 8, 24, 128, 136, 200, 256, 260, 384, 520, 1000])
        parts = []
        for k in range(rng.choice([1, 1, 2, 3])):
            rows = rng.choice([1, 7, 64, 100, 128, 129, 255, 256, 300, 384, 511])
            params.append(Param(f"o{o}p{k}", rows, cols, _split(rng, rows, shards)))
            parts.append(len(params) - 1)
        m = sum(params[p].rows for p in parts)
        fp8 = rng.random() < 0.7
        ndst = rng.randint(1, 3)
        dst = tuple(rng.randrange(ranks) for _ in range(ndst))
        slices = None
        if rng.random() < 0.4:
            slices = tuple(None if rng.random() < 0.3 else
                           _slice(rng, m if dim == 0 else cols, dim)
                           for dim in [rng.randint(0, 1) for _ in range(ndst)])
        outputs.append(Output(f"o{o}", tuple(parts), fp8, dst, slices=slices))
    vals = ValueRecipe("student_t3", 0.02, 5000 + seed, zero_tile_eighths=1,
                       outlier_tile_eighths=1, outlier=3.0e4)
    return Workload(f"random_{seed}", params, outputs, ranks, vals)
