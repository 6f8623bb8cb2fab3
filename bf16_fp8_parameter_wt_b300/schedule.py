"""Source assignment across training GPUs.

On the page "Weight transfer for RL post-training in under 2 seconds"
(section "High-level workflow") the controller's static schedule maps each
parameter to the training GPU that sends it; with FSDP every GPU of a
DeviceMesh can rebuild any full parameter (section "DeviceMesh and mesh
groups"), so any of them can be the source. Outputs are independent, so
the preparation stage partitions over source GPUs with no exchange on the
data path beyond the full_tensor() gather itself.

assign_sources() is that choice: a deterministic greedy balance of the
outputs' bytes (read + written) over `world` sources, largest first, ties
to the lower rank. rank_view() is the sub-workload one source prepares.
"""
from __future__ import annotations

import heapq
from typing import List


def output_bytes(w, o: int) -> int:
    out = w.outputs[o]
    m, n = w.output_shape(o)
    written = (m * n + 4 * (-(-m // 128)) * (-(-n // 128))) if out.fp8 else 2 * m * n
    return 2 * m * n + written * len(out.dst_ranks)


def assign_sources(w, world: int) -> List[int]:
    """Source rank of every output."""
    if world < 1:
        raise ValueError("world must be >= 1")
    order = sorted(range(len(w.outputs)), key=lambda o: (-output_bytes(w, o), o))
    heap = [(0, r) for r in range(world)]
    src = [0] * len(w.outputs)
    for o in order:
        load, r = heapq.heappop(heap)
        src[o] = r
        heapq.heappush(heap, (load + output_bytes(w, o), r))
    return src


def rank_view(w, world: int, rank: int):
    """The outputs (in plan order) that `rank` prepares, as a workload."""
    src = assign_sources(w, world)
    mine = [o for o in range(len(w.outputs)) if src[o] == rank]
    return w.subset(mine, name=f"{w.name}[source {rank}/{world}]"), mine
