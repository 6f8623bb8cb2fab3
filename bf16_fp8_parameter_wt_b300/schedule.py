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

The other partition keeps FSDP's own placement: rank r of a group holds
shard r of every parameter and prepares, with a shard-local plan, the
128-row block rows that start in its shard. Where a shard boundary is off
the 128-row grid, the block row that spans it also needs the leading rows
of the next shard(s) -- at most 127 rows per boundary instead of the
whole parameter that full_tensor() gathers. halo_transfers() lists those
row runs for the whole group (from the plans' own wt_plan_shard_rows_read
answers) and exchange_halos() moves them with point-to-point sends over a
torch.distributed group.
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


def halo_transfers(w, fsdp: int) -> List[tuple]:
    """(src rank, dst rank, param, shard, rows) for every halo the
    shard-local plans of an FSDP group of `fsdp` ranks read: rank dst needs
    the first `rows` rows of shard `shard` of param `param`, held by rank
    src == shard. Host-only plans; the same list on every rank."""
    from . import wt
    out = []
    for r in range(fsdp):
        with wt.Plan(w, device=-1, local_shard=r, halo=True) as p:
            for i, par in enumerate(w.params):
                for k in range(len(par.shard_rows)):
                    if k == r:
                        continue
                    n = p.shard_rows_read(i, k)
                    if n:
                        if k >= fsdp:
                            raise ValueError(f"{par.name}: shard {k} has no rank in a group of {fsdp}")
                        out.append((k, r, i, k, n))
    return out


def halo_buffers(w, transfers, rank: int, device) -> dict:
    """Receive buffers for this rank's halos, {(param, shard): [rows, cols]
    BF16 tensor}: allocated once, so that every step's exchange lands at the
    same addresses (a plan then reuses its pointer tables)."""
    import torch
    return {(p, k): torch.empty((n, w.params[p].cols), dtype=torch.bfloat16, device=device)
            for src, dst, p, k, n in transfers if dst == rank and src != rank}


def exchange_halos(w, transfers, rank: int, own_shards, group=None, out=None) -> dict:
    """Send the leading rows of this rank's shards that other ranks need and
    receive this rank's halos. own_shards[p] is this rank's shard of param p
    (a [shard_rows, cols] BF16 tensor on the group's device). Returns
    {(param, shard): [rows, cols] tensor} of the received halo rows, written
    into `out` (from halo_buffers) when given, else into new tensors."""
    import torch
    import torch.distributed as dist
    ops, got = [], {}
    dev = next((t.device for t in own_shards if t is not None), torch.device("cpu"))
    # raw 16-bit payloads (no reduction happens, so the dtype is only a
    # size); every rank walks the same list in the same order, so sends
    # and receives pair up, and one tag per transfer where the backend
    # uses tags; posted as one batch (a group of point-to-point calls for
    # NCCL, where separately posted sends and receives can wait on each
    # other)
    for tag, (src, dst, p, k, n) in enumerate(transfers):
        if src == rank and dst != rank:
            t = own_shards[p][:n].contiguous().view(torch.int16)
            ops.append(dist.P2POp(dist.isend, t, dst, group=group, tag=tag))
        elif dst == rank and src != rank:
            if out is not None:
                got[(p, k)] = out[(p, k)]
                buf = out[(p, k)].view(torch.int16)
            else:
                buf = torch.empty((n, w.params[p].cols), dtype=torch.int16, device=dev)
                got[(p, k)] = buf.view(torch.bfloat16)
            ops.append(dist.P2POp(dist.irecv, buf, src, group=group, tag=tag))
    if ops:
        for q in dist.batch_isend_irecv(ops):
            q.wait()
    return got
