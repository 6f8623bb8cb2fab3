"""The benchmark's multi-rank partitions, host logic on two gloo ranks (no
GPU): what bench.rank_work gives each rank and, for FSDP groups with
halos, the per-step exchange into fixed buffers that the timed loop
repeats. The CPU oracle stands in for the device.

- sources: one model shared by the ranks; each prepares the outputs that
  schedule.assign_sources gives it; the union covers every output exactly
  once and matches the single-process bytes.
- shard-local with halos: each rank receives its halo rows three times in
  a row into the same buffers (so a plan's pointer tables never change
  between steps), the buffers always hold the right rows, and the oracle
  run on what each rank holds reproduces the full output's blocks.
"""
import hashlib
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from shard_helpers import assembled_oracle_blocks, full_oracle_blocks
from workloads import halo_mix, make_shards, shards_to_host_u16, tiny_dense


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _digest(data, scales):
    h = hashlib.sha256(data.tobytes())
    if scales is not None:
        h.update(scales.tobytes())
    return h.hexdigest()


def _run(target, world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=target, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = q.get(timeout=300)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    return got


def _sources_worker(rank, world, port, q):
    import bench
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, kw, note = bench.rank_work("tiny_dense", "sources", world, rank)
    assert kw == {} and f"source {rank} of {world}" in note
    m = oracle.Model(w)
    host = shards_to_host_u16(make_shards(w))
    local = {out.name: _digest(*m.prepare_output(i, host)) for i, out in enumerate(w.outputs)}
    gathered = [None] * world
    dist.all_gather_object(gathered, local)
    if rank == 0:
        q.put(gathered)
    dist.barrier()
    dist.destroy_process_group()


def test_sources_partition_covers_the_model_once(oracle_mod):
    gathered = _run(_sources_worker, 2)
    w = tiny_dense()
    seen = {}
    for part in gathered:
        assert part, "a source with nothing to prepare"
        for name, h in part.items():
            assert name not in seen
            seen[name] = h
    m = oracle_mod.Model(w)
    host = shards_to_host_u16(make_shards(w))
    assert seen == {out.name: _digest(*m.prepare_output(i, host)) for i, out in enumerate(w.outputs)}


def _halo_worker(rank, world, port, q):
    import bench
    import oracle
    from bf16_fp8_parameter_wt_b300.schedule import exchange_halos, halo_buffers, halo_transfers
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, kw, note = bench.rank_work(halo_mix(world), "shard-local", world, rank, halo=True)
    assert kw == {"local_shard": rank, "halo": True}
    full = make_shards(w)
    own = [per[rank] for per in full]
    transfers = halo_transfers(w, world)
    bufs = halo_buffers(w, transfers, rank, "cpu")
    addrs = {k: b.data_ptr() for k, b in bufs.items()}
    for step in range(3):
        for b in bufs.values():
            b.fill_(float("nan"))
        got = exchange_halos(w, transfers, rank, own, out=bufs)
        assert {k: t.data_ptr() for k, t in got.items()} == addrs
        for (p, k), t in got.items():
            assert torch.equal(t.view(torch.int16), full[p][k][:t.shape[0]].view(torch.int16)), step

    def rows_of(p, k, a, b):
        t = own[p][a:b] if k == rank else bufs[(p, k)][a:b]
        assert k == rank or b <= bufs[(p, k)].shape[0]
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    local = assembled_oracle_blocks(oracle, w, rank, rows_of)
    msg = {k: _digest(*v) for k, v in local.items()}
    gathered = [None] * world
    dist.all_gather_object(gathered, msg)
    if rank == 0:
        q.put(gathered)
    dist.barrier()
    dist.destroy_process_group()


def test_halo_exchange_each_step_into_fixed_buffers(oracle_mod):
    gathered = _run(_halo_worker, 2)
    w = halo_mix(2)
    full = full_oracle_blocks(oracle_mod, w, shards_to_host_u16(make_shards(w)))
    seen = {}
    for g in gathered:
        for k, h in g.items():
            assert k not in seen
            seen[k] = h
    assert seen == {k: _digest(*v) for k, v in full.items()}
