"""Shard-local plans on the host (no GPU).

With FSDP dim-0 shards whose boundaries fall on multiples of 128 rows of
their output, every 128x128 block draws its rows from one shard, so the
rank holding shard s can quantize those blocks with no exchange (the
page "Weight transfer for RL post-training in under 2 seconds", section
"DeviceMesh and mesh groups": each rank holds one dim-0 shard; the
full_tensor() gather is what the shortcut avoids).

- The oracle fixes the arithmetic claim: quantizing only the rows of
  shard s, fused in part order, gives exactly the block rows of the full
  output that come from shard s (block scales never mix shards).
- The plan compiler partitions the work: the S local plans' units,
  bytes, element counts and per-rank expected blocks add up to the full
  plan's, the layout is the full plan's, and the counts match an
  ownership count made here from the workload.
- Two or four gloo ranks each compile their own local plan and run the oracle on
  their own shards only; rank 0 checks the union against the full oracle.
- Misaligned shards, offload and bad arguments are refused.
- With halos (WT_FLAG_SHARD_HALO) boundaries may be off the grid: a block
  row belongs to the shard holding its first row, and the plan reports,
  per shard, the leading rows it reads; those match a count made here,
  the local plans still partition the full plan, and two or four gloo ranks that
  exchange exactly those rows (schedule.exchange_halos) and run the
  oracle on what they hold reproduce the full oracle output.
"""
import ctypes
import hashlib
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bf16_fp8_parameter_wt_b300 as wt
from bf16_fp8_parameter_wt_b300.schedule import exchange_halos, halo_transfers
from shard_helpers import (_cdiv, assembled_oracle_blocks, full_oracle_blocks, halo_rows_needed,
                           local_counts, owned_block_rows, same_blocks)
from workloads import (TILE, Output, Param, Workload, halo_mix, kimi_k2_moe_layer, llama_dense,
                       make_shards, shard_local_mix, shards_to_host_u16, tiny_dense)


def local_view(w, s):
    """The workload made of shard s alone: each param replaced by its shard
    s (one shard), empty parts and outputs dropped, same formats, ranks and
    column slices. Returns (workload, kept output indices, kept params)."""
    params, outs, kept, keep_p = [], [], [], []
    for o, out in enumerate(w.outputs):
        parts = []
        for p in out.parts:
            n = w.params[p].shard_rows[s] if s < len(w.params[p].shard_rows) else 0
            if n:
                params.append(Param(w.params[p].name + f"#s{s}", n, w.params[p].cols, (n,)))
                keep_p.append(p)
                parts.append(len(params) - 1)
        if parts:
            assert out.slices is None or all(x is None or x[0] == 1 for x in out.slices)
            outs.append(Output(out.name, tuple(parts), out.fp8, out.dst_ranks, slices=out.slices))
            kept.append(o)
    return Workload(w.name + f"[shard {s}]", params, outs, w.num_ranks, w.values), kept, keep_p


def local_oracle_blocks(oracle_mod, w, s, flat_full):
    """{(output, block row): (data rows bytes, scale row)} computed by the
    oracle from shard s's rows alone."""
    sub, kept, keep_p = local_view(w, s)
    slot_base, k = [], 0
    for p in w.params:
        slot_base.append(k)
        k += len(p.shard_rows)
    flat_local = [flat_full[slot_base[p] + s] for p in keep_p]
    m = oracle_mod.Model(sub)
    res = {}
    for i, o in enumerate(kept):
        data, scales = m.prepare_output(i, flat_local)
        rows_local, n = sub.output_shape(i)
        esz = 1 if w.outputs[o].fp8 else 2
        data = data.reshape(rows_local, n * esz)
        bn = _cdiv(n, TILE)
        lr = 0
        for bi in owned_block_rows(w, o, s):
            h = min(TILE, w.output_shape(o)[0] - bi * TILE)
            srow = scales.reshape(-1, bn)[lr // TILE].copy() if scales is not None else None
            res[(o, bi)] = (data[lr:lr + h].copy(), srow)
            lr += h
        assert lr == rows_local
    return res


@pytest.mark.parametrize("shards", [4, 2])
def test_oracle_shard_rows_alone_give_the_full_block_rows(oracle_mod, shards):
    w = shard_local_mix(shards)
    flat = shards_to_host_u16(make_shards(w))
    full = full_oracle_blocks(oracle_mod, w, flat)
    seen = set()
    for s in range(shards):
        for key, blk in local_oracle_blocks(oracle_mod, w, s, flat).items():
            assert key not in seen
            seen.add(key)
            assert same_blocks(blk, full[key]), f"shard {s}, output {key[0]}, block row {key[1]}"
    assert seen == set(full)


def test_oracle_pin_fails_when_a_block_mixes_shards(oracle_mod):
    """The pin above is not vacuous: with a boundary off the 128 grid the
    locally computed block row differs from the full one (its scale sees
    only part of the rows)."""
    w = Workload("mixed", [Param("x", 256, 128, (100, 156))],
                 [Output("x", (0,), True, (0,))], 1, shard_local_mix().values)
    flat = shards_to_host_u16(make_shards(w))
    flat[1][0] = 0x4780                        # 65536 in fused row 100: the block amax
    full = full_oracle_blocks(oracle_mod, w, flat)
    sub = Workload("x0", [Param("x#0", 100, 128, (100,))], [Output("x", (0,), True, (0,))], 1,
                   w.values)
    data, scales = oracle_mod.Model(sub).prepare_output(0, [flat[0]])
    fdata, fscale = full[(0, 0)]
    assert not (np.array_equal(data.reshape(100, 128), fdata[:100]) and
                np.array_equal(scales[:1], fscale))


def _stats(w, s=-1, halo=False):
    with wt.Plan(w, device=-1, local_shard=s, halo=halo) as p:
        st = p.stats
        exp = [p.expected_count(r) for r in range(w.num_ranks)]
        lay = [p.output_layout(o, d) for o in range(len(w.outputs))
               for d in range(len(w.outputs[o].dst_ranks))]
        pools = [p.pool_bytes(r) for r in range(w.num_ranks)]
    return st, exp, lay, pools


@pytest.mark.parametrize("make,shards", [(shard_local_mix, 4), (lambda: shard_local_mix(2), 2),
                                         (kimi_k2_moe_layer, 8),
                                         (lambda: kimi_k2_moe_layer(16, shards=2), 2)])
def test_local_plans_partition_the_full_plan(make, shards):
    w = make()
    full, full_exp, full_lay, full_pools = _stats(w)
    tot = {k: 0 for k in ("num_units", "num_params_total", "bytes_read", "bytes_written")}
    tot_exp = [0] * w.num_ranks
    for s in range(shards):
        st, exp, lay, pools = _stats(w, s)
        assert lay == full_lay and pools == full_pools     # same layout as the full plan
        assert st["num_slots"] == full["num_slots"] and st["host_bytes"] == full["host_bytes"]
        units, elems, written, per_rank = local_counts(w, s)
        assert (st["num_units"], st["num_params_total"], st["bytes_read"], st["bytes_written"]) == (
            units, elems, 2 * elems, written)
        assert exp == per_rank
        for k in tot:
            tot[k] += st[k]
        tot_exp = [a + b for a, b in zip(tot_exp, exp)]
    for k in tot:
        assert tot[k] == full[k], k
    assert tot_exp == full_exp
    assert full["bytes_read"] == w.bytes_read and full["bytes_written"] == w.bytes_written


def test_shard_index_past_the_last_shard_is_an_empty_plan():
    st, exp, _, _ = _stats(shard_local_mix(), 7)
    assert st["num_units"] == 0 and st["bytes_read"] == 0 and exp == [0, 0, 0]


@pytest.mark.parametrize("make", [tiny_dense, llama_dense])
def test_block_spanning_two_shards_is_refused(make):
    # tiny: 64-row shards of q; llama: the 128256-row vocabulary in 16032-row shards
    with pytest.raises(wt.WTError) as ei:
        wt.Plan(make(), device=-1, local_shard=0)
    assert ei.value.name == "WT_ERR_SHAPE" and "spans shards" in str(ei.value)


def test_bad_shard_local_arguments():
    w = shard_local_mix()
    with pytest.raises(wt.WTError) as ei:
        wt.Plan(w, device=-1, local_shard=0, offload_chunk_bytes=1 << 20)
    assert ei.value.name == "WT_ERR_INVALID_ARGUMENT"
    d = wt.PlanDesc(w, flags=wt.WT_FLAG_SHARD_LOCAL)
    d.c.local_shard = -2
    h = ctypes.c_void_p()
    st = wt.lib().wt_plan_create(ctypes.byref(d.c), -1, ctypes.byref(h))
    assert wt.wt_status_string(st) == "WT_ERR_INVALID_ARGUMENT"
    # without the flag local_shard is ignored: a full plan
    d = wt.PlanDesc(w)
    d.c.local_shard = -2
    h = ctypes.c_void_p()
    assert wt.lib().wt_plan_create(ctypes.byref(d.c), -1, ctypes.byref(h)) == 0
    wt.wt_plan_destroy(h.value)


# ---- gloo ranks, each with its own shard -----------------------------------

def _free_port():
    sk = socket.socket()
    sk.bind(("127.0.0.1", 0))
    port = sk.getsockname()[1]
    sk.close()
    return port


def _digest(blk):
    h = hashlib.sha256(blk[0].tobytes())
    if blk[1] is not None:
        h.update(blk[1].tobytes())
    return h.hexdigest()


def _worker(rank, world, port, q):
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = shard_local_mix(world)
    flat = shards_to_host_u16(make_shards(w))
    # this rank touches its own shard only: the other slots are dropped
    slot = 0
    mine = []
    for p in w.params:
        mine += [a if k == rank else None for k, a in enumerate(flat[slot:slot + len(p.shard_rows)])]
        slot += len(p.shard_rows)
    local = local_oracle_blocks(oracle, w, rank, mine)
    with wt.Plan(w, device=-1, local_shard=rank) as p:
        st = p.stats
        exp = [p.expected_count(r) for r in range(w.num_ranks)]
    msg = {"digests": {k: _digest(v) for k, v in local.items()}, "stats": st, "expected": exp}
    gathered = [None] * world
    dist.all_gather_object(gathered, msg)
    if rank == 0:
        q.put(gathered)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_gloo_ranks_prepare_their_own_shards(oracle_mod, world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    gathered = q.get(timeout=300)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    w = shard_local_mix(world)
    full = full_oracle_blocks(oracle_mod, w, shards_to_host_u16(make_shards(w)))
    seen = {}
    for g in gathered:
        for k, h in g["digests"].items():
            assert k not in seen
            seen[k] = h
    assert seen == {k: _digest(v) for k, v in full.items()}
    fst, fexp, _, _ = _stats(w)
    assert sum(g["stats"]["bytes_read"] for g in gathered) == fst["bytes_read"]
    assert sum(g["stats"]["num_units"] for g in gathered) == fst["num_units"]
    assert [sum(g["expected"][r] for g in gathered) for r in range(w.num_ranks)] == fexp


# ---- halos ------------------------------------------------------------------

HALO_CASES = [(halo_mix, 4), (lambda: halo_mix(2), 2), (tiny_dense, 4), (llama_dense, 8),
              (shard_local_mix, 4)]


@pytest.mark.parametrize("make,shards", HALO_CASES)
def test_halo_plans_partition_the_full_plan_and_read_only_their_halos(make, shards):
    w = make()
    full, full_exp, full_lay, full_pools = _stats(w)
    tot = {k: 0 for k in ("num_units", "num_params_total", "bytes_read", "bytes_written")}
    tot_exp = [0] * w.num_ranks
    for s in range(shards):
        st, exp, lay, pools = _stats(w, s, halo=True)
        assert lay == full_lay and pools == full_pools
        units, elems, written, per_rank = local_counts(w, s, halo=True)
        assert (st["num_units"], st["num_params_total"], st["bytes_written"]) == (units, elems, written)
        assert exp == per_rank
        need = halo_rows_needed(w, s)
        with wt.Plan(w, device=-1, local_shard=s, halo=True) as p:
            for i, par in enumerate(w.params):
                for k, n in enumerate(par.shard_rows):
                    want = n if k == s else need.get((i, k), 0)
                    assert p.shard_rows_read(i, k) == want, (par.name, k)
                    assert want < TILE or k == s
        for k in tot:
            tot[k] += st[k]
        tot_exp = [a + b for a, b in zip(tot_exp, exp)]
    for k in tot:
        assert tot[k] == full[k], k
    assert tot_exp == full_exp


def test_halo_flag_on_an_aligned_layout_equals_the_strict_plan():
    w = kimi_k2_moe_layer(4)
    for s in range(8):
        assert _stats(w, s, halo=True)[:2] == _stats(w, s)[:2]
        with wt.Plan(w, device=-1, local_shard=s, halo=True) as p:
            assert all(p.shard_rows_read(i, k) == 0 for i in range(len(w.params))
                       for k in range(8) if k != s)


def test_halo_flag_alone_is_refused():
    with pytest.raises(wt.WTError) as ei:
        wt.Plan(halo_mix(), device=-1, flags=wt.WT_FLAG_SHARD_HALO)
    assert ei.value.name == "WT_ERR_INVALID_ARGUMENT"
    with wt.Plan(halo_mix(), device=-1) as p:          # a full plan reads every row
        assert p.shard_rows_read(0, 1) == 20
        with pytest.raises(wt.WTError):
            p.shard_rows_read(0, 4)


def test_halo_transfer_list():
    w = halo_mix()
    tr = halo_transfers(w, 4)
    for src, dst, p, k, n in tr:
        assert src == k != dst and 0 < n < TILE
    for s in range(4):
        assert {(p, k): n for src, dst, p, k, n in tr if dst == s} == halo_rows_needed(w, s)
    assert halo_transfers(kimi_k2_moe_layer(2), 8) == []
    with pytest.raises(ValueError):
        halo_transfers(halo_mix(), 2)                  # shards 2 and 3 would have no rank


def _halo_worker(rank, world, port, q):
    import oracle
    import torch
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = halo_mix(world)
    full = make_shards(w)
    own = [per[rank] for per in full]            # what this FSDP rank holds
    del full
    halos = exchange_halos(w, halo_transfers(w, world), rank, own)

    def rows_of(p, k, a, b):
        if k == rank:
            t = own[p][a:b]
        else:
            assert b <= halos[(p, k)].shape[0], "read past the received halo"
            t = halos[(p, k)][a:b]
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    local = assembled_oracle_blocks(oracle, w, rank, rows_of)
    msg = {k: _digest(v) for k, v in local.items()}
    gathered = [None] * world
    dist.all_gather_object(gathered, msg)
    if rank == 0:
        q.put(gathered)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_gloo_ranks_exchange_halos_and_prepare_their_blocks(oracle_mod, world):
    # world 4: block row 0 of A starts in shard 0 and runs through the
    # 20-row shard 1 into shard 2, so rank 0 receives from two ranks
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_halo_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    gathered = q.get(timeout=300)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    w = halo_mix(world)
    full = full_oracle_blocks(oracle_mod, w, shards_to_host_u16(make_shards(w)))
    seen = {}
    for g in gathered:
        for k, h in g.items():
            assert k not in seen
            seen[k] = h
    assert seen == {k: _digest(v) for k, v in full.items()}
