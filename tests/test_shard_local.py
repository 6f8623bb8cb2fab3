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
- Two gloo ranks each compile their own local plan and run the oracle on
  their own shards only; rank 0 checks the union against the full oracle.
- Misaligned shards, offload and bad arguments are refused.
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
from workloads import (TILE, Output, Param, Workload, kimi_k2_moe_layer, llama_dense,
                       make_shards, shard_local_mix, shards_to_host_u16, tiny_dense)


def _cdiv(a, b):
    return -(-a // b)


def shard_runs(w, o, s):
    """(fused row begin, rows, param index) of every shard-s run of output o."""
    out, row = [], 0
    for p in w.outputs[o].parts:
        par = w.params[p]
        r = row
        for k, n in enumerate(par.shard_rows):
            if k == s and n:
                out.append((r, n, p))
            r += n
        row += par.rows
    return out


def owned_block_rows(w, o, s):
    """Block rows of output o whose rows all come from shard s."""
    return [b for (r0, n, _) in shard_runs(w, o, s) for b in range(r0 // TILE, _cdiv(r0 + n, TILE))]


def held_blocks(w, o, d, block_rows):
    """Blocks of block_rows that destination d of output o holds."""
    m, n = w.output_shape(o)
    out = w.outputs[o]
    bn = _cdiv(n, TILE)
    sl = out.slices[d] if out.slices is not None else None
    held = []
    for bi in block_rows:
        for bj in range(bn):
            if sl is not None:
                dim, ranges = sl
                idx = bi if dim == 0 else bj
                if not any(b // TILE <= idx < _cdiv(b + l, TILE) for b, l in ranges):
                    continue
            held.append((bi, bj))
    return held


def local_counts(w, s):
    """Units, elements, bytes written and per-rank blocks of shard s's work."""
    units = elems = written = 0
    per_rank = [0] * w.num_ranks
    for o, out in enumerate(w.outputs):
        m, n = w.output_shape(o)
        rows = owned_block_rows(w, o, s)
        for bi in rows:
            for bj in range(_cdiv(n, TILE)):
                units += 1
                elems += (min(TILE, m - bi * TILE)) * (min(TILE, n - bj * TILE))
        for d, r in enumerate(out.dst_ranks):
            for bi, bj in held_blocks(w, o, d, rows):
                e = min(TILE, m - bi * TILE) * min(TILE, n - bj * TILE)
                written += e + 4 if out.fp8 else 2 * e
                per_rank[r] += 1
    return units, elems, written, per_rank


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


def full_oracle_blocks(oracle_mod, w, flat_full):
    m = oracle_mod.Model(w)
    res = {}
    for o in range(len(w.outputs)):
        data, scales = m.prepare_output(o, flat_full)
        rows, n = w.output_shape(o)
        esz = 1 if w.outputs[o].fp8 else 2
        data = data.reshape(rows, n * esz)
        bn = _cdiv(n, TILE)
        for bi in range(_cdiv(rows, TILE)):
            srow = scales.reshape(-1, bn)[bi].copy() if scales is not None else None
            res[(o, bi)] = (data[bi * TILE:(bi + 1) * TILE].copy(), srow)
    return res


def _same(a, b):
    return np.array_equal(a[0], b[0]) and (a[1] is None) == (b[1] is None) and (
        a[1] is None or np.array_equal(a[1].view(np.uint32), b[1].view(np.uint32)))


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
            assert _same(blk, full[key]), f"shard {s}, output {key[0]}, block row {key[1]}"
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


def _stats(w, s=-1):
    with wt.Plan(w, device=-1, local_shard=s) as p:
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


# ---- two gloo ranks, each with its own shard ------------------------------

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


def test_two_gloo_ranks_prepare_their_own_shards(oracle_mod):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    gathered = q.get(timeout=300)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    w = shard_local_mix(2)
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
