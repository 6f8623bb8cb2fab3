"""Randomized structures on the host (no GPU): seeded random workloads
(random fusion groups, ragged shapes, random FSDP splits with empty
shards, both formats, 1-3 destinations on 1-4 ranks, random 128-aligned
row or column slices) checked against the oracle and against counts made
from the workload description.

- The plan's layout (every offset, every pool size) equals the oracle's.
- Its stats equal the workload's bytes, blocks and elements; its per-rank
  expected counts equal the oracle's.
- Shard-local plans with halos partition the full plan, read exactly the
  halo rows counted here, and (oracle pin) the blocks each shard owns,
  computed by the oracle from its own rows and those halo rows only, are
  the full output's.
"""
import numpy as np
import pytest

import bf16_fp8_parameter_wt_b300 as wt
from shard_helpers import (assembled_oracle_blocks, full_oracle_blocks, halo_rows_needed,
                           local_counts, same_blocks)
from workloads import make_shards, random_workload, shards_to_host_u16

SEEDS = range(120)


@pytest.mark.parametrize("seed", SEEDS)
def test_random_layout_and_counts_equal_oracle(oracle_mod, seed):
    w = random_workload(seed)
    m = oracle_mod.Model(w)
    d, s, pools = m.layout()
    with wt.Plan(w, device=-1) as p:
        assert [p.pool_bytes(r) for r in range(w.num_ranks)] == pools
        for o, out in enumerate(w.outputs):
            for k, rank in enumerate(out.dst_ranks):
                rr, dd, ss = p.output_layout(o, k)
                assert (rr, dd) == (rank, d[o][k])
                if out.fp8:
                    assert ss == s[o][k]
        st = p.stats
        assert (st["bytes_read"], st["bytes_written"], st["num_units"], st["num_params_total"]) == (
            w.bytes_read, w.bytes_written, w.num_tiles, w.num_params_total)
        assert [p.expected_count(r) for r in range(w.num_ranks)] == \
               [m.expected_blocks(r) for r in range(w.num_ranks)]


@pytest.mark.parametrize("seed", SEEDS)
def test_random_halo_plans_partition_the_full_plan(seed):
    w = random_workload(seed)
    shards = len(w.params[0].shard_rows)
    with wt.Plan(w, device=-1) as full:
        fst = full.stats
        fexp = [full.expected_count(r) for r in range(w.num_ranks)]
    tot = {k: 0 for k in ("num_units", "bytes_read", "bytes_written", "num_params_total")}
    texp = [0] * w.num_ranks
    for s in range(shards):
        with wt.Plan(w, device=-1, local_shard=s, halo=True) as p:
            st = p.stats
            units, elems, written, per_rank = local_counts(w, s, halo=True)
            assert (st["num_units"], st["num_params_total"], st["bytes_written"]) == (units, elems, written)
            assert [p.expected_count(r) for r in range(w.num_ranks)] == per_rank
            need = halo_rows_needed(w, s)
            for i, par in enumerate(w.params):
                for k, n in enumerate(par.shard_rows):
                    assert p.shard_rows_read(i, k) == (n if k == s else need.get((i, k), 0))
            for k in tot:
                tot[k] += st[k]
            texp = [a + b for a, b in zip(texp, per_rank)]
    assert all(tot[k] == fst[k] for k in tot) and texp == fexp


@pytest.mark.parametrize("seed", range(0, 120, 6))
def test_random_oracle_blocks_from_own_and_halo_rows(oracle_mod, seed):
    w = random_workload(seed)
    flat = shards_to_host_u16(make_shards(w))
    base, k = [], 0
    for p in w.params:
        base.append(k)
        k += len(p.shard_rows)
    full = full_oracle_blocks(oracle_mod, w, flat)
    seen = set()
    for s in range(len(w.params[0].shard_rows)):
        need = halo_rows_needed(w, s)

        def rows_of(p, k, a, b):
            assert k == s or b <= need[(p, k)]          # only its own rows and its halos
            return flat[base[p] + k][a:b]

        for key, blk in assembled_oracle_blocks(oracle_mod, w, s, rows_of).items():
            assert key not in seen
            seen.add(key)
            assert same_blocks(blk, full[key]), (seed, s, key)
    assert seen == set(full)
