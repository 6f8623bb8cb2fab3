"""GPU tests of shard-local plans (each FSDP rank quantizes the blocks of
its own dim-0 shard, no exchange).

- Every local plan writes only its own blocks, computed from its own
  shard: the other shard slots point at decoys (the same shards negated),
  so a block read from the wrong shard would come out with flipped signs.
  What a plan writes is found by running it on pools filled with two
  different canaries: the bytes that agree are the written ones. Those
  bytes equal the oracle's, count to the plan's bytes_written, are
  disjoint across shards, and together are exactly what the full plan
  writes.
- All local plans run one after another into the same pools, with NULL
  for the shards they do not read, give the oracle's pools; per-rank
  completion counters then read the full plan's expected counts.
- At the full Kimi-K2 layer size the union of the 8 local plans is
  byte-identical to the full plan's output.
- Halo plans (shard boundaries off the 128-row grid): the same checks,
  with each halo slot pointing at a copy of the shard whose rows past the
  reported halo are negated (a read past the halo changes the result),
  then with halo buffers holding exactly the rows reported and NULL for
  every other shard; on the Llama stack the 8 halo plans together (with
  decoys past the halos) equal the full plan.
"""
import pytest
import torch

import bf16_fp8_parameter_wt_b300 as wt
from gpu_helpers import CANARY, assert_pools_equal, device_pools, oracle_pools
from workloads import halo_mix, kimi_k2_moe_layer, llama_dense, make_shards, shard_local_mix

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from bf16_fp8_parameter_wt_b300 import build
    build.build()
    assert torch.cuda.is_available()


def _ptrs(shards, s, other):
    """Flat shard pointers: shard index s from `shards`, the others from
    `other` (a list of the same shape) or 0 when other is None."""
    out = []
    for per, alt in zip(shards, other if other is not None else [None] * len(shards)):
        for k, x in enumerate(per):
            if k == s:
                out.append(x.data_ptr() if x.numel() else 0)
            elif alt is not None and alt[k].numel():
                out.append(alt[k].data_ptr())
            else:
                out.append(0)
    return out


def _all(shards):
    return [x.data_ptr() if x.numel() else 0 for per in shards for x in per]


def _run(plan, ptrs, pools):
    plan.prepare(ptrs, [p.data_ptr() for p in pools], torch.cuda.current_stream().cuda_stream)
    plan.check()
    torch.cuda.synchronize()


def _written(plan, ptrs, n_ranks):
    """(pools after a run on 0xA5 canaries, per-rank mask of written bytes)."""
    a = device_pools(plan, n_ranks, fill=CANARY)
    b = device_pools(plan, n_ranks, fill=0x5A)
    _run(plan, ptrs, a)
    _run(plan, ptrs, b)
    return a, [x == y for x, y in zip(a, b)]


@pytest.mark.parametrize("shards", [4, 2])
def test_each_local_plan_writes_its_own_blocks_from_its_own_shard(oracle_mod, shards):
    w = shard_local_mix(shards)
    src = make_shards(w, device="cuda:0")
    decoy = [[-x for x in per] for per in src]
    want = [torch.from_numpy(x).to("cuda:0") for x in oracle_pools(oracle_mod, w, src)]
    with wt.Plan(w, device=0) as full:
        _, full_mask = _written(full, _all(src), w.num_ranks)
    union = [torch.zeros_like(m) for m in full_mask]
    for s in range(shards):
        with wt.Plan(w, device=0, local_shard=s) as plan:
            got, mask = _written(plan, _ptrs(src, s, decoy), w.num_ranks)
            n = 0
            for r in range(w.num_ranks):
                k = want[r].numel()
                m = mask[r][:k]
                assert not bool(mask[r][k:].any()), f"shard {s}: write past pool {r}"
                assert torch.equal(got[r][:k][m], want[r][m]), f"shard {s}, rank {r}"
                assert not bool((union[r][:k] & m).any()), f"shard {s} rewrote another's bytes"
                union[r][:k] |= m
                n += int(m.sum())
            assert n == plan.stats["bytes_written"]
    for r in range(w.num_ranks):
        assert torch.equal(union[r], full_mask[r]), f"rank {r}: union differs from the full plan"


@pytest.mark.parametrize("mode", [wt.WT_COUNT_PER_LAUNCH, wt.WT_COUNT_PER_RANK])
def test_local_plans_together_give_the_oracle_pools(oracle_mod, mode):
    w = kimi_k2_moe_layer(8)
    src = make_shards(w, device="cuda:0")
    want = oracle_pools(oracle_mod, w, src)
    with wt.Plan(w, device=-1) as full:
        expected = [full.expected_count(r) for r in range(w.num_ranks)]
    counters = torch.zeros(w.num_ranks, dtype=torch.int32, device="cuda:0")
    plans = [wt.Plan(w, device=0, local_shard=s) for s in range(8)]
    pools = device_pools(plans[0], w.num_ranks)
    for s, plan in enumerate(plans):
        plan.set_counters(counters.data_ptr(), mode)
        _run(plan, _ptrs(src, s, None), pools)     # other shards: NULL
    assert [int(v) for v in counters.cpu()] == expected
    assert_pools_equal(pools, want)
    for p in plans:
        p.close()


def test_kimi_k2_layer_full_size_union_equals_full_plan():
    w = kimi_k2_moe_layer()
    src = make_shards(w, device="cuda:0")
    with wt.Plan(w, device=0) as full:
        ref = device_pools(full, w.num_ranks)
        _run(full, _all(src), ref)
    pools = [torch.full_like(p, CANARY) for p in ref]
    total = 0
    for s in range(8):
        with wt.Plan(w, device=0, local_shard=s) as plan:
            total += plan.stats["bytes_read"]
            _run(plan, _ptrs(src, s, None), pools)
    assert total == w.bytes_read
    for r in range(w.num_ranks):
        assert torch.equal(pools[r], ref[r]), f"rank {r}"


def _halo_ptrs(w, plan, src, s, exact, keep):
    """Pointers for halo plan s: its own shards, halo buffers (a copy of the
    shard with the rows past the halo negated, or exactly the halo rows),
    and for the rest the negated shard (exact=False) or NULL."""
    out = []
    for i, per in enumerate(src):
        for k, x in enumerate(per):
            n = plan.shard_rows_read(i, k)
            if k == s or not x.numel():
                out.append(x.data_ptr() if x.numel() else 0)
            elif n and exact:
                t = x[:n].clone()
                keep.append(t)
                out.append(t.data_ptr())
            elif n:
                t = x.clone()
                t[n:] = -t[n:]
                keep.append(t)
                out.append(t.data_ptr())
            elif exact:
                out.append(0)
            else:
                t = -x
                keep.append(t)
                out.append(t.data_ptr())
    return out


@pytest.mark.parametrize("shards", [4, 2])
def test_halo_plans_write_their_own_blocks_from_own_and_halo_rows(oracle_mod, shards):
    w = halo_mix(shards)
    src = make_shards(w, device="cuda:0")
    want = [torch.from_numpy(x).to("cuda:0") for x in oracle_pools(oracle_mod, w, src)]
    with wt.Plan(w, device=0) as full:
        _, full_mask = _written(full, _all(src), w.num_ranks)
    union = [torch.zeros_like(m) for m in full_mask]
    for s in range(shards):
        with wt.Plan(w, device=0, local_shard=s, halo=True) as plan:
            keep = []
            got, mask = _written(plan, _halo_ptrs(w, plan, src, s, False, keep), w.num_ranks)
            n = 0
            for r in range(w.num_ranks):
                k = want[r].numel()
                m = mask[r][:k]
                assert not bool(mask[r][k:].any()), f"shard {s}: write past pool {r}"
                assert torch.equal(got[r][:k][m], want[r][m]), f"shard {s}, rank {r}"
                assert not bool((union[r][:k] & m).any()), f"shard {s} rewrote another's bytes"
                union[r][:k] |= m
                n += int(m.sum())
            assert n == plan.stats["bytes_written"]
    for r in range(w.num_ranks):
        assert torch.equal(union[r], full_mask[r]), f"rank {r}: union differs from the full plan"
    # exactly-sized halo buffers and NULL for every shard a plan does not read
    with wt.Plan(w, device=0) as full:
        pools = device_pools(full, w.num_ranks)
    for s in range(shards):
        with wt.Plan(w, device=0, local_shard=s, halo=True) as plan:
            keep = []
            _run(plan, _halo_ptrs(w, plan, src, s, True, keep), pools)
    assert_pools_equal(pools, [x.cpu().numpy() for x in want])


def test_llama_halo_plans_together_equal_the_full_plan():
    w = llama_dense()
    src = make_shards(w, device="cuda:0")
    with wt.Plan(w, device=0) as full:
        ref = device_pools(full, w.num_ranks)
        _run(full, _all(src), ref)
    pools = [torch.full_like(p, CANARY) for p in ref]
    for s in range(8):
        with wt.Plan(w, device=0, local_shard=s, halo=True) as plan:
            keep = []                               # full-size buffers, decoys past the halo
            _run(plan, _halo_ptrs(w, plan, src, s, False, keep), pools)
    for r in range(w.num_ranks):
        assert torch.equal(pools[r], ref[r]), f"rank {r}"
