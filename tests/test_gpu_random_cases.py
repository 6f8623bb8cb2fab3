"""Randomized structures on the GPU: seeded random workloads (see
workloads.random_cases) prepared through the C ABI, byte for byte against
the CPU oracle -- the full plan, the full plan on the element path
(WT_FLAG_FORCE_NARROW), and every shard-local plan with halos run into the
same pools (with the rows past each halo, and every shard a plan does not
read, replaced by negated decoys)."""
import pytest
import torch

import bf16_fp8_parameter_wt_b300 as wt
from gpu_helpers import CANARY, assert_pools_equal, device_pools, oracle_pools, run_gpu
from workloads import make_shards, random_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from bf16_fp8_parameter_wt_b300 import build
    build.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("seed", range(60))
def test_random_workload_equals_oracle(oracle_mod, seed):
    w = random_workload(seed)
    shards = make_shards(w, device="cuda:0")
    want = oracle_pools(oracle_mod, w, shards)
    flags = wt.WT_FLAG_FORCE_NARROW if seed % 3 == 2 else 0
    plan, pools = run_gpu(w, shards, flags=flags)
    plan.check()
    assert_pools_equal(pools, want)
    plan.close()


@pytest.mark.parametrize("seed", range(0, 60, 2))
def test_random_halo_plans_together_equal_oracle(oracle_mod, seed):
    w = random_workload(seed)
    src = make_shards(w, device="cuda:0")
    want = oracle_pools(oracle_mod, w, src)
    nshards = len(w.params[0].shard_rows)
    pools = None
    for s in range(nshards):
        with wt.Plan(w, device=0, local_shard=s, halo=True) as plan:
            if pools is None:
                pools = device_pools(plan, w.num_ranks)
            keep, ptrs = [], []
            for i, per in enumerate(src):
                for k, x in enumerate(per):
                    n = plan.shard_rows_read(i, k)
                    if not x.numel():
                        ptrs.append(0)
                        continue
                    t = x if k == s else x.clone()
                    if k != s:
                        t[n:] = -t[n:]              # past the halo (all of it when n = 0)
                    keep.append(t)
                    ptrs.append(t.data_ptr())
            plan.prepare(ptrs, [p.data_ptr() for p in pools], torch.cuda.current_stream().cuda_stream)
            plan.check()
            torch.cuda.synchronize()
    assert_pools_equal(pools, want)
