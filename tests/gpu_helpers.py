"""Helpers shared by the GPU tests: run a workload through the C ABI and
through the CPU oracle on the same seeded inputs, compare byte for byte."""
import os

import numpy as np
import torch

import bf16_fp8_parameter_wt_b300 as wt
from workloads import make_shards, shards_to_host_u16

CANARY = 0xA5


def ncores() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def device_pools(plan, num_ranks, fill=CANARY, dev="cuda:0"):
    return [torch.full((max(1, plan.pool_bytes(r)) + 256,), fill, dtype=torch.uint8, device=dev)
            for r in range(num_ranks)]


def run_gpu(w, shards, pools=None, flags=0, stream=None, plan=None):
    """Run one wt_prepare; returns (plan, pools)."""
    own = plan is None
    if own:
        plan = wt.Plan(w, device=0, flags=flags)
    if pools is None:
        pools = device_pools(plan, w.num_ranks)
    flat = [s for per in shards for s in per]
    st = stream or torch.cuda.current_stream()
    plan.prepare([s.data_ptr() if s.numel() else 0 for s in flat], [p.data_ptr() for p in pools],
                 st.cuda_stream)
    torch.cuda.synchronize()
    return plan, pools


def oracle_pools(oracle_mod, w, shards, fill=CANARY):
    return oracle_mod.Model(w).prepare(shards_to_host_u16(shards), nthreads=ncores(), fill=fill)


def assert_pools_equal(gpu_pools, want, fill=CANARY):
    for r, exp in enumerate(want):
        got = gpu_pools[r].cpu().numpy()
        n = len(exp)
        if not np.array_equal(got[:n], exp):
            bad = np.nonzero(got[:n] != exp)[0]
            raise AssertionError(f"rank {r}: {bad.size} bytes differ, first at {int(bad[0])}: "
                                 f"gpu {got[bad[0]]:#x} oracle {exp[bad[0]]:#x}")
        # the guard band after the pool is never written
        assert np.all(got[n:] == fill), f"rank {r}: write past the pool end"


def full_check(oracle_mod, w, flags=0, dev="cuda:0"):
    shards = make_shards(w, device=dev)
    plan, pools = run_gpu(w, shards, flags=flags)
    want = oracle_pools(oracle_mod, w, shards)
    assert_pools_equal(pools, want)
    plan.close()
    return shards
