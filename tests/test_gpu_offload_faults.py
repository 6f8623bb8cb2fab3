"""GPU tests of the CPU-offload pipeline and of failure reporting.

- wt_prepare_offload (pinned host image -> two staging buffers on a copy
  stream, preparation on a compute stream) writes the same pools as the CPU
  oracle on an offload layer split into several chunks, twice in a row.
- A chunk failure injected on the host drains both streams, reports
  WT_ERR_CUDA, and leaves the plan usable.
- A kernel wait that runs out (one unit's stage is left unfilled on
  purpose, with a short wait limit) is reported by wt_plan_check as
  WT_ERR_TIMEOUT; the kernel returns on its own and the next step is
  correct. Nothing here faults or hangs the GPU: every wait in the kernel
  is bounded.
"""
import time

import pytest
import torch

import bf16_fp8_parameter_wt_b300 as wt
from gpu_helpers import CANARY, assert_pools_equal, device_pools, oracle_pools, run_gpu
from workloads import kimi_k2_moe_layer, make_shards, offload_layer, tiny_dense

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from bf16_fp8_parameter_wt_b300 import build
    build.build()
    assert torch.cuda.is_available()


def _host_image(plan, shards):
    """The packed pinned image that wt_prepare_offload reads."""
    host = torch.zeros(plan.stats["host_bytes"], dtype=torch.uint8, pin_memory=True)
    for p, per in enumerate(shards):
        for k, s in enumerate(per):
            off = plan.shard_host_offset(p, k)
            n = s.numel() * 2
            host[off:off + n].copy_(s.reshape(-1).view(torch.uint8))
    return host


def _offload(plan, host, pools, copy_s, comp_s):
    plan.prepare_offload(host.data_ptr(), [p.data_ptr() for p in pools], copy_s.cuda_stream,
                         comp_s.cuda_stream)
    comp_s.synchronize()


def test_offload_equals_oracle_over_several_chunks(oracle_mod):
    w = offload_layer(3)                       # qkv, o and 3 experts + the shared one
    shards = make_shards(w, device="cuda:0")
    want = oracle_pools(oracle_mod, w, shards)
    plan = wt.Plan(w, device=0, offload_chunk_bytes=160 << 20)
    assert plan.stats["num_chunks"] >= 4      # the 308 MB qkv is a chunk of its own
    host = _host_image(plan, shards)
    del shards
    pools = device_pools(plan, w.num_ranks)
    copy_s, comp_s = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(2):                         # staging buffers and pools reused
        for p in pools:
            p.fill_(CANARY)
        _offload(plan, host, pools, copy_s, comp_s)
        plan.check(comp_s.cuda_stream)
        assert_pools_equal(pools, want)
    plan.close()


def test_injected_offload_failure_drains_and_recovers(oracle_mod):
    w = offload_layer(1)
    shards = make_shards(w, device="cuda:0")
    want = oracle_pools(oracle_mod, w, shards)
    plan = wt.Plan(w, device=0, offload_chunk_bytes=96 << 20)
    assert plan.stats["num_chunks"] >= 3
    host = _host_image(plan, shards)
    pools = device_pools(plan, w.num_ranks)
    copy_s, comp_s = torch.cuda.Stream(), torch.cuda.Stream()
    wt.wt_debug_fail_offload_chunk(plan.handle, 2)
    with pytest.raises(wt.WTError) as ei:
        _offload(plan, host, pools, copy_s, comp_s)
    assert ei.value.name == "WT_ERR_CUDA"
    assert "chunk 2" in str(ei.value)
    wt.wt_debug_fail_offload_chunk(plan.handle, -1)
    for p in pools:
        p.fill_(CANARY)
    _offload(plan, host, pools, copy_s, comp_s)
    plan.check(comp_s.cuda_stream)
    assert_pools_equal(pools, want)
    plan.close()


@pytest.mark.parametrize("make,unit", [(tiny_dense, 3), (lambda: kimi_k2_moe_layer(4), 1000)])
def test_stalled_wait_reports_timeout_then_recovers(oracle_mod, make, unit):
    w = make()
    shards = make_shards(w, device="cuda:0")
    want = oracle_pools(oracle_mod, w, shards)
    plan = wt.Plan(w, device=0)
    pools = device_pools(plan, w.num_ranks)
    wt.wt_debug_stall_unit(plan.handle, unit, 50_000_000)      # 50 ms wait limit
    t0 = time.perf_counter()
    run_gpu(w, shards, pools=pools, plan=plan)
    with pytest.raises(wt.WTError) as ei:
        plan.check()
    assert ei.value.name == "WT_ERR_TIMEOUT"
    assert time.perf_counter() - t0 < 10.0     # a few wait limits, not the default 2 s each
    # the error was cleared and the plan works again
    wt.wt_debug_stall_unit(plan.handle, -1, 0)
    for p in pools:
        p.fill_(CANARY)
    run_gpu(w, shards, pools=pools, plan=plan)
    plan.check()
    assert_pools_equal(pools, want)
    plan.close()


def test_allocation_failure_is_reported_and_leaves_no_stale_error(oracle_mod):
    """Offload staging larger than the GPU (two buffers of a 300 GB chunk):
    the plan is refused with WT_ERR_OUT_OF_MEMORY, its tables are freed, and
    the failed cudaMalloc does not surface as an error of the next plan's
    step."""
    from gpu_helpers import full_check
    from workloads import Output, Param, Workload
    huge = Workload("huge", [Param("x", 150_000, 1_000_000, (150_000,))],
                    [Output("x", (0,), True, (0,))], 1)
    free0 = torch.cuda.mem_get_info(0)[0]
    with pytest.raises(wt.WTError) as ei:
        wt.Plan(huge, device=0, offload_chunk_bytes=1 << 40)
    assert ei.value.name == "WT_ERR_OUT_OF_MEMORY"
    assert "offload staging" in str(ei.value)
    assert torch.cuda.mem_get_info(0)[0] >= free0 - (64 << 20)     # nothing left behind
    full_check(oracle_mod, tiny_dense())


def test_offload_with_row_by_row_blocks_keeps_each_chunk_in_its_range(oracle_mod):
    """Outputs with blocks gathered row by row (4100-byte rows, block rows
    spanning shards, a 1-column norm) are handed out first within each
    offload chunk; over several chunks, twice in a row, the pools equal the
    oracle's."""
    from workloads import Output, Param, ValueRecipe, Workload
    params = [Param("a", 700, 2050, (301, 399)), Param("b", 300, 264, (1,) * 44 + (256,)),
              Param("n", 512, 1, (100, 300, 112)), Param("c", 1000, 1024, (500, 500)),
              Param("d", 640, 2049, (640,))]
    outs = [Output("a", (0,), True, (0,)), Output("b", (1,), True, (1,)),
            Output("n", (2,), False, (0,)), Output("c", (3,), True, (1,)),
            Output("d", (4,), False, (0,))]
    w = Workload("offload_slow_first", params, outs, 2,
                 ValueRecipe("student_t3", 0.02, 93, zero_tile_eighths=1, outlier_tile_eighths=1,
                             outlier=3.0e4))
    shards = make_shards(w, device="cuda:0")
    want = oracle_pools(oracle_mod, w, shards)
    plan = wt.Plan(w, device=0, offload_chunk_bytes=2 << 20)
    assert plan.stats["num_chunks"] >= 4
    host = _host_image(plan, shards)
    pools = device_pools(plan, w.num_ranks)
    copy_s, comp_s = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(2):
        for p in pools:
            p.fill_(CANARY)
        _offload(plan, host, pools, copy_s, comp_s)
        plan.check(comp_s.cuda_stream)
        assert_pools_equal(pools, want)
    plan.close()
