"""GPU tests of the completion counters (the transfer stage's receive-side
count) and of the bounded device-side wait for a consumer.

The waiting kernel is always queued after the preparation on the same
stream, or waits for a target that nothing will reach and must give up:
no test runs a kernel that depends on another one running at the same time.
"""
import time

import numpy as np
import pytest
import torch

import bf16_fp8_parameter_wt_b300 as wt
from bf16_fp8_parameter_wt_b300.wt import STATUS_NAMES
from gpu_helpers import CANARY, assert_pools_equal, device_pools, oracle_pools, run_gpu
from workloads import kimi_k2_moe_layer, make_shards, offload_layer, tiny_dense, tp_slices_small

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from bf16_fp8_parameter_wt_b300 import build
    build.build()
    assert torch.cuda.is_available()


def _counters(n):
    return torch.zeros(max(1, n), dtype=torch.int32, device="cuda:0")


def _read(c, n):
    torch.cuda.synchronize()
    return [int(v) & 0xFFFFFFFF for v in c[:n].cpu().tolist()]


MODES = [wt.WT_COUNT_PER_LAUNCH, wt.WT_COUNT_PER_RANK]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("make", [tiny_dense, tp_slices_small, lambda: kimi_k2_moe_layer(4)])
def test_counters_count_every_block_of_every_step(oracle_mod, make, mode):
    w = make()
    shards = make_shards(w, device="cuda:0")
    want = oracle_pools(oracle_mod, w, shards)
    plan = wt.Plan(w, device=0)
    pools = device_pools(plan, w.num_ranks)
    c = _counters(w.num_ranks)
    plan.set_counters(c.data_ptr(), mode)
    expected = [plan.expected_count(r) for r in range(w.num_ranks)]
    for step in (1, 2):
        for p in pools:
            p.fill_(CANARY)
        run_gpu(w, shards, pools=pools, plan=plan)
        plan.check()
        assert _read(c, w.num_ranks) == [step * e for e in expected]
        assert_pools_equal(pools, want)
    plan.set_counters(0)                      # signalling off: the counters stay put
    run_gpu(w, shards, pools=pools, plan=plan)
    assert _read(c, w.num_ranks) == [2 * e for e in expected]
    plan.close()


def test_wait_after_the_step_on_the_same_stream(oracle_mod):
    w = tiny_dense()
    shards = make_shards(w, device="cuda:0")
    plan = wt.Plan(w, device=0)
    pools = device_pools(plan, w.num_ranks)
    c = _counters(w.num_ranks)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda:0")
    plan.set_counters(c.data_ptr())
    s = torch.cuda.Stream()
    flat = [x.data_ptr() for per in shards for x in per]
    plan.prepare(flat, [p.data_ptr() for p in pools], s.cuda_stream)
    targets = [plan.expected_count(r) for r in range(w.num_ranks)]
    wt.wt_wait_counters(c.data_ptr(), targets, 1_000_000_000, status.data_ptr(), s.cuda_stream)
    s.synchronize()
    assert int(status.item()) == 0
    # one more than any step will deliver: the wait gives up and says so
    status.fill_(-1)
    t0 = time.perf_counter()
    wt.wt_wait_counters(c.data_ptr(), [t + 1 for t in targets], 20_000_000, status.data_ptr(),
                        s.cuda_stream)
    s.synchronize()
    assert int(status.item()) == STATUS_NAMES.index("WT_ERR_TIMEOUT")
    assert time.perf_counter() - t0 < 5.0
    plan.close()


@pytest.mark.parametrize("mode", MODES)
def test_offload_steps_signal_too(oracle_mod, mode):
    w = offload_layer(1)
    shards = make_shards(w, device="cuda:0")
    want = oracle_pools(oracle_mod, w, shards)
    plan = wt.Plan(w, device=0, offload_chunk_bytes=96 << 20)
    host = torch.zeros(plan.stats["host_bytes"], dtype=torch.uint8, pin_memory=True)
    for p_, per in enumerate(shards):
        for k, sh in enumerate(per):
            off = plan.shard_host_offset(p_, k)
            host[off:off + sh.numel() * 2].copy_(sh.reshape(-1).view(torch.uint8))
    pools = device_pools(plan, w.num_ranks)
    c = _counters(w.num_ranks)
    plan.set_counters(c.data_ptr(), mode)
    copy_s, comp_s = torch.cuda.Stream(), torch.cuda.Stream()
    plan.prepare_offload(host.data_ptr(), [p.data_ptr() for p in pools], copy_s.cuda_stream,
                         comp_s.cuda_stream)
    comp_s.synchronize()
    assert _read(c, w.num_ranks) == [plan.expected_count(r) for r in range(w.num_ranks)]
    assert_pools_equal(pools, want)
    plan.close()


@pytest.mark.parametrize("mode", MODES)
def test_a_stalled_step_leaves_its_block_uncounted(oracle_mod, mode):
    """Per rank, the stalled step's counts stay short of a step; per launch,
    the step counts nothing. Either way the next good step adds exactly one
    step's counts once wt_plan_check has reported the timeout."""
    w = kimi_k2_moe_layer(4)
    shards = make_shards(w, device="cuda:0")
    plan = wt.Plan(w, device=0)
    pools = device_pools(plan, w.num_ranks)
    c = _counters(w.num_ranks)
    plan.set_counters(c.data_ptr(), mode)
    expected = [plan.expected_count(r) for r in range(w.num_ranks)]
    wt.wt_debug_stall_unit(plan.handle, 1000, 50_000_000)
    run_gpu(w, shards, pools=pools, plan=plan)
    with pytest.raises(wt.WTError) as ei:
        plan.check()
    assert ei.value.name == "WT_ERR_TIMEOUT"
    partial = _read(c, w.num_ranks)
    assert sum(partial) < sum(expected)
    assert all(p <= e for p, e in zip(partial, expected))
    if mode == wt.WT_COUNT_PER_LAUNCH:
        assert sum(partial) == 0
    wt.wt_debug_stall_unit(plan.handle, -1, 0)
    run_gpu(w, shards, pools=pools, plan=plan)
    plan.check()
    assert [a - b for a, b in zip(_read(c, w.num_ranks), partial)] == expected
    plan.close()


def test_per_rank_counting_completes_the_ranks_in_order(oracle_mod):
    """Counting per rank runs the step rank group by rank group: when a unit
    of rank 2's group stalls, ranks 0 and 1 have already received their
    whole step's count and the later ranks nothing."""
    w = kimi_k2_moe_layer(4)                   # experts 0..3 on ranks 0..3
    shards = make_shards(w, device="cuda:0")
    plan = wt.Plan(w, device=0)
    pools = device_pools(plan, w.num_ranks)
    c = _counters(w.num_ranks)
    plan.set_counters(c.data_ptr(), wt.WT_COUNT_PER_RANK)
    expected = [plan.expected_count(r) for r in range(w.num_ranks)]
    per_expert = (4096 // 128) * (7168 // 128) + (7168 // 128) * (2048 // 128)
    wt.wt_debug_stall_unit(plan.handle, 2 * per_expert + 100, 50_000_000)   # expert 2's gate_up
    run_gpu(w, shards, pools=pools, plan=plan)
    with pytest.raises(wt.WTError):
        plan.check()
    assert _read(c, w.num_ranks) == expected[:2] + [0] * (w.num_ranks - 2)
    wt.wt_debug_stall_unit(plan.handle, -1, 0)
    plan.close()


def test_per_rank_counting_replays_from_a_cuda_graph(oracle_mod):
    """A step counted per rank (rank-group launches queued as programmatic
    dependents, each followed by its count kernel) captured into a CUDA
    graph: every replay writes the oracle's bytes and adds one step's counts."""
    w = kimi_k2_moe_layer(4)
    shards = make_shards(w, device="cuda:0")
    want = oracle_pools(oracle_mod, w, shards)
    plan = wt.Plan(w, device=0)
    pools = device_pools(plan, w.num_ranks)
    c = _counters(w.num_ranks)
    plan.set_counters(c.data_ptr(), wt.WT_COUNT_PER_RANK)
    expected = [plan.expected_count(r) for r in range(w.num_ranks)]
    stream = torch.cuda.Stream()
    sp, pp = plan.bind([s.data_ptr() for per in shards for s in per], [p.data_ptr() for p in pools])
    plan.prepare(sp, pp, stream.cuda_stream)          # stages the pointers (one step counted)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        plan.prepare(sp, pp, stream.cuda_stream)
    for step in (2, 3):
        for p in pools:
            p.fill_(CANARY)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert _read(c, w.num_ranks) == [step * e for e in expected]
        assert_pools_equal(pools, want)
    plan.close()
