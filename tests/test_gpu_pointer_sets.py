"""wt_prepare with changing buffer addresses: a plan keeps several uploaded
pointer-table sets, so a caller that alternates between buffer sets (FSDP
double buffering: two sets of shards, two sets of pools) reuses them with no
upload and no host-side wait; more sets than the plan holds are rebuilt
least-recently-used first, always with the right bytes; a set that a
captured CUDA graph replays is never rebuilt."""
import statistics
import time

import pytest
import torch

import bf16_fp8_parameter_wt_b300 as wt
from gpu_helpers import CANARY, assert_pools_equal, device_pools, oracle_pools
from workloads import llama_dense, make_shards, tiny_dense

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from bf16_fp8_parameter_wt_b300 import build
    build.build()
    assert torch.cuda.is_available()


def test_alternating_two_buffer_sets_never_waits_on_the_host(oracle_mod):
    """Ten steps of the Llama stack alternating between two shard sets and
    two pool sets: both pool sets hold the oracle's bytes, and once both sets
    are staged a call returns in a small fraction of one step's kernel time
    (the host runs ahead of the GPU instead of waiting for it)."""
    w = llama_dense()
    shards_a = make_shards(w, device="cuda:0")
    want = oracle_pools(oracle_mod, w, shards_a)
    shards_b = [[s.clone() for s in per] for per in shards_a]
    plan = wt.Plan(w, device=0)
    pools = [device_pools(plan, w.num_ranks), device_pools(plan, w.num_ranks)]
    bound = [plan.bind([s.data_ptr() for per in sh for s in per], [p.data_ptr() for p in pl])
             for sh, pl in ((shards_a, pools[0]), (shards_b, pools[1]))]
    stream = torch.cuda.Stream()
    sp = stream.cuda_stream
    for i in range(2):                       # stage both sets
        plan.prepare(*bound[i], sp)
    stream.synchronize()
    for pl in pools:
        for p in pl:
            p.fill_(CANARY)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(10)]
    host = []
    for i in range(10):
        ev[i][0].record(stream)
        t0 = time.perf_counter()
        plan.prepare(*bound[i % 2], sp)
        host.append(time.perf_counter() - t0)
        ev[i][1].record(stream)
    still_running = not stream.query()
    stream.synchronize()
    plan.check(sp)
    kernel_s = statistics.median(s.elapsed_time(e) for s, e in ev) * 1e-3
    assert still_running, "the host waited for the GPU"
    assert statistics.median(host) < 0.1 * kernel_s, (host, kernel_s)
    assert max(host) < 0.5 * kernel_s, (host, kernel_s)
    assert_pools_equal(pools[0], want)
    assert_pools_equal(pools[1], want)
    plan.close()


def test_more_buffer_sets_than_the_plan_holds(oracle_mod):
    """Seven pool sets cycled three times (the plan keeps four): every step
    writes the oracle's bytes into its own pools."""
    w = tiny_dense()
    shards = make_shards(w, device="cuda:0")
    want = oracle_pools(oracle_mod, w, shards)
    plan = wt.Plan(w, device=0)
    sets = [device_pools(plan, w.num_ranks) for _ in range(7)]
    flat = [s.data_ptr() for per in shards for s in per]
    stream = torch.cuda.current_stream()
    for _ in range(3):
        for pl in sets:
            for p in pl:
                p.fill_(CANARY)
            plan.prepare(flat, [p.data_ptr() for p in pl], stream.cuda_stream)
        torch.cuda.synchronize()
        for pl in sets:
            assert_pools_equal(pl, want)
    plan.close()


def test_captured_set_is_kept_while_others_come_and_go(oracle_mod):
    """A graph captured with one pool set replays correctly after six other
    pool sets have been used (its set is never rebuilt); once every set is
    held by a captured graph, new addresses are refused."""
    w = tiny_dense()
    shards = make_shards(w, device="cuda:0")
    want = oracle_pools(oracle_mod, w, shards)
    plan = wt.Plan(w, device=0)
    flat = [s.data_ptr() for per in shards for s in per]
    stream = torch.cuda.Stream()
    sp = stream.cuda_stream
    held = device_pools(plan, w.num_ranks)
    ptrs = [p.data_ptr() for p in held]
    plan.prepare(flat, ptrs, sp)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        plan.prepare(flat, ptrs, sp)
    others = [device_pools(plan, w.num_ranks) for _ in range(6)]
    for pl in others:
        plan.prepare(flat, [p.data_ptr() for p in pl], sp)
    stream.synchronize()
    for p in held:
        p.fill_(CANARY)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    assert_pools_equal(held, want)
    for pl in others:
        assert_pools_equal(pl, want)
    # capture three more sets: all four are then pinned by graphs
    graphs = [graph]
    for pl in others[:3]:
        ptr = [p.data_ptr() for p in pl]
        plan.prepare(flat, ptr, sp)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            plan.prepare(flat, ptr, sp)
        graphs.append(g)
    with pytest.raises(wt.WTError) as ei:
        plan.prepare(flat, [p.data_ptr() for p in others[5]], sp)
    assert ei.value.name == "WT_ERR_INVALID_ARGUMENT"
    assert "captured" in str(ei.value)
    for p in held:
        p.fill_(CANARY)
    torch.cuda.synchronize()
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()
    assert_pools_equal(held, want)
    plan.close()
