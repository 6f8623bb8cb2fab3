"""wt_prepare_noalloc against wt_prepare.

wt_prepare_noalloc is for callers that cannot let a library call cudaMalloc
(code running inside a memory pool it does not own, or beside an engine that
has reserved all device memory): it keeps its schedule tables in a fixed
array inside the library instead. Its results must be the bytes wt_prepare
writes, bit for bit (the tolerance of every parity test here), on two calls
in a row -- the second call reuses the array the first one left behind.
This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import bf16_fp8_parameter_wt_b300 as wt
from workloads import (Output, Param, ValueRecipe, Workload, kimi_k2_moe_layer, make_shards,
                       tiny_dense, tp_slices_small)

pytestmark = pytest.mark.gpu

CANARY = 0xA5


@pytest.fixture(scope="module", autouse=True)
def built():
    from bf16_fp8_parameter_wt_b300 import build
    build.build()
    assert torch.cuda.is_available()


def _pools(plan, num_ranks, fill):
    return [torch.full((max(1, plan.pool_bytes(r)) + 256,), fill, dtype=torch.uint8, device="cuda:0")
            for r in range(num_ranks)]


def _small_shapes():
    # ragged edges, a 2050-column element-path output, multi-shard block rows,
    # an empty shard, BF16 pass-through and a replicated destination
    params = [Param("a", 300, 264, (1,) * 44 + (256,)), Param("b", 3, 2050, (2, 0, 1)),
              Param("c1", 50, 130, (17, 33)), Param("c2", 79, 130, (1, 0, 40, 38)),
              Param("n", 256, 1, (100, 100, 56))]
    outs = [Output("a", (0,), True, (0, 1)), Output("b", (1,), True, (1,)),
            Output("c", (2, 3), True, (0,)), Output("n", (4,), False, (1,))]
    return Workload("noalloc_small", params, outs, 2, ValueRecipe("student_t3", 0.02, 31))


@pytest.mark.parametrize("make", [tiny_dense, _small_shapes, tp_slices_small])
def test_noalloc_matches_prepare_on_two_calls(make):
    w = make()
    shards = make_shards(w, device="cuda:0")
    flat = [s.data_ptr() if s.numel() else 0 for per in shards for s in per]
    stream = torch.cuda.current_stream().cuda_stream
    plan = wt.Plan(w, device=0)
    want = _pools(plan, w.num_ranks, CANARY)
    plan.prepare(flat, [p.data_ptr() for p in want], stream)
    torch.cuda.synchronize()
    want_host = [p.cpu().numpy() for p in want]
    # which pool bytes the schedule writes (the rest is alignment padding)
    masks = [np.zeros(plan.pool_bytes(r) + 256, bool) for r in range(w.num_ranks)]
    for o, out in enumerate(w.outputs):
        for k in range(len(out.dst_ranks)):
            m_, n_ = w.dst_shape(o, k)
            data = m_ * n_ * (1 if out.fp8 else 2)
            scales = 4 * (-(-m_ // 128)) * (-(-n_ // 128)) if out.fp8 else 0
            rank, doff, soff = plan.output_layout(o, k)
            masks[rank][doff:doff + data] = True
            masks[rank][soff:soff + scales] = True
    desc = wt.PlanDesc(w)
    for call in range(2):
        # a different fill each call: every scheduled byte must be rewritten,
        # and nothing else may be touched
        fill = CANARY if call == 0 else 0x5A
        got = _pools(plan, w.num_ranks, fill)
        wt.wt_prepare_noalloc(desc, flat, [p.data_ptr() for p in got], stream)
        torch.cuda.synchronize()
        for r in range(w.num_ranks):
            g = got[r].cpu().numpy()
            assert np.array_equal(g[masks[r]], want_host[r][masks[r]]), (call, r)
            assert np.all(g[~masks[r]] == fill), (call, r)
    plan.close()


def test_noalloc_rejects_schedules_beyond_its_array():
    w = kimi_k2_moe_layer()          # about a million blocks: 33 MB of tables
    with pytest.raises(wt.WTError) as ei:
        wt.wt_prepare_noalloc(wt.PlanDesc(w), [], [0] * w.num_ranks)
    assert ei.value.name == "WT_ERR_INVALID_ARGUMENT"
    assert "at most" in str(ei.value)


@pytest.mark.parametrize("halo", [False, True])
def test_noalloc_runs_shard_local_plans(halo):
    from workloads import halo_mix, shard_local_mix
    w = halo_mix() if halo else shard_local_mix()
    shards = make_shards(w, device="cuda:0")
    flat = [s.data_ptr() if s.numel() else 0 for per in shards for s in per]
    stream = torch.cuda.current_stream().cuda_stream
    for s in range(4):
        plan = wt.Plan(w, device=0, local_shard=s, halo=halo)
        want = _pools(plan, w.num_ranks, CANARY)
        plan.prepare(flat, [p.data_ptr() for p in want], stream)
        got = _pools(plan, w.num_ranks, CANARY)
        wt.wt_prepare_noalloc(wt.PlanDesc(w, local_shard=s, halo=halo), flat,
                              [p.data_ptr() for p in got], stream)
        torch.cuda.synchronize()
        for r in range(w.num_ranks):
            assert torch.equal(got[r], want[r]), (s, r)
        plan.close()


def test_noalloc_reports_a_wait_that_gave_up_then_recovers():
    """A kernel wait that runs out (one unit's stage left unfilled on the
    host's request, 50 ms wait limit) is kept outside the uploaded tables and
    reported by wt_noalloc_check, even after a later call; the check clears
    it and the next step is complete again."""
    w = tiny_dense()
    shards = make_shards(w, device="cuda:0")
    flat = [s.data_ptr() for per in shards for s in per]
    stream = torch.cuda.current_stream().cuda_stream
    plan = wt.Plan(w, device=0)
    want = _pools(plan, w.num_ranks, CANARY)
    plan.prepare(flat, [p.data_ptr() for p in want], stream)
    desc = wt.PlanDesc(w)
    got = _pools(plan, w.num_ranks, CANARY)
    wt.wt_noalloc_check(stream)                  # nothing recorded before
    try:
        wt.wt_debug_noalloc_stall_unit(3, 50_000_000)
        wt.wt_prepare_noalloc(desc, flat, [p.data_ptr() for p in got], stream)
    finally:
        wt.wt_debug_noalloc_stall_unit(-1, 0)
    # a second, normal call in between does not wipe the record
    wt.wt_prepare_noalloc(desc, flat, [p.data_ptr() for p in got], stream)
    with pytest.raises(wt.WTError) as ei:
        wt.wt_noalloc_check(stream)
    assert ei.value.name == "WT_ERR_TIMEOUT"
    wt.wt_noalloc_check(stream)                  # cleared by the report
    for p in got:
        p.fill_(CANARY)
    wt.wt_prepare_noalloc(desc, flat, [p.data_ptr() for p in got], stream)
    wt.wt_noalloc_check(stream)
    for r in range(w.num_ranks):
        assert torch.equal(got[r], want[r]), r
    plan.close()


def test_noalloc_refuses_stream_capture():
    """The call uploads a host image that lives only for the call, so a
    captured copy would read freed memory at replay: it is refused."""
    w = tiny_dense()
    shards = make_shards(w, device="cuda:0")
    flat = [s.data_ptr() for per in shards for s in per]
    plan = wt.Plan(w, device=0, pool_capacity=None)
    pools = _pools(plan, w.num_ranks, CANARY)
    plan.close()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        wt.wt_prepare_noalloc(wt.PlanDesc(w), flat, [p.data_ptr() for p in pools], stream.cuda_stream)
    stream.synchronize()
    with pytest.raises(wt.WTError) as ei:
        with torch.cuda.graph(torch.cuda.CUDAGraph(), stream=stream):
            pools[0].add_(0)
            wt.wt_prepare_noalloc(wt.PlanDesc(w), flat, [p.data_ptr() for p in pools],
                                  stream.cuda_stream)
    assert ei.value.name == "WT_ERR_INVALID_ARGUMENT"
    assert "captured" in str(ei.value)
    torch.cuda.synchronize()


def test_noalloc_takes_no_device_memory():
    """After a first call on the device (which loads the library's module
    and its fixed array), further calls -- including a larger schedule --
    leave the device's free memory unchanged: nothing is allocated."""
    ws = [tiny_dense(), kimi_k2_moe_layer(40)]
    bufs = []
    for w in ws:
        shards = make_shards(w, device="cuda:0")
        flat = [s.data_ptr() for per in shards for s in per]
        plan = wt.Plan(w, device=-1)
        pools = _pools(plan, w.num_ranks, CANARY)
        plan.close()
        bufs.append((w, shards, flat, pools, wt.PlanDesc(w)))
    stream = torch.cuda.current_stream().cuda_stream
    w, _, flat, pools, desc = bufs[0]
    wt.wt_prepare_noalloc(desc, flat, [p.data_ptr() for p in pools], stream)
    wt.wt_noalloc_check(stream)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info(0)[0]
    for _ in range(3):
        for w, _, flat, pools, desc in reversed(bufs):
            wt.wt_prepare_noalloc(desc, flat, [p.data_ptr() for p in pools], stream)
        wt.wt_noalloc_check(stream)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(0)[0] == free0


def test_noalloc_calls_from_two_host_threads_on_one_stream():
    """Two host threads queue calls onto one stream at the same time (ctypes
    releases the interpreter lock during the call): the library keeps each
    call's table upload and kernel adjacent, so every call's pools hold the
    bytes wt_prepare writes."""
    import threading
    w = tiny_dense()
    shards = make_shards(w, device="cuda:0")
    flat = [s.data_ptr() for per in shards for s in per]
    stream = torch.cuda.current_stream().cuda_stream
    plan = wt.Plan(w, device=0)
    want = _pools(plan, w.num_ranks, CANARY)
    plan.prepare(flat, [p.data_ptr() for p in want], stream)
    torch.cuda.synchronize()
    desc = wt.PlanDesc(w)
    per_thread = [[_pools(plan, w.num_ranks, CANARY) for _ in range(12)] for _ in range(2)]
    errors = []

    def run(sets):
        try:
            for pools in sets:
                wt.wt_prepare_noalloc(desc, flat, [p.data_ptr() for p in pools], stream)
        except Exception as e:                 # reported below, in the test's thread
            errors.append(e)

    threads = [threading.Thread(target=run, args=(sets,)) for sets in per_thread]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    wt.wt_noalloc_check(stream)
    torch.cuda.synchronize()
    for sets in per_thread:
        for pools in sets:
            for r in range(w.num_ranks):
                assert torch.equal(pools[r], want[r]), r
    plan.close()


def test_noalloc_equals_the_oracle(oracle_mod):
    """The no-alloc call's pools against the CPU oracle directly (every
    scheduled byte; padding left untouched)."""
    from gpu_helpers import assert_pools_equal, oracle_pools
    w = _small_shapes()
    shards = make_shards(w, device="cuda:0")
    flat = [s.data_ptr() if s.numel() else 0 for per in shards for s in per]
    plan = wt.Plan(w, device=-1)
    pools = _pools(plan, w.num_ranks, CANARY)
    plan.close()
    wt.wt_prepare_noalloc(wt.PlanDesc(w), flat, [p.data_ptr() for p in pools],
                          torch.cuda.current_stream().cuda_stream)
    wt.wt_noalloc_check(torch.cuda.current_stream().cuda_stream)
    assert_pools_equal(pools, oracle_pools(oracle_mod, w, shards))
