"""GPU parity: wt_prepare's destination pools equal the CPU oracle's byte for
byte (FP8 codes, fp32 scales, BF16 pass-through, untouched padding) on the
seeded workloads, and on every (block amax, element) pair of BF16 values."""
import numpy as np
import pytest
import torch

import bf16_fp8_parameter_wt_b300 as wt
from gpu_helpers import (CANARY, assert_pools_equal, device_pools, full_check, ncores,
                         oracle_pools, run_gpu)
from workloads import (Output, Param, ValueRecipe, Workload, edge_stress, llama_dense,
                       llama_dense_tp4, make_shards, tiny_dense, tp_slices_small)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from bf16_fp8_parameter_wt_b300 import build
    build.build()
    assert torch.cuda.is_available()


def test_tiny_dense(oracle_mod):
    full_check(oracle_mod, tiny_dense())


def test_tiny_dense_narrow_path_and_debug_checks(oracle_mod):
    w = tiny_dense()
    shards = make_shards(w, device="cuda:0")
    want = oracle_pools(oracle_mod, w, shards)
    for flags in (wt.WT_FLAG_FORCE_NARROW, wt.WT_FLAG_DEBUG_CHECKS,
                  wt.WT_FLAG_FORCE_NARROW | wt.WT_FLAG_DEBUG_CHECKS):
        plan, pools = run_gpu(w, shards, flags=flags)
        plan.check()
        assert_pools_equal(pools, want)
        plan.close()


def test_llama_dense_full(oracle_mod):
    full_check(oracle_mod, llama_dense())


def test_edge_stress_full(oracle_mod):
    full_check(oracle_mod, edge_stress())


def test_tensor_parallel_slices_small(oracle_mod):
    """Row and column slices, in and out of order, ending at the edge,
    mixed with whole-tensor destinations and replicas; through the single-
    destination fast path, the general path, the element path and the
    debug-checked kernel."""
    w = tp_slices_small()
    shards = make_shards(w, device="cuda:0")
    want = oracle_pools(oracle_mod, w, shards)
    for flags in (0, wt.WT_FLAG_FORCE_NARROW, wt.WT_FLAG_DEBUG_CHECKS):
        plan, pools = run_gpu(w, shards, flags=flags)
        plan.check()
        assert_pools_equal(pools, want)
        plan.close()


def test_llama_dense_tp4_full(oracle_mod):
    """The Llama-style stack laid out for 4-way tensor parallelism: every
    Linear layer sliced per rank, norms replicated."""
    full_check(oracle_mod, llama_dense_tp4())


def test_small_shapes_and_special_values(oracle_mod):
    """1x1, 3x5, 129x130 fused, 256x1, shards of 0 and 1 rows, -0.0 blocks,
    subnormal scales, outliers, replicated destinations on two ranks; 64-column
    outputs narrower than one block (FP8 from two shards, BF16 from one) and a
    fused BF16 output whose partial blocks span three shards."""
    params = [Param("a", 1, 1, (1,)), Param("b", 3, 5, (2, 0, 1)),
              Param("c1", 50, 130, (17, 33)), Param("c2", 79, 130, (1, 0, 40, 38)),
              Param("d", 256, 1, (100, 100, 56)), Param("e", 300, 264, (1,) * 44 + (256,)),
              Param("negzero", 130, 136, (130,)), Param("tiny", 128, 128, (128,)),
              Param("f", 40, 64, (17, 23)), Param("g", 200, 64, (200,)),
              Param("h1", 70, 72, (70,)), Param("h2", 90, 72, (0, 45, 45))]
    outs = [Output("a", (0,), True, (0,)), Output("b", (1,), True, (1, 0)),
            Output("c", (2, 3), True, (1,)), Output("d", (4,), False, (0, 1)),
            Output("e", (5,), True, (0, 1)), Output("negzero", (6,), True, (0,)),
            Output("tiny", (7,), True, (1,)), Output("f", (8,), True, (0,)),
            Output("g", (9,), False, (1,)), Output("h", (10, 11), False, (0, 1))]
    w = Workload("small", params, outs, 2, ValueRecipe("student_t3", 0.02, 77))
    shards = make_shards(w, device="cuda:0")
    shards[6] = [torch.full((130, 136), -0.0, dtype=torch.bfloat16, device="cuda:0")]
    shards[7] = [(torch.randn(128, 128, device="cuda:0") * 1e-39).to(torch.bfloat16)]
    shards[2][0][3, 7] = 29952.0
    plan, pools = run_gpu(w, shards)
    assert_pools_equal(pools, oracle_pools(oracle_mod, w, shards))
    plan.close()


def test_pointer_tables_follow_new_buffers(oracle_mod):
    w = tiny_dense()
    shards = make_shards(w, device="cuda:0")
    want = oracle_pools(oracle_mod, w, shards)
    plan = wt.Plan(w, device=0)
    pools_a = device_pools(plan, w.num_ranks)
    pools_b = device_pools(plan, w.num_ranks)
    run_gpu(w, shards, pools=pools_a, plan=plan)
    # new shard buffers holding the same values, new pools
    shards2 = [[s.clone() for s in per] for per in shards]
    run_gpu(w, shards2, pools=pools_b, plan=plan)
    assert_pools_equal(pools_a, want)
    assert_pools_equal(pools_b, want)
    # repeat into the first pools after zeroing them: same bytes again
    for p in pools_a:
        p.fill_(CANARY)
    run_gpu(w, shards2, pools=pools_a, plan=plan)
    assert_pools_equal(pools_a, want)
    plan.close()


def _exhaustive_workload():
    """One output per group of amax values; each 128x128 block holds one
    amax a (placed first) followed by every BF16 pattern x with |x| <= a,
    both signs, padded with a."""
    groups = 16
    amaxes = np.arange(1, 0x7F80, dtype=np.int64)         # every positive finite bf16
    split = np.array_split(amaxes, groups)
    blocks = []
    for g in split:
        tiles = []
        for a in g.tolist():
            vals = np.concatenate([np.arange(0, a + 1), np.arange(0x8000, 0x8000 + a + 1)])
            per = 128 * 128 - 1
            n = -(-vals.size // per)
            buf = np.full(n * per, a, dtype=np.int64)
            buf[:vals.size] = vals
            buf = buf.reshape(n, per)
            tiles.append(np.concatenate([np.full((n, 1), a, np.int64), buf], axis=1))
        blocks.append(np.concatenate(tiles).astype(np.uint16))
    params, outs = [], []
    for i, b in enumerate(blocks):
        rows = b.shape[0] * 128
        params.append(Param(f"g{i}", rows, 128, (rows,)))
        outs.append(Output(f"g{i}", (i,), True, (i % 4,)))
    w = Workload("exhaustive_pairs", params, outs, 4)
    return w, blocks


def test_every_amax_element_pair_bit_exact(oracle_mod):
    """Each code depends only on (block amax, element); this covers every
    pair of positive finite BF16 amax and BF16 element |x| <= amax, so it
    covers every input the FP8 path can ever see."""
    w, blocks = _exhaustive_workload()
    host = [[np.ascontiguousarray(b.reshape(-1, 128))] for b in blocks]
    shards = [[torch.from_numpy(h[0].view(np.int16)).view(torch.bfloat16).to("cuda:0")]
              for h in host]
    plan, pools = run_gpu(w, shards)
    want = oracle_mod.Model(w).prepare([h[0] for h in host], nthreads=ncores(), fill=CANARY)
    assert_pools_equal(pools, want)
    plan.close()


def test_captured_step_replays_from_a_cuda_graph(oracle_mod):
    """A wt_prepare captured into a CUDA graph (after an uncaptured call has
    staged the same pointers) writes the same bytes on every replay; new
    pointers inside a capture are refused."""
    w = tiny_dense()
    shards = make_shards(w, device="cuda:0")
    want = oracle_pools(oracle_mod, w, shards)
    plan = wt.Plan(w, device=0)
    pools = device_pools(plan, w.num_ranks)
    stream = torch.cuda.Stream()
    shard_arr, pool_arr = plan.bind([s.data_ptr() for per in shards for s in per],
                                    [p.data_ptr() for p in pools])
    plan.prepare(shard_arr, pool_arr, stream.cuda_stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        plan.prepare(shard_arr, pool_arr, stream.cuda_stream)
    for _ in range(2):
        for p in pools:
            p.fill_(CANARY)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert_pools_equal(pools, want)
    other = device_pools(plan, w.num_ranks)
    with pytest.raises(wt.WTError) as ei:
        with torch.cuda.graph(torch.cuda.CUDAGraph(), stream=stream):
            other[0].add_(0)
            plan.prepare(shard_arr, [p.data_ptr() for p in other], stream.cuda_stream)
    assert ei.value.name == "WT_ERR_INVALID_ARGUMENT"
    torch.cuda.synchronize()
    plan.close()


def test_all_zero_plan_and_misuse_errors():
    w = Workload("empty", [], [], 2)
    plan = wt.Plan(w, device=0)
    plan.prepare([], [0, 0], torch.cuda.current_stream().cuda_stream)
    plan.close()
    w = tiny_dense()
    shards = make_shards(w, device="cuda:0")
    plan = wt.Plan(w, device=0)
    pools = device_pools(plan, w.num_ranks)
    flat = [s.data_ptr() for per in shards for s in per]
    bad = list(flat)
    bad[1] += 2                                      # breaks 16-byte alignment
    with pytest.raises(wt.WTError) as ei:
        plan.prepare(bad, [p.data_ptr() for p in pools])
    assert ei.value.name == "WT_ERR_ALIGNMENT"
    with pytest.raises(wt.WTError) as ei:
        plan.prepare(flat, [pools[0].data_ptr(), 0])
    assert ei.value.name == "WT_ERR_INVALID_ARGUMENT"
    with pytest.raises(wt.WTError) as ei:
        plan.prepare(flat, [pools[0].data_ptr() + 4, pools[1].data_ptr()])
    assert ei.value.name == "WT_ERR_ALIGNMENT"
    # the plan is still usable after refusals
    plan.prepare(flat, [p.data_ptr() for p in pools])
    torch.cuda.synchronize()
    plan.close()


def test_unaligned_rows_view_maps_and_fallbacks(oracle_mod):
    """Rows that are not 16-byte aligned: N = 2050, 2052, 2049 and 141 (view
    rows of 4, 2, 8 and 8 shard rows), shards whose row counts leave a
    partial view row at the end, a 9-column output too narrow for a view
    map, blocks spanning shards; then the same shards copied to addresses 2
    bytes past a 16-byte boundary, which must take the row-by-row path."""
    params = [Param("a", 700, 2050, (301, 399)), Param("b", 390, 2052, (390,)),
              Param("c", 260, 2049, (130, 130)), Param("d", 300, 141, (300,)),
              Param("e", 140, 9, (140,))]
    outs = [Output("a", (0,), True, (0,)), Output("b", (1,), True, (1,)),
            Output("c", (2,), False, (0,)), Output("d", (3,), True, (1,)),
            Output("e", (4,), True, (0,))]
    w = Workload("views", params, outs, 2, ValueRecipe("student_t3", 0.02, 91, zero_tile_eighths=1,
                                                       outlier_tile_eighths=1, outlier=3.0e4))
    shards = make_shards(w, device="cuda:0")
    want = oracle_pools(oracle_mod, w, shards)
    plan, pools = run_gpu(w, shards)
    plan.check()
    assert_pools_equal(pools, want)
    plan.close()
    # the same values at addresses 2 bytes past a 16-byte boundary
    keep = []
    moved = []
    for per in shards:
        row = []
        for s in per:
            buf = torch.empty(s.numel() + 16, dtype=torch.bfloat16, device="cuda:0")
            t = buf[1:1 + s.numel()].view(s.shape)
            t.copy_(s)
            assert t.data_ptr() % 16 == 2
            keep.append(buf)
            row.append(t)
        moved.append(row)
    plan, pools = run_gpu(w, moved)
    plan.check()
    assert_pools_equal(pools, want)
    plan.close()
