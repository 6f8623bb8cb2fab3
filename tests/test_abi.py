"""C-ABI tests that need no GPU: the library loads and exports every entry
point include/wt.h declares; host-only plans (device -1) compile the same
layout as the oracle; invalid descriptors return their status codes."""
import ctypes
import os
import re

import pytest

import bf16_fp8_parameter_wt_b300 as wt
from bf16_fp8_parameter_wt_b300 import build as wt_build
from workloads import (Output, Param, ValueRecipe, Workload, edge_stress, kimi_k2_moe_layer,
                       llama_dense, llama_dense_tp4, offload_layer, tiny_dense, tp_slices_small)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    wt_build.build()
    wt.lib()


def _declared():
    with open(os.path.join(ROOT, "include", "wt.h")) as f:
        src = f.read()
    return sorted(set(re.findall(r"^\s*(?:wt_status|const char\*)\s+(wt_\w+)\s*\(", src, re.M)))


def test_exports_every_declared_symbol():
    names = _declared()
    assert len(names) >= 12
    assert sorted(wt.EXPORTS) == names
    L = wt.lib()
    for n in names:
        assert hasattr(L, n), n


def test_status_strings():
    assert wt.wt_status_string(0) == "WT_OK"
    assert wt.wt_status_string(3) == "WT_ERR_LAYOUT_OVERLAP"


@pytest.mark.parametrize("make", [tiny_dense, llama_dense, kimi_k2_moe_layer, edge_stress,
                                  lambda: offload_layer(4), llama_dense_tp4, tp_slices_small])
def test_host_plan_layout_equals_oracle(oracle_mod, make):
    w = make()
    d, s, pools = oracle_mod.Model(w).layout()
    with wt.Plan(w, device=-1) as p:
        for r in range(w.num_ranks):
            assert p.pool_bytes(r) == pools[r]
        for o, out in enumerate(w.outputs):
            for k, rank in enumerate(out.dst_ranks):
                rr, dd, ss = p.output_layout(o, k)
                assert rr == rank and dd == d[o][k]
                if out.fp8:
                    assert ss == s[o][k]
        st = p.stats
        assert st["bytes_read"] == w.bytes_read
        assert st["bytes_written"] == w.bytes_written
        assert st["num_units"] == w.num_tiles
        assert st["num_params_total"] == w.num_params_total


def test_host_plan_explicit_offsets_equal_oracle(oracle_mod):
    params = [Param("a", 128, 256, (128,)), Param("b", 64, 64, (64,))]
    outs = [Output("a", (0,), True, (0, 1), data_off=(4096, None), scale_off=(0, None)),
            Output("b", (1,), False, (0, 0))]
    w = Workload("explicit", params, outs, 2)
    d, s, pools = oracle_mod.Model(w).layout()
    with wt.Plan(w, device=-1) as p:
        assert [p.pool_bytes(r) for r in range(2)] == pools
        assert [p.output_layout(0, k)[1:] for k in range(2)] == list(zip(d[0], s[0]))
        assert [p.output_layout(1, k)[1] for k in range(2)] == d[1]


def test_host_image_offsets_and_chunks():
    w = offload_layer(6)
    with wt.Plan(w, device=-1, offload_chunk_bytes=2 << 30) as p:
        offs = []
        for o in w.outputs:
            for q in o.parts:
                for k in range(len(w.params[q].shard_rows)):
                    offs.append((p.shard_host_offset(q, k), w.params[q].shard_rows[k] * w.params[q].cols * 2))
        for (a, n), (b, _) in zip(offs, offs[1:]):
            assert a % 256 == 0 and b >= a + n and b - (a + n) < 256
        st = p.stats
        assert st["host_bytes"] >= w.bytes_read and st["host_bytes"] % 256 == 0
        # qkv (308 MB) + o + 6 experts (88 MB each) fit in one 2 GiB chunk
        assert st["num_chunks"] == 1
    with wt.Plan(w, device=-1, offload_chunk_bytes=100 << 20) as p:
        # every output is a chunk of its own except pairs of expert downs that fit
        assert p.stats["num_chunks"] >= len(w.outputs) // 2


def _simple(**over):
    params = [Param("a", 256, 256, (128, 128)), Param("b", 256, 256, (256,))]
    outs = [Output("ab", (0, 1), True, (0,))]
    w = Workload("s", params, outs, 1, ValueRecipe())
    for k, v in over.items():
        setattr(w, k, v)
    return w


def _err(w, **kw):
    with pytest.raises(wt.WTError) as ei:
        wt.Plan(w, device=-1, **kw)
    return ei.value.name


def test_validation_errors():
    assert _err(Workload("x", [Param("a", 10, 8, (5, 4))], [Output("a", (0,), True, (0,))], 1)) == "WT_ERR_SHAPE"
    assert _err(Workload("x", [Param("a", 10, 8, (5, 5)), Param("b", 10, 16, (10,))],
                         [Output("ab", (0, 1), True, (0,))], 1)) == "WT_ERR_SHAPE"
    assert _err(Workload("x", [Param("a", 10, 8, (10,))], [Output("a", (0,), True, (1,))], 1)) == "WT_ERR_INVALID_ARGUMENT"
    assert _err(Workload("x", [Param("a", 10, 8, (10,))], [Output("a", (0,), True, (0,)),
                                                           Output("b", (0,), True, (0,))], 1)) == "WT_ERR_INVALID_ARGUMENT"
    assert _err(Workload("x", [Param("a", 10, 8, (10,)), Param("b", 10, 8, (10,))],
                         [Output("a", (0,), True, (0,))], 1)) == "WT_ERR_INVALID_ARGUMENT"
    assert _err(Workload("x", [Param("a", 0, 8, (0,))], [Output("a", (0,), True, (0,))], 1)) == "WT_ERR_SHAPE"
    # overlapping explicit ranges
    assert _err(Workload("x", [Param("a", 128, 128, (128,)), Param("b", 128, 128, (128,))],
                         [Output("a", (0,), False, (0,), data_off=(0,)),
                          Output("b", (1,), False, (0,), data_off=(1024,))], 1)) == "WT_ERR_LAYOUT_OVERLAP"
    # misaligned explicit offsets
    assert _err(Workload("x", [Param("a", 128, 128, (128,))],
                         [Output("a", (0,), True, (0,), data_off=(8,))], 1)) == "WT_ERR_ALIGNMENT"
    assert _err(Workload("x", [Param("a", 128, 128, (128,))],
                         [Output("a", (0,), True, (0,), scale_off=(2,))], 1)) == "WT_ERR_ALIGNMENT"
    # pool capacity
    assert _err(_simple(), pool_capacity=[1000]) == "WT_ERR_POOL_TOO_SMALL"
    with wt.Plan(_simple(), device=-1, pool_capacity=[512 * 256 + 256]) as p:
        assert p.pool_bytes(0) == 512 * 256 + 256


def test_empty_plan_and_empty_ranks():
    with wt.Plan(Workload("empty", [], [], 3), device=-1) as p:
        assert [p.pool_bytes(r) for r in range(3)] == [0, 0, 0]
        assert p.stats["num_units"] == 0
    with wt.Plan(edge_stress(), device=-1) as p:
        assert p.pool_bytes(3) == 0 and p.pool_bytes(4) == 0


def test_host_only_plan_refuses_to_run():
    with wt.Plan(_simple(), device=-1) as p:
        with pytest.raises(wt.WTError) as ei:
            p.prepare([0, 0, 0], [0])
        assert ei.value.name == "WT_ERR_INVALID_ARGUMENT"


def test_null_arguments():
    L = wt.lib()
    assert L.wt_plan_create(None, -1, None) == 1
    assert L.wt_plan_pool_bytes(None, 0, None) == 1
    assert L.wt_prepare(None, None, None, None, None) == 1
    assert L.wt_plan_destroy(None) == 0


def test_testing_hooks_validate_their_arguments():
    L = wt.lib()
    assert L.wt_debug_stall_unit(None, 0, 0) == 1
    assert L.wt_debug_fail_offload_chunk(None, 0) == 1
    with wt.Plan(_simple(), device=-1) as p:
        n = p.stats["num_units"]
        for bad in (-2, n):
            with pytest.raises(wt.WTError) as ei:
                wt.wt_debug_stall_unit(p.handle, bad, 0)
            assert ei.value.name == "WT_ERR_INVALID_ARGUMENT"
        wt.wt_debug_stall_unit(p.handle, n - 1, 1000)
        wt.wt_debug_stall_unit(p.handle, -1, 0)


@pytest.mark.parametrize("sl,status", [((0, ((64, 128),)), "WT_ERR_SHAPE"),
                                       ((0, ((0, 100), (128, 128))), "WT_ERR_SHAPE"),
                                       ((0, ((0, 256), (128, 128))), "WT_ERR_SHAPE"),
                                       ((0, ((256, 128),)), "WT_ERR_SHAPE"),
                                       ((1, ((0, 200),)), "WT_ERR_SHAPE"),
                                       ((2, ((0, 128),)), "WT_ERR_INVALID_ARGUMENT"),
                                       ((0, ((0, 0),)), "WT_ERR_SHAPE")])
def test_invalid_slices_are_rejected(sl, status):
    w = Workload("bad", [Param("p", 300, 260, (300,))],
                 [Output("p", (0,), True, (0,), slices=(sl,))], 1)
    with pytest.raises(wt.WTError) as ei:
        wt.Plan(w, device=-1)
    assert ei.value.name == status


def test_tensor_parallel_blocks_have_one_destination():
    """Every block of a sliced Linear layer of the TP stack goes to exactly
    one rank: the pool sizes add up to the unsliced tensors once, plus the
    replicated norms."""
    w = llama_dense_tp4()
    with wt.Plan(w, device=-1) as p:
        assert p.stats["bytes_written"] == w.bytes_written
    one = llama_dense()
    norms = sum(2 * 4096 for o in one.outputs if o.name.endswith("norm"))
    assert w.bytes_written == one.bytes_written + 3 * norms


def test_token_codec_validates_arguments_before_touching_a_device():
    L = wt.lib()
    assert L.wt_quantize_tokens(None, -1, 128, 128, None, None, None, None) == 1
    assert L.wt_quantize_tokens(None, 4, 0, 128, None, None, None, None) == 1
    assert L.wt_quantize_tokens(None, 4, 256, 128, None, None, None, None) == 1     # ld < hidden
    assert L.wt_quantize_tokens(None, 4, 128, 128, None, None, None, None) == 1     # NULL buffers
    assert L.wt_quantize_tokens(None, 0, 128, 128, None, None, None, None) == 0     # nothing to do
    assert L.wt_quantize_tokens(2, 1 << 25, 1 << 13, 1 << 13, 16, 16, None, None) == 1  # > 2^31 groups
    align = wt.lib().wt_status_string
    assert align(L.wt_quantize_tokens(2, 4, 128, 128, 16, 16, 6, None)) == b"WT_ERR_ALIGNMENT"  # ticket
    # the testing hook of the codec's bounded waits: -1 (off) and groups >= 0
    # are accepted, anything below -1 refused, all without a device
    assert L.wt_debug_tokens_stall_group(-2, 0) == 1
    assert L.wt_debug_tokens_stall_group(5, 1000) == 0
    assert L.wt_debug_tokens_stall_group(-1, 0) == 0


@pytest.mark.parametrize("make", [tiny_dense, llama_dense_tp4, tp_slices_small,
                                  lambda: kimi_k2_moe_layer(12)])
def test_expected_counts_equal_oracle(oracle_mod, make):
    w = make()
    m = oracle_mod.Model(w)
    with wt.Plan(w, device=-1) as p:
        assert [p.expected_count(r) for r in range(w.num_ranks)] == \
               [m.expected_blocks(r) for r in range(w.num_ranks)]


def test_counter_calls_validate_arguments():
    L = wt.lib()
    assert L.wt_plan_set_counters(None, None, 0) == 1
    with wt.Plan(_simple(), device=-1) as p:
        with pytest.raises(wt.WTError):
            p.set_counters(256)                    # host-only plan
        p.set_counters(0)                          # turning counting off is always fine
        with pytest.raises(wt.WTError):
            p.set_counters(0, 7)                   # unknown mode
        with pytest.raises(wt.WTError):
            p.expected_count(5)
    t = (ctypes.c_uint32 * 1)(0)
    assert L.wt_wait_counters(None, 1001, t, 0, None, None) == 1
    assert L.wt_wait_counters(None, 1, t, 0, None, None) == 1
    assert L.wt_wait_counters(16, 1, None, 0, 16, None) == 1
    assert L.wt_wait_counters(18, 1, t, 0, 16, None) == 5         # misaligned counters


def test_plan_owns_a_copy_of_its_descriptor(oracle_mod):
    """wt_plan_create deep-copies the descriptor: after every array the
    descriptor points to has been overwritten and freed, the plan's layout,
    stats and errors are unchanged."""
    import gc
    w = llama_dense_tp4()
    d, s, pools = oracle_mod.Model(w).layout()
    desc = wt.PlanDesc(w)
    h = wt.wt_plan_create(desc, -1)
    try:
        keep, params, outs = desc._keep
        for arr in keep:
            if isinstance(arr, ctypes.Array):
                ctypes.memset(arr, 0xFF, ctypes.sizeof(arr))
        ctypes.memset(params, 0xFF, ctypes.sizeof(params))
        ctypes.memset(outs, 0xFF, ctypes.sizeof(outs))
        del keep, params, outs, desc
        gc.collect()
        for r in range(w.num_ranks):
            assert wt.wt_plan_pool_bytes(h, r) == pools[r]
        for o, out in enumerate(w.outputs):
            for k in range(len(out.dst_ranks)):
                rr, dd, ss = wt.wt_plan_output_layout(h, o, k)
                assert (rr, dd) == (out.dst_ranks[k], d[o][k])
                if out.fp8:
                    assert ss == s[o][k]
        st = wt.wt_plan_get_stats(h)
        assert st["bytes_read"] == w.bytes_read and st["bytes_written"] == w.bytes_written
    finally:
        wt.wt_plan_destroy(h)
