"""Descriptor fuzzing on the host: random workloads with one random defect
each (bad shapes, shard splits that do not add up, out-of-range or reused
parts, unknown formats, ranks out of range, misaligned or colliding
explicit offsets, broken slices, empty lists) go to wt_plan_create. Every
call must come back with a status -- WT_OK only when the defect happened
to leave a valid descriptor, then with the oracle's layout -- and never
crash; the library keeps working afterwards."""
import ctypes
import dataclasses
import random

import pytest

import bf16_fp8_parameter_wt_b300 as wt
from workloads import Output, Param, random_workload

STATUSES = {"WT_OK", "WT_ERR_INVALID_ARGUMENT", "WT_ERR_SHAPE", "WT_ERR_LAYOUT_OVERLAP",
            "WT_ERR_POOL_TOO_SMALL", "WT_ERR_ALIGNMENT"}


def _mutate(w, rng):
    params, outs = list(w.params), list(w.outputs)
    kind = rng.randrange(12)
    i = rng.randrange(len(params))
    o = rng.randrange(len(outs))
    p, out = params[i], outs[o]
    if kind == 0:                                   # rows that the shards do not add up to
        params[i] = dataclasses.replace(p, rows=p.rows + rng.choice([-1, 1, 128]))
    elif kind == 1:                                 # a negative shard
        sr = list(p.shard_rows)
        sr[0] = -1 - rng.randrange(5)
        params[i] = dataclasses.replace(p, shard_rows=tuple(sr))
    elif kind == 2:                                 # zero or negative columns
        params[i] = dataclasses.replace(p, cols=rng.choice([0, -7]))
    elif kind == 3:                                 # a part index out of range
        outs[o] = dataclasses.replace(out, parts=out.parts + (len(params) + rng.randrange(3),))
    elif kind == 4:                                 # a parameter used twice
        outs[o] = dataclasses.replace(out, parts=out.parts + (out.parts[0],))
    elif kind == 5:                                 # a rank out of range
        outs[o] = dataclasses.replace(out, dst_ranks=out.dst_ranks[:-1] + (w.num_ranks + rng.randrange(3),))
    elif kind == 6:                                 # no destinations
        outs[o] = dataclasses.replace(out, dst_ranks=(), slices=None)
    elif kind == 7:                                 # a misaligned explicit data offset
        outs[o] = dataclasses.replace(out, data_off=tuple(8 + 16 * rng.randrange(100) for _ in out.dst_ranks))
    elif kind == 8:                                 # two outputs at the same explicit offset on one rank
        outs[o] = dataclasses.replace(out, dst_ranks=(0,) * len(out.dst_ranks),
                                      data_off=(0,) * len(out.dst_ranks), slices=None)
    elif kind == 9:                                 # a slice range off the 128 grid
        m, n = w.output_shape(o)
        outs[o] = dataclasses.replace(out, slices=tuple((rng.randint(0, 1), ((1 + rng.randrange(100), 64),))
                                                        for _ in out.dst_ranks))
    elif kind == 10:                                # a slice past the tensor's end
        m, n = w.output_shape(o)
        outs[o] = dataclasses.replace(out, slices=tuple((0, ((0, m + 128),)) for _ in out.dst_ranks))
    else:                                           # an output with no parts
        outs[o] = dataclasses.replace(out, parts=())
    return dataclasses.replace(w, params=params, outputs=outs), kind


def _create(w):
    d = wt.PlanDesc(w)
    h = ctypes.c_void_p()
    st = wt.lib().wt_plan_create(ctypes.byref(d.c), -1, ctypes.byref(h))
    return wt.wt_status_string(st), h.value


@pytest.mark.parametrize("seed", range(300))
def test_random_defects_return_a_status(oracle_mod, seed):
    rng = random.Random(10_000 + seed)
    w, kind = _mutate(random_workload(seed % 120), rng)
    name, h = _create(w)
    assert name in STATUSES, (kind, name)
    if name == "WT_OK":
        # a defect that left a valid descriptor: the plan is the oracle's
        d, s, pools = oracle_mod.Model(w).layout()
        assert [wt.wt_plan_pool_bytes(h, r) for r in range(w.num_ranks)] == pools
        wt.wt_plan_destroy(h)
    else:
        assert h is None
        assert wt.wt_last_error()                      # a message says why
    assert kind not in (0, 1, 2, 3, 4, 5, 6, 11) or name != "WT_OK", kind


def test_library_still_works_after_the_fuzzing():
    name, h = _create(random_workload(3))
    assert name == "WT_OK"
    wt.wt_plan_destroy(h)
