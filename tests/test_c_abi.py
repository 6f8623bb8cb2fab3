"""The C ABI from plain C: tests/c/plan_host.c is compiled with gcc against
include/wt.h and linked to libwt.so, and builds host-only plans (no GPU,
no Python in the caller). What it prints is checked against the oracle's
layout and per-rank counts and against the shard bookkeeping of
tests/shard_helpers.py, for the full plan and for both shard-local plans
with halos; the strict shard-local plan is refused."""
import os
import subprocess

import pytest

import bf16_fp8_parameter_wt_b300 as wt
from shard_helpers import halo_rows_needed, local_counts
from workloads import Output, Param, Workload

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _workload():
    """The model plan_host.c describes, as a workload."""
    params = [Param("q", 256, 256, (128, 128)), Param("k", 128, 256, (64, 64)),
              Param("v", 128, 256, (64, 64)), Param("gate", 512, 256, (256, 256)),
              Param("up", 512, 256, (256, 256)), Param("norm", 256, 1, (200, 56))]
    outs = [Output("qkv", (0, 1, 2), True, (0, 1)),
            Output("gate_up", (3, 4), True, (0, 1), slices=((0, ((0, 512),)), (0, ((512, 512),)))),
            Output("norm", (5,), False, (1,))]
    return Workload("c_example", params, outs, 2)


@pytest.fixture(scope="module")
def printed(tmp_path_factory):
    wt.lib()                                   # the library exists (built by the session)
    exe = str(tmp_path_factory.mktemp("c") / "plan_host")
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(HERE, "c", "plan_host.c"), wt.LIB_PATH,
                    "-Wl,-rpath," + os.path.dirname(wt.LIB_PATH), "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    out = {}
    for line in r.stdout.splitlines():
        k, _, v = line.partition(" ")
        out[k] = v
    return out


def test_full_plan_from_c_equals_oracle(printed, oracle_mod):
    w = _workload()
    m = oracle_mod.Model(w)
    d, s, pools = m.layout()
    assert [int(printed[f"full.pool{r}"]) for r in range(2)] == pools
    assert [int(printed[f"full.count{r}"]) for r in range(2)] == [m.expected_blocks(r) for r in range(2)]
    for o, out in enumerate(w.outputs):
        for k, rank in enumerate(out.dst_ranks):
            r, doff, soff = map(int, printed[f"full.layout{o}.{k}"].split())
            assert (r, doff) == (rank, d[o][k]) and (not out.fp8 or soff == s[o][k])
    assert int(printed["full.bytes_read"]) == w.bytes_read
    assert int(printed["full.bytes_written"]) == w.bytes_written
    assert int(printed["full.slots"]) == 12
    assert printed["full.prepare"] == "WT_ERR_INVALID_ARGUMENT"


def test_halo_plans_from_c(printed):
    w = _workload()
    units = 0
    for s in range(2):
        n_units, elems, written, per_rank = local_counts(w, s, halo=True)
        assert int(printed[f"halo{s}.units"]) == n_units
        assert int(printed[f"halo{s}.bytes_written"]) == written
        assert [int(printed[f"halo{s}.count{r}"]) for r in range(2)] == per_rank
        need = halo_rows_needed(w, s)
        for i, par in enumerate(w.params):
            for k, n in enumerate(par.shard_rows):
                assert int(printed[f"halo{s}.read{i}.{k}"]) == (n if k == s else need.get((i, k), 0))
        units += n_units
    assert units == int(printed["full.units"])
    # block rows 2 and 3 of qkv and row 1 of the norm start in shard 0 and
    # run into shard 1: 64 rows of k, 64 of v and 56 of the norm
    assert (printed["halo0.read1.1"], printed["halo0.read2.1"], printed["halo0.read5.1"]) == ("64", "64", "56")


def test_errors_from_c(printed):
    assert printed["null"] == "WT_ERR_INVALID_ARGUMENT"
    assert printed["error"].startswith("wt_plan_create(&d, -1, &p) WT_ERR_SHAPE")
