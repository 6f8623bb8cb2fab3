"""Write tests/golden/oracle_small.json from the CPU oracle alone.

No page prints a worked example of the quantisation, so this fixture is not
the pages' numbers: it freezes the oracle's output on one small seeded case
(a fused 3-part output with uneven shards, a ragged 130x129 edge, a
BF16 pass-through norm, two ranks) so that any later change to the oracle's
arithmetic shows up as a failing test and has to be justified.

Run from the repository root:  python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from workloads import Output, Param, ValueRecipe, Workload, make_shards, shards_to_host_u16  # noqa: E402


def small_case() -> Workload:
    params = [Param("q", 64, 129, (30, 34)), Param("k", 33, 129, (33, 0)),
              Param("v", 33, 129, (1, 32)), Param("norm", 129, 1, (43, 43, 43)),
              Param("w", 3, 5, (2, 1))]
    outs = [Output("qkv", (0, 1, 2), True, (0,)), Output("norm", (3,), False, (1,)),
            Output("w", (4,), True, (1, 0))]
    return Workload("golden_small", params, outs, 2,
                    ValueRecipe("student_t3", 0.02, 4242, zero_tile_eighths=0))


def main():
    w = small_case()
    shards = shards_to_host_u16(make_shards(w))
    m = oracle.Model(w)
    d, s, pool_bytes = m.layout()
    pools = m.prepare(shards, nthreads=1, fill=0)
    doc = {
        "what": "CPU oracle output on a small seeded case (regression pin of the oracle)",
        "inputs_sha256": hashlib.sha256(b"".join(a.tobytes() for a in shards)).hexdigest(),
        "data_off": d, "scale_off": s, "pool_bytes": pool_bytes,
        "pools_hex": [p.tobytes().hex() for p in pools],
    }
    with open(os.path.join(HERE, "oracle_small.json"), "w") as f:
        json.dump(doc, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
