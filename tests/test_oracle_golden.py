"""The oracle still produces the frozen output of tests/golden/oracle_small.json."""
import hashlib
import json
import os

from golden.make_golden import small_case
from workloads import make_shards, shards_to_host_u16

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_matches_frozen_small_case(oracle_mod):
    with open(os.path.join(HERE, "golden", "oracle_small.json")) as f:
        doc = json.load(f)
    w = small_case()
    shards = shards_to_host_u16(make_shards(w))
    assert hashlib.sha256(b"".join(a.tobytes() for a in shards)).hexdigest() == doc["inputs_sha256"]
    m = oracle_mod.Model(w)
    d, s, pool_bytes = m.layout()
    assert d == doc["data_off"] and s == doc["scale_off"] and pool_bytes == doc["pool_bytes"]
    pools = m.prepare(shards, nthreads=2, fill=0)
    assert [p.tobytes().hex() for p in pools] == doc["pools_hex"]
