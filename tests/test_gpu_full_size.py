"""Full-size parity: every byte of every pool, at the full sizes of the
Kimi-K2-shaped MoE layer (770 outputs, 17 GB of pools, in the launch
configuration the benchmark times) and of one whole layer of the streamed
offload stack (772 outputs through wt_prepare_offload with 2 GiB chunks),
equals the CPU oracle's.

The oracle runs output by output on host copies of the shards (its
prepare_output, one output per thread; ctypes releases the GIL), a batch of
outputs at a time so that host memory holds one batch of source copies.
Every scheduled byte is compared, and every byte between scheduled ranges
and in the guard band after each pool is checked to hold the canary.
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import bf16_fp8_parameter_wt_b300 as wt
from gpu_helpers import CANARY, device_pools, ncores, run_gpu
from workloads import kimi_k2_moe_layer, make_shards, offload_layer

pytestmark = pytest.mark.gpu

GiB = 1 << 30


@pytest.fixture(scope="module", autouse=True)
def built():
    from bf16_fp8_parameter_wt_b300 import build
    build.build()
    assert torch.cuda.is_available()


def _slot_base(w):
    return np.cumsum([0] + [len(p.shard_rows) for p in w.params]).tolist()


def compare_every_output(oracle_mod, w, plan, pools, slot_host, batch=64):
    """Byte-compare every destination of every output with the oracle, and
    check that nothing outside the scheduled ranges was written.
    slot_host(p, k) gives shard k of param p as a host uint16 array."""
    host_pools = [p.cpu().numpy() for p in pools]
    m = oracle_mod.Model(w)
    base = _slot_base(w)
    nslots = base[-1]
    ranges = [[] for _ in range(w.num_ranks)]
    for b0 in range(0, len(w.outputs), batch):
        outs = list(range(b0, min(len(w.outputs), b0 + batch)))
        flat = [None] * nslots
        for o in outs:
            for q in w.outputs[o].parts:
                for k in range(len(w.params[q].shard_rows)):
                    flat[base[q] + k] = slot_host(q, k)
        with ThreadPoolExecutor(ncores()) as ex:
            results = list(ex.map(lambda o: m.prepare_output(o, flat), outs))
        for o, (data, scales) in zip(outs, results):
            out = w.outputs[o]
            for d in range(len(out.dst_ranks)):
                rank, doff, soff = plan.output_layout(o, d)
                got = host_pools[rank][doff:doff + data.size]
                if not np.array_equal(got, data):
                    bad = int(np.nonzero(got != data)[0][0])
                    raise AssertionError(f"{out.name} -> rank {rank}: data differs at byte {bad}")
                ranges[rank].append((doff, doff + data.size))
                if scales is not None:
                    gs = host_pools[rank][soff:soff + 4 * scales.size].view(np.uint32)
                    assert np.array_equal(gs, scales.view(np.uint32)), f"{out.name}: scales differ"
                    ranges[rank].append((soff, soff + 4 * scales.size))
        del flat, results
    # padding between scheduled ranges and the guard band: never written
    for r, hp in enumerate(host_pools):
        cur = 0
        for b, e in sorted(ranges[r]):
            assert b >= cur, f"rank {r}: scheduled ranges overlap at {b}"
            assert np.all(hp[cur:b] == CANARY), f"rank {r}: padding at {cur}..{b} written"
            cur = e
        assert cur <= plan.pool_bytes(r)
        assert np.all(hp[cur:] == CANARY), f"rank {r}: bytes after {cur} written"


def test_kimi_k2_layer_every_output_bit_exact(oracle_mod):
    """The benchmark's workload and launch (one wt_prepare over 1,034,880
    blocks, one CTA per SM), all 770 outputs byte for byte."""
    w = kimi_k2_moe_layer()
    shards = make_shards(w, device="cuda:0")
    plan = wt.Plan(w, device=0)
    pools = device_pools(plan, w.num_ranks)
    run_gpu(w, shards, pools=pools, plan=plan)
    plan.check()

    def slot_host(q, k):
        return shards[q][k].cpu().view(torch.int16).numpy().view(np.uint16)

    compare_every_output(oracle_mod, w, plan, pools, slot_host)
    plan.close()


def test_offload_layer_every_output_bit_exact_with_2gib_chunks(oracle_mod):
    """One whole layer of the streamed-offload stack (q/k/v fused into
    21504x7168 qkv, o, and the 385 experts: 34.3 GB of BF16 in pinned host
    memory) through wt_prepare_offload with the stack's 2 GiB chunks, every
    output byte for byte against the oracle run on the same pinned image."""
    w = offload_layer(385)
    plan = wt.Plan(w, device=0, offload_chunk_bytes=2 * GiB)
    st = plan.stats
    assert st["num_chunks"] >= 16
    host = torch.empty(st["host_bytes"], dtype=torch.uint8, pin_memory=True)
    shards = make_shards(w, device="cuda:0")
    for p, per in enumerate(shards):
        for k, t in enumerate(per):
            off = plan.shard_host_offset(p, k)
            host[off:off + t.numel() * 2].copy_(t.reshape(-1).view(torch.uint8))
    del shards
    torch.cuda.empty_cache()
    pools = device_pools(plan, w.num_ranks)
    copy_s, comp_s = torch.cuda.Stream(), torch.cuda.Stream()
    plan.prepare_offload(host.data_ptr(), [p.data_ptr() for p in pools], copy_s.cuda_stream,
                         comp_s.cuda_stream)
    plan.check(comp_s.cuda_stream)
    torch.cuda.synchronize()
    hn = host.numpy()

    def slot_host(q, k):
        off = plan.shard_host_offset(q, k)
        n = w.params[q].shard_rows[k] * w.params[q].cols
        return hn[off:off + 2 * n].view(np.uint16)

    compare_every_output(oracle_mod, w, plan, pools, slot_host)
    plan.close()
