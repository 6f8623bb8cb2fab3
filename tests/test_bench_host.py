"""Host-side pieces of bench.py (no GPU): the bounded CPU-oracle sample, the
CPU-baseline record and the single-rank reductions."""
import bench
from workloads import edge_stress, kimi_k2_moe_layer, llama_dense, tiny_dense


def test_sample_outputs_are_bounded_and_representative():
    k = kimi_k2_moe_layer()
    assert bench.sample_outputs(k, 8) == list(range(16))           # the first 8 experts
    for w in (llama_dense(), edge_stress(), tiny_dense()):
        outs = bench.sample_outputs(w, 8)
        assert outs and len(set(outs)) == len(outs)
        total = sum(2 * w.output_shape(o)[0] * w.output_shape(o)[1] for o in outs)
        assert total <= 700_000_000
    # the dense stack's sample is its layers, not its 1 GB embedding alone
    l = llama_dense()
    assert [l.outputs[o].name for o in bench.sample_outputs(l, 8)][:2] == ["l0.qkv", "l0.o"]


def test_cpu_baseline_record(oracle_mod):
    rec = bench.cpu_baseline(tiny_dense(), 8)
    assert rec["kind"] == "oracle" and rec["unit"] == "GB/s" and rec["value"] > 0
    assert rec["cores"] >= 1 and rec["single_thread"]["cores"] == 1
    assert "15 of 15 outputs" in rec["sample"]


def test_single_rank_reductions_are_identities():
    assert bench.max_over_ranks(1, 3.5, None) == 3.5
    assert bench.sum_over_ranks(1, 7.0, None) == 7.0


def test_end_to_end_leg_fits_the_pinned_budget():
    import bf16_fp8_parameter_wt_b300 as wt
    w = kimi_k2_moe_layer()
    shards = [[None] * len(p.shard_rows) for p in w.params]
    with wt.Plan(w, device=-1, offload_chunk_bytes=2 << 30) as p:
        full = p.stats["host_bytes"]
    assert bench.e2e_subset(w, shards, full, full)[2] is None          # fits: the whole layer
    sub, sh, note = bench.e2e_subset(w, shards, full, full / 8)
    assert note and len(sh) == len(sub.params) and sub.params == w.params[:len(sh)]
    with wt.Plan(sub, device=-1, offload_chunk_bytes=2 << 30) as p:
        assert p.stats["host_bytes"] <= full / 8
    assert len(sub.outputs) == 2 * (385 // 8)
    assert bench.e2e_subset(llama_dense(), [], 10 ** 12, 1.0)[2] is None   # only the MoE layer is cut


def test_rank_groups_counts_the_launches_of_a_step_counted_per_rank():
    """A step counted per rank is one launch per non-empty rank group (the
    blocks whose lowest holding rank is g): the bench's launch count."""
    import bench
    from workloads import edge_stress, kimi_k2_moe_layer, llama_dense_tp4, tiny_dense, tp_slices_small
    assert bench.rank_groups(kimi_k2_moe_layer()) == 8
    assert bench.rank_groups(kimi_k2_moe_layer(3)) == 3
    assert bench.rank_groups(tiny_dense()) == 2
    assert bench.rank_groups(edge_stress()) == 3          # ranks 3 and 4 receive nothing
    assert bench.rank_groups(llama_dense_tp4()) == 4
    # every block there has a destination on rank 0 (a whole-tensor replica,
    # or a row slice covering every row): one group
    assert bench.rank_groups(tp_slices_small()) == 1


def test_kernel_hash_ignores_comments_and_whitespace_only():
    """The traffic figure stays tied to the kernel's code: comments and
    layout do not change the hash, code (string literals included) does."""
    base = b'asm volatile("ld.global.nc.v4.u32 {%0}, [%1];");\nint a = 1;  // one\n'
    same = b'/* a block\n comment */ asm volatile("ld.global.nc.v4.u32 {%0}, [%1];");\n\n  int a = 1; // two\n'
    assert bench._code_only(base) == bench._code_only(same)
    assert bench._code_only(base) != bench._code_only(base.replace(b"a = 1", b"a = 2"))
    assert bench._code_only(base) != bench._code_only(base.replace(b"v4.u32", b"v2.u32"))
    kept = bench._code_only(b'const char* s = "a // b /* c */";')
    assert kept == b'const char* s = "a // b /* c */";'


def test_token_cpu_baseline_record(oracle_mod):
    rec = bench.token_cpu_baseline(64, 256, steps=1)
    assert rec["kind"] == "oracle" and rec["unit"] == "GB/s" and rec["value"] > 0
    assert rec["cores"] >= 1 and "64 tokens x 256" in rec["sample"]
