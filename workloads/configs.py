"""Workload descriptors: parameter shapes, FSDP dim-0 shard splits, fusion
groups, output formats and destination ranks.

This module holds shapes and bookkeeping only; it does none of the stage's
arithmetic. Both the CUDA library (through its binding) and the CPU oracle
(through its own wrapper) receive the same descriptor and compute the
layout and the outputs independently.

The five named workloads mirror the shapes the stage is quoted on:
a tiny two-layer dense transformer, a four-layer Llama-style stack, one
Kimi-K2-shaped MoE layer (384 routed experts plus one shared expert,
hidden 7168 -- the hidden size also appears on the page "Enabling
trillion-parameter models on AWS EFA", section on dispatch/combine
kernels), an edge/value-stress set, and an eight-layer CPU-offloaded stack.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Sequence

TILE = 128


def chunk_rows(rows: int, shards: int) -> tuple:
    """Dim-0 split with torch.chunk semantics: ceil(rows/shards) rows per
    shard, the remainder in the last non-empty one; trailing shards that
    get nothing are kept with 0 rows so every parameter has `shards`
    entries (the FSDP placement of the page "Weight transfer for RL
    post-training in under 2 seconds", section "DeviceMesh and mesh
    groups", with empty shards allowed)."""
    per = -(-rows // shards)
    out, left = [], rows
    for _ in range(shards):
        n = min(per, left)
        out.append(n)
        left -= n
    return tuple(out)


@dataclass(frozen=True)
class Param:
    name: str
    rows: int
    cols: int
    shard_rows: tuple

    @property
    def numel(self) -> int:
        return self.rows * self.cols


@dataclass(frozen=True)
class Output:
    name: str
    parts: tuple            # param indices, fusion order
    fp8: bool               # True: e4m3 + 128x128 fp32 scales; False: BF16 bytes
    dst_ranks: tuple
    data_off: Optional[tuple] = None    # None or per-destination offset / None=auto
    scale_off: Optional[tuple] = None
    # None, or per destination: None (whole tensor) or (dim, ((begin, length), ...)),
    # the row (dim 0) or column (dim 1) ranges that destination takes
    slices: Optional[tuple] = None


@dataclass(frozen=True)
class ValueRecipe:
    """How source values are drawn (see workloads.values)."""
    dist: str = "normal"        # "normal" or "student_t3"
    sigma: float = 0.02
    seed: int = 0
    zero_tile_eighths: int = 0      # blocks whose seeded hash % 8 lands here are all zero
    outlier_tile_eighths: int = 0   # blocks that get one +-outlier
    outlier: float = 3.0e4


@dataclass
class Workload:
    name: str
    params: list
    outputs: list
    num_ranks: int
    values: ValueRecipe = field(default_factory=ValueRecipe)

    # --- derived sizes (bookkeeping only) ---------------------------------
    def output_shape(self, o: int) -> tuple:
        out = self.outputs[o]
        cols = {self.params[p].cols for p in out.parts}
        if len(cols) != 1:
            raise ValueError(f"fusion parts of {out.name} differ in cols")
        return sum(self.params[p].rows for p in out.parts), cols.pop()

    def dst_shape(self, o: int, d: int) -> tuple:
        """(rows, cols) that destination d of output o holds."""
        m, n = self.output_shape(o)
        out = self.outputs[o]
        if out.slices is None or out.slices[d] is None:
            return m, n
        dim, ranges = out.slices[d]
        total = sum(r[1] for r in ranges)
        return (total, n) if dim == 0 else (m, total)

    @property
    def num_params_total(self) -> int:
        return sum(p.numel for p in self.params)

    @property
    def bytes_read(self) -> int:
        """BF16 source bytes read by one pass."""
        return 2 * sum(self.params[p].numel for o in self.outputs for p in o.parts)

    @property
    def bytes_written(self) -> int:
        """Destination bytes written by one pass (data + scales, all dsts)."""
        total = 0
        for o, out in enumerate(self.outputs):
            for d in range(len(out.dst_ranks)):
                m, n = self.dst_shape(o, d)
                total += m * n if out.fp8 else 2 * m * n
                if out.fp8:
                    total += 4 * (-(-m // TILE)) * (-(-n // TILE))
        return total

    @property
    def num_tiles(self) -> int:
        t = 0
        for o in range(len(self.outputs)):
            m, n = self.output_shape(o)
            t += (-(-m // TILE)) * (-(-n // TILE))
        return t

    def subset(self, outputs: Sequence[int], name: Optional[str] = None) -> "Workload":
        """A workload made of some outputs (and only the params they use),
        keeping each output's destination ranks."""
        keep_params = []
        for o in outputs:
            for p in self.outputs[o].parts:
                if p not in keep_params:
                    keep_params.append(p)
        remap = {p: i for i, p in enumerate(keep_params)}
        outs = []
        for o in outputs:
            out = self.outputs[o]
            outs.append(Output(out.name, tuple(remap[p] for p in out.parts), out.fp8,
                               out.dst_ranks, out.data_off, out.scale_off, out.slices))
        return Workload(name or f"{self.name}[subset]", [self.params[p] for p in keep_params],
                        outs, self.num_ranks, self.values)


class _Builder:
    def __init__(self, name, num_ranks, shards, values):
        self.w = Workload(name, [], [], num_ranks, values)
        self.shards = shards

    def param(self, name, rows, cols, shard_rows=None):
        sr = shard_rows if shard_rows is not None else chunk_rows(rows, self.shards)
        self.w.params.append(Param(name, rows, cols, tuple(sr)))
        return len(self.w.params) - 1

    def output(self, name, parts, fp8, dst_ranks, data_off=None, scale_off=None, slices=None):
        self.w.outputs.append(Output(name, tuple(parts), fp8, tuple(dst_ranks),
                                     data_off, scale_off, slices))

    def round_robin_rank(self):
        """Outputs go round-robin over the ranks in plan order."""
        return len(self.w.outputs) % self.w.num_ranks


def dense_transformer(name, layers, hidden, q_heads, kv_heads, head_dim, ffn, vocab,
                      shards, ranks, values, lm_head_fp8=True) -> Workload:
    """Embedding (BF16), per layer [qkv, o, gate_up, down (FP8), two norms
    (BF16, [hidden, 1])], final norm (BF16), untied lm_head (FP8 unless
    lm_head_fp8 is False)."""
    b = _Builder(name, ranks, shards, values)

    def out(name, parts, fp8):
        b.output(name, parts, fp8, (b.round_robin_rank(),))

    out("embed", [b.param("embed", vocab, hidden)], False)
    for l in range(layers):
        q = b.param(f"l{l}.q", q_heads * head_dim, hidden)
        k = b.param(f"l{l}.k", kv_heads * head_dim, hidden)
        v = b.param(f"l{l}.v", kv_heads * head_dim, hidden)
        out(f"l{l}.qkv", [q, k, v], True)
        out(f"l{l}.o", [b.param(f"l{l}.o", hidden, q_heads * head_dim)], True)
        g = b.param(f"l{l}.gate", ffn, hidden)
        u = b.param(f"l{l}.up", ffn, hidden)
        out(f"l{l}.gate_up", [g, u], True)
        out(f"l{l}.down", [b.param(f"l{l}.down", hidden, ffn)], True)
        out(f"l{l}.attn_norm", [b.param(f"l{l}.attn_norm", hidden, 1)], False)
        out(f"l{l}.mlp_norm", [b.param(f"l{l}.mlp_norm", hidden, 1)], False)
    out("final_norm", [b.param("final_norm", hidden, 1)], False)
    out("lm_head", [b.param("lm_head", vocab, hidden)], lm_head_fp8)
    return b.w


def tiny_dense() -> Workload:
    """Two layers, hidden 256, 4 q heads / 2 kv heads of 64, FFN 512,
    vocab 1024, 4 shards, 2 destination ranks, N(0, 0.02), seed 1001."""
    return dense_transformer("tiny_dense_2l_h256", 2, 256, 4, 2, 64, 512, 1024,
                             shards=4, ranks=2, values=ValueRecipe("normal", 0.02, 1001))


def llama_dense(lm_head_fp8=True) -> Workload:
    """Four layers, hidden 4096, 32 q heads / 8 kv heads of 128, FFN 14336,
    vocab 128256, 8 shards, 4 destination ranks, N(0, 0.02), seed 1002."""
    return dense_transformer("llama_dense_4l_h4096", 4, 4096, 32, 8, 128, 14336, 128256,
                             shards=8, ranks=4, values=ValueRecipe("normal", 0.02, 1002),
                             lm_head_fp8=lm_head_fp8)


def tp_split(extent: int, tp: int) -> list:
    """(begin, length) of each of tp 128-aligned pieces covering [0, extent):
    ceil(extent / tp) rounded up to 128 each, the remainder last."""
    per = -(-(-(-extent // tp)) // TILE) * TILE
    out, b = [], 0
    for _ in range(tp):
        n = max(0, min(per, extent - b))
        out.append((b, n))
        b += n
    return out


def dense_transformer_tp(name, layers, hidden, q_heads, kv_heads, head_dim, ffn, vocab,
                         shards, tp, values) -> Workload:
    """The dense stack of dense_transformer laid out for tensor-parallel
    inference on tp ranks: every rank takes its slice of every Linear layer
    (column-parallel qkv and gate_up: its heads / its FFN rows of each
    fusion part; row-parallel o and down: its input columns), the
    vocabulary-parallel embedding and lm_head are split along rows, and the
    norms are replicated. Every 128x128 block of a sliced tensor goes to
    exactly one rank."""
    b = _Builder(name, tp, shards, values)
    ranks = tuple(range(tp))

    def rows_of(parts_rows):
        """Per rank, its row range of each fusion part, as fused-row ranges."""
        per_rank = [[] for _ in range(tp)]
        base = 0
        for n in parts_rows:
            for r, (bg, ln) in enumerate(tp_split(n, tp)):
                if ln:
                    per_rank[r].append((base + bg, ln))
            base += n
        return tuple((0, tuple(x)) for x in per_rank)

    def cols_of(n):
        return tuple((1, (rng,)) for rng in tp_split(n, tp))

    b.output("embed", [b.param("embed", vocab, hidden)], False, ranks, slices=rows_of([vocab]))
    qd, kvd = q_heads * head_dim, kv_heads * head_dim
    for l in range(layers):
        q = b.param(f"l{l}.q", qd, hidden)
        k = b.param(f"l{l}.k", kvd, hidden)
        v = b.param(f"l{l}.v", kvd, hidden)
        b.output(f"l{l}.qkv", [q, k, v], True, ranks, slices=rows_of([qd, kvd, kvd]))
        b.output(f"l{l}.o", [b.param(f"l{l}.o", hidden, qd)], True, ranks, slices=cols_of(qd))
        g = b.param(f"l{l}.gate", ffn, hidden)
        u = b.param(f"l{l}.up", ffn, hidden)
        b.output(f"l{l}.gate_up", [g, u], True, ranks, slices=rows_of([ffn, ffn]))
        b.output(f"l{l}.down", [b.param(f"l{l}.down", hidden, ffn)], True, ranks,
                 slices=cols_of(ffn))
        b.output(f"l{l}.attn_norm", [b.param(f"l{l}.attn_norm", hidden, 1)], False, ranks)
        b.output(f"l{l}.mlp_norm", [b.param(f"l{l}.mlp_norm", hidden, 1)], False, ranks)
    b.output("final_norm", [b.param("final_norm", hidden, 1)], False, ranks)
    b.output("lm_head", [b.param("lm_head", vocab, hidden)], True, ranks, slices=rows_of([vocab]))
    return b.w


def tp_slices_small() -> Workload:
    """Small slicing cases: an FP8 output fused from two parts (300 x 260,
    partial blocks in both dimensions) and a BF16 output (200 x 136), each
    sent whole and as row / column slices, in and out of order, with ranges
    that end at the tensor's edge, replicated on two ranks."""
    params = [Param("a1", 172, 260, (100, 72)), Param("a2", 128, 260, (128,)),
              Param("b", 200, 136, (64, 136))]
    fp8_slices = (None, (0, ((128, 128), (0, 128))), (0, ((256, 44),)),
                  (1, ((128, 132),)), (1, ((0, 128), (256, 4))))
    bf16_slices = (None, (0, ((0, 128), (128, 72))), (1, ((128, 8),)))
    outs = [Output("a", (0, 1), True, (0, 1, 0, 1, 0), slices=fp8_slices),
            Output("b", (2,), False, (1, 0, 1), slices=bf16_slices)]
    return Workload("tp_slices_small", params, outs, 2, ValueRecipe("student_t3", 0.02, 41))


def llama_dense_tp4() -> Workload:
    """The four-layer Llama-style stack of llama_dense, laid out for 4-way
    tensor-parallel inference (see dense_transformer_tp)."""
    return dense_transformer_tp("llama_dense_4l_h4096_tp4", 4, 4096, 32, 8, 128, 14336, 128256,
                                shards=8, tp=4, values=ValueRecipe("normal", 0.02, 1002))


def _moe_experts(b: _Builder, prefix: str, experts: int, hidden: int, inter: int,
                 rank_of=None):
    for e in range(experts):
        rank = (e % b.w.num_ranks) if rank_of is None else rank_of(e)
        w1 = b.param(f"{prefix}e{e}.w1", inter, hidden)
        w3 = b.param(f"{prefix}e{e}.w3", inter, hidden)
        b.output(f"{prefix}e{e}.gate_up", [w1, w3], True, (rank,))
        w2 = b.param(f"{prefix}e{e}.w2", hidden, inter)
        b.output(f"{prefix}e{e}.down", [w2], True, (rank,))


def kimi_k2_moe_layer(experts: int = 385, seed: int = 1003, shards: int = 8) -> Workload:
    """One Kimi-K2-shaped MoE layer: 384 routed experts plus the shared one
    (index 384), each w1/w3 2048x7168 fused into gate_up 4096x7168 and w2
    7168x2048, 8 dim-0 shards per weight, expert e on rank e % 8, all FP8,
    N(0, 0.006). `experts` < 385 gives the first `experts` of them;
    `shards` changes the FSDP degree (the values do not depend on it)."""
    name = f"kimi_k2_moe_layer_e{experts}" + ("" if shards == 8 else f"_s{shards}")
    b = _Builder(name, 8, shards, ValueRecipe("normal", 0.006, seed))
    _moe_experts(b, "", experts, 7168, 2048)
    return b.w


def edge_stress() -> Workload:
    """7168x2050 (ragged last column block, 4100-byte rows) and 1000x7168
    (ragged last row block) FP8, a 163840x7168 BF16 embedding, 3 uneven
    shards each, 5 ranks of which 3 and 4 receive nothing. Values
    Student-t(3) x 0.02; one block in eight all-zero, one in eight with a
    single +-3e4 outlier. Seed 1004."""
    vals = ValueRecipe("student_t3", 0.02, 1004, zero_tile_eighths=1,
                       outlier_tile_eighths=1, outlier=3.0e4)
    b = _Builder("edge_stress", 5, 3, vals)
    b.output("A", [b.param("A", 7168, 2050)], True, (0,))
    b.output("B", [b.param("B", 1000, 7168)], True, (1,))
    b.output("C_embed", [b.param("C_embed", 163840, 7168)], False, (2,))
    return b.w


def edge_narrow(copies: int = 8) -> Workload:
    """Rows that are not 16-byte aligned, at a size larger than L2: `copies`
    outputs shaped like the edge set's 7168x2050 FP8 matrix (4100-byte
    rows, a 2-column last block column), 3 uneven shards each, one rank
    per output, the edge set's value recipe (seed 1009). copies=1 is the
    edge set's matrix alone (L2-resident)."""
    vals = ValueRecipe("student_t3", 0.02, 1009, zero_tile_eighths=1,
                       outlier_tile_eighths=1, outlier=3.0e4)
    b = _Builder(f"edge_narrow_x{copies}", copies, 3, vals)
    for i in range(copies):
        b.output(f"A{i}", [b.param(f"A{i}", 7168, 2050)], True, (i,))
    return b.w


def shard_local_mix(shards: int = 4) -> Workload:
    """Cases for shard-local preparation, where every FSDP shard boundary
    falls on a multiple of 128 rows of its output: empty shards, a ragged
    last block row, a fused qkv whose parts live on different shards,
    narrow (cols % 8 != 0) and 16-byte rows, a ragged last column block,
    FP8 and BF16, dim-1 tensor-parallel slices, a replicated output and a
    1-column norm; 4 shards (2: neighbouring pairs merged), 3 ranks.
    Student-t(3) x 0.02 values, one block in eight all-zero and one in
    eight with a +-3e4 outlier, seed 1007."""
    splits = {"A": (384, 0, 512, 104), "B": (128, 128, 0, 264), "q": (256, 256, 0, 0),
              "k": (0, 0, 128, 0), "v": (0, 0, 0, 128), "emb": (128, 256, 256, 0),
              "norm": (256, 44, 0, 0)}
    if shards == 2:
        splits = {k: (v[0] + v[1], v[2] + v[3]) for k, v in splits.items()}
    elif shards != 4:
        raise ValueError("shard_local_mix has 4 or 2 shards")
    vals = ValueRecipe("student_t3", 0.02, 1007, zero_tile_eighths=1,
                       outlier_tile_eighths=1, outlier=3.0e4)
    b = _Builder(f"shard_local_mix_s{shards}", 3, shards, vals)
    b.output("A", [b.param("A", 1000, 2050, splits["A"])], True, (0,))
    b.output("B", [b.param("B", 520, 1040, splits["B"])], True, (0, 2))
    qkv = [b.param(n, r, 1024, splits[n]) for n, r in (("q", 512), ("k", 128), ("v", 128))]
    b.output("qkv", qkv, True, (1, 2), slices=((1, ((0, 512),)), (1, ((512, 512),))))
    b.output("emb", [b.param("emb", 640, 132, splits["emb"])], False, (2,))
    b.output("norm", [b.param("norm", 300, 1, splits["norm"])], False, (0, 1))
    return b.w


def halo_mix(shards: int = 4) -> Workload:
    """Cases for shard-local preparation with halos, where shard boundaries
    fall off the 128-row grid: a block row spanning three shards (a 20-row
    shard in the middle), an empty shard, a fused qkv whose parts end
    mid-block, narrow and 16-byte rows, FP8 and BF16, dim-1 slices, a
    replicated 1-column norm; 4 shards (2: neighbouring pairs merged),
    3 ranks. Student-t(3) x 0.02 values, one block in eight all-zero and
    one in eight with a +-3e4 outlier, seed 1008."""
    splits = {"A": (100, 20, 500, 380), "q": (64, 100, 136, 0), "k": (0, 0, 72, 128),
              "v": (50, 50, 0, 0), "emb": (175, 175, 175, 175), "norm": (75, 75, 75, 75)}
    if shards == 2:
        splits = {k: (v[0] + v[1], v[2] + v[3]) for k, v in splits.items()}
    elif shards != 4:
        raise ValueError("halo_mix has 4 or 2 shards")
    vals = ValueRecipe("student_t3", 0.02, 1008, zero_tile_eighths=1,
                       outlier_tile_eighths=1, outlier=3.0e4)
    b = _Builder(f"halo_mix_s{shards}", 3, shards, vals)
    b.output("A", [b.param("A", 1000, 2050, splits["A"])], True, (0,))
    qkv = [b.param(n, r, 1024, splits[n]) for n, r in (("q", 300), ("k", 200), ("v", 100))]
    b.output("qkv", qkv, True, (1, 2), slices=((1, ((0, 512),)), (1, ((512, 512),))))
    b.output("emb", [b.param("emb", 700, 136, splits["emb"])], False, (2,))
    b.output("norm", [b.param("norm", 300, 1, splits["norm"])], False, (0, 1))
    return b.w


def offload_layer(experts: int = 385, seed: int = 1005) -> Workload:
    """One layer of the streamed-offload stack: the MoE layer above plus
    attention projections q, k, v, o of 7168x7168 (q/k/v fused into qkv
    21504x7168), all FP8, 8 shards, 8 ranks."""
    b = _Builder(f"offload_layer_e{experts}", 8, 8, ValueRecipe("normal", 0.006, seed))
    q = b.param("q", 7168, 7168)
    k = b.param("k", 7168, 7168)
    v = b.param("v", 7168, 7168)
    b.output("qkv", [q, k, v], True, (b.round_robin_rank(),))
    b.output("o", [b.param("o", 7168, 7168)], True, (b.round_robin_rank(),))
    _moe_experts(b, "", experts, 7168, 2048)
    return b.w


WORKLOADS = {
    "tiny_dense": tiny_dense,
    "llama_dense": llama_dense,
    "llama_dense_tp4": llama_dense_tp4,
    "tp_slices_small": tp_slices_small,
    "shard_local_mix": shard_local_mix,
    "halo_mix": halo_mix,
    "kimi_k2_moe_layer": kimi_k2_moe_layer,
    "edge_stress": edge_stress,
    "edge_narrow": edge_narrow,
    "edge_narrow_1": lambda: edge_narrow(1),
    "offload_layer": offload_layer,
}
