"""Synthetic workloads (shapes, shard splits, fusion groups, ranks) and
their seeded source values. Shared by the tests, the benchmark and both
sides of the parity check; holds none of the stage's arithmetic."""
from .configs import (TILE, Output, Param, ValueRecipe, Workload, WORKLOADS, chunk_rows,
                      edge_narrow, edge_stress, halo_mix, kimi_k2_moe_layer, llama_dense, llama_dense_tp4,
                      offload_layer, shard_local_mix, tiny_dense, tp_slices_small, tp_split)
from .random_cases import random_workload
from .values import make_shards, param_values, shards_to_host_u16, split_shards

__all__ = [
    "TILE", "Output", "Param", "ValueRecipe", "Workload", "WORKLOADS", "chunk_rows",
    "edge_narrow", "edge_stress", "kimi_k2_moe_layer", "llama_dense", "llama_dense_tp4", "offload_layer",
    "halo_mix", "shard_local_mix", "tiny_dense", "tp_slices_small", "tp_split",
    "random_workload", "make_shards", "param_values", "shards_to_host_u16", "split_shards",
]
