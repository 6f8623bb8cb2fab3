"""Seeded synthetic source values for the workloads in workloads.configs.

Only random-number draws live here: no reassembly, fusion, scaling or
encoding. Each parameter is drawn whole from its own seeded generator,
rounded to BF16 (round-to-nearest-even, torch's cast) and then cut along
dim 0 into separately allocated shards, so shard base pointers are as
unrelated as FSDP's.

Recipes (ValueRecipe.dist):
  normal      N(0, sigma^2) in fp32, then BF16.
  student_t3  sigma * z / sqrt(chi2_3 / 3) with z and the three chi-square
              terms standard normals; heavy tails with finite variance.
Block patterns (per 128x128 block of each parameter, drawn from a CPU
generator so they do not depend on the device):
  category 0 .. zero_tile_eighths-1                      -> block set to 0
  next outlier_tile_eighths categories                    -> one element set
                                                             to +-outlier
"""
from __future__ import annotations

import zlib

import numpy as np
import torch

from .configs import TILE, Workload


def _param_seed(seed: int, name: str) -> int:
    """Seed of one parameter: depends on the recipe seed and the parameter's
    name only, so any subset of a workload draws the same values."""
    return (seed * 1_000_003 + zlib.crc32(name.encode()) * 7919 + 17) % (2**63 - 1)


def param_values(w: Workload, p: int, device="cpu") -> torch.Tensor:
    """The full BF16 value of parameter p, shape [rows, cols]."""
    par = w.params[p]
    rec = w.values
    g = torch.Generator(device=device)
    g.manual_seed(_param_seed(rec.seed, par.name))
    shape = (par.rows, par.cols)
    if rec.dist == "normal":
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        x.mul_(rec.sigma)
    elif rec.dist == "student_t3":
        z = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        chi = torch.zeros(shape, device=device, dtype=torch.float32)
        for _ in range(3):
            n = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
            chi.addcmul_(n, n)
        x = z.mul_(rec.sigma).div_(chi.div_(3.0).sqrt_())
        del chi
    else:
        raise ValueError(rec.dist)
    xb = x.to(torch.bfloat16)
    del x
    if rec.zero_tile_eighths or rec.outlier_tile_eighths:
        _apply_block_patterns(w, p, xb)
    return xb


def _apply_block_patterns(w: Workload, p: int, xb: torch.Tensor) -> None:
    par = w.params[p]
    rec = w.values
    tr, tc = -(-par.rows // TILE), -(-par.cols // TILE)
    g = torch.Generator(device="cpu")
    g.manual_seed(_param_seed(rec.seed, par.name) ^ 0x5DEECE66D)
    cat = torch.randint(0, 8, (tr, tc), generator=g)
    pos_r = torch.randint(0, TILE, (tr, tc), generator=g)
    pos_c = torch.randint(0, TILE, (tr, tc), generator=g)
    sign = torch.randint(0, 2, (tr, tc), generator=g)
    zero_cut = rec.zero_tile_eighths
    out_cut = zero_cut + rec.outlier_tile_eighths
    cat_np = cat.numpy()
    for bi, bj in zip(*np.nonzero(cat_np < out_cut)):
        r0, c0 = int(bi) * TILE, int(bj) * TILE
        r1, c1 = min(r0 + TILE, par.rows), min(c0 + TILE, par.cols)
        if cat_np[bi, bj] < zero_cut:
            xb[r0:r1, c0:c1] = 0
        else:
            r = r0 + int(pos_r[bi, bj]) % (r1 - r0)
            c = c0 + int(pos_c[bi, bj]) % (c1 - c0)
            v = rec.outlier if int(sign[bi, bj]) else -rec.outlier
            xb[r, c] = v


def split_shards(w: Workload, p: int, full: torch.Tensor) -> list:
    """Cut a parameter into its dim-0 shards, each its own allocation."""
    out, r = [], 0
    for n in w.params[p].shard_rows:
        out.append(full[r:r + n].clone())
        r += n
    return out


def make_shards(w: Workload, device="cpu") -> list:
    """Per parameter, the list of its BF16 shard tensors (plan order)."""
    shards = []
    for p in range(len(w.params)):
        full = param_values(w, p, device)
        shards.append(split_shards(w, p, full))
        del full
    return shards


def shards_to_host_u16(shards: list) -> list:
    """Host uint16 numpy views of every shard (param-major, then shard)."""
    flat = []
    for per_param in shards:
        for s in per_param:
            flat.append(np.ascontiguousarray(s.detach().cpu().view(torch.int16).numpy()).view(np.uint16))
    return flat
