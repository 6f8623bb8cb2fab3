"""Bookkeeping shared by the shard-local tests: which block rows a shard
owns, which halo rows it needs, what its plan should count, and the
oracle's block rows computed from a given set of rows. Computed here from
the workload description alone, independently of the plan compiler."""
import numpy as np

from workloads import TILE, Output, Param, Workload


def _cdiv(a, b):
    return -(-a // b)


def shard_runs(w, o, s):
    """(fused row begin, rows, param index) of every shard-s run of output o."""
    out, row = [], 0
    for p in w.outputs[o].parts:
        par = w.params[p]
        r = row
        for k, n in enumerate(par.shard_rows):
            if k == s and n:
                out.append((r, n, p))
            r += n
        row += par.rows
    return out


def owned_block_rows(w, o, s, halo=False):
    """Block rows of output o whose rows all come from shard s (halo: whose
    first row does)."""
    if halo:
        # the multiples of 128 that fall inside one of shard s's runs
        return sorted(start // TILE for (r0, n, _) in shard_runs(w, o, s)
                      for start in range(_cdiv(r0, TILE) * TILE, r0 + n, TILE))
    return [b for (r0, n, _) in shard_runs(w, o, s) for b in range(r0 // TILE, _cdiv(r0 + n, TILE))]


def all_runs(w, o):
    """(fused row begin, rows, param, shard) of every non-empty shard of output o."""
    out, row = [], 0
    for p in w.outputs[o].parts:
        for k, n in enumerate(w.params[p].shard_rows):
            if n:
                out.append((row, n, p, k))
            row += n
    return out


def halo_rows_needed(w, s):
    """{(param, shard): leading rows} that shard s's halo plan reads from
    shards of other indices."""
    need = {}
    for o in range(len(w.outputs)):
        m, _ = w.output_shape(o)
        for bi in owned_block_rows(w, o, s, halo=True):
            lo, hi = bi * TILE, min(m, bi * TILE + TILE)
            for r0, n, p, k in all_runs(w, o):
                if k != s and r0 < hi and r0 + n > lo:
                    assert r0 > lo                     # a halo is always a prefix
                    need[(p, k)] = max(need.get((p, k), 0), min(n, hi - r0))
    return need


def held_blocks(w, o, d, block_rows):
    """Blocks of block_rows that destination d of output o holds."""
    m, n = w.output_shape(o)
    out = w.outputs[o]
    bn = _cdiv(n, TILE)
    sl = out.slices[d] if out.slices is not None else None
    held = []
    for bi in block_rows:
        for bj in range(bn):
            if sl is not None:
                dim, ranges = sl
                idx = bi if dim == 0 else bj
                if not any(b // TILE <= idx < _cdiv(b + l, TILE) for b, l in ranges):
                    continue
            held.append((bi, bj))
    return held


def local_counts(w, s, halo=False):
    """Units, elements, bytes written and per-rank blocks of shard s's work."""
    units = elems = written = 0
    per_rank = [0] * w.num_ranks
    for o, out in enumerate(w.outputs):
        m, n = w.output_shape(o)
        rows = owned_block_rows(w, o, s, halo)
        for bi in rows:
            for bj in range(_cdiv(n, TILE)):
                units += 1
                elems += (min(TILE, m - bi * TILE)) * (min(TILE, n - bj * TILE))
        for d, r in enumerate(out.dst_ranks):
            for bi, bj in held_blocks(w, o, d, rows):
                e = min(TILE, m - bi * TILE) * min(TILE, n - bj * TILE)
                written += e + 4 if out.fp8 else 2 * e
                per_rank[r] += 1
    return units, elems, written, per_rank


def assembled_oracle_blocks(oracle_mod, w, s, rows_of):
    """{(output, block row): (data, scale row)} of the block rows shard s
    owns under the halo rule, computed by the oracle from the rows that
    rows_of(param, shard, begin, end) hands out."""
    res = {}
    for o, out in enumerate(w.outputs):
        m, n = w.output_shape(o)
        own = owned_block_rows(w, o, s, halo=True)
        if not own:
            continue
        pieces = []
        for bi in own:
            lo, hi = bi * TILE, min(m, bi * TILE + TILE)
            for r0, cnt, p, k in all_runs(w, o):
                a, b = max(lo, r0), min(hi, r0 + cnt)
                if a < b:
                    pieces.append(rows_of(p, k, a - r0, b - r0))
        x = np.ascontiguousarray(np.concatenate(pieces, axis=0))
        sub = Workload("local", [Param("local", x.shape[0], n, (x.shape[0],))],
                       [Output(out.name, (0,), out.fp8, (0,))], 1, w.values)
        data, scales = oracle_mod.Model(sub).prepare_output(0, [x])
        esz = 1 if out.fp8 else 2
        data = data.reshape(x.shape[0], n * esz)
        bn = _cdiv(n, TILE)
        for j, bi in enumerate(own):
            h = min(TILE, m - bi * TILE)
            srow = scales.reshape(-1, bn)[j].copy() if scales is not None else None
            res[(o, bi)] = (data[j * TILE:j * TILE + h].copy(), srow)
    return res


def full_oracle_blocks(oracle_mod, w, flat_full):
    m = oracle_mod.Model(w)
    res = {}
    for o in range(len(w.outputs)):
        data, scales = m.prepare_output(o, flat_full)
        rows, n = w.output_shape(o)
        esz = 1 if w.outputs[o].fp8 else 2
        data = data.reshape(rows, n * esz)
        bn = _cdiv(n, TILE)
        for bi in range(_cdiv(rows, TILE)):
            srow = scales.reshape(-1, bn)[bi].copy() if scales is not None else None
            res[(o, bi)] = (data[bi * TILE:(bi + 1) * TILE].copy(), srow)
    return res


def same_blocks(a, b):
    return np.array_equal(a[0], b[0]) and (a[1] is None) == (b[1] is None) and (
        a[1] is None or np.array_equal(a[1].view(np.uint32), b[1].view(np.uint32)))


