// Plan compiler: validates the descriptor and turns it into the static
// schedule that every wt_prepare replays ("Weight transfer for RL
// post-training in under 2 seconds", sections "High-level workflow" --
// metadata in, schedule computed by the controller -- and "Why it is fast
// and simple / static schedule" -- computed once, replayed each step).
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <limits>

#include "plan.h"

namespace wt {

namespace {

uint64_t align_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

std::string pname(const wt_param_desc& d, int i) {
  return d.name ? std::string(d.name) : "param " + std::to_string(i);
}
std::string oname(const wt_output_desc& d, int i) {
  return d.name ? std::string(d.name) : "output " + std::to_string(i);
}

wt_status fail(wt_status s, const std::string& msg) {
  set_error(msg);
  return s;
}

struct Range {
  uint64_t off, bytes;
  int32_t out, dst;
  bool scale;
};

// Destination k of output oi: the slice it takes (if any) and its sizes.
// A slice is the listed 128-aligned row (dim 0) or column (dim 1) ranges
// of the fused tensor, concatenated; only the last range may end off the
// 128 grid, at the tensor's edge; ranges do not overlap.
wt_status parse_slice(const wt_slice_desc* sd, OutputInfo& oi, int k) {
  DstInfo& ds = oi.dsts[k];
  const std::string where = oi.name + ", destination " + std::to_string(k) + ": ";
  ds.rows = oi.rows;
  ds.cols = oi.cols;
  if (sd && sd->num_ranges != 0) {
    if (sd->num_ranges < 0 || !sd->begin || !sd->length)
      return fail(WT_ERR_INVALID_ARGUMENT, where + "slice ranges missing");
    if (sd->dim != 0 && sd->dim != 1) return fail(WT_ERR_INVALID_ARGUMENT, where + "slice dim must be 0 or 1");
    const int64_t extent = sd->dim == 0 ? oi.rows : oi.cols;
    int64_t total = 0;
    for (int32_t r = 0; r < sd->num_ranges; ++r) {
      const int64_t b = sd->begin[r], n = sd->length[r];
      if (b < 0 || n < 1 || b + n > extent)
        return fail(WT_ERR_SHAPE, where + "slice range " + std::to_string(r) + " is outside the tensor");
      if (b % kTile) return fail(WT_ERR_SHAPE, where + "slice range does not start on a multiple of 128");
      if (n % kTile && !(b + n == extent && r == sd->num_ranges - 1))
        return fail(WT_ERR_SHAPE, where + "only the last slice range may end off the 128 grid, at the edge");
      for (int32_t q = 0; q < r; ++q)
        if (b < sd->begin[q] + sd->length[q] && sd->begin[q] < b + n)
          return fail(WT_ERR_SHAPE, where + "slice ranges overlap");
      total += n;
    }
    ds.slice_dim = sd->dim;
    ds.slice_begin.assign(sd->begin, sd->begin + sd->num_ranges);
    ds.slice_len.assign(sd->length, sd->length + sd->num_ranges);
    if (sd->dim == 0) ds.rows = total; else ds.cols = total;
  }
  const bool fp8 = oi.format == WT_OUT_FP8_E4M3_B128;
  ds.data_bytes = uint64_t(ds.rows * ds.cols) * (fp8 ? 1u : 2u);
  ds.scale_bytes = fp8 ? uint64_t(ceil_div(ds.rows, kTile) * ceil_div(ds.cols, kTile)) * 4u : 0u;
  return WT_OK;
}

}  // namespace

wt_status compile_plan(const wt_plan_desc* d, Plan* p) {
  const int64_t kMaxDim = (int64_t(1) << 31) - 1;
  if (!d) return fail(WT_ERR_INVALID_ARGUMENT, "descriptor is NULL");
  if (d->num_params < 0 || d->num_outputs < 0 || d->num_ranks < 0)
    return fail(WT_ERR_INVALID_ARGUMENT, "negative count in descriptor");
  if ((d->num_params > 0 && !d->params) || (d->num_outputs > 0 && !d->outputs))
    return fail(WT_ERR_INVALID_ARGUMENT, "params/outputs array is NULL");
  if (d->flags & ~(WT_FLAG_FORCE_NARROW | WT_FLAG_DEBUG_CHECKS | WT_FLAG_SHARD_LOCAL | WT_FLAG_SHARD_HALO))
    return fail(WT_ERR_INVALID_ARGUMENT, "unknown flag bits");
  if ((d->flags & WT_FLAG_SHARD_HALO) && !(d->flags & WT_FLAG_SHARD_LOCAL))
    return fail(WT_ERR_INVALID_ARGUMENT, "WT_FLAG_SHARD_HALO needs WT_FLAG_SHARD_LOCAL");
  p->local_shard = -1;
  if (d->flags & WT_FLAG_SHARD_LOCAL) {
    if (d->local_shard < 0) return fail(WT_ERR_INVALID_ARGUMENT, "local_shard must be >= 0");
    if (d->offload_chunk_bytes)
      return fail(WT_ERR_INVALID_ARGUMENT, "a shard-local plan does not stage offloaded shards");
    p->local_shard = d->local_shard;
  }
  p->flags = d->flags;
  p->num_ranks = d->num_ranks;

  // ---- params: shapes and dim-0 shards ---------------------------------
  p->params.resize(d->num_params);
  int64_t slot = 0;
  for (int i = 0; i < d->num_params; ++i) {
    const wt_param_desc& pd = d->params[i];
    ParamInfo& pi = p->params[i];
    pi.name = pname(pd, i);
    if (pd.rows < 0 || pd.cols < 1 || pd.rows > kMaxDim || pd.cols > kMaxDim)
      return fail(WT_ERR_SHAPE, pi.name + ": rows must be >= 0 and cols >= 1");
    if (pd.num_shards < 1 || !pd.shard_rows)
      return fail(WT_ERR_INVALID_ARGUMENT, pi.name + ": needs at least one shard");
    int64_t sum = 0;
    for (int s = 0; s < pd.num_shards; ++s) {
      if (pd.shard_rows[s] < 0) return fail(WT_ERR_SHAPE, pi.name + ": negative shard rows");
      sum += pd.shard_rows[s];
    }
    if (sum != pd.rows)
      return fail(WT_ERR_SHAPE, pi.name + ": shard rows sum to " + std::to_string(sum) +
                                    ", expected " + std::to_string(pd.rows));
    pi.rows = pd.rows;
    pi.cols = pd.cols;
    pi.shard_rows.assign(pd.shard_rows, pd.shard_rows + pd.num_shards);
    pi.slot_base = (int32_t)slot;
    slot += pd.num_shards;
    if (slot > std::numeric_limits<int32_t>::max())
      return fail(WT_ERR_INVALID_ARGUMENT, "too many shards");
  }
  p->num_slots = (int32_t)slot;

  // ---- outputs: fusion groups, formats, destinations --------------------
  p->outputs.resize(d->num_outputs);
  int64_t units = 0;
  for (int o = 0; o < d->num_outputs; ++o) {
    const wt_output_desc& od = d->outputs[o];
    OutputInfo& oi = p->outputs[o];
    oi.name = oname(od, o);
    if (od.num_parts < 1 || !od.part_params)
      return fail(WT_ERR_INVALID_ARGUMENT, oi.name + ": needs at least one part");
    if (od.format != WT_OUT_BF16 && od.format != WT_OUT_FP8_E4M3_B128)
      return fail(WT_ERR_INVALID_ARGUMENT, oi.name + ": unknown format");
    if (od.num_dsts < 1 || !od.dst_ranks)
      return fail(WT_ERR_INVALID_ARGUMENT, oi.name + ": needs at least one destination");
    oi.format = od.format;
    int64_t rows = 0, cols = -1;
    for (int k = 0; k < od.num_parts; ++k) {
      int32_t q = od.part_params[k];
      if (q < 0 || q >= d->num_params)
        return fail(WT_ERR_INVALID_ARGUMENT, oi.name + ": part index out of range");
      ParamInfo& pi = p->params[q];
      if (pi.output >= 0)
        return fail(WT_ERR_INVALID_ARGUMENT,
                    pi.name + ": used by more than one output (or twice in one)");
      pi.output = o;
      if (cols < 0) cols = pi.cols;
      if (pi.cols != cols)
        return fail(WT_ERR_SHAPE, oi.name + ": fusion parts differ in cols");
      rows += pi.rows;
      oi.parts.push_back(q);
    }
    if (rows < 1 || rows > kMaxDim)
      return fail(WT_ERR_SHAPE, oi.name + ": fused tensor has no rows");
    if (rows * cols > (int64_t(1) << 46))
      return fail(WT_ERR_SHAPE, oi.name + ": tensor too large");
    oi.rows = rows;
    oi.cols = cols;
    const bool fp8 = od.format == WT_OUT_FP8_E4M3_B128;
    oi.data_bytes = uint64_t(rows * cols) * (fp8 ? 1u : 2u);
    oi.scale_bytes = fp8 ? uint64_t(ceil_div(rows, kTile) * ceil_div(cols, kTile)) * 4u : 0u;
    oi.unit_begin = units;
    oi.num_units = ceil_div(rows, kTile) * ceil_div(cols, kTile);
    units += oi.num_units;
    oi.vec = (cols % 8 == 0) && !(d->flags & WT_FLAG_FORCE_NARROW);
    oi.dsts.resize(od.num_dsts);
    for (int k = 0; k < od.num_dsts; ++k) {
      int32_t r = od.dst_ranks[k];
      if (r < 0 || r >= d->num_ranks)
        return fail(WT_ERR_INVALID_ARGUMENT, oi.name + ": destination rank out of range");
      oi.dsts[k].rank = r;
      uint64_t doff = od.dst_data_off ? od.dst_data_off[k] : WT_OFFSET_AUTO;
      uint64_t soff = (fp8 && od.dst_scale_off) ? od.dst_scale_off[k] : WT_OFFSET_AUTO;
      if (doff != WT_OFFSET_AUTO && doff % 16)
        return fail(WT_ERR_ALIGNMENT, oi.name + ": explicit data offset not a multiple of 16");
      if (soff != WT_OFFSET_AUTO && soff % 4)
        return fail(WT_ERR_ALIGNMENT, oi.name + ": explicit scale offset not a multiple of 4");
      if ((doff != WT_OFFSET_AUTO && doff > (uint64_t(1) << 56)) ||
          (soff != WT_OFFSET_AUTO && soff > (uint64_t(1) << 56)))
        return fail(WT_ERR_INVALID_ARGUMENT, oi.name + ": explicit offset out of range");
      oi.dsts[k].data_off = doff;
      oi.dsts[k].scale_off = soff;
      wt_status st = parse_slice(od.dst_slices ? &od.dst_slices[k] : nullptr, oi, k);
      if (st != WT_OK) return st;
    }
  }
  for (int i = 0; i < d->num_params; ++i)
    if (p->params[i].output < 0)
      return fail(WT_ERR_INVALID_ARGUMENT, p->params[i].name + ": not used by any output");
  p->num_units = units;
  if (units > std::numeric_limits<uint32_t>::max() / 2)
    return fail(WT_ERR_SHAPE, "too many 128x128 units");

  // ---- destination layout: explicit ranges, then auto-pack per rank ------
  p->pool_bytes.assign(d->num_ranks, 0);
  std::vector<uint64_t> cursor(d->num_ranks, 0);
  for (auto& oi : p->outputs)
    for (auto& ds : oi.dsts) {
      if (ds.data_off != WT_OFFSET_AUTO)
        cursor[ds.rank] = std::max(cursor[ds.rank], ds.data_off + ds.data_bytes);
      if (oi.format == WT_OUT_FP8_E4M3_B128 && ds.scale_off != WT_OFFSET_AUTO)
        cursor[ds.rank] = std::max(cursor[ds.rank], ds.scale_off + ds.scale_bytes);
    }
  for (auto& oi : p->outputs)
    for (auto& ds : oi.dsts) {
      uint64_t& c = cursor[ds.rank];
      if (ds.data_off == WT_OFFSET_AUTO) {
        ds.data_off = align_up(c, 256);
        c = ds.data_off + ds.data_bytes;
      }
      if (oi.format == WT_OUT_FP8_E4M3_B128) {
        if (ds.scale_off == WT_OFFSET_AUTO) {
          ds.scale_off = align_up(c, 256);
          c = ds.scale_off + ds.scale_bytes;
        }
      } else {
        ds.scale_off = 0;
      }
    }
  // prove the ranges of every rank disjoint, and size the pools
  std::vector<std::vector<Range>> per_rank(d->num_ranks);
  for (int o = 0; o < (int)p->outputs.size(); ++o) {
    auto& oi = p->outputs[o];
    for (int k = 0; k < (int)oi.dsts.size(); ++k) {
      auto& ds = oi.dsts[k];
      per_rank[ds.rank].push_back({ds.data_off, ds.data_bytes, o, k, false});
      if (oi.format == WT_OUT_FP8_E4M3_B128)
        per_rank[ds.rank].push_back({ds.scale_off, ds.scale_bytes, o, k, true});
    }
  }
  for (int r = 0; r < d->num_ranks; ++r) {
    auto& v = per_rank[r];
    std::sort(v.begin(), v.end(), [](const Range& a, const Range& b) { return a.off < b.off; });
    uint64_t end = 0;
    for (size_t i = 0; i < v.size(); ++i) {
      if (i > 0 && v[i].off < v[i - 1].off + v[i - 1].bytes)
        return fail(WT_ERR_LAYOUT_OVERLAP,
                    "rank " + std::to_string(r) + ": destination of " +
                        p->outputs[v[i].out].name + " overlaps " +
                        p->outputs[v[i - 1].out].name);
      end = std::max(end, v[i].off + v[i].bytes);
    }
    p->pool_bytes[r] = end ? align_up(end, 256) : 0;
    if (d->pool_capacity && p->pool_bytes[r] > d->pool_capacity[r])
      return fail(WT_ERR_POOL_TOO_SMALL, "rank " + std::to_string(r) + ": needs " +
                                             std::to_string(p->pool_bytes[r]) + " bytes");
  }

  // ---- device tables: units, row runs, per-slot shapes -------------------
  p->h_units.clear();
  p->h_runs.clear();
  p->h_geom.clear();
  p->h_blockmap.clear();
  p->expected_blocks.assign((size_t)p->num_ranks, 0);
  p->group_counts.assign((size_t)p->num_ranks * (size_t)p->num_ranks, 0);
  std::vector<int32_t> unit_group, held_ranks;
  p->h_units.reserve((size_t)units);
  p->slot_rows.assign(p->num_slots, 0);
  p->slot_cols.assign(p->num_slots, 0);
  p->slot_tmap.assign(p->num_slots, 0);
  p->slot_view_k.assign(p->num_slots, 1);
  // the element-path test flag keeps every unaligned row on the row-by-row path
  const bool views = !(p->flags & WT_FLAG_FORCE_NARROW);
  p->slot_used.assign(p->num_slots, 0);
  p->slot_read_rows.assign(p->num_slots, 0);
  for (const auto& pi : p->params)
    for (size_t s = 0; s < pi.shard_rows.size(); ++s) {
      // a shard-local plan reads the shards of its own index whole (and,
      // with halos, leading rows of others: found below)
      const bool own = p->local_shard < 0 || (int64_t)s == p->local_shard;
      p->slot_rows[pi.slot_base + s] = pi.shard_rows[s];
      p->slot_cols[pi.slot_base + s] = pi.cols;
      p->slot_read_rows[pi.slot_base + s] = own ? pi.shard_rows[s] : 0;
      // tensor maps only for whole shards: a one-shard block lies in a shard
      // of this plan's own index. Rows that are not 16-byte aligned get a
      // view map (k consecutive rows per view row, see tmap.cpp) when the
      // shard holds a whole view row and a view row is at least one box wide.
      const auto& oi = p->outputs[pi.output];
      const int32_t k = view_rows(pi.cols);
      p->slot_view_k[pi.slot_base + s] = k;
      if (own && pi.shard_rows[s] > 0) {
        if (oi.vec)
          p->slot_tmap[pi.slot_base + s] = 1;
        else if (views && pi.shard_rows[s] >= k && (int64_t)k * pi.cols >= kViewBoxCols)
          p->slot_tmap[pi.slot_base + s] = 2;
      }
    }
  const bool halo = (p->flags & WT_FLAG_SHARD_HALO) != 0;
  p->bytes_read = p->bytes_written = 0;
  p->num_params_total = 0;
  int32_t dst_entries = 0;
  for (int o = 0; o < (int)p->outputs.size(); ++o) {
    auto& oi = p->outputs[o];
    oi.dst_begin = dst_entries;
    dst_entries += (int32_t)oi.dsts.size();
    // where each block lands in each destination
    const int64_t tiles_m = ceil_div(oi.rows, kTile), tiles_n_all = ceil_div(oi.cols, kTile);
    bool sliced = false;
    for (const DstInfo& ds : oi.dsts) {
      DevDstGeom g;
      g.dim = ds.slice_dim;
      g.map_off = -1;
      g.ld = (uint32_t)ds.cols;
      g.sld = (uint32_t)ceil_div(ds.cols, kTile);
      if (ds.slice_dim >= 0) {
        sliced = true;
        g.map_off = (int32_t)p->h_blockmap.size();
        const int64_t nblk = ds.slice_dim == 0 ? tiles_m : tiles_n_all;
        p->h_blockmap.resize(p->h_blockmap.size() + (size_t)nblk, -1);
        int32_t at = 0;
        for (size_t r = 0; r < ds.slice_begin.size(); ++r)
          for (int64_t b = ds.slice_begin[r] / kTile; b < ceil_div(ds.slice_begin[r] + ds.slice_len[r], kTile); ++b)
            p->h_blockmap[(size_t)g.map_off + (size_t)b] = at++;
      }
      p->h_geom.push_back(g);
    }
    // the runs of this output: shards of its parts in fusion order, empty
    // shards skipped (reassembly: row r of the part comes from the shard
    // whose row range holds r)
    const size_t first_run = p->h_runs.size();
    int64_t row = 0;
    for (int32_t q : oi.parts) {
      auto& pi = p->params[q];
      for (size_t s = 0; s < pi.shard_rows.size(); ++s) {
        if (pi.shard_rows[s] == 0) continue;
        p->h_runs.push_back({row, pi.shard_rows[s], pi.slot_base + (int32_t)s, (int32_t)s});
        row += pi.shard_rows[s];
      }
    }
    const int64_t tiles_n = ceil_div(oi.cols, kTile);
    const uint32_t flags = (oi.format == WT_OUT_FP8_E4M3_B128 ? kUnitFp8 : 0u) |
                           (oi.vec ? kUnitVec : 0u);
    size_t k = first_run;
    oi.unit_begin = (int64_t)p->h_units.size();
    const uint64_t esize = oi.format == WT_OUT_FP8_E4M3_B128 ? 1u : 2u;
    for (int64_t bi = 0; bi * kTile < oi.rows; ++bi) {
      const int64_t r0 = bi * kTile;
      const int64_t nrows = std::min<int64_t>(kTile, oi.rows - r0);
      while (p->h_runs[k].row0 + p->h_runs[k].rows <= r0) ++k;
      const DevRun& run = p->h_runs[k];
      const bool single = run.row0 + run.rows >= r0 + nrows;
      if (p->local_shard >= 0) {
        // shard-local: a block row belongs to the shard holding its first
        // row; without halos it must lie wholly in that shard
        if (!single && !halo)
          return fail(WT_ERR_SHAPE, oi.name + ": block row " + std::to_string(bi) +
                                        " spans shards; shard-local preparation needs shard "
                                        "boundaries on multiples of 128 rows of every output "
                                        "(or WT_FLAG_SHARD_HALO)");
        if (run.shard != p->local_shard) continue;
        // the leading rows of later shards that this block reads (its halo)
        for (size_t q = k + 1; q < p->h_runs.size() && p->h_runs[q].row0 < r0 + nrows; ++q) {
          const DevRun& hr = p->h_runs[q];
          int64_t& got = p->slot_read_rows[(size_t)hr.slot];
          got = std::max(got, std::min(hr.rows, r0 + nrows - hr.row0));
        }
      }
      // one shard and 16-byte rows: one 2-D tensor copy from that shard
      const bool tma = single && oi.vec;
      // unaligned rows from one shard whose view map holds all of the
      // block's rows: k tensor copies instead of a bulk copy per row
      bool view = false;
      if (single && !oi.vec && p->slot_tmap[(size_t)run.slot] == 2) {
        const int64_t k = p->slot_view_k[(size_t)run.slot];
        const int64_t s0 = r0 - run.row0;
        view = s0 + nrows <= (run.rows / k) * k;
      }
      // rows gathered one by one that the consumers load straight from the
      // shards instead of through a bulk copy per row: 16-byte rows from
      // several shards, and rows at most one 16-byte chunk wide
      const bool direct = (!single && oi.vec) || (!oi.vec && oi.cols <= 8);
      const uint32_t f = flags | (single ? 0u : kUnitMulti) | (sliced ? kUnitSliced : 0u) |
                         (view ? kUnitView : 0u) | (direct ? kUnitDirect : 0u);
      for (int64_t bj = 0; bj < tiles_n; ++bj) {
        const int64_t ncols = std::min<int64_t>(kTile, oi.cols - bj * kTile);
        DevUnit u;
        u.src = tma ? (uint32_t)run.slot : (uint32_t)k;
        u.src_row = tma ? (uint32_t)(r0 - run.row0) : (uint32_t)r0;
        u.bi = (uint32_t)bi;
        u.bj = (uint32_t)bj;
        u.cols = (uint32_t)oi.cols;
        u.shape = (uint32_t)(nrows - 1) | ((uint32_t)(ncols - 1) << 8) | (f << 16);
        u.num_dsts = (uint32_t)oi.dsts.size();
        u.dst_begin = (uint32_t)oi.dst_begin;
        // the destinations that hold this block; what the step moves is
        // counted from the units it runs
        int32_t held = 0, which = -1, min_rank = -1;
        const uint64_t elems = uint64_t(nrows * ncols);
        held_ranks.clear();
        for (size_t d = 0; d < oi.dsts.size(); ++d) {
          const DevDstGeom& g = p->h_geom[(size_t)oi.dst_begin + d];
          const bool in = g.dim < 0 || p->h_blockmap[(size_t)g.map_off + (size_t)(g.dim == 0 ? bi : bj)] >= 0;
          if (!in) continue;
          ++held;
          which = (int32_t)d;
          const int32_t rk = oi.dsts[d].rank;
          p->expected_blocks[(size_t)rk] += 1;
          p->bytes_written += elems * esize + (esize == 1 ? 4u : 0u);
          held_ranks.push_back(rk);
          if (min_rank < 0 || rk < min_rank) min_rank = rk;
        }
        // rank groups: a unit belongs to the group of the lowest rank that
        // holds its block (group 0 if none does)
        const int32_t grp = std::max(min_rank, 0);
        unit_group.push_back(grp);
        for (int32_t rk : held_ranks) ++p->group_counts[(size_t)grp * (size_t)p->num_ranks + (size_t)rk];
        p->bytes_read += elems * 2u;
        p->num_params_total += (int64_t)elems;
        // when exactly one destination holds it, the unit names that one
        // alone (the kernel's single-destination path)
        if (sliced && held <= 1) {
          u.num_dsts = (uint32_t)held;
          u.dst_begin = (uint32_t)(oi.dst_begin + std::max(which, 0));
        }
        p->h_units.push_back(u);
      }
    }
    oi.num_units = (int64_t)p->h_units.size() - oi.unit_begin;
  }
  p->num_dst_entries = dst_entries;
  p->num_units = (int64_t)p->h_units.size();
  // Units whose rows are gathered row by row (rows from several shards, or
  // rows that are not 16-byte aligned: a bulk copy per row, or loads by the
  // consumers from published row addresses) take longer than a
  // tensor-copied block; a launch hands them out first, so that they
  // overlap the streaming blocks instead of forming its tail.
  auto slow = [&](int64_t u) {
    const uint32_t f = p->h_units[(size_t)u].shape >> 16;
    return (f & kUnitMulti) || !(f & kUnitVec);
  };
  // units in rank-group order, slow units first within a group, plan order
  // otherwise, and where each group starts
  p->rank_perm.resize((size_t)p->num_units);
  p->group_begin.assign((size_t)p->num_ranks + 1, 0);
  for (int32_t g : unit_group) ++p->group_begin[(size_t)g + 1];
  for (int32_t r = 0; r < p->num_ranks; ++r) p->group_begin[(size_t)r + 1] += p->group_begin[(size_t)r];
  {
    std::vector<int64_t> at(p->group_begin.begin(), p->group_begin.end() - 1);
    for (int pass = 0; pass < 2; ++pass)
      for (int64_t u = 0; u < p->num_units; ++u)
        if (slow(u) == (pass == 0)) p->rank_perm[(size_t)at[(size_t)unit_group[(size_t)u]]++] = (uint32_t)u;
  }
  // the order of a whole-step launch (and of each offload chunk, whose unit
  // range it keeps): slow units first; left empty when there are none
  p->launch_perm.clear();
  for (int32_t s = 0; s < p->num_slots; ++s) p->slot_used[(size_t)s] = p->slot_read_rows[(size_t)s] > 0;

  // ---- packed host image for offload and its chunks ----------------------
  p->shard_host_off.assign(p->num_slots, 0);
  uint64_t hcur = 0;
  std::vector<uint64_t> out_host_begin(p->outputs.size() + 1, 0);
  for (int o = 0; o < (int)p->outputs.size(); ++o) {
    auto& oi = p->outputs[o];
    out_host_begin[o] = hcur;
    for (int32_t q : oi.parts) {
      auto& pi = p->params[q];
      for (size_t s = 0; s < pi.shard_rows.size(); ++s) {
        hcur = align_up(hcur, 256);
        p->shard_host_off[pi.slot_base + s] = hcur;
        hcur += uint64_t(pi.shard_rows[s] * pi.cols) * 2u;
      }
    }
    hcur = align_up(hcur, 256);
  }
  out_host_begin[p->outputs.size()] = hcur;
  p->host_bytes = hcur;
  p->chunk_bytes = d->offload_chunk_bytes;
  p->chunks.clear();
  p->staging_bytes = 0;
  if (p->chunk_bytes > 0) {
    int o = 0;
    const int n = (int)p->outputs.size();
    while (o < n) {
      Chunk c;
      c.out_begin = o;
      c.host_begin = out_host_begin[o];
      int e = o + 1;
      while (e < n && out_host_begin[e + 1] - c.host_begin <= p->chunk_bytes) ++e;
      c.out_end = e;
      c.host_bytes = out_host_begin[e] - c.host_begin;
      c.unit_begin = p->outputs[o].unit_begin;
      c.unit_end = p->outputs[e - 1].unit_begin + p->outputs[e - 1].num_units;
      p->staging_bytes = std::max(p->staging_bytes, c.host_bytes);
      p->chunks.push_back(c);
      o = e;
    }
  }
  bool any_slow = false;
  for (int64_t u = 0; u < p->num_units && !any_slow; ++u) any_slow = slow(u);
  if (any_slow) {
    std::vector<std::pair<int64_t, int64_t>> ranges;
    for (const Chunk& c : p->chunks) ranges.push_back({c.unit_begin, c.unit_end});
    if (ranges.empty()) ranges.push_back({0, p->num_units});
    p->launch_perm.reserve((size_t)p->num_units);
    for (const auto& rg : ranges)
      for (int pass = 0; pass < 2; ++pass)
        for (int64_t u = rg.first; u < rg.second; ++u)
          if (slow(u) == (pass == 0)) p->launch_perm.push_back((uint32_t)u);
  }
  return WT_OK;
}

}  // namespace wt
