// C ABI of the preparation library (declared in include/wt.h): plan
// creation and upload, the per-step wt_prepare, the CPU-offload pipeline
// (host-to-device copies on one stream overlapping preparation on another,
// "Weight transfer for RL post-training in under 2 seconds", sections
// "Task pipeline" and "GPU memory usage control"), checks and teardown.
#include <algorithm>
#include <cstring>
#include <new>
#include <string>

#include <nvtx3/nvToolsExt.h>

#include "plan.h"

namespace wt {

namespace {
thread_local std::string g_last_error;

struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

// An NVTX range over one host-side entry point (plan compilation, the
// queueing of a step), for timelines taken with a profiler; without one
// attached the calls do nothing.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

wt_status fail(wt_status s, const std::string& msg) {
  set_error(msg);
  return s;
}

wt_status cuda_fail(cudaError_t e, const char* what) {
  return fail(WT_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

void free_device(Plan& p) {
  if (p.device < 0) return;
  DeviceGuard g(p.device);
  if (p.d_tables) cudaFree(p.d_tables);
  for (PtrSet& ps : p.sets) {
    if (ps.h_pinned) cudaFreeHost(ps.h_pinned);
    if (ps.upload_done) cudaEventDestroy(ps.upload_done);
    ps.h_pinned = nullptr;
    ps.upload_done = nullptr;
  }
  for (int b = 0; b < 2; ++b) {
    if (p.staging[b]) cudaFree(p.staging[b]);
    if (p.h2d_done[b]) cudaEventDestroy(p.h2d_done[b]);
    if (p.prep_done[b]) cudaEventDestroy(p.prep_done[b]);
  }
  if (p.last_done) cudaEventDestroy(p.last_done);
  p.d_tables = nullptr;
}

// Layout of a pointer-table block (identical on the device and in its
// pinned staging buffer): shard pointers, their tensor maps, destinations,
// and per shard whether its map is a view map.
struct DynLayout {
  size_t shards = 0, tmaps = 0, dsts = 0, views = 0, bytes = 0;
};

DynLayout dyn_layout(const Plan& p) {
  DynLayout d;
  d.shards = 0;
  d.tmaps = align256(d.shards + (size_t)p.num_slots * sizeof(void*));
  d.dsts = align256(d.tmaps + (size_t)p.num_slots * kTmapBytes);
  d.views = align256(d.dsts + (size_t)p.num_dst_entries * sizeof(DevDstPtr));
  d.bytes = align256(d.views + (size_t)p.num_slots);
  return d;
}

// A failed allocation leaves its (non-sticky) error as the runtime's last
// error; take it back so that a later call's launch check does not report
// it as its own failure.
wt_status alloc_fail(const char* what) {
  (void)cudaGetLastError();
  return fail(WT_ERR_OUT_OF_MEMORY, what);
}

// Upload the static tables and allocate what the per-step calls need, so
// that wt_prepare and wt_prepare_offload never allocate.
wt_status upload(Plan& p, int device) {
  int count = 0;
  cudaError_t e = cudaGetDeviceCount(&count);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceCount");
  if (device >= count) return fail(WT_ERR_INVALID_ARGUMENT, "device index out of range");
  DeviceGuard g(device);
  if (!g.ok) return fail(WT_ERR_CUDA, "cudaSetDevice failed");
  p.device = device;
  e = cudaDeviceGetAttribute(&p.sm_count, cudaDevAttrMultiProcessorCount, device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  if ((e = prep_kernel_setup()) != cudaSuccess) return cuda_fail(e, "preparation kernel set-up");

  const size_t n_slots = (size_t)p.num_slots;
  const bool offload = p.chunk_bytes > 0;
  const DynLayout dl = dyn_layout(p);
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
  const size_t o_dyn = take(dl.bytes * kPtrSets);
  const size_t o_units = take(p.h_units.size() * sizeof(DevUnit));
  const size_t o_units_rank = take(p.h_units.size() * sizeof(DevUnit));
  const size_t o_runs = take(p.h_runs.size() * sizeof(DevRun));
  const size_t o_geom = take(p.h_geom.size() * sizeof(DevDstGeom));
  const size_t o_bmap = take(p.h_blockmap.size() * sizeof(int32_t));
  const size_t o_gcounts = take(p.group_counts.size() * sizeof(uint32_t));
  // per-rank block counts of a whole step and of each offload chunk
  std::vector<uint32_t> lc((1 + p.chunks.size()) * (size_t)p.num_ranks, 0);
  for (int32_t r = 0; r < p.num_ranks; ++r) lc[(size_t)r] = (uint32_t)p.expected_blocks[(size_t)r];
  for (size_t c = 0; c < p.chunks.size(); ++c)
    for (int32_t o = p.chunks[c].out_begin; o < p.chunks[c].out_end; ++o)
      for (const DstInfo& ds : p.outputs[o].dsts)
        lc[(1 + c) * (size_t)p.num_ranks + (size_t)ds.rank] +=
            (uint32_t)(((ds.rows + kTile - 1) / kTile) * ((ds.cols + kTile - 1) / kTile));
  const size_t o_lc = take(lc.size() * sizeof(uint32_t));
  const size_t o_err = take(sizeof(int32_t));
  const size_t o_ticket = take(2 * sizeof(uint32_t) * (1 + (size_t)p.num_ranks));
  const size_t o_offl_s = take(offload ? n_slots * sizeof(void*) : 0);
  const size_t o_offl_t = take(offload ? n_slots * kTmapBytes : 0);
  const size_t o_offl_v = take(offload ? n_slots : 0);
  e = cudaMalloc(&p.d_tables, std::max<size_t>(off, 256));
  if (e != cudaSuccess) return alloc_fail("cudaMalloc of plan tables failed");
  char* base = static_cast<char*>(p.d_tables);
  auto put = [&](size_t o, const void* src, size_t bytes) {
    return bytes ? cudaMemcpy(base + o, src, bytes, cudaMemcpyHostToDevice) : cudaSuccess;
  };
  // the unit table in launch order and in rank-group order
  std::vector<DevUnit> ordered(p.h_units.size());
  const std::vector<DevUnit>* launch_units = &p.h_units;
  if (!p.launch_perm.empty()) {
    for (size_t i = 0; i < ordered.size(); ++i) ordered[i] = p.h_units[p.launch_perm[i]];
    launch_units = &ordered;
  }
  if ((e = cudaMemset(base + o_dyn, 0, dl.bytes * kPtrSets)) != cudaSuccess ||
      (e = put(o_units, launch_units->data(), p.h_units.size() * sizeof(DevUnit))) != cudaSuccess)
    return cuda_fail(e, "uploading plan tables");
  for (size_t i = 0; i < ordered.size(); ++i) ordered[i] = p.h_units[p.rank_perm[i]];
  if ((e = put(o_units_rank, ordered.data(), ordered.size() * sizeof(DevUnit))) != cudaSuccess ||
      (e = put(o_runs, p.h_runs.data(), p.h_runs.size() * sizeof(DevRun))) != cudaSuccess ||
      (e = put(o_geom, p.h_geom.data(), p.h_geom.size() * sizeof(DevDstGeom))) != cudaSuccess ||
      (e = put(o_bmap, p.h_blockmap.data(), p.h_blockmap.size() * sizeof(int32_t))) != cudaSuccess ||
      (e = put(o_gcounts, p.group_counts.data(), p.group_counts.size() * sizeof(uint32_t))) != cudaSuccess ||
      (e = put(o_lc, lc.data(), lc.size() * sizeof(uint32_t))) != cudaSuccess ||
      (e = cudaMemset(base + o_err, 0, sizeof(int32_t))) != cudaSuccess ||
      (e = cudaMemset(base + o_ticket, 0, 2 * sizeof(uint32_t) * (1 + (size_t)p.num_ranks))) != cudaSuccess)
    return cuda_fail(e, "uploading plan tables");
  p.dyn_bytes = dl.bytes;
  p.d_error = reinterpret_cast<int32_t*>(base + o_err);
  p.d_units_launch = reinterpret_cast<const DevUnit*>(base + o_units);
  p.d_units_rank = reinterpret_cast<const DevUnit*>(base + o_units_rank);
  p.args.units = p.d_units_launch;
  p.args.runs = reinterpret_cast<const DevRun*>(base + o_runs);
  p.d_tickets = reinterpret_cast<uint32_t*>(base + o_ticket);
  p.args.ticket = p.d_tickets;
  p.args.geom = reinterpret_cast<const DevDstGeom*>(base + o_geom);
  p.d_group_counts = reinterpret_cast<const uint32_t*>(base + o_gcounts);
  p.d_launch_counts = reinterpret_cast<uint32_t*>(base + o_lc);
  p.args.blockmap = reinterpret_cast<const int32_t*>(base + o_bmap);
  p.args.error_word = p.d_error;
  p.args.timeout_ns = kDefaultTimeoutNs;

  for (int j = 0; j < kPtrSets; ++j) {
    PtrSet& ps = p.sets[j];
    ps.d_block = reinterpret_cast<unsigned char*>(base + o_dyn + (size_t)j * dl.bytes);
    e = cudaHostAlloc(&ps.h_pinned, std::max<size_t>(dl.bytes, 256), cudaHostAllocDefault);
    if (e != cudaSuccess) return alloc_fail("pinned pointer staging allocation failed");
    std::memset(ps.h_pinned, 0, std::max<size_t>(dl.bytes, 256));
    if ((e = cudaEventCreateWithFlags(&ps.upload_done, cudaEventDisableTiming)) != cudaSuccess)
      return cuda_fail(e, "cudaEventCreate");
    ps.shards.assign(n_slots, nullptr);
    ps.pools.assign((size_t)p.num_ranks, nullptr);
  }
  if ((e = cudaEventCreateWithFlags(&p.last_done, cudaEventDisableTiming)) != cudaSuccess)
    return cuda_fail(e, "cudaEventCreate");

  if (offload) {
    // the watermark: two staging buffers of the largest chunk
    for (int b = 0; b < 2; ++b) {
      if (p.staging_bytes && cudaMalloc(&p.staging[b], p.staging_bytes) != cudaSuccess)
        return alloc_fail("offload staging allocation failed");
      if ((e = cudaEventCreateWithFlags(&p.h2d_done[b], cudaEventDisableTiming)) != cudaSuccess ||
          (e = cudaEventCreateWithFlags(&p.prep_done[b], cudaEventDisableTiming)) != cudaSuccess)
        return cuda_fail(e, "cudaEventCreate");
    }
    // static tables: chunk c's shards live in staging[c % 2]
    std::vector<const void*> tbl(n_slots, nullptr);
    for (size_t c = 0; c < p.chunks.size(); ++c) {
      const Chunk& ch = p.chunks[c];
      char* st = static_cast<char*>(p.staging[c % 2]);
      for (int o = ch.out_begin; o < ch.out_end; ++o)
        for (int32_t q : p.outputs[o].parts) {
          const ParamInfo& pi = p.params[q];
          for (size_t s = 0; s < pi.shard_rows.size(); ++s) {
            const size_t slot = pi.slot_base + s;
            tbl[slot] = st + (p.shard_host_off[slot] - ch.host_begin);
          }
        }
    }
    std::vector<unsigned char> maps(n_slots * kTmapBytes);
    std::vector<uint8_t> views(n_slots, 0);
    if (n_slots) {
      wt_status st = encode_tmaps(p, tbl.data(), maps.data(), views.data());
      if (st != WT_OK) return st;
    }
    p.d_offload_shard_ptrs = reinterpret_cast<const uint16_t**>(base + o_offl_s);
    p.d_offload_tmaps = reinterpret_cast<unsigned char*>(base + o_offl_t);
    p.d_offload_view_ok = reinterpret_cast<const uint8_t*>(base + o_offl_v);
    if ((e = put(o_offl_s, tbl.data(), n_slots * sizeof(void*))) != cudaSuccess ||
        (e = put(o_offl_t, maps.data(), n_slots * kTmapBytes)) != cudaSuccess ||
        (e = put(o_offl_v, views.data(), n_slots)) != cudaSuccess)
      return cuda_fail(e, "uploading offload tables");
    p.offload_tmaps_dirty = true;
  }
  return WT_OK;
}

// Check the caller's pointers and find the pointer-table set that holds
// them; when none does, rebuild the least recently used set on the host
// (shard pointers, the shards' tensor maps, absolute destination addresses,
// each part only if it changed) and queue one copy of it on s. shards ==
// NULL (offload): only the destinations matter. The only host wait is for
// the earlier upload from the replaced set's staging buffer, kPtrSets
// uploads back.
wt_status stage_pointers(Plan& p, const void* const* shards, void* const* pools, cudaStream_t s,
                         bool capturing, int* set_out) {
  const size_t n_slots = (size_t)p.num_slots, n_ranks = (size_t)p.num_ranks;
  auto same_shards = [&](const PtrSet& ps) {
    return ps.shards_valid && std::equal(ps.shards.begin(), ps.shards.end(), shards);
  };
  auto same_pools = [&](const PtrSet& ps) {
    return ps.pools_valid && std::equal(ps.pools.begin(), ps.pools.end(), pools);
  };
  for (int j = 0; j < kPtrSets; ++j) {
    PtrSet& ps = p.sets[j];
    if (same_pools(ps) && (!shards || same_shards(ps))) {
      ps.last_use = ++p.use_clock;
      // a graph replays this set's addresses: it must stay as it is
      if (capturing) ps.captured = true;
      *set_out = j;
      return WT_OK;
    }
  }
  // a captured copy would read the staging buffer at every replay, after
  // later calls may have rewritten it
  if (capturing)
    return fail(WT_ERR_INVALID_ARGUMENT,
                "new shard or pool pointers inside a stream capture: stage them with an uncaptured call first");
  int victim = -1;
  for (int j = 0; j < kPtrSets; ++j)
    if (!p.sets[j].captured && (victim < 0 || p.sets[j].last_use < p.sets[victim].last_use)) victim = j;
  if (victim < 0)
    return fail(WT_ERR_INVALID_ARGUMENT,
                "every pointer-table set holds addresses that a captured CUDA graph replays");
  PtrSet& ps = p.sets[victim];
  const bool shards_changed = shards && !same_shards(ps);
  const bool pools_changed = !same_pools(ps);
  if (pools_changed)
    for (size_t r = 0; r < n_ranks; ++r) {
      if (p.pool_bytes[r] == 0) continue;
      if (!pools[r]) return fail(WT_ERR_INVALID_ARGUMENT, "pool " + std::to_string(r) + " is NULL");
      if (reinterpret_cast<uintptr_t>(pools[r]) % 16)
        return fail(WT_ERR_ALIGNMENT, "pool " + std::to_string(r) + " is not 16-byte aligned");
    }
  if (shards_changed)
    for (const ParamInfo& pi : p.params) {
      const bool vec = p.outputs[pi.output].vec;
      for (size_t k = 0; k < pi.shard_rows.size(); ++k) {
        const void* ptr = shards[pi.slot_base + k];
        if (!p.slot_used[pi.slot_base + k]) continue;   // empty, or not this plan's shard
        if (!ptr) return fail(WT_ERR_INVALID_ARGUMENT, pi.name + ": shard " + std::to_string(k) + " is NULL");
        if (reinterpret_cast<uintptr_t>(ptr) % (vec ? 16 : 2))
          return fail(WT_ERR_ALIGNMENT, pi.name + ": shard " + std::to_string(k) + " is misaligned");
      }
    }
  // the staging buffer may still be read by this set's previous upload
  cudaError_t e = ps.uploaded ? cudaEventSynchronize(ps.upload_done) : cudaSuccess;
  if (e != cudaSuccess) return cuda_fail(e, "waiting for an earlier pointer upload");
  const DynLayout dl = dyn_layout(p);
  char* h = static_cast<char*>(ps.h_pinned);
  if (shards_changed) {
    ps.shards_valid = false;
    std::memcpy(h + dl.shards, shards, n_slots * sizeof(void*));
    wt_status st = encode_tmaps(p, shards, reinterpret_cast<unsigned char*>(h + dl.tmaps),
                                reinterpret_cast<uint8_t*>(h + dl.views));
    if (st != WT_OK) return st;
    ps.tmaps_dirty = true;
  }
  if (pools_changed) {
    ps.pools_valid = false;
    DevDstPtr* dp = reinterpret_cast<DevDstPtr*>(h + dl.dsts);
    for (const OutputInfo& oi : p.outputs)
      for (size_t k = 0; k < oi.dsts.size(); ++k) {
        const DstInfo& ds = oi.dsts[k];
        uint8_t* pool = static_cast<uint8_t*>(pools[ds.rank]);
        DevDstPtr& d = dp[oi.dst_begin + k];
        d.data = pool + ds.data_off;
        d.scale = oi.format == WT_OUT_FP8_E4M3_B128 ? reinterpret_cast<float*>(pool + ds.scale_off) : nullptr;
        d.pool_begin = pool;
        d.pool_end = pool + p.pool_bytes[ds.rank];
      }
  }
  e = cudaMemcpyAsync(ps.d_block, h, dl.bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "pointer table upload");
  if ((e = cudaEventRecord(ps.upload_done, s)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  ps.uploaded = true;
  if (shards_changed) {
    std::copy(shards, shards + n_slots, ps.shards.begin());
    ps.shards_valid = true;
  }
  std::copy(pools, pools + n_ranks, ps.pools.begin());
  ps.pools_valid = true;
  ps.last_use = ++p.use_clock;
  *set_out = victim;
  return WT_OK;
}

// The kernel's view of one pointer-table set.
void bind_set(const Plan& p, const PtrSet& ps, PrepArgs& a) {
  const DynLayout dl = dyn_layout(p);
  a.shard_ptrs = reinterpret_cast<const uint16_t* const*>(ps.d_block + dl.shards);
  a.tmaps = ps.d_block + dl.tmaps;
  a.dst_ptrs = reinterpret_cast<const DevDstPtr*>(ps.d_block + dl.dsts);
  a.view_ok = ps.d_block + dl.views;
}

// One persistent CTA per SM (each holds a 128 KiB shared-memory ring).
int grid_for(const Plan& p, int64_t units) {
  return (int)std::max<int64_t>(1, std::min<int64_t>(units, p.sm_count));
}

}  // namespace

void set_error(const std::string& msg) { g_last_error = msg; }

}  // namespace wt

using namespace wt;

extern "C" {

wt_status wt_plan_create(const wt_plan_desc* desc, int device, wt_plan** out) {
  NvtxRange range("wt_plan_create");
  if (!out) return fail(WT_ERR_INVALID_ARGUMENT, "out is NULL");
  if (device < -1) return fail(WT_ERR_INVALID_ARGUMENT, "device must be >= -1");
  wt_plan* h = new (std::nothrow) wt_plan;
  if (!h) return fail(WT_ERR_OUT_OF_MEMORY, "host allocation failed");
  wt_status st;
  try {
    st = compile_plan(desc, &h->p);
  } catch (const std::bad_alloc&) {
    st = fail(WT_ERR_OUT_OF_MEMORY, "host allocation failed");
  }
  if (st == WT_OK && device >= 0) {
    st = upload(h->p, device);
    if (st != WT_OK) free_device(h->p);
  }
  if (st != WT_OK) {
    delete h;
    return st;
  }
  *out = h;
  return WT_OK;
}

wt_status wt_plan_pool_bytes(const wt_plan* h, int32_t rank, uint64_t* bytes) {
  if (!h || !bytes) return fail(WT_ERR_INVALID_ARGUMENT, "NULL argument");
  if (rank < 0 || rank >= h->p.num_ranks) return fail(WT_ERR_INVALID_ARGUMENT, "rank out of range");
  *bytes = h->p.pool_bytes[rank];
  return WT_OK;
}

wt_status wt_plan_output_layout(const wt_plan* h, int32_t out, int32_t dst, int32_t* rank,
                                uint64_t* data_off, uint64_t* scale_off) {
  if (!h || !rank || !data_off || !scale_off) return fail(WT_ERR_INVALID_ARGUMENT, "NULL argument");
  if (out < 0 || out >= (int32_t)h->p.outputs.size()) return fail(WT_ERR_INVALID_ARGUMENT, "output out of range");
  const OutputInfo& oi = h->p.outputs[out];
  if (dst < 0 || dst >= (int32_t)oi.dsts.size()) return fail(WT_ERR_INVALID_ARGUMENT, "destination out of range");
  *rank = oi.dsts[dst].rank;
  *data_off = oi.dsts[dst].data_off;
  *scale_off = oi.dsts[dst].scale_off;
  return WT_OK;
}

wt_status wt_plan_shard_host_offset(const wt_plan* h, int32_t param, int32_t shard, uint64_t* off) {
  if (!h || !off) return fail(WT_ERR_INVALID_ARGUMENT, "NULL argument");
  if (param < 0 || param >= (int32_t)h->p.params.size()) return fail(WT_ERR_INVALID_ARGUMENT, "param out of range");
  const ParamInfo& pi = h->p.params[param];
  if (shard < 0 || shard >= (int32_t)pi.shard_rows.size()) return fail(WT_ERR_INVALID_ARGUMENT, "shard out of range");
  *off = h->p.shard_host_off[pi.slot_base + shard];
  return WT_OK;
}

wt_status wt_plan_shard_rows_read(const wt_plan* h, int32_t param, int32_t shard, int64_t* rows) {
  if (!h || !rows) return fail(WT_ERR_INVALID_ARGUMENT, "NULL argument");
  if (param < 0 || param >= (int32_t)h->p.params.size()) return fail(WT_ERR_INVALID_ARGUMENT, "param out of range");
  const ParamInfo& pi = h->p.params[param];
  if (shard < 0 || shard >= (int32_t)pi.shard_rows.size()) return fail(WT_ERR_INVALID_ARGUMENT, "shard out of range");
  *rows = h->p.slot_read_rows[pi.slot_base + shard];
  return WT_OK;
}

wt_status wt_plan_get_stats(const wt_plan* h, wt_plan_stats* st) {
  if (!h || !st) return fail(WT_ERR_INVALID_ARGUMENT, "NULL argument");
  st->num_units = h->p.num_units;
  st->num_params_total = h->p.num_params_total;
  st->bytes_read = h->p.bytes_read;
  st->bytes_written = h->p.bytes_written;
  st->host_bytes = h->p.host_bytes;
  st->num_chunks = (int32_t)h->p.chunks.size();
  st->num_slots = h->p.num_slots;
  return WT_OK;
}

wt_status wt_prepare(wt_plan* h, const void* const* shard_ptrs, void* const* pools, void* stream) {
  NvtxRange range("wt_prepare");
  if (!h) return fail(WT_ERR_INVALID_ARGUMENT, "plan is NULL");
  Plan& p = h->p;
  if (p.device < 0) return fail(WT_ERR_INVALID_ARGUMENT, "host-only plan cannot run");
  if ((p.num_slots > 0 && !shard_ptrs) || (p.num_ranks > 0 && !pools))
    return fail(WT_ERR_INVALID_ARGUMENT, "shard_ptrs or pools is NULL");
  DeviceGuard g(p.device);
  if (!g.ok) return fail(WT_ERR_CUDA, "cudaSetDevice failed");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cap);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  const bool capturing = cap != cudaStreamCaptureStatusNone;
  int set = 0;
  wt_status st = stage_pointers(p, shard_ptrs, pools, s, capturing, &set);
  if (st != WT_OK) return st;
  PtrSet& ps = p.sets[set];
  PrepArgs a = p.args;
  bind_set(p, ps, a);
  a.timeout_ns = p.wait_limit_ns ? p.wait_limit_ns : kDefaultTimeoutNs;
  a.tmap_fence = ps.tmaps_dirty ? 1u : 0u;
  const bool debug = p.flags & WT_FLAG_DEBUG_CHECKS;
  if (p.counters && p.count_mode == WT_COUNT_PER_RANK) {
    // rank by rank: the units whose lowest holding rank is g, then their
    // counts; after launch g, ranks 0..g have all their blocks. Every launch
    // after the first may start while the one before drains (programmatic
    // dependent launch: the groups touch disjoint bytes and each has its
    // own ticket words); each count kernel first waits for its group's
    // launch to complete.
    a.units = p.d_units_rank;
    a.stall_unit = p.stall_pos_rank;
    bool first = true;
    for (int32_t g = 0; g < p.num_ranks; ++g) {
      a.unit_begin = p.group_begin[(size_t)g];
      a.unit_end = p.group_begin[(size_t)g + 1];
      if (a.unit_end == a.unit_begin) continue;
      const int grid = grid_for(p, a.unit_end - a.unit_begin);
      a.ticket = tickets_for(p.d_tickets + 2 * (1 + (size_t)g), a.unit_end - a.unit_begin, grid);
      if ((e = launch_prepare(a, grid, s, debug, !first)) != cudaSuccess)
        return cuda_fail(e, "preparation kernel launch");
      first = false;
      if ((e = launch_add_counts(p.counters, p.d_group_counts + (size_t)g * (size_t)p.num_ranks, p.num_ranks,
                                 p.d_error, s, true)) != cudaSuccess)
        return cuda_fail(e, "completion count launch");
    }
  } else {
    a.stall_unit = p.stall_pos_launch;
    a.unit_begin = 0;
    a.unit_end = p.num_units;
    const int grid = grid_for(p, p.num_units);
    a.ticket = tickets_for(p.d_tickets, p.num_units, grid);
    e = launch_prepare(a, grid, s, debug, false);
    if (e != cudaSuccess) return cuda_fail(e, "preparation kernel launch");
    if (p.counters &&
        (e = launch_add_counts(p.counters, p.d_launch_counts, p.num_ranks, p.d_error, s, false)) != cudaSuccess)
      return cuda_fail(e, "completion count launch");
  }
  if (capturing) return WT_OK;         // the graph's replays are the caller's to track
  ps.tmaps_dirty = false;
  if ((e = cudaEventRecord(p.last_done, s)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  p.ran = true;
  return WT_OK;
}

wt_status wt_prepare_offload(wt_plan* h, const void* host_image, void* const* pools,
                             void* copy_stream, void* compute_stream) {
  NvtxRange range("wt_prepare_offload");
  if (!h) return fail(WT_ERR_INVALID_ARGUMENT, "plan is NULL");
  Plan& p = h->p;
  if (p.device < 0) return fail(WT_ERR_INVALID_ARGUMENT, "host-only plan cannot run");
  if (p.chunk_bytes == 0) return fail(WT_ERR_INVALID_ARGUMENT, "plan was built without offload_chunk_bytes");
  if ((p.host_bytes > 0 && !host_image) || (p.num_ranks > 0 && !pools))
    return fail(WT_ERR_INVALID_ARGUMENT, "host_image or pools is NULL");
  DeviceGuard g(p.device);
  if (!g.ok) return fail(WT_ERR_CUDA, "cudaSetDevice failed");
  cudaStream_t cs = static_cast<cudaStream_t>(copy_stream);
  cudaStream_t ks = static_cast<cudaStream_t>(compute_stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(ks, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone ||
      cudaStreamIsCapturing(cs, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
    return fail(WT_ERR_INVALID_ARGUMENT, "wt_prepare_offload cannot be captured into a CUDA graph");
  int set = 0;
  wt_status st = stage_pointers(p, nullptr, pools, ks, false, &set);
  if (st != WT_OK) return st;
  PrepArgs a = p.args;
  bind_set(p, p.sets[set], a);
  a.shard_ptrs = p.d_offload_shard_ptrs;
  a.view_ok = p.d_offload_view_ok;
  a.tmaps = p.d_offload_tmaps;
  a.stall_unit = p.stall_pos_launch;
  a.timeout_ns = p.wait_limit_ns ? p.wait_limit_ns : kDefaultTimeoutNs;
  const char* host = static_cast<const char*>(host_image);
  auto drain = [&](wt_status s_, const std::string& msg) {
    cudaStreamSynchronize(cs);
    cudaStreamSynchronize(ks);
    return fail(s_, msg);
  };
  cudaError_t e;
  for (size_t i = 0; i < p.chunks.size(); ++i) {
    const Chunk& c = p.chunks[i];
    const int b = (int)(i & 1);
    if ((int32_t)i == p.fail_chunk)
      return drain(WT_ERR_CUDA, "injected failure before queueing chunk " + std::to_string(i));
    // the staging buffer is free once the preparation that last read it ended
    if (p.prep_recorded[b] && (e = cudaStreamWaitEvent(cs, p.prep_done[b], 0)) != cudaSuccess)
      return drain(WT_ERR_CUDA, std::string("cudaStreamWaitEvent: ") + cudaGetErrorString(e));
    if (c.host_bytes &&
        (e = cudaMemcpyAsync(p.staging[b], host + c.host_begin, c.host_bytes,
                             cudaMemcpyHostToDevice, cs)) != cudaSuccess)
      return drain(WT_ERR_CUDA, std::string("host-to-device copy: ") + cudaGetErrorString(e));
    if ((e = cudaEventRecord(p.h2d_done[b], cs)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(ks, p.h2d_done[b], 0)) != cudaSuccess)
      return drain(WT_ERR_CUDA, std::string("event: ") + cudaGetErrorString(e));
    a.unit_begin = c.unit_begin;
    a.unit_end = c.unit_end;
    a.tmap_fence = p.offload_tmaps_dirty ? 1u : 0u;
    const int grid = grid_for(p, c.unit_end - c.unit_begin);
    a.ticket = tickets_for(p.d_tickets, c.unit_end - c.unit_begin, grid);
    if ((e = launch_prepare(a, grid, ks, p.flags & WT_FLAG_DEBUG_CHECKS, false)) != cudaSuccess)
      return drain(WT_ERR_CUDA, std::string("preparation kernel launch: ") + cudaGetErrorString(e));
    if (c.unit_end > c.unit_begin) p.offload_tmaps_dirty = false;
    if (p.counters &&
        (e = launch_add_counts(p.counters, p.d_launch_counts + (1 + i) * (size_t)p.num_ranks, p.num_ranks,
                               p.d_error, ks, false)) != cudaSuccess)
      return drain(WT_ERR_CUDA, std::string("completion count launch: ") + cudaGetErrorString(e));
    if ((e = cudaEventRecord(p.prep_done[b], ks)) != cudaSuccess)
      return drain(WT_ERR_CUDA, std::string("cudaEventRecord: ") + cudaGetErrorString(e));
    p.prep_recorded[b] = true;
  }
  if ((e = cudaEventRecord(p.last_done, ks)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  p.ran = true;
  return WT_OK;
}

wt_status wt_plan_check(wt_plan* h, void* stream) {
  if (!h) return fail(WT_ERR_INVALID_ARGUMENT, "plan is NULL");
  Plan& p = h->p;
  if (p.device < 0) return fail(WT_ERR_INVALID_ARGUMENT, "host-only plan");
  DeviceGuard g(p.device);
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int32_t word = 0;
  if ((e = cudaMemcpy(&word, p.d_error, sizeof word, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "reading the error word");
  if (word) {
    cudaMemset(p.d_error, 0, sizeof(int32_t));
    if (word & kErrTimeout)
      return fail(WT_ERR_TIMEOUT, "a wait inside the preparation kernel gave up; its output is incomplete");
    return fail(WT_ERR_INTERNAL, "a store fell outside its destination range");
  }
  return WT_OK;
}

wt_status wt_debug_fail_offload_chunk(wt_plan* h, int32_t chunk) {
  if (!h) return fail(WT_ERR_INVALID_ARGUMENT, "plan is NULL");
  h->p.fail_chunk = chunk;
  return WT_OK;
}

wt_status wt_plan_set_counters(wt_plan* h, uint32_t* counters, uint32_t mode) {
  if (!h) return fail(WT_ERR_INVALID_ARGUMENT, "plan is NULL");
  if (h->p.device < 0 && counters) return fail(WT_ERR_INVALID_ARGUMENT, "host-only plan cannot signal");
  if (mode != WT_COUNT_PER_LAUNCH && mode != WT_COUNT_PER_RANK)
    return fail(WT_ERR_INVALID_ARGUMENT, "unknown counting mode");
  if (reinterpret_cast<uintptr_t>(counters) % 4) return fail(WT_ERR_ALIGNMENT, "counters must be 4-byte aligned");
  h->p.counters = counters;
  h->p.count_mode = mode;
  return WT_OK;
}

wt_status wt_plan_expected_count(const wt_plan* h, int32_t rank, uint64_t* count) {
  if (!h || !count) return fail(WT_ERR_INVALID_ARGUMENT, "NULL argument");
  if (rank < 0 || rank >= h->p.num_ranks) return fail(WT_ERR_INVALID_ARGUMENT, "rank out of range");
  *count = h->p.expected_blocks[(size_t)rank];
  return WT_OK;
}

wt_status wt_debug_stall_unit(wt_plan* h, int64_t unit, uint64_t wait_limit_ns) {
  if (!h) return fail(WT_ERR_INVALID_ARGUMENT, "plan is NULL");
  if (unit < -1 || unit >= h->p.num_units) return fail(WT_ERR_INVALID_ARGUMENT, "unit out of range");
  Plan& p = h->p;
  p.stall_unit = unit;
  p.stall_pos_launch = p.stall_pos_rank = -1;
  for (int64_t i = 0; unit >= 0 && i < p.num_units; ++i) {
    if ((p.launch_perm.empty() ? i : (int64_t)p.launch_perm[(size_t)i]) == unit) p.stall_pos_launch = i;
    if ((int64_t)p.rank_perm[(size_t)i] == unit) p.stall_pos_rank = i;
  }
  p.wait_limit_ns = wait_limit_ns;
  return WT_OK;
}

wt_status wt_plan_destroy(wt_plan* h) {
  if (!h) return WT_OK;
  wt_status st = WT_OK;
  if (h->p.device >= 0 && h->p.ran) {
    DeviceGuard g(h->p.device);
    cudaError_t e = cudaEventSynchronize(h->p.last_done);
    if (e != cudaSuccess) st = cuda_fail(e, "waiting for the plan's last step");
  }
  free_device(h->p);
  delete h;
  return st;
}

const char* wt_status_string(wt_status s) {
  switch (s) {
    case WT_OK: return "WT_OK";
    case WT_ERR_INVALID_ARGUMENT: return "WT_ERR_INVALID_ARGUMENT";
    case WT_ERR_SHAPE: return "WT_ERR_SHAPE";
    case WT_ERR_LAYOUT_OVERLAP: return "WT_ERR_LAYOUT_OVERLAP";
    case WT_ERR_POOL_TOO_SMALL: return "WT_ERR_POOL_TOO_SMALL";
    case WT_ERR_ALIGNMENT: return "WT_ERR_ALIGNMENT";
    case WT_ERR_OUT_OF_MEMORY: return "WT_ERR_OUT_OF_MEMORY";
    case WT_ERR_CUDA: return "WT_ERR_CUDA";
    case WT_ERR_TIMEOUT: return "WT_ERR_TIMEOUT";
    case WT_ERR_INTERNAL: return "WT_ERR_INTERNAL";
  }
  return "WT_ERR_UNKNOWN";
}

const char* wt_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
