// wt_prepare_noalloc: one preparation step that allocates no device memory.
//
// wt_plan_create keeps its schedule tables (unit descriptors, row runs,
// pointer tables, an error word) in device memory it obtains with
// cudaMalloc. Some callers cannot allow that: code that runs inside a
// memory pool or arena it does not own, a process whose device memory is
// fully reserved up front by an inference engine, or a host path that must
// not touch the device allocator at all. For them this entry point compiles
// the schedule on the host on every call and copies its tables into one
// fixed scratch array that lives in the library image on each device, then
// runs the same preparation kernel as wt_prepare. The caller passes inputs
// (shards) and outputs (pools) as usual.
//
// The array's last 256 bytes hold the kernel's error word. Uploads never
// reach it, so a wait that gave up stays recorded until wt_noalloc_check
// reads and clears it. A library mutex spans each call's upload and launch,
// so calls that several host threads queue on one stream stay paired.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "plan.h"

namespace wt {
namespace {

// Maximum size of the schedule tables one call may use. Every device that
// loads the library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;   // 4 MiB
// the error word's offset: the last 256 bytes, never uploaded over
constexpr size_t kErrorOffset = kNoAllocScratchBytes - 256;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;                          // set-up, and each call's upload + launch
void* g_scratch_addr[kMaxDevices] = {};   // device address of the array, per device
int g_sm_count[kMaxDevices] = {};
// testing hook (wt_debug_noalloc_stall_unit), read under g_mu
int64_t g_stall_unit = -1;
uint64_t g_wait_limit_ns = 0;

size_t up256(size_t v) { return (v + 255) & ~size_t(255); }

wt_status fail_na(wt_status s, const std::string& msg) {
  set_error(msg);
  return s;
}

// With `device` current: the array's device address (host code only sees a
// host-side stand-in under its name) and the launch geometry, once per device.
// Called with g_mu held.
wt_status device_setup(int device) {
  if (g_scratch_addr[device]) return WT_OK;
  void* ptr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (e != cudaSuccess || !ptr)
    return fail_na(WT_ERR_CUDA, std::string("cudaGetSymbolAddress of the scratch array: ") +
                                    cudaGetErrorString(e));
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (e != cudaSuccess) return fail_na(WT_ERR_CUDA, std::string("cudaDeviceGetAttribute: ") + cudaGetErrorString(e));
  if ((e = prep_kernel_setup()) != cudaSuccess)
    return fail_na(WT_ERR_CUDA, std::string("preparation kernel set-up: ") + cudaGetErrorString(e));
  g_sm_count[device] = sms;
  g_scratch_addr[device] = ptr;
  return WT_OK;
}

}  // namespace
}  // namespace wt

using namespace wt;

extern "C" wt_status wt_prepare_noalloc(const wt_plan_desc* desc, const void* const* shard_ptrs,
                                        void* const* pools, void* stream) {
  if (!desc) return fail_na(WT_ERR_INVALID_ARGUMENT, "descriptor is NULL");
  if (desc->offload_chunk_bytes != 0)
    return fail_na(WT_ERR_INVALID_ARGUMENT, "wt_prepare_noalloc does not stage offloaded shards");
  if (desc->flags & WT_FLAG_DEBUG_CHECKS)
    return fail_na(WT_ERR_INVALID_ARGUMENT, "wt_prepare_noalloc has no debug-check readback");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the upload reads a host image that lives only for this call; a graph
  // node would read it again at every replay, after it is gone
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t ce = cudaStreamIsCapturing(s, &cap);
  if (ce != cudaSuccess)
    return fail_na(WT_ERR_CUDA, std::string("cudaStreamIsCapturing: ") + cudaGetErrorString(ce));
  if (cap != cudaStreamCaptureStatusNone)
    return fail_na(WT_ERR_INVALID_ARGUMENT, "wt_prepare_noalloc cannot be captured into a CUDA graph");
  Plan p;
  wt_status st = compile_plan(desc, &p);
  if (st != WT_OK) return st;

  // table image: shard pointers, their tensor maps, destinations, unit
  // descriptors, row runs, destination geometry and block maps, and the
  // kernel's ticket counter (zero, like every launch needs it)
  const size_t n_slots = (size_t)p.num_slots;
  const size_t o_shards = 0;
  const size_t o_tmaps = up256(o_shards + n_slots * sizeof(void*));
  const size_t o_dsts = up256(o_tmaps + n_slots * kTmapBytes);
  const size_t o_views = up256(o_dsts + (size_t)p.num_dst_entries * sizeof(DevDstPtr));
  const size_t o_units = up256(o_views + n_slots);
  const size_t o_runs = up256(o_units + p.h_units.size() * sizeof(DevUnit));
  const size_t o_geom = up256(o_runs + p.h_runs.size() * sizeof(DevRun));
  const size_t o_bmap = up256(o_geom + p.h_geom.size() * sizeof(DevDstGeom));
  const size_t o_ticket = up256(o_bmap + p.h_blockmap.size() * sizeof(int32_t));
  const size_t total = o_ticket + 256;
  if (total > kErrorOffset)
    return fail_na(WT_ERR_INVALID_ARGUMENT,
                   "schedule tables need " + std::to_string(total) +
                       " bytes; wt_prepare_noalloc holds at most " +
                       std::to_string(kErrorOffset) + " bytes (use wt_plan_create)");
  if ((n_slots > 0 && !shard_ptrs) || (p.num_ranks > 0 && !pools))
    return fail_na(WT_ERR_INVALID_ARGUMENT, "shard_ptrs or pools is NULL");
  for (int32_t r = 0; r < p.num_ranks; ++r) {
    if (p.pool_bytes[r] == 0) continue;
    if (!pools[r]) return fail_na(WT_ERR_INVALID_ARGUMENT, "pool " + std::to_string(r) + " is NULL");
    if (reinterpret_cast<uintptr_t>(pools[r]) % 16)
      return fail_na(WT_ERR_ALIGNMENT, "pool " + std::to_string(r) + " is not 16-byte aligned");
  }
  for (const ParamInfo& pi : p.params) {
    const bool vec = p.outputs[pi.output].vec;
    for (size_t k = 0; k < pi.shard_rows.size(); ++k) {
      const void* ptr = shard_ptrs[pi.slot_base + k];
      if (!p.slot_used[pi.slot_base + k]) continue;   // empty, or not this plan's shard
      if (!ptr) return fail_na(WT_ERR_INVALID_ARGUMENT, pi.name + ": shard " + std::to_string(k) + " is NULL");
      if (reinterpret_cast<uintptr_t>(ptr) % (vec ? 16 : 2))
        return fail_na(WT_ERR_ALIGNMENT, pi.name + ": shard " + std::to_string(k) + " is misaligned");
    }
  }

  int device = -1;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return fail_na(WT_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (device < 0 || device >= kMaxDevices) return fail_na(WT_ERR_INVALID_ARGUMENT, "device index out of range");

  std::vector<unsigned char> img(total, 0);   // host image of the tables
  unsigned char* h = img.data();
  if (n_slots) {
    std::memcpy(h + o_shards, shard_ptrs, n_slots * sizeof(void*));
    if ((st = encode_tmaps(p, shard_ptrs, h + o_tmaps, h + o_views)) != WT_OK) return st;
  }
  DevDstPtr* dp = reinterpret_cast<DevDstPtr*>(h + o_dsts);
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
  if (!p.h_units.empty()) std::memcpy(h + o_units, p.h_units.data(), p.h_units.size() * sizeof(DevUnit));
  if (!p.h_runs.empty()) std::memcpy(h + o_runs, p.h_runs.data(), p.h_runs.size() * sizeof(DevRun));
  if (!p.h_geom.empty()) std::memcpy(h + o_geom, p.h_geom.data(), p.h_geom.size() * sizeof(DevDstGeom));
  if (!p.h_blockmap.empty())
    std::memcpy(h + o_bmap, p.h_blockmap.data(), p.h_blockmap.size() * sizeof(int32_t));

  // one thread at a time from here to the launch: another thread's upload
  // queued between this call's upload and its kernel would overwrite the
  // tables that kernel reads
  std::lock_guard<std::mutex> lock(g_mu);
  if ((st = device_setup(device)) != WT_OK) return st;
  char* dbase = static_cast<char*>(g_scratch_addr[device]);
  // from pageable memory: the call returns once the image has been staged
  e = cudaMemcpyAsync(dbase, h, total, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return fail_na(WT_ERR_CUDA, std::string("scratch upload: ") + cudaGetErrorString(e));

  PrepArgs a{};
  a.units = reinterpret_cast<const DevUnit*>(dbase + o_units);
  a.tmaps = reinterpret_cast<const unsigned char*>(dbase + o_tmaps);
  a.view_ok = reinterpret_cast<const uint8_t*>(dbase + o_views);
  a.tmap_fence = 1;                    // the maps were just rewritten
  a.timeout_ns = g_wait_limit_ns ? g_wait_limit_ns : kDefaultTimeoutNs;
  a.stall_unit = g_stall_unit;
  a.runs = reinterpret_cast<const DevRun*>(dbase + o_runs);
  a.shard_ptrs = reinterpret_cast<const uint16_t* const*>(dbase + o_shards);
  a.dst_ptrs = reinterpret_cast<const DevDstPtr*>(dbase + o_dsts);
  a.geom = reinterpret_cast<const DevDstGeom*>(dbase + o_geom);
  a.blockmap = reinterpret_cast<const int32_t*>(dbase + o_bmap);
  a.unit_begin = 0;
  a.unit_end = p.num_units;
  a.error_word = reinterpret_cast<int32_t*>(dbase + kErrorOffset);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(p.num_units, g_sm_count[device]));
  a.ticket = tickets_for(reinterpret_cast<uint32_t*>(dbase + o_ticket), p.num_units, grid);
  e = launch_prepare(a, grid, s, false, false);
  if (e != cudaSuccess) return fail_na(WT_ERR_CUDA, std::string("preparation kernel launch: ") + cudaGetErrorString(e));
  return WT_OK;
}

extern "C" wt_status wt_noalloc_check(void* stream) {
  int device = -1;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return fail_na(WT_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (device < 0 || device >= kMaxDevices) return fail_na(WT_ERR_INVALID_ARGUMENT, "device index out of range");
  if ((e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream))) != cudaSuccess)
    return fail_na(WT_ERR_CUDA, std::string("cudaStreamSynchronize: ") + cudaGetErrorString(e));
  char* dbase;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    dbase = static_cast<char*>(g_scratch_addr[device]);
  }
  if (!dbase) return WT_OK;            // no call has run on this device
  int32_t word = 0;
  if ((e = cudaMemcpy(&word, dbase + kErrorOffset, sizeof word, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return fail_na(WT_ERR_CUDA, std::string("reading the error word: ") + cudaGetErrorString(e));
  if (!word) return WT_OK;
  const int32_t zero = 0;
  if ((e = cudaMemcpy(dbase + kErrorOffset, &zero, sizeof zero, cudaMemcpyHostToDevice)) != cudaSuccess)
    return fail_na(WT_ERR_CUDA, std::string("clearing the error word: ") + cudaGetErrorString(e));
  return fail_na(WT_ERR_TIMEOUT, "a wait inside the preparation kernel gave up; its output is incomplete");
}

extern "C" wt_status wt_debug_noalloc_stall_unit(int64_t unit, uint64_t wait_limit_ns) {
  if (unit < -1) return fail_na(WT_ERR_INVALID_ARGUMENT, "unit out of range");
  std::lock_guard<std::mutex> lock(g_mu);
  g_stall_unit = unit;
  g_wait_limit_ns = wait_limit_ns;
  return WT_OK;
}
