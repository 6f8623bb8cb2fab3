// Internal definitions of the preparation library: the device tables the
// plan compiler builds once and the kernels replay every step (the static
// schedule of "Weight transfer for RL post-training in under 2 seconds",
// section "Why it is fast and simple / static schedule").
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <string>
#include <vector>

#include "../../include/wt.h"

namespace wt {

constexpr int kTile = 128;        // block edge (rows and cols)
constexpr int kTmapBytes = 128;   // one CUtensorMap
constexpr int kViewBoxCols = 136; // columns of a view-map box: a block's 128 and 8 for the misalignment

// DevUnit.shape flag bits (bits 16..23)
constexpr uint32_t kUnitFp8 = 1u;    // e4m3 codes + scale, else BF16 bytes
constexpr uint32_t kUnitVec = 2u;    // rows are 16-byte aligned: bulk-copy path, else element path
constexpr uint32_t kUnitMulti = 4u;  // block rows come from more than one shard
constexpr uint32_t kUnitSliced = 8u; // some destination of the output takes a slice
constexpr uint32_t kUnitView = 16u;  // unaligned rows from one shard, inside its view map (see tmap.cpp)
// The consumers load the block's rows themselves, from row addresses the
// producer resolves: 16-byte rows from several shards, and rows one chunk
// (at most 8 elements) wide. One copy per row cost about 5 us per block.
constexpr uint32_t kUnitDirect = 32u;
constexpr uint32_t kUnitEnd = 0x80u; // in the kernel only: a stage that ends the CTA's units

// Error word bits set by the kernel
constexpr int32_t kErrBadStore = 1;  // debug checks: a store fell outside its pool range
constexpr int32_t kErrTimeout = 2;   // a bounded wait gave up

// Static descriptor of one 128x128 work unit, 32 bytes (eight words that
// one warp fetches with one coalesced load). Where the block's rows come
// from:
//   vec, one shard  : src = shard slot (its tensor map), src_row = first
//                     row of the block inside that shard;
//   otherwise       : src = first row run that touches the block, src_row =
//                     first fused row of the block (bi * 128).
struct DevUnit {
  uint32_t src;
  uint32_t src_row;
  uint32_t bi, bj;     // block row / column inside the output
  uint32_t cols;       // N: elements per row of the output
  uint32_t shape;      // (nrows - 1) | (ncols - 1) << 8 | flags << 16
  uint32_t num_dsts;
  uint32_t dst_begin;  // first entry of the destination pointer table
};
static_assert(sizeof(DevUnit) == 32, "layout");

// A run of consecutive fused rows that come from one shard.
struct DevRun {
  int64_t row0;            // first fused row of the run
  int64_t rows;            // number of rows
  int32_t slot;            // index into the shard pointer table
  int32_t shard;           // index of that shard within its parameter
};
static_assert(sizeof(DevRun) == 24, "layout");

// Absolute addresses of one (output, destination), rebuilt on the host
// whenever the caller's pools change.
struct DevDstPtr {
  uint8_t* data;
  float* scale;
  const uint8_t* pool_begin;   // for the debug bounds check
  const uint8_t* pool_end;
};
static_assert(sizeof(DevDstPtr) == 32, "layout");

// Where the blocks of an output land in one destination (static). A block
// (bi, bj) of the output is block (bi, bj) of a whole-tensor destination,
// (map[bi], bj) of a row slice, (bi, map[bj]) of a column slice; a -1 map
// entry means the destination does not hold that block row / column.
struct DevDstGeom {
  int32_t dim;         // -1 whole tensor, 0 row slice, 1 column slice
  int32_t map_off;     // first entry of this destination's block map
  uint32_t ld;         // elements per row of the destination tensor
  uint32_t sld;        // scales per row of the destination's scale grid
};
static_assert(sizeof(DevDstGeom) == 16, "layout");

// Everything one launch of the preparation kernel reads.
struct PrepArgs {
  const DevUnit* units;
  const DevRun* runs;
  const uint16_t* const* shard_ptrs;
  const unsigned char* tmaps;        // kTmapBytes per slot, 64-byte aligned
  const uint8_t* view_ok;            // per slot: its map is a view map (unaligned rows)
  const DevDstPtr* dst_ptrs;
  const DevDstGeom* geom;            // per destination entry, like dst_ptrs
  const int32_t* blockmap;
  int64_t unit_begin, unit_end;
  int32_t* error_word;               // kErr* bits
  uint64_t timeout_ns;               // limit of every wait inside the kernel
  uint32_t tmap_fence;               // tensor maps were rewritten since the last launch
  int64_t stall_unit;                // testing: this unit is never filled (-1: none)
  // Two words, zero before a launch and reset to zero by its last CTA: the
  // next ticket (a batch of kBatch consecutive units) and the CTAs done.
  // NULL: units are assigned statically (CTA b takes b, b + grid, ...).
  uint32_t* ticket;
};

// Host-side copy of one param.
struct ParamInfo {
  std::string name;
  int64_t rows = 0, cols = 0;
  std::vector<int64_t> shard_rows;
  int32_t slot_base = 0;    // index of its first shard in the pointer table
  int32_t output = -1;      // the output that uses it
};

struct DstInfo {
  int32_t rank = 0;
  uint64_t data_off = 0, scale_off = 0;
  int32_t slice_dim = -1;                    // -1: the whole tensor
  std::vector<int64_t> slice_begin, slice_len;
  int64_t rows = 0, cols = 0;                // what this destination holds
  uint64_t data_bytes = 0, scale_bytes = 0;
};

struct OutputInfo {
  std::string name;
  std::vector<int32_t> parts;
  int32_t format = 0;
  int64_t rows = 0, cols = 0;
  std::vector<DstInfo> dsts;
  uint64_t data_bytes = 0, scale_bytes = 0;
  int64_t unit_begin = 0, num_units = 0;
  int32_t dst_begin = 0;    // first entry of the destination pointer table
  bool vec = false;
};

// An offload chunk: a run of whole outputs, contiguous in the host image.
struct Chunk {
  int32_t out_begin = 0, out_end = 0;
  int64_t unit_begin = 0, unit_end = 0;
  uint64_t host_begin = 0, host_bytes = 0;
};

// One set of the caller's buffer addresses as the kernel reads them:
// shard pointers, one tensor map per shard, absolute destination
// addresses (a block on the device, its pinned staging on the host). A plan
// keeps kPtrSets of them, so that a caller alternating between a few
// buffer sets (FSDP double buffering) reuses uploaded tables and never
// waits for an upload.
constexpr int kPtrSets = 4;
struct PtrSet {
  unsigned char* d_block = nullptr;
  void* h_pinned = nullptr;
  cudaEvent_t upload_done = nullptr;  // the last upload from h_pinned
  bool uploaded = false;              // upload_done has been recorded
  std::vector<const void*> shards;
  std::vector<void*> pools;
  bool shards_valid = false, pools_valid = false;
  bool tmaps_dirty = false;           // maps rewritten since a launch used them
  bool captured = false;              // a captured graph reads it: never replaced
  uint64_t last_use = 0;
};

// Everything the host side of a plan owns.
struct Plan {
  int device = -1;
  uint32_t flags = 0;
  int32_t num_ranks = 0;
  std::vector<ParamInfo> params;
  std::vector<OutputInfo> outputs;
  std::vector<uint64_t> pool_bytes;
  std::vector<uint64_t> shard_host_off;   // per slot
  uint64_t host_bytes = 0;
  int32_t num_slots = 0;
  int32_t num_dst_entries = 0;
  int64_t num_units = 0;
  uint64_t bytes_read = 0, bytes_written = 0;
  int64_t num_params_total = 0;

  // host images of the static device tables
  std::vector<DevUnit> h_units;
  std::vector<DevRun> h_runs;
  std::vector<DevDstGeom> h_geom;           // per destination entry
  std::vector<int32_t> h_blockmap;
  std::vector<uint64_t> expected_blocks;    // per rank and step
  // Rank groups (counting per rank): group g holds the units whose lowest
  // holding rank is g; rank_perm lists the units group by group (plan order
  // within a group), group g is rank_perm[group_begin[g] .. group_begin[g+1]),
  // and group_counts[g * num_ranks + r] is what it adds to rank r's counter.
  std::vector<uint32_t> rank_perm;
  std::vector<int64_t> group_begin;
  std::vector<uint32_t> group_counts;
  // The unit order of whole-step and offload-chunk launches when some
  // units are slow (gathered row by row): those first, within each chunk's
  // range; empty (plan order) otherwise.
  std::vector<uint32_t> launch_perm;
  // per slot: rows and cols of the shard, whether the plan reads it
  // (non-empty, and of the local index in a shard-local plan) and whether a
  // tensor map is encoded for it (vec outputs, read shards)
  std::vector<int64_t> slot_rows, slot_cols;
  std::vector<int64_t> slot_read_rows;      // leading rows of the shard read
  std::vector<uint8_t> slot_used, slot_tmap;   // slot_tmap: 0 none, 1 block map, 2 view map
  std::vector<int32_t> slot_view_k;            // rows per view row of a view map
  int32_t local_shard = -1;                 // >= 0: shard-local plan

  // device side: one allocation for the static tables and kPtrSets
  // pointer-table blocks that follow the caller's buffers
  void* d_tables = nullptr;
  PrepArgs args{};                   // static parts filled at upload
  size_t dyn_bytes = 0;              // size of one pointer-table block
  PtrSet sets[kPtrSets];
  uint64_t use_clock = 0;            // for least-recently-used replacement
  int32_t* d_error = nullptr;
  cudaEvent_t last_done = nullptr;
  bool ran = false;
  int sm_count = 0;

  // offload
  uint64_t chunk_bytes = 0;
  std::vector<Chunk> chunks;
  uint64_t staging_bytes = 0;
  void* staging[2] = {nullptr, nullptr};
  const uint16_t** d_offload_shard_ptrs = nullptr;
  unsigned char* d_offload_tmaps = nullptr;
  const uint8_t* d_offload_view_ok = nullptr;
  bool offload_tmaps_dirty = false;
  cudaEvent_t h2d_done[2] = {nullptr, nullptr};
  cudaEvent_t prep_done[2] = {nullptr, nullptr};
  bool prep_recorded[2] = {false, false};
  int32_t fail_chunk = -1;
  uint32_t* counters = nullptr;     // wt_plan_set_counters
  uint32_t count_mode = 0;          // WT_COUNT_PER_LAUNCH or WT_COUNT_PER_RANK
  uint32_t* d_launch_counts = nullptr;   // [1 + chunks][ranks]: a step, then each chunk
  // the unit table in the order of whole-step and offload launches
  // (launch_perm, or plan order), and in rank-group order (rank_perm)
  const DevUnit* d_units_launch = nullptr;
  const DevUnit* d_units_rank = nullptr;
  uint32_t* d_tickets = nullptr;    // two words per launch of a step: [0] whole step, [1 + g] group g
  const uint32_t* d_group_counts = nullptr; // group_counts on the device
  // testing hooks (wt_debug_stall_unit): the unit, and its position in
  // the launch-order and rank-order tables
  int64_t stall_unit = -1, stall_pos_launch = -1, stall_pos_rank = -1;
  uint64_t wait_limit_ns = 0;        // 0: kDefaultTimeoutNs
};

// plan.cpp
wt_status compile_plan(const wt_plan_desc* d, Plan* p);   // host only
void set_error(const std::string& msg);

// tmap.cpp: the 2-D tensor map of every slot that has one (zeros for the
// others), kTmapBytes each, into out (64-byte aligned), and per slot in
// view_ok whether its map is a view map (a slot with slot_tmap == 2 whose
// pointer is 16-byte aligned).
wt_status encode_tmaps(const Plan& p, const void* const* shards, unsigned char* out, uint8_t* view_ok);
// The rows per view row of an output with `cols` columns whose rows are
// not 16-byte aligned: the smallest k with k * cols * 2 a multiple of 16.
inline int32_t view_rows(int64_t cols) { return (cols & 1) ? 8 : (cols & 2) ? 4 : (cols & 4) ? 2 : 1; }

// prep_kernel.cu
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;   // 2 s per wait

// The ticket counter pays once CTAs take many units each. Each producer
// takes its first three batches of four units at once, so in a launch with
// fewer units per CTA the CTAs that start first would hold them all while
// the rest had none (a 114-unit launch on 114 CTAs ran about ten times
// longer than with one unit per CTA). Below this many units per CTA the
// units are assigned statically: CTA b takes b, b + grid, ...
constexpr int64_t kTicketMinUnitsPerCta = 48;
inline uint32_t* tickets_for(uint32_t* ticket, int64_t units, int grid) {
  return units >= kTicketMinUnitsPerCta * (int64_t)grid ? ticket : nullptr;
}
// One-time per-device set-up of the kernel (shared-memory size); call with
// the device current.
cudaError_t prep_kernel_setup();
// Launch over units [a.unit_begin, a.unit_end) of a.units with grid CTAs
// (at most one per SM is resident). pdl: the launch may begin while the
// kernel before it on s is still running (programmatic dependent launch);
// only for work that reads nothing that kernel writes.
cudaError_t launch_prepare(const PrepArgs& a, int grid, cudaStream_t s, bool debug, bool pdl);

// counters.cu: counters[i] += counts[i] for i < n, queued on s after one
// device-scope fence (everything before it on s is complete and visible);
// nothing is added while error_word holds kErrTimeout. pdl: launched as a
// programmatic dependent of the kernel before it, which it waits for (and
// lets the kernel after it begin at once).
cudaError_t launch_add_counts(uint32_t* counters, const uint32_t* counts, int32_t n, const int32_t* error_word,
                              cudaStream_t s, bool pdl);

}  // namespace wt

struct wt_plan {
  wt::Plan p;
};
