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
constexpr int kThreads = 256;     // threads per CTA of the preparation kernel

// One output tensor (device table entry).
struct DevOutput {
  int64_t rows, cols;      // M x N of the fused tensor
  int64_t unit_begin;      // global index of its first 128x128 unit
  int32_t tiles_n;         // ceil(N / 128)
  int32_t fp8;             // 1: e4m3 codes + scales, 0: BF16 bytes
  int32_t vec;             // 1: 16-byte vector path, 0: element path
  int32_t num_dsts;
  int32_t dst_begin;       // first entry in the DevDst table
  int32_t trow_begin;      // first entry in the tile-row table
};
static_assert(sizeof(DevOutput) == 48, "layout");

// A run of consecutive fused rows that come from one shard.
struct DevRun {
  int64_t row0;            // first fused row of the run
  int64_t rows;            // number of rows
  int32_t slot;            // index into the shard pointer table
  int32_t pad;
};
static_assert(sizeof(DevRun) == 24, "layout");

// One destination of one output.
struct DevDst {
  int32_t rank;
  int32_t pad;
  uint64_t data_off;
  uint64_t scale_off;
};
static_assert(sizeof(DevDst) == 24, "layout");

// Everything one launch of the preparation kernel reads.
struct PrepArgs {
  const DevOutput* outs;
  const DevRun* runs;
  const int32_t* trow_first_run;   // per tile row: first run that touches it
  const DevDst* dsts;
  const uint32_t* unit_out;        // per unit: its output
  const uint16_t* const* shard_ptrs;
  uint8_t* const* pool_ptrs;
  const uint64_t* pool_bytes;
  int64_t unit_begin, unit_end;
  int32_t* error_word;             // debug checks: set to 1 on a bad store
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
};

struct OutputInfo {
  std::string name;
  std::vector<int32_t> parts;
  int32_t format = 0;
  int64_t rows = 0, cols = 0;
  std::vector<DstInfo> dsts;
  uint64_t data_bytes = 0, scale_bytes = 0;
  int64_t unit_begin = 0, num_units = 0;
  bool vec = false;
};

// An offload chunk: a run of whole outputs, contiguous in the host image.
struct Chunk {
  int32_t out_begin = 0, out_end = 0;
  int64_t unit_begin = 0, unit_end = 0;
  uint64_t host_begin = 0, host_bytes = 0;
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
  int64_t num_units = 0;
  uint64_t bytes_read = 0, bytes_written = 0;
  int64_t num_params_total = 0;

  // host images of the device tables
  std::vector<DevOutput> h_outs;
  std::vector<DevRun> h_runs;
  std::vector<int32_t> h_trow;
  std::vector<DevDst> h_dsts;
  std::vector<uint32_t> h_unit_out;

  // device side
  void* d_tables = nullptr;          // one allocation for all static tables
  PrepArgs args{};                   // pointers into d_tables
  const uint16_t** d_shard_ptrs = nullptr;
  uint8_t** d_pool_ptrs = nullptr;
  uint64_t* d_pool_bytes = nullptr;
  int32_t* d_error = nullptr;
  void* h_pinned_ptrs = nullptr;     // pinned staging for pointer uploads
  std::vector<const void*> cached_shards;
  std::vector<void*> cached_pools;
  bool ptrs_valid = false;
  cudaEvent_t ptr_upload_done = nullptr;
  cudaEvent_t last_done = nullptr;
  bool ran = false;
  int sm_count = 0;
  int grid_per_sm = 4;

  // offload
  uint64_t chunk_bytes = 0;
  std::vector<Chunk> chunks;
  uint64_t staging_bytes = 0;
  void* staging[2] = {nullptr, nullptr};
  const uint16_t** d_offload_shard_ptrs = nullptr;
  cudaEvent_t h2d_done[2] = {nullptr, nullptr};
  cudaEvent_t prep_done[2] = {nullptr, nullptr};
  bool prep_recorded[2] = {false, false};
  int32_t fail_chunk = -1;
};

// plan.cpp
wt_status compile_plan(const wt_plan_desc* d, Plan* p);   // host only
void set_error(const std::string& msg);

// prep_kernel.cu
cudaError_t launch_prepare(const PrepArgs& a, int grid, cudaStream_t s, bool debug);
int prep_blocks_per_sm();

}  // namespace wt

struct wt_plan {
  wt::Plan p;
};
