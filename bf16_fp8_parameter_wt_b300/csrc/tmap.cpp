// Tensor maps of the shards: one 2-D map per shard of an output whose rows
// are 16-byte aligned, so that the preparation kernel moves each 128x128
// BF16 block of a one-shard block row with a single TMA copy. Built on the
// host whenever the caller's shard pointers change (the maps hold the
// addresses), through the driver's cuTensorMapEncodeTiled, which is looked
// up once through the runtime (no link against the driver library).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>
#include <string>

#include "plan.h"

namespace wt {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;
cudaError_t g_lookup_err = cudaSuccess;

void lookup() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q{};
  g_lookup_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                  cudaEnableDefault, &q);
  if (g_lookup_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

}  // namespace

wt_status encode_tmaps(const Plan& p, const void* const* shards, unsigned char* out) {
  static_assert(sizeof(CUtensorMap) == kTmapBytes, "tensor map size");
  std::call_once(g_once, lookup);
  if (!g_encode) {
    set_error(std::string("cuTensorMapEncodeTiled is unavailable: ") + cudaGetErrorString(g_lookup_err));
    return WT_ERR_CUDA;
  }
  for (int32_t s = 0; s < p.num_slots; ++s) {
    unsigned char* m = out + (size_t)s * kTmapBytes;
    if (!p.slot_tmap[s]) {
      std::memset(m, 0, kTmapBytes);
      continue;
    }
    // dim 0 = columns (contiguous), dim 1 = the shard's rows; a box is one
    // 128x128 block (256-byte rows); rows or columns past the shard's
    // edge read as zero
    const cuuint64_t dims[2] = {(cuuint64_t)p.slot_cols[s], (cuuint64_t)p.slot_rows[s]};
    const cuuint64_t strides[1] = {(cuuint64_t)p.slot_cols[s] * 2u};
    const cuuint32_t box[2] = {(cuuint32_t)kTile, (cuuint32_t)kTile};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(reinterpret_cast<CUtensorMap*>(m), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                          const_cast<void*>(shards[s]), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      set_error("cuTensorMapEncodeTiled failed for shard slot " + std::to_string(s) + " (CUresult " +
                std::to_string((int)r) + ")");
      return WT_ERR_CUDA;
    }
  }
  return WT_OK;
}

}  // namespace wt
