// Tensor maps of the shards: one 2-D map per shard of an output whose rows
// are 16-byte aligned, so that the preparation kernel moves each 128x128
// BF16 block of a one-shard block row with a single TMA copy. Built on the
// host whenever the caller's shard pointers change (the maps hold the
// addresses), through the driver's cuTensorMapEncodeTiled, which is looked
// up once through the runtime (no link against the driver library).
//
// Rows that are not 16-byte aligned (N % 8 != 0 columns) cannot be a map's
// rows: a map's row pitch must be a multiple of 16 bytes. Their shard gets
// a view map instead, whose rows are k consecutive shard rows (k = 8 /
// gcd(N, 8), the fewest whose bytes are a multiple of 16): view row v holds
// shard rows k v .. k v + k - 1, shard row r at column (r % k) N. A block's
// rows fall into k residue classes r = j mod k, each class k-strided in the
// shard and so one box of 128 / k consecutive view rows; its columns start
// at (c N + 128 bj) for the class's column offset c N, rounded down to a
// multiple of 8 (a map's box must start 16-byte aligned), so a box is 136
// columns wide and the block's 128 sit at an offset of 0..7 in it. The map
// covers the shard's whole view rows only (rows / k of them), needs a
// 16-byte-aligned shard, and columns past a view row's end read as zero.
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

wt_status encode_tmaps(const Plan& p, const void* const* shards, unsigned char* out, uint8_t* view_ok) {
  static_assert(sizeof(CUtensorMap) == kTmapBytes, "tensor map size");
  std::call_once(g_once, lookup);
  if (!g_encode) {
    set_error(std::string("cuTensorMapEncodeTiled is unavailable: ") + cudaGetErrorString(g_lookup_err));
    return WT_ERR_CUDA;
  }
  for (int32_t s = 0; s < p.num_slots; ++s) {
    unsigned char* m = out + (size_t)s * kTmapBytes;
    view_ok[s] = 0;
    const bool view = p.slot_tmap[s] == 2;
    if (!p.slot_tmap[s] || (view && reinterpret_cast<uintptr_t>(shards[s]) % 16)) {
      std::memset(m, 0, kTmapBytes);   // an unaligned shard keeps the row-by-row path
      continue;
    }
    // dim 0 = columns (contiguous), dim 1 = the shard's rows; a box is one
    // 128x128 block (256-byte rows); rows or columns past the shard's
    // edge read as zero. A view map: dim 0 = k rows' columns, dim 1 = whole
    // view rows, a box 136 columns by 128 / k view rows.
    const cuuint64_t k = view ? (cuuint64_t)p.slot_view_k[s] : 1u;
    const cuuint64_t dims[2] = {(cuuint64_t)p.slot_cols[s] * k, (cuuint64_t)p.slot_rows[s] / k};
    const cuuint64_t strides[1] = {(cuuint64_t)p.slot_cols[s] * k * 2u};
    const cuuint32_t box[2] = {view ? (cuuint32_t)kViewBoxCols : (cuuint32_t)kTile, (cuuint32_t)(kTile / k)};
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
    view_ok[s] = view ? 1 : 0;
  }
  return WT_OK;
}

}  // namespace wt
