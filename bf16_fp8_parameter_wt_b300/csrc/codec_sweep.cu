// Testing hook for the e4m3 convert that every code of the library goes
// through (codec.cuh: the packed round-to-nearest-even, saturating convert
// of two fp32 values): applied to a range of fp32 bit patterns, so that a
// test can compare it with the CPU definition over all 2^32 inputs.
#include <algorithm>
#include <string>

#include "codec.cuh"
#include "plan.h"

namespace wt {
namespace {

__global__ void __launch_bounds__(256) e4m3_sweep_kernel(uint32_t first, uint64_t n, uint8_t* out) {
  const uint64_t stride = 2ull * gridDim.x * blockDim.x;
  for (uint64_t i = 2ull * (blockIdx.x * (uint64_t)blockDim.x + threadIdx.x); i < n; i += stride) {
    const float lo = __uint_as_float(first + (uint32_t)i);
    const float hi = i + 1 < n ? __uint_as_float(first + (uint32_t)i + 1u) : 0.0f;
    const uint32_t c = e4m3x2(lo, hi);
    out[i] = (uint8_t)c;
    if (i + 1 < n) out[i + 1] = (uint8_t)(c >> 8);
  }
}

}  // namespace
}  // namespace wt

using namespace wt;

extern "C" wt_status wt_debug_e4m3_encode(uint32_t first_bits, uint64_t n, uint8_t* codes, void* stream) {
  if (n == 0) return WT_OK;
  if (!codes) {
    set_error("wt_debug_e4m3_encode: codes is NULL");
    return WT_ERR_INVALID_ARGUMENT;
  }
  if (n > (1ull << 32) - first_bits) {
    set_error("wt_debug_e4m3_encode: first_bits + n exceeds 2^32");
    return WT_ERR_INVALID_ARGUMENT;
  }
  const uint64_t pairs = (n + 1) / 2;
  const unsigned grid = (unsigned)std::min<uint64_t>((pairs + 255) / 256, 148ull * 16);
  e4m3_sweep_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(first_bits, n, codes);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error(std::string("wt_debug_e4m3_encode: launch: ") + cudaGetErrorString(e));
    return WT_ERR_CUDA;
  }
  return WT_OK;
}
