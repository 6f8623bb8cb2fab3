// The activation codec of the MoE dispatch: tokens x hidden BF16 ->
// e4m3 codes with one fp32 scale per token per group of 128 channels
// ("Enabling trillion-parameter models on AWS EFA", section on the
// dispatch/combine kernels: block-scaled FP8 dispatch at hidden 7168), with
// the weight path's scale and code (codec.cuh).
//
// A streaming kernel: four lanes own one group of 128 channels, each lane
// four 16-byte chunks of it (chunk c of lane l is chunk 4c + l % 4 of the
// group, so every load instruction reads whole 64-byte runs, and every
// store writes whole 32-byte sectors); a warp takes eight groups per slot
// and four slots per pass, so 256 bytes per lane are in flight (two slots
// reached 86 % of the copy bandwidth, four 99 %). The group's
// amax is a two-step shuffle; its scale and reciprocal are computed once
// per 32 elements of a lane. Loops are warp-uniform so the shuffles never
// see an exited lane. Contiguous batches whose hidden size is a multiple of
// 128 index groups as one flat sequence (no division); other shapes split
// the group index into token and group, and rows that are not 16-byte
// aligned are read and written element by element.
#include <algorithm>
#include <string>

#include "codec.cuh"
#include "plan.h"

namespace wt {
namespace {

constexpr int kTokThreads = 256;
constexpr int kTokSlots = 4;        // groups in flight per lane
constexpr int kTokLanes = 4;        // lanes per group
constexpr int kTokChunks = kTile / 8 / kTokLanes;   // 16-byte chunks per lane and group
constexpr int kTokGroupsPerWarp = 32 / kTokLanes;

enum TokMode { kTokFlat = 0, kTokVec = 1, kTokElem = 2 };

struct TokArgs {
  const uint16_t* x;
  uint8_t* codes;
  float* scales;
  int64_t hidden, ld;
  uint32_t groups_per_token;
  uint32_t num_groups;
};

template <int kMode>
__global__ void __launch_bounds__(kTokThreads) token_kernel(const __grid_constant__ TokArgs a) {
  const int lane = threadIdx.x & 31, sub = lane % kTokLanes;
  const uint32_t gw = (uint32_t)(lane / kTokLanes);
  const uint32_t warp = (blockIdx.x * kTokThreads + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * kTokThreads) >> 5;
  for (uint32_t p = warp; kTokGroupsPerWarp * p < a.num_groups; p += kTokSlots * nwarps) {
    uint4 v[kTokSlots][kTokChunks];
    int64_t xoff[kTokSlots], coff[kTokSlots];
    int64_t cols[kTokSlots];                      // valid channels of the group
    uint32_t g[kTokSlots];
#pragma unroll
    for (int k = 0; k < kTokSlots; ++k) {
      g[k] = kTokGroupsPerWarp * (p + (uint32_t)k * nwarps) + gw;
      cols[k] = 0;
      xoff[k] = coff[k] = 0;
      if (g[k] < a.num_groups) {
        if (kMode == kTokFlat) {
          xoff[k] = coff[k] = (int64_t)g[k] * kTile;
          cols[k] = kTile;
        } else {
          const uint32_t t = g[k] / a.groups_per_token;
          const int64_t c0 = (int64_t)(g[k] - t * a.groups_per_token) * kTile;
          cols[k] = min((int64_t)kTile, a.hidden - c0);
          xoff[k] = (int64_t)t * a.ld + c0;
          coff[k] = (int64_t)t * a.hidden + c0;
        }
      }
#pragma unroll
      for (int c = 0; c < kTokChunks; ++c) {
        const int col = (c * kTokLanes + sub) * 8;
        v[k][c] = make_uint4(0, 0, 0, 0);
        if (kMode != kTokElem) {
          if (col < cols[k]) v[k][c] = ld_nc_v4(a.x + xoff[k] + col);
        } else {
          uint16_t e[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) e[j] = col + j < cols[k] ? ld_nc_u16(a.x + xoff[k] + col + j) : (uint16_t)0;
          v[k][c] = make_uint4(e[0] | ((uint32_t)e[1] << 16), e[2] | ((uint32_t)e[3] << 16),
                               e[4] | ((uint32_t)e[5] << 16), e[6] | ((uint32_t)e[7] << 16));
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kTokSlots; ++k) {
      uint32_t m2 = 0;
#pragma unroll
      for (int c = 0; c < kTokChunks; ++c)
        m2 = absmax_bf16x2(absmax_bf16x2(m2, absmax_bf16x2(v[k][c].x, v[k][c].y)),
                           absmax_bf16x2(v[k][c].z, v[k][c].w));
      m2 &= 0x7FFF7FFFu;
      float amax = fmaxf(bf16_lo(m2), bf16_hi(m2));
#pragma unroll
      for (int off = kTokLanes / 2; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
      const float s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
      const bool corr = scale_in_range(s);
      const float r = corr ? __frcp_rn(s) : 0.0f;
#pragma unroll
      for (int c = 0; c < kTokChunks; ++c) {
        const int col = (c * kTokLanes + sub) * 8;
        if (col >= cols[k]) continue;
        const uint2 q = corr ? quant_chunk(v[k][c], s, r) : quant_exact(v[k][c], s);
        uint8_t* dst = a.codes + coff[k] + col;
        if (kMode != kTokElem) {
          *reinterpret_cast<uint2*>(dst) = q;
        } else {
          const uint32_t wds[2] = {q.x, q.y};
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (col + j < cols[k]) dst[j] = (uint8_t)(wds[j >> 2] >> (8 * (j & 3)));
        }
      }
      if (sub == 0 && g[k] < a.num_groups) a.scales[g[k]] = s;
    }
  }
}

int g_sm_count[64] = {};
int g_ctas_per_sm[64][3] = {};

}  // namespace
}  // namespace wt

using namespace wt;

extern "C" wt_status wt_quantize_tokens(const void* x, int64_t tokens, int64_t hidden, int64_t x_ld,
                                        void* codes, float* scales, void* stream) {
  if (tokens < 0 || hidden < 1 || x_ld < hidden) {
    set_error("wt_quantize_tokens: need tokens >= 0, hidden >= 1 and x_ld >= hidden");
    return WT_ERR_INVALID_ARGUMENT;
  }
  if (tokens == 0) return WT_OK;
  if (!x || !codes || !scales) {
    set_error("wt_quantize_tokens: x, codes and scales must not be NULL");
    return WT_ERR_INVALID_ARGUMENT;
  }
  const int64_t gpt = (hidden + kTile - 1) / kTile;
  if (tokens * gpt >= (int64_t(1) << 31)) {
    set_error("wt_quantize_tokens: more than 2^31 - 1 groups of 128 channels in one call");
    return WT_ERR_INVALID_ARGUMENT;
  }
  if (reinterpret_cast<uintptr_t>(x) % 2 || reinterpret_cast<uintptr_t>(scales) % 4) {
    set_error("wt_quantize_tokens: x must be 2-byte and scales 4-byte aligned");
    return WT_ERR_ALIGNMENT;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    set_error(std::string("wt_quantize_tokens: cudaGetDevice: ") + cudaGetErrorString(e));
    return WT_ERR_CUDA;
  }
  if (!g_sm_count[dev]) {
    int n = 0, c0 = 0, c1 = 0, c2 = 0;
    if ((e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&c0, token_kernel<kTokFlat>, kTokThreads, 0)) != cudaSuccess ||
        (e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&c1, token_kernel<kTokVec>, kTokThreads, 0)) != cudaSuccess ||
        (e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&c2, token_kernel<kTokElem>, kTokThreads, 0)) != cudaSuccess) {
      set_error(std::string("wt_quantize_tokens: device query: ") + cudaGetErrorString(e));
      return WT_ERR_CUDA;
    }
    g_ctas_per_sm[dev][0] = std::max(1, c0);
    g_ctas_per_sm[dev][1] = std::max(1, c1);
    g_ctas_per_sm[dev][2] = std::max(1, c2);
    g_sm_count[dev] = n;
  }
  TokArgs a;
  a.x = static_cast<const uint16_t*>(x);
  a.codes = static_cast<uint8_t*>(codes);
  a.scales = scales;
  a.hidden = hidden;
  a.ld = x_ld;
  a.groups_per_token = (uint32_t)gpt;
  a.num_groups = (uint32_t)(tokens * gpt);
  const bool vec = hidden % 8 == 0 && x_ld % 8 == 0 && reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(codes) % 8 == 0;
  const bool flat = vec && hidden % kTile == 0 && x_ld == hidden;
  // eight groups per warp per slot; one wave of resident CTAs at most
  const int mode = flat ? kTokFlat : vec ? kTokVec : kTokElem;
  const int64_t warps = (a.num_groups + kTokGroupsPerWarp - 1) / kTokGroupsPerWarp;
  const int64_t want = (warps + (kTokThreads / 32) - 1) / (kTokThreads / 32);
  const int grid = (int)std::max<int64_t>(
      1, std::min<int64_t>(want, (int64_t)g_sm_count[dev] * g_ctas_per_sm[dev][mode]));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (flat)
    token_kernel<kTokFlat><<<grid, kTokThreads, 0, s>>>(a);
  else if (vec)
    token_kernel<kTokVec><<<grid, kTokThreads, 0, s>>>(a);
  else
    token_kernel<kTokElem><<<grid, kTokThreads, 0, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error(std::string("wt_quantize_tokens: launch: ") + cudaGetErrorString(e));
    return WT_ERR_CUDA;
  }
  return WT_OK;
}
