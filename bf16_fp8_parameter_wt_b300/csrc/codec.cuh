// The e4m3 block codec shared by the preparation kernel (128x128 weight
// blocks) and the token kernel (1x128 activation groups): BF16 unpacking,
// packed abs-max, the quotient fl32(x / s) and the packed convert.
//
// FP8 = e4m3 "fn" (bias 7, no infinities, largest finite 448), RNE,
// saturating; scale s = amax / 448 as an IEEE binary32 division (1.0 for an
// all-zero group); code = E(fl32(x / s)) ("Weight transfer for RL
// post-training in under 2 seconds", section "Task pipeline": quantize if
// needed; "Enabling trillion-parameter models on AWS EFA": block-scaled FP8
// dispatch).
//
// Division. The code of x must be E(fl32(x / s)). The scale is the same for
// a whole block or group, so the kernels form r = RN(1/s) once per scale
// and get each quotient with one reciprocal-based correction step
// (Markstein):
//   q0 = RN(x r),  e = x - q0 s (one fma),  y = fma(e, r, q0).
// q0 is within one ulp of x/s, so the remainder e = x - q0 s is exact, and
// y = RN(x/s + (x/s - q0) d) where d, the relative error of r, is at most
// 2^-24: y differs from fl32(x/s) only if x/s lies within 2^-47 (relative)
// of a binary32 rounding boundary without being on it. x/s can never sit
// exactly on such a boundary (x has 8 significant bits, s 24), and exact
// e4m3 ties (x/s equal to an e4m3 midpoint, which BF16 inputs hit often)
// are binary32 numbers, which the correction reproduces exactly. Whether a
// near-boundary quotient exists is settled by the GPU tests that run every
// pair (amax, element) of BF16 values through both kernels and compare each
// code with the CPU oracle's division. The remainder is exact only
// while it stays normal, so blocks with s < 2^-87 (amax < 4.5e-24) or a
// subnormal 1/s take the IEEE division instead; below that range x/s
// rounds to a signed zero code on both paths.
//
#pragma once

#include <cuda_fp8.h>

#include <cstdint>

namespace wt {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
// biased exponents of the scales the correction step handles: 2^-87 <= s
// and 1/s normal
constexpr uint32_t kMinScaleExp = 40u, kMaxScaleExp = 252u;

__device__ __forceinline__ uint32_t ld_nc_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint16_t ld_nc_u16(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// max(|a|, |b|) per bf16 half; the result's sign bits are meaningless
// (xorsign), only magnitudes are kept.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 values -> two e4m3 codes (first value in the low byte), RNE, satfinite.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// fl32(x / s) from r = RN(1/s): one correction step (see the header),
// written with t = -e so that x = -0 gives -0 (-0 + -0), not +0.
__device__ __forceinline__ float quotient(float x, float s, float r) {
  const float q0 = __fmul_rn(x, r);
  const float t = __fmaf_rn(q0, s, -x);
  return __fmaf_rn(t, -r, q0);
}

// 8 BF16 elements (one 16-byte chunk) -> 8 codes by the correction step.
__device__ __forceinline__ uint2 quant_chunk(const uint4& v, float s, float r) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) c[k] = e4m3x2(quotient(bf16_lo(w[k]), s, r), quotient(bf16_hi(w[k]), s, r));
  return make_uint2(__byte_perm(c[0], c[1], 0x5410), __byte_perm(c[2], c[3], 0x5410));
}

// 8 BF16 elements (one 16-byte chunk) -> 8 codes with the IEEE division.
__device__ __forceinline__ uint2 quant_exact(const uint4& v, float s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) c[k] = e4m3x2(__fdiv_rn(bf16_lo(w[k]), s), __fdiv_rn(bf16_hi(w[k]), s));
  return make_uint2(__byte_perm(c[0], c[1], 0x5410), __byte_perm(c[2], c[3], 0x5410));
}

// Codes of a group with scale s: the correction step when s is in its
// range, else the IEEE division.
__device__ __forceinline__ bool scale_in_range(float s) {
  const uint32_t se = (__float_as_uint(s) >> 23) & 0xFFu;
  return se >= kMinScaleExp && se <= kMaxScaleExp;
}

}  // namespace
}  // namespace wt
